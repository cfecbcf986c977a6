// Shared pieces of the pipelined kernels (decode and short rows).
//
// Persistent CTAs walk units = (row, value head, CW-column tile).  A unit's
// state tile is copied into shared memory with cp.async, 16-byte chunks, the
// chunk index XOR-ed by (row / 8) so that the warp layout (lane kl = 8-row
// group, lane vl = C columns) reads it without bank conflicts, and written
// back to HBM from shared memory with fully coalesced rows.
#pragma once

#include "gdr_device.cuh"

namespace gdr {

template <typename ST, int K, int NWMAX = 8> struct PipeShape {
    static constexpr int V = K;
    static constexpr int LK = K / 8;
    static constexpr int LV = 32 / LK;
    static constexpr int C = 16 / (int)sizeof(ST);          // one 16-byte vector per row
    static constexpr bool OK = C <= V / LV;
    static constexpr int WC = LV * C;                       // columns per warp
    static constexpr int NW = OK ? cmin(NWMAX, V / WC) : 1;  // warps per CTA
    static constexpr int NT = 32 * NW;
    static constexpr int CW = NW * WC;                      // columns per unit
    static constexpr int USL = V / CW;                      // units per (row, head)
    static constexpr int CPR = CW * (int)sizeof(ST) / 16;   // 16-byte chunks per tile row
    static constexpr int S_STATE = K * CPR;                 // stage layout, in 16-byte chunks
    static constexpr int S_Q = K / 4, S_K = K / 4, S_V = CW / 4;
    static constexpr int SC = S_STATE + S_Q + S_K + S_V + 1;
    static constexpr int SMEM1 = SC * 16;                   // bytes per stage
};

// What a CTA needs to know about one unit.  hu = h * USL + us; a unit past the
// end of the batch is an empty row (t0 == t1 == 0).
struct UnitMeta {
    int hu, t0, t1, slot;
};

// Unit index -> (row b, head h, tile us), us fastest; 32-bit arithmetic.
template <int USL>
__device__ __forceinline__ UnitMeta unit_meta(const StepParams &p, int u, int nunits) {
    UnitMeta m{};
    if (u >= nunits) return m;
    const int bh = u / USL;
    const int b = bh / p.nv;
    m.hu = u - b * p.nv * USL;
    m.t0 = p.offsets[b];
    m.t1 = p.offsets[b + 1];
    m.slot = p.slot_idx[b];
    return m;
}

// Asynchronous copy of one unit's state tile (K rows x CW columns starting at
// src, rows st_k elements apart) into shared memory, swizzled: chunk c of row
// r is stored at chunk c ^ ((r >> SWS) & (CPR - 1)).  SWS = 3 suits lanes that
// own one 8-row group, SWS = 4 lanes that own runs of 16 or more rows.  Every
// thread of the CTA takes S_STATE / NT chunks; consecutive threads read
// consecutive 16-byte chunks of a row.
template <typename ST, int K, int NT = PipeShape<ST, K>::NT, int NWMAX = 8, int SWS = 3>
__device__ __forceinline__ void tile_issue(const ST *src, long long st_k, uint4 *tile) {
    using Sh = PipeShape<ST, K, NWMAX>;
    constexpr int CPR = Sh::CPR, RPI = NT / CPR, NJ = Sh::S_STATE / NT;
    static_assert(NT % CPR == 0 && Sh::S_STATE % NT == 0, "tile split");
    const int r0 = threadIdx.x / CPR, c0 = threadIdx.x % CPR;
    // row r0 + j*RPI lands at a per-thread shared base plus a constant per j,
    // and (when RPI is a multiple of 2^SWS) its swizzle is (r0 >> SWS) plus a
    // constant per j
    const unsigned base = (unsigned)__cvta_generic_to_shared(tile) + (unsigned)(r0 * CPR) * 16u;
    const char *g = reinterpret_cast<const char *>(src + (long long)r0 * st_k + c0 * (16 / (int)sizeof(ST)));
    const long long gstep = (long long)RPI * st_k * (long long)sizeof(ST);
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
        int sw;
        if constexpr (RPI % (1 << SWS) == 0)
            sw = ((r0 >> SWS) + j * (RPI >> SWS)) & (CPR - 1);
        else
            sw = ((r0 + j * RPI) >> SWS) & (CPR - 1);
        cp_async16_s(base + (unsigned)(j * RPI * CPR * 16) + (unsigned)(c0 ^ sw) * 16u, g + j * gstep);
    }
}

// This lane's chunk of tile row 8*kl + i: rows of one 8-row group share the
// swizzle (row / 8 == kl), so it is a fixed base plus i * CPR.
template <typename ST, int K, int NWMAX = 8>
__device__ __forceinline__ uint4 *tile_lane_base(uint4 *tile, int kl, int col) {
    using Sh = PipeShape<ST, K, NWMAX>;
    return tile + kl * 8 * Sh::CPR + ((col / Sh::C) ^ (kl & (Sh::CPR - 1)));
}

// Coalesced copy of a tile held in a stage to HBM: dst points at element
// (row 0, column 0) of the unit's tile, rows st_k elements apart.
template <typename ST, int K, int NT = PipeShape<ST, K>::NT, int NWMAX = 8, int SWS = 3>
__device__ __forceinline__ void tile_store(ST *dst, long long st_k, const uint4 *tile) {
    using Sh = PipeShape<ST, K, NWMAX>;
    constexpr int CPR = Sh::CPR, RPI = NT / CPR, NJ = Sh::S_STATE / NT;
    const int r0 = threadIdx.x / CPR, c0 = threadIdx.x % CPR;
    char *g = reinterpret_cast<char *>(dst + (long long)r0 * st_k + c0 * (16 / (int)sizeof(ST)));
    const long long gstep = (long long)RPI * st_k * (long long)sizeof(ST);
    const uint4 *base = tile + r0 * CPR;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
        int sw;
        if constexpr (RPI % (1 << SWS) == 0)
            sw = ((r0 >> SWS) + j * (RPI >> SWS)) & (CPR - 1);
        else
            sw = ((r0 + j * RPI) >> SWS) & (CPR - 1);
        *reinterpret_cast<uint4 *>(g + j * gstep) = base[j * RPI * CPR + (c0 ^ sw)];
    }
}

// Round C float32 values to the pool type and store them as one vector (bf16
// pairs use one round-to-nearest-even instruction per pair; same bits).
template <typename ST, int C>
__device__ __forceinline__ void pack_store(uint4 *dst, const float (&n)[C]) {
    using VT = typename Pack<ST, C>::VT;
    if constexpr (sizeof(ST) == 2 && C % 2 == 0) {
        uint32_t w[C / 2];
#pragma unroll
        for (int j = 0; j < C / 2; ++j) {
            const __nv_bfloat162 h2 = __floats2bfloat162_rn(n[2 * j], n[2 * j + 1]);
            w[j] = *reinterpret_cast<const uint32_t *>(&h2);
        }
        *reinterpret_cast<VT *>(dst) = *reinterpret_cast<const VT *>(w);
    } else {
        Pack<ST, C> x;
#pragma unroll
        for (int c = 0; c < C; ++c) x.set(c, n[c]);
        *reinterpret_cast<VT *>(dst) = x.u.v;
    }
}

// Reduce-scatter of the per-lane partials a[C], b[C] over the LK lanes that
// share columns (kl = lane % LK, LK == 2C): at the level pairing lanes (l, l^m)
// each lane keeps half of its values and adds the partner's partials for them
// -- the same pairwise tree as tree_lanes, in 2C-1 shuffles.  Afterwards the
// lane pair (kl, kl^1) holds the full sums (A, B) = (a_c, b_c) of column
// c = rs_column(kl); both lanes of the pair return the same A and B.
template <int LK, int C>
__device__ __forceinline__ int rs_column(int kl) {
    int c = 0;
#pragma unroll
    for (int m = 2, w = C / 2; m < LK; m <<= 1, w >>= 1) c += (kl & m) ? w : 0;
    return c;
}

template <int LK, int C>
__device__ __forceinline__ void rs_reduce(const float (&a)[C], const float (&b)[C], int kl, float &A,
                                          float &B) {
    static_assert(LK == 2 * C, "reduce-scatter layout");
    float x[2 * C];
#pragma unroll
    for (int c = 0; c < C; ++c) {
        x[c] = a[c];
        x[C + c] = b[c];
    }
#pragma unroll
    for (int m = 1, n = 2 * C; m < LK; m <<= 1, n >>= 1) {
        const bool hi = (kl & m) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
            const float send = hi ? x[i] : x[n / 2 + i];
            const float keep = hi ? x[n / 2 + i] : x[i];
            x[i] = __fadd_rn(keep, __shfl_xor_sync(kFull, send, m));
        }
    }
    const float other = __shfl_xor_sync(kFull, x[0], 1);
    A = (kl & 1) ? other : x[0];
    B = (kl & 1) ? x[0] : other;
}

// Every lane of a column group receives the values uc of columns 0..C-1 from
// the lanes that computed them (after rs_reduce).
template <int LK, int C>
__device__ __forceinline__ void rs_broadcast(float uc, int lane, float (&u)[C]) {
#pragma unroll
    for (int cc = 0; cc < C; ++cc) {
        int src = 0;
#pragma unroll
        for (int m = 2, w = C / 2; m < LK; m <<= 1, w >>= 1) src |= (cc & w) ? m : 0;
        u[cc] = __shfl_sync(kFull, uc, (lane & ~(LK - 1)) | src);
    }
}

}  // namespace gdr
