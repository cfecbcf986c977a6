// Single-token (decode) forward kernel.
//
// "gated_delta_recurrence_fwd_gpu" (summary) gives one CTA per (row, value
// head) with one thread per state column.  Here the unit of work is a WARP
// that owns a slice of columns of one (row, value head) and all K rows of it:
// lane kl = lane % (K/8) holds the 8 consecutive rows of group kl, lane
// vl = lane / (K/8) holds C consecutive columns (one 16-byte vector per row).
// Both K-reductions of the token finish with xor-shuffles inside the warp, so
// no shared memory and no block barrier is needed, and every warp streams its
// 128-row x 16-column bf16 tile (4 KiB) in and out once.  The state stays in
// its storage format in registers and is widened on use.
#include "gdr_pipe.cuh"

namespace gdr {

template <typename ST, int K> struct DecodeShape {
    static constexpr int V = K;
    static constexpr int NG = K / 8;          // row groups (= lanes along K)
    static constexpr int LK = NG;
    static constexpr int LV = 32 / LK;        // lanes along V
    static constexpr int C = cmin(16 / (int)sizeof(ST), V / LV);
    static constexpr int WC = LV * C;         // columns per warp
    static constexpr int SLICES = V / WC;     // warps per (row, head)
};

constexpr int kDecodeThreads = 256;

template <typename ST, int K>
__global__ void __launch_bounds__(kDecodeThreads) k_decode(const StepParams p) {
    using Sh = DecodeShape<ST, K>;
    constexpr int V = K, LK = Sh::LK, C = Sh::C, WC = Sh::WC, SLICES = Sh::SLICES;
    const int lane = threadIdx.x & 31;
    const int kl = lane % LK, vl = lane / LK;
    const long long unit = (long long)blockIdx.x * (kDecodeThreads / 32) + (threadIdx.x >> 5);
    const long long nunits = (long long)p.batch * p.nv * SLICES;
    if (unit >= nunits) return;
    const int slice = (int)(unit % SLICES);
    const long long bh = unit / SLICES;
    const int h = (int)(bh % p.nv);
    const int b = (int)(bh / p.nv);
    const bool leader = lane == 0 && slice == 0 && h == 0;

    const int t0 = p.offsets[b], t1 = p.offsets[b + 1];
    if (t0 < 0 || t1 < t0 || t1 > p.T) {
        if (leader) flag(p.status, GDR_STATUS_BAD_OFFSETS);
        return;
    }
    if (t1 == t0) return;
    const int col0 = slice * WC + vl * C;
    float *orow = p.out + (long long)t0 * p.out_ss + (long long)(h * V + col0) * p.out_vs;
    if (t1 - t0 > 1) {  // longer than the caller's bound: zero output, nothing else
        if (leader) flag(p.status, GDR_STATUS_ROW_TOO_LONG);
        if (kl == 0) zero_rows<C>(orow, t1 - t0, p);
        return;
    }
    const int slot = p.slot_idx[b];
    if (slot < 0 || slot >= p.max_slots) {
        if (slot != -1 && leader) flag(p.status, GDR_STATUS_BAD_SLOT);
        if (kl == 0) zero_rows<C>(orow, 1, p);
        return;
    }

    // State tile: rows 8*kl .. 8*kl+7, columns col0 .. col0+C-1, issued first.
    ST *sp = reinterpret_cast<ST *>(p.state) + (long long)slot * p.st_slot +
             (long long)h * p.st_head + (long long)(kl * 8) * p.st_k + col0;
    Pack<ST, C> s[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) s[i].load(sp + i * p.st_k);

    const int hk = h / p.r;
    const float *row = p.qkv + (long long)t0 * p.qkv_ss;
    float q[8], k[8], v[C];
    load_f32<8>(row + (long long)(hk * K + kl * 8) * p.qkv_cs, p.qkv_cs, p.qkv_vec, q);
    load_f32<8>(row + (long long)(p.nk * K + hk * K + kl * 8) * p.qkv_cs, p.qkv_cs, p.qkv_vec, k);
    load_f32<C>(row + (long long)(2 * p.nk * K + h * V + col0) * p.qkv_cs, p.qkv_cs, p.qkv_vec, v);
    const float alpha = gdr_alpha(p.decay[(long long)t0 * p.tok_ss + (long long)h * p.tok_hs],
                                  p.decay_is_log);
    const float beta = p.beta[(long long)t0 * p.tok_ss + (long long)h * p.tok_hs];

    // |q|^2, |k|^2, k.q: this lane's group partial, then the tree across groups.
    float ssq = chain_first(q[0], q[0]), ssk = chain_first(k[0], k[0]), kqr = chain_first(k[0], q[0]);
#pragma unroll
    for (int i = 1; i < 8; ++i) {
        ssq = chain_next(q[i], q[i], ssq);
        ssk = chain_next(k[i], k[i], ssk);
        kqr = chain_next(k[i], q[i], kqr);
    }
    ssq = tree_lanes<LK>(ssq);
    ssk = tree_lanes<LK>(ssk);
    kqr = tree_lanes<LK>(kqr);
    float inv_k, qsc, kq;
    gdr_norm_scalars(ssq, ssk, kqr, p.l2norm, p.scale, p.eps, inv_k, qsc, kq);
    float kh[8], qt[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        kh[i] = __fmul_rn(k[i], inv_k);
        qt[i] = __fmul_rn(q[i], qsc);
    }

    // a = S^T k^, b = S^T q~ over this lane's group, then across groups.
    float a[C], bq[C];
#pragma unroll
    for (int c = 0; c < C; ++c) {
        const float x = s[0].get(c);
        a[c] = chain_first(x, kh[0]);
        bq[c] = chain_first(x, qt[0]);
    }
#pragma unroll
    for (int i = 1; i < 8; ++i) {
#pragma unroll
        for (int c = 0; c < C; ++c) {
            const float x = s[i].get(c);
            a[c] = chain_next(x, kh[i], a[c]);
            bq[c] = chain_next(x, qt[i], bq[c]);
        }
    }
    float u[C], o[C];
#pragma unroll
    for (int c = 0; c < C; ++c) {
        a[c] = tree_lanes<LK>(a[c]);
        bq[c] = tree_lanes<LK>(bq[c]);
        u[c] = gdr_u(beta, alpha, a[c], v[c]);
        o[c] = gdr_o(alpha, bq[c], kq, u[c]);
    }
    if (kl == 0) store_f32<C>(orow, p.out_vs, p.out_vec, o);

    // S <- k^ u^T + alpha S, rounded to the pool's type, written in place.
#pragma unroll
    for (int i = 0; i < 8; ++i) {
#pragma unroll
        for (int c = 0; c < C; ++c) s[i].set(c, gdr_advance(s[i].get(c), kh[i], u[c], alpha));
        s[i].store(sp + i * p.st_k);
    }
}

// Warps per CTA (each owns 16 bf16 / 8 f32 columns of a tile) and the
// pipeline's depth and residency.
constexpr int kDecodeWarps = 4;
constexpr int kDecodeMinBlocks = 4;

// ---------------------------------------------------------------------------
// Pipelined variant for the common layouts (16-byte state vectors, unit-stride
// Q/K/V rows).  Persistent CTAs walk (row, value head, tile) units with a
// stride of gridDim.x; NS shared-memory stages keep NS-1 units' copies in
// flight while one is computed.  Same arithmetic as k_decode.

__device__ __forceinline__ bool decode_unit_streams(const StepParams &p, const UnitMeta &m) {
    return m.t0 >= 0 && m.t1 == m.t0 + 1 && m.t1 <= p.T && m.slot >= 0 && m.slot < p.max_slots;
}

// Queue the copies of one unit into a stage (always commits one group).
template <typename ST, int K>
__device__ __forceinline__ void unit_issue(const StepParams &p, const UnitMeta &m, uint4 *stage) {
    using Sh = PipeShape<ST, K, kDecodeWarps>;
    if (decode_unit_streams(p, m)) {
        const int tid = threadIdx.x;
        const int h = m.hu / Sh::USL, us = m.hu % Sh::USL;
        tile_issue<ST, K, PipeShape<ST, K, kDecodeWarps>::NT, kDecodeWarps>(reinterpret_cast<const ST *>(p.state) + (long long)m.slot * p.st_slot +
                              (long long)h * p.st_head + us * Sh::CW,
                          p.st_k, stage);
        const int hk = h / p.r;
        const float *trow = p.qkv + (long long)m.t0 * p.qkv_ss;
        for (int ch = tid; ch < Sh::S_Q + Sh::S_K + Sh::S_V; ch += Sh::NT) {
            const float *g = ch < Sh::S_Q ? trow + hk * K + 4 * ch
                             : ch < Sh::S_Q + Sh::S_K ? trow + (p.nk + hk) * K + 4 * (ch - Sh::S_Q)
                                                      : trow + 2 * p.nk * K + h * K + us * Sh::CW +
                                                            4 * (ch - Sh::S_Q - Sh::S_K);
            cp_async16(stage + Sh::S_STATE + ch, g);
        }
        if (tid == 0) {
            float *ab = reinterpret_cast<float *>(stage + Sh::SC - 1);
            const long long o = (long long)m.t0 * p.tok_ss + (long long)h * p.tok_hs;
            cp_async4(ab, p.decay + o);
            cp_async4(ab + 1, p.beta + o);
        }
    }
    cp_async_commit();
}

template <typename ST, int K>
__device__ __forceinline__ void unit_compute(const StepParams &p, const UnitMeta &m, uint4 *stage) {
    using Sh = PipeShape<ST, K, kDecodeWarps>;
    constexpr int V = K, LK = Sh::LK, C = Sh::C, CPR = Sh::CPR;
    using VT = typename Pack<ST, C>::VT;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int kl = lane % LK, vl = lane / LK;
    const int h = m.hu / Sh::USL, us = m.hu % Sh::USL;
    const bool leader = tid == 0 && m.hu == 0;
    if (m.t0 < 0 || m.t1 < m.t0 || m.t1 > p.T) {
        if (leader) flag(p.status, GDR_STATUS_BAD_OFFSETS);
        return;
    }
    if (m.t1 == m.t0) return;
    const int col = warp * Sh::WC + vl * C;  // inside the unit's tile
    float *orow = p.out + (long long)m.t0 * p.out_ss + (long long)(h * V + us * Sh::CW + col) * p.out_vs;
    if (m.t1 - m.t0 > 1) {  // longer than the caller's bound: zero output, nothing else
        if (leader) flag(p.status, GDR_STATUS_ROW_TOO_LONG);
        if (kl == 0) zero_rows<C>(orow, m.t1 - m.t0, p);
        return;
    }
    if (m.slot < 0 || m.slot >= p.max_slots) {
        if (m.slot != -1 && leader) flag(p.status, GDR_STATUS_BAD_SLOT);
        if (kl == 0) zero_rows<C>(orow, 1, p);
        return;
    }
    const float *qs = reinterpret_cast<const float *>(stage + Sh::S_STATE);
    const float *ks = qs + K;
    const float *vs = ks + K;
    const float *ab = reinterpret_cast<const float *>(stage + Sh::SC - 1);
    float q[8], k[8];
#pragma unroll
    for (int i = 0; i < 8; i += 4) {
        const float4 a4 = *reinterpret_cast<const float4 *>(qs + kl * 8 + i);
        const float4 b4 = *reinterpret_cast<const float4 *>(ks + kl * 8 + i);
        q[i] = a4.x; q[i + 1] = a4.y; q[i + 2] = a4.z; q[i + 3] = a4.w;
        k[i] = b4.x; k[i + 1] = b4.y; k[i + 2] = b4.z; k[i + 3] = b4.w;
    }
    float ssq = chain_first(q[0], q[0]), ssk = chain_first(k[0], k[0]), kqr = chain_first(k[0], q[0]);
#pragma unroll
    for (int i = 1; i < 8; ++i) {
        ssq = chain_next(q[i], q[i], ssq);
        ssk = chain_next(k[i], k[i], ssk);
        kqr = chain_next(k[i], q[i], kqr);
    }
    ssq = tree_lanes<LK>(ssq);
    ssk = tree_lanes<LK>(ssk);
    kqr = tree_lanes<LK>(kqr);
    float inv_k, qsc, kq;
    gdr_norm_scalars(ssq, ssk, kqr, p.l2norm, p.scale, p.eps, inv_k, qsc, kq);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        k[i] = __fmul_rn(k[i], inv_k);  // k^
        q[i] = __fmul_rn(q[i], qsc);    // q~
    }
    uint4 *mine = tile_lane_base<ST, K, kDecodeWarps>(stage, kl, col);
    float a[C], bq[C];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        Pack<ST, C> x;
        x.u.v = *reinterpret_cast<const VT *>(mine + i * CPR);
        float sr[C];
#pragma unroll
        for (int c = 0; c < C; ++c) sr[c] = x.get(c);
        if (i == 0) {
            chain_first_cols<C>(sr, k[0], a);
            chain_first_cols<C>(sr, q[0], bq);
        } else {
            chain_next_cols<C>(sr, k[i], a);
            chain_next_cols<C>(sr, q[i], bq);
        }
    }
    const float alpha = gdr_alpha(ab[0], p.decay_is_log);
    const float beta = ab[1];
    float u[C];
    if constexpr (LK == 2 * C) {
        float A, B;
        rs_reduce<LK, C>(a, bq, kl, A, B);
        const int c = rs_column<LK, C>(kl);
        const float uc = gdr_u(beta, alpha, A, vs[col + c]);
        if (!(kl & 1)) orow[(long long)c * p.out_vs] = gdr_o(alpha, B, kq, uc);
        rs_broadcast<LK, C>(uc, lane, u);
    } else {
#pragma unroll
        for (int c = 0; c < C; ++c) {
            const float A = tree_lanes<LK>(a[c]);
            const float B = tree_lanes<LK>(bq[c]);
            u[c] = gdr_u(beta, alpha, A, vs[col + c]);
            a[c] = gdr_o(alpha, B, kq, u[c]);  // the output
        }
        if (kl == 0) store_f32<C>(orow, p.out_vs, p.out_vec, a);
    }
    // New state back into the same (lane-private) chunks of the stage; the CTA
    // then writes the whole tile to HBM with coalesced rows.
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        Pack<ST, C> x;
        x.u.v = *reinterpret_cast<const VT *>(mine + i * CPR);
        float n[C];
#pragma unroll
        for (int c = 0; c < C; ++c) n[c] = x.get(c);
        advance_cols<C>(n, k[i], u, alpha);
        pack_store<ST, C>(mine + i * CPR, n);
    }
}

template <typename ST, int K, int NS>
__global__ void __launch_bounds__(PipeShape<ST, K, kDecodeWarps>::NT, kDecodeMinBlocks)
    k_decode_pipe(const StepParams p, const int nunits) {
    using Sh = PipeShape<ST, K, kDecodeWarps>;
    extern __shared__ uint4 smem_pipe[];
    const int G = gridDim.x;
    // mq[s] holds units i .. i+NS-1 (i = this CTA's current unit)
    UnitMeta mq[NS];
#pragma unroll
    for (int s = 0; s < NS; ++s) {
        const long long us_ = (long long)blockIdx.x + (long long)s * G;
        mq[s] = unit_meta<Sh::USL>(p, us_ < nunits ? (int)us_ : nunits, nunits);
    }
#pragma unroll
    for (int s = 0; s < NS - 1; ++s) unit_issue<ST, K>(p, mq[s], smem_pipe + s * Sh::SC);
    int cur = 0;  // stage of unit i
    for (int u = blockIdx.x; u < nunits; u += G) {
        const int nxt = cur == 0 ? NS - 1 : cur - 1;  // stage of unit i+NS-1
        unit_issue<ST, K>(p, mq[NS - 1], smem_pipe + nxt * Sh::SC);
        const long long ul = (long long)u + (long long)NS * G;
        const UnitMeta later = unit_meta<Sh::USL>(p, ul < nunits ? (int)ul : nunits, nunits);
        cp_async_wait<NS - 1>();
        __syncthreads();
        uint4 *stage = smem_pipe + cur * Sh::SC;
        unit_compute<ST, K>(p, mq[0], stage);
        __syncthreads();
        if (decode_unit_streams(p, mq[0])) {
            const int h = mq[0].hu / Sh::USL, us = mq[0].hu % Sh::USL;
            tile_store<ST, K, PipeShape<ST, K, kDecodeWarps>::NT, kDecodeWarps>(reinterpret_cast<ST *>(p.state) + (long long)mq[0].slot * p.st_slot +
                                  (long long)h * p.st_head + us * Sh::CW,
                              p.st_k, stage);
        }
        __syncthreads();
#pragma unroll
        for (int s = 0; s < NS - 1; ++s) mq[s] = mq[s + 1];
        mq[NS - 1] = later;
        cur = cur == NS - 1 ? 0 : cur + 1;
    }
    cp_async_wait<0>();
}

// Pipeline depth of the decode kernel (shared-memory stages per CTA).
constexpr int kDecodeStages = 3;
static_assert(kDecodeWarps >= 1, "decode CTA");

template <typename ST, int K> static cudaError_t launch_pipe_t(const StepParams &p, cudaStream_t st) {
    using Sh = PipeShape<ST, K, kDecodeWarps>;
    constexpr int NS = kDecodeStages;
    constexpr int SMEM = NS * Sh::SMEM1;
    static LaunchCache cache;
    LaunchInfo li;
    cudaError_t e = launch_info(cache, &li, [](LaunchInfo &x) {
        cudaError_t r = cudaFuncSetAttribute(k_decode_pipe<ST, K, NS>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
        if (r != cudaSuccess) return r;
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(&x.occ, k_decode_pipe<ST, K, NS>, Sh::NT, SMEM);
    });
    if (e != cudaSuccess) return e;
    const long long nunits = (long long)p.batch * p.nv * Sh::USL;
    long long grid = (long long)li.sms * li.occ;
    if (grid > nunits) grid = nunits;
    if (grid > 0) k_decode_pipe<ST, K, NS><<<(unsigned)grid, Sh::NT, SMEM, st>>>(p, (int)nunits);
    return cudaGetLastError();
}

template <typename ST, int K> static cudaError_t launch_decode_t(const StepParams &p, cudaStream_t st) {
    const long long nunits = (long long)p.batch * p.nv * DecodeShape<ST, K>::SLICES;
    const long long blocks = (nunits + kDecodeThreads / 32 - 1) / (kDecodeThreads / 32);
    if (blocks > 0) k_decode<ST, K><<<(unsigned)blocks, kDecodeThreads, 0, st>>>(p);
    return cudaGetLastError();
}

template <typename ST, int K> static cudaError_t launch_decode_any(const StepParams &p, cudaStream_t s) {
    if constexpr (PipeShape<ST, K, kDecodeWarps>::OK) {
        // the pipelined kernel counts units in 32 bits
        if (p.qkv_vec && (long long)p.batch * p.nv * PipeShape<ST, K, kDecodeWarps>::USL < (1ll << 31))
            return launch_pipe_t<ST, K>(p, s);
    }
    return launch_decode_t<ST, K>(p, s);
}

cudaError_t launch_decode(const StepParams &p, int K, bool bf16, cudaStream_t s) {
#define GDR_CASE(KK)                                                                            \
    case KK:                                                                                    \
        return bf16 ? launch_decode_any<uint16_t, KK>(p, s) : launch_decode_any<float, KK>(p, s);
    switch (K) {
        GDR_CASE(16)
        GDR_CASE(32)
        GDR_CASE(64)
        GDR_CASE(128)
    }
#undef GDR_CASE
    return cudaErrorInvalidValue;
}

}  // namespace gdr
