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
#include "gdr_device.cuh"

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
    if (t1 - t0 > 1) {
        if (leader) flag(p.status, GDR_STATUS_ROW_TOO_LONG);
        return;
    }
    const int col0 = slice * WC + vl * C;
    float *orow = p.out + (long long)t0 * p.out_ss + (long long)(h * V + col0) * p.out_vs;
    const int slot = p.slot_idx[b];
    if (slot < 0 || slot >= p.max_slots) {
        if (slot != -1 && leader) flag(p.status, GDR_STATUS_BAD_SLOT);
        if (kl == 0) {
            float z[C];
#pragma unroll
            for (int c = 0; c < C; ++c) z[c] = 0.0f;
            store_f32<C>(orow, p.out_vs, p.out_vec, z);
        }
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

// ---------------------------------------------------------------------------
// Pipelined variant for the common layouts (16-byte state vectors, unit-stride
// Q/K/V rows).  Persistent CTAs walk units = (row, value head, CW-column tile)
// with a stride of gridDim.x.  While a unit is computed, the next unit's state
// tile and operands are already in flight into the other shared-memory stage
// through cp.async, so every SM keeps tens of KiB of loads outstanding.  The
// state tile is stored with the 16-byte chunk index XOR-ed by (row / 8), which
// makes the warp-layout reads below free of bank conflicts.  The arithmetic is
// the same sequence of operations as k_decode.
template <typename ST, int K> struct PipeShape {
    static constexpr int V = K;
    static constexpr int LK = K / 8;
    static constexpr int LV = 32 / LK;
    static constexpr int C = 16 / (int)sizeof(ST);          // one 16-byte vector per row
    static constexpr bool OK = C <= V / LV;
    static constexpr int WC = LV * C;                       // columns per warp
    static constexpr int NW = OK ? cmin(8, V / WC) : 1;      // warps per CTA
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

__device__ __forceinline__ bool unit_streams(const StepParams &p, const UnitMeta &m) {
    return m.t0 >= 0 && m.t1 == m.t0 + 1 && m.t1 <= p.T && m.slot >= 0 && m.slot < p.max_slots;
}

// Per-thread share of a tile copy: chunk j (j < NJ) of this thread is tile row
// r0 + j*RPI, 16-byte column chunk c0; its shared-memory slot is swizzled.
template <typename ST, int K> struct TileLane {
    using Sh = PipeShape<ST, K>;
    static constexpr int CPR = Sh::CPR;
    static constexpr int RPI = Sh::NT / CPR;
    static constexpr int NJ = Sh::S_STATE / Sh::NT;
    static_assert(Sh::NT % CPR == 0 && Sh::S_STATE % Sh::NT == 0, "tile split");
    int r0, c0;
    long long goff;  // element offset of chunk 0 inside the (slot, head) block
    long long gstep; // element offset between consecutive chunks of this thread
    __device__ __forceinline__ void init(const StepParams &p) {
        r0 = threadIdx.x / CPR;
        c0 = threadIdx.x % CPR;
        goff = (long long)r0 * p.st_k + c0 * (16 / (int)sizeof(ST));
        gstep = (long long)RPI * p.st_k;
    }
    __device__ __forceinline__ int soff(int j) const {
        const int row = r0 + j * RPI;
        return row * CPR + (c0 ^ ((row >> 3) & (CPR - 1)));
    }
};

// Queue the copies of one unit into a stage (always commits one group).
template <typename ST, int K>
__device__ __forceinline__ void unit_issue(const StepParams &p, const UnitMeta &m, uint4 *stage) {
    using Sh = PipeShape<ST, K>;
    if (unit_streams(p, m)) {
        TileLane<ST, K> tl;  // recomputed per unit: cheaper than keeping it live
        tl.init(p);
        const int tid = threadIdx.x;
        const int h = m.hu / Sh::USL, us = m.hu % Sh::USL;
        const ST *src = reinterpret_cast<const ST *>(p.state) + (long long)m.slot * p.st_slot +
                        (long long)h * p.st_head + us * Sh::CW + tl.goff;
#pragma unroll
        for (int j = 0; j < TileLane<ST, K>::NJ; ++j) cp_async16(stage + tl.soff(j), src + j * tl.gstep);
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
    using Sh = PipeShape<ST, K>;
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
    if (m.t1 - m.t0 > 1) {
        if (leader) flag(p.status, GDR_STATUS_ROW_TOO_LONG);
        return;
    }
    const int col = warp * Sh::WC + vl * C;  // inside the unit's tile
    float *orow = p.out + (long long)m.t0 * p.out_ss + (long long)(h * V + us * Sh::CW + col) * p.out_vs;
    if (m.slot < 0 || m.slot >= p.max_slots) {
        if (m.slot != -1 && leader) flag(p.status, GDR_STATUS_BAD_SLOT);
        if (kl == 0) {
            float z[C];
#pragma unroll
            for (int c = 0; c < C; ++c) z[c] = 0.0f;
            store_f32<C>(orow, p.out_vs, p.out_vec, z);
        }
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
    // Rows 8*kl .. 8*kl+7 share the swizzle (row / 8 == kl), so this lane's
    // chunk of row 8*kl + i sits at a fixed base plus i*CPR.
    uint4 *mine = stage + kl * 8 * CPR + ((col / C) ^ (kl & (CPR - 1)));
    float a[C], bq[C];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        Pack<ST, C> x;
        x.u.v = *reinterpret_cast<const VT *>(mine + i * CPR);
#pragma unroll
        for (int c = 0; c < C; ++c) {
            const float s = x.get(c);
            a[c] = i == 0 ? chain_first(s, k[i]) : chain_next(s, k[i], a[c]);
            bq[c] = i == 0 ? chain_first(s, q[i]) : chain_next(s, q[i], bq[c]);
        }
    }
    const float alpha = gdr_alpha(ab[0], p.decay_is_log);
    const float beta = ab[1];
    float u[C];
    if constexpr (LK == 2 * C) {
        // Reduce-scatter over the LK lanes of a column group: at the level that
        // pairs lanes (l, l^m) each lane keeps half of its values and adds the
        // partner's partials for them -- the same pairwise tree as tree_lanes,
        // in 2C-1 shuffles instead of 2C*log2(LK).  Lane kl ends with value
        // j = bit-reverse(kl) of [a_0..a_{C-1}, b_0..b_{C-1}].
        float x[2 * C];
#pragma unroll
        for (int c = 0; c < C; ++c) {
            x[c] = a[c];
            x[C + c] = bq[c];
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
        // lane pair (kl, kl^1) holds (a_c, b_c) with c = bits 1..3 of kl reversed
        int c = 0;
#pragma unroll
        for (int m = 2, w = C / 2; m < LK; m <<= 1, w >>= 1) c += (kl & m) ? w : 0;
        const float other = __shfl_xor_sync(kFull, x[0], 1);
        const float A = (kl & 1) ? other : x[0];
        const float B = (kl & 1) ? x[0] : other;
        const float uc = gdr_u(beta, alpha, A, vs[col + c]);
        if (!(kl & 1)) orow[(long long)c * p.out_vs] = gdr_o(alpha, B, kq, uc);
#pragma unroll
        for (int cc = 0; cc < C; ++cc) {
            int src = 0;
#pragma unroll
            for (int m = 2, w = C / 2; m < LK; m <<= 1, w >>= 1) src |= (cc & w) ? m : 0;
            u[cc] = __shfl_sync(kFull, uc, (lane & ~(LK - 1)) | src);
        }
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
    // then writes the whole tile to HBM with coalesced rows (unit_store).
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        Pack<ST, C> x;
        x.u.v = *reinterpret_cast<const VT *>(mine + i * CPR);
        float n[C];
#pragma unroll
        for (int c = 0; c < C; ++c) n[c] = gdr_advance(x.get(c), k[i], u[c], alpha);
        if constexpr (sizeof(ST) == 2 && C % 2 == 0) {
            // two round-to-nearest-even conversions per instruction (same bits as one at a time)
            uint32_t w[C / 2];
#pragma unroll
            for (int j = 0; j < C / 2; ++j) {
                const __nv_bfloat162 h2 = __floats2bfloat162_rn(n[2 * j], n[2 * j + 1]);
                w[j] = *reinterpret_cast<const uint32_t *>(&h2);
            }
            *reinterpret_cast<VT *>(mine + i * CPR) = *reinterpret_cast<const VT *>(w);
        } else {
#pragma unroll
            for (int c = 0; c < C; ++c) x.set(c, n[c]);
            *reinterpret_cast<VT *>(mine + i * CPR) = x.u.v;
        }
    }
}

// Coalesced write-back of a computed tile: consecutive threads store
// consecutive 16-byte chunks of a row.
template <typename ST, int K>
__device__ __forceinline__ void unit_store(const StepParams &p, const UnitMeta &m, const uint4 *stage) {
    using Sh = PipeShape<ST, K>;
    if (!unit_streams(p, m)) return;
    TileLane<ST, K> tl;
    tl.init(p);
    const int h = m.hu / Sh::USL, us = m.hu % Sh::USL;
    ST *dst = reinterpret_cast<ST *>(p.state) + (long long)m.slot * p.st_slot + (long long)h * p.st_head +
              us * Sh::CW + tl.goff;
#pragma unroll
    for (int j = 0; j < TileLane<ST, K>::NJ; ++j)
        *reinterpret_cast<uint4 *>(dst + j * tl.gstep) = stage[tl.soff(j)];
}

template <typename ST, int K, int NS>
__global__ void __launch_bounds__(PipeShape<ST, K>::NT, NS == 2 ? 3 : 2)
    k_decode_pipe(const StepParams p, const int nunits) {
    using Sh = PipeShape<ST, K>;
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
        unit_compute<ST, K>(p, mq[0], smem_pipe + cur * Sh::SC);
        __syncthreads();
        unit_store<ST, K>(p, mq[0], smem_pipe + cur * Sh::SC);
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

template <typename ST, int K> static cudaError_t launch_pipe_t(const StepParams &p, cudaStream_t st) {
    using Sh = PipeShape<ST, K>;
    constexpr int NS = kDecodeStages;
    constexpr int SMEM = NS * Sh::SMEM1;
    static int configured[64] = {0};
    static int sms[64] = {0}, occ[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        e = cudaFuncSetAttribute(k_decode_pipe<ST, K, NS>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
        if (e != cudaSuccess) return e;
        e = cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ[dev], k_decode_pipe<ST, K, NS>, Sh::NT, SMEM);
        if (e != cudaSuccess) return e;
        if (occ[dev] < 1) occ[dev] = 1;
        configured[dev] = 1;
    }
    const long long nunits = (long long)p.batch * p.nv * Sh::USL;
    long long grid = (long long)sms[dev] * occ[dev];
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
    if constexpr (PipeShape<ST, K>::OK) {
        // the pipelined kernel counts units in 32 bits
        if (p.qkv_vec && (long long)p.batch * p.nv * PipeShape<ST, K>::USL < (1ll << 31))
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
