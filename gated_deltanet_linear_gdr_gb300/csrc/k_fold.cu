// Fold (commit the accepted prefix of a verify window) and rollback (restore a
// snapshot) kernels.  Both are pure streams over the state: no reductions, so
// threads are laid out for 16-byte coalesced access along the value dimension.
//
// Fold ("gated_delta_recurrence_verify_ring_gpu", summary): for a live row
// with 0 < count <= ring_len, S <- k^_t u_t^T + alpha_t S for t < count, using
// the records the verify pass wrote, then the state is written back once.  The
// advance is the same float32 operation the forward pass applies, so with a
// float32 ring the result is the forward pass over the accepted prefix, bit for
// bit.
//
// Rollback ("core.ssm.ops.gdp.fused_recurrent", intermediate_states): a copy of
// the accepted draft's snapshot over the live state.
#include "gdr_pipe.cuh"

namespace gdr {

constexpr int kFoldThreads = 256;

template <typename ST, int K> struct FoldShape {
    static constexpr int V = K;
    static constexpr int CF = cmin(16 / (int)sizeof(ST), V);  // columns per thread (16 B)
    static constexpr int LVF = V / CF;                         // threads along a row
    static constexpr int RPP = kFoldThreads / LVF;             // rows per pass of the CTA
    static constexpr int RF0 = K / RPP;
    static constexpr int RF = RF0 < 1 ? 1 : (RF0 > 4 ? 4 : RF0);  // rows per thread
    static constexpr int RB = RPP * RF;                           // rows per CTA
    static constexpr int BLOCKS = K / RB < 1 ? 1 : K / RB;         // CTAs per (row, head)
};

template <typename ST, int K>
__global__ void __launch_bounds__(kFoldThreads) k_fold(const FoldParams p) {
    using Sh = FoldShape<ST, K>;
    constexpr int V = K, CF = Sh::CF, LVF = Sh::LVF, RPP = Sh::RPP, RF = Sh::RF, RB = Sh::RB;
    constexpr int BLOCKS = Sh::BLOCKS;
    // records of this row, sized by ring_len: k^ [len][K], u [len][V], alpha [len]
    extern __shared__ __align__(16) float fold_smem[];
    float(*kh_s)[K] = reinterpret_cast<float(*)[K]>(fold_smem);
    float(*u_s)[V] = reinterpret_cast<float(*)[V]>(fold_smem + p.ring_len * K);
    float *a_s = fold_smem + p.ring_len * (K + V);

    const int tid = threadIdx.x;
    const int blk = (int)(blockIdx.x % BLOCKS);
    const long long bh = blockIdx.x / BLOCKS;
    const int h = (int)(bh % p.nv);
    const int b = (int)(bh / p.nv);
    const bool leader = tid == 0 && blk == 0 && h == 0;
    const int slot = p.slot_idx[b];
    const int c = p.counts[b];
    if (slot == -1 || c == 0 || c > p.ring_len) return;
    if (c < 0) {
        if (leader) flag(p.status, GDR_STATUS_BAD_COUNT);
        return;
    }
    if (slot < 0 || slot >= p.max_slots) {
        if (leader) flag(p.status, GDR_STATUS_BAD_SLOT);
        return;
    }
    const int rs = p.ring_slot[b];
    if (rs < 0 || rs >= p.ring_rows) {
        if (leader) flag(p.status, GDR_STATUS_BAD_RING_SLOT);
        return;
    }
    const int hk = h / p.r, jr = h % p.r;
    const float *rrow = p.ring + ((long long)rs * p.nk + hk) * p.ring_len * p.stride;
    for (int idx = tid; idx < c * K; idx += kFoldThreads) {
        const int t = idx / K, i = idx - t * K;
        kh_s[t][i] = rrow[(long long)t * p.stride + i];
    }
    for (int idx = tid; idx < c * V; idx += kFoldThreads) {
        const int t = idx / V, j = idx - t * V;
        u_s[t][j] = rrow[(long long)t * p.stride + p.u_off + jr * V + j];
    }
    for (int t = tid; t < c; t += kFoldThreads) a_s[t] = rrow[(long long)t * p.stride + p.alpha_off + jr];
    __syncthreads();

    const int lv = tid % LVF, rsub = tid / LVF;
    const int col = lv * CF;
    ST *base = reinterpret_cast<ST *>(p.state) + (long long)slot * p.st_slot + (long long)h * p.st_head + col;
    float s[RF][CF];
    int rows[RF];
#pragma unroll
    for (int i = 0; i < RF; ++i) {
        rows[i] = blk * RB + rsub + i * RPP;
        if (rows[i] < K) {
            Pack<ST, CF> x;
            x.load(base + (long long)rows[i] * p.st_k);
#pragma unroll
            for (int cc = 0; cc < CF; ++cc) s[i][cc] = x.get(cc);
        }
    }
    for (int t = 0; t < c; ++t) {
        const float alpha = a_s[t];
        float u[CF];
#pragma unroll
        for (int cc = 0; cc < CF; ++cc) u[cc] = u_s[t][col + cc];
#pragma unroll
        for (int i = 0; i < RF; ++i) {
            if (rows[i] < K) advance_cols<CF>(s[i], kh_s[t][rows[i]], u, alpha);
        }
    }
#pragma unroll
    for (int i = 0; i < RF; ++i) {
        if (rows[i] < K) {
            Pack<ST, CF> x;
#pragma unroll
            for (int cc = 0; cc < CF; ++cc) x.set(cc, s[i][cc]);
            x.store(base + (long long)rows[i] * p.st_k);
        }
    }
}

template <typename ST, int K>
__global__ void __launch_bounds__(kFoldThreads) k_rollback(const RollbackParams p) {
    using Sh = FoldShape<ST, K>;
    constexpr int V = K, CF = Sh::CF, LVF = Sh::LVF, RPP = Sh::RPP, RB = Sh::RB, BLOCKS = Sh::BLOCKS;
    const int tid = threadIdx.x;
    const int blk = (int)(blockIdx.x % BLOCKS);
    const long long bh = blockIdx.x / BLOCKS;
    const int h = (int)(bh % p.nv);
    const int b = (int)(bh / p.nv);
    const bool leader = tid == 0 && blk == 0 && h == 0;
    const int slot = p.slot_idx[b];
    const int a = p.accepted[b];
    if (slot == -1 || a == -1) return;
    if (slot < 0 || slot >= p.max_slots) {
        if (leader) flag(p.status, GDR_STATUS_BAD_SLOT);
        return;
    }
    if (a < 0 || a >= p.n_inter) {
        if (leader) flag(p.status, GDR_STATUS_BAD_ACCEPTED);
        return;
    }
    const int lv = tid % LVF, rsub = tid / LVF;
    const ST *src = reinterpret_cast<const ST *>(p.inter) + (long long)slot * p.s_slot +
                    (long long)a * p.s_tok + (long long)h * p.s_head + lv * CF;
    ST *dst = reinterpret_cast<ST *>(p.state) + (long long)slot * p.st_slot + (long long)h * p.st_head + lv * CF;
    for (int r = blk * RB + rsub; r < (blk + 1) * RB && r < K; r += RPP) {
        Pack<ST, CF> x;
        x.load(src + (long long)r * V);
        x.store(dst + (long long)r * p.st_k);
    }
}

// ---------------------------------------------------------------------------
// Pipelined fold for the common layouts: persistent CTAs walk (row, head,
// tile) units; a unit's stage holds its state tile and its first `count`
// records (k^, the tile's u columns, alpha), copied with cp.async while the
// previous unit computes; the new tile leaves through the stage as coalesced
// rows.  Lane layout and arithmetic as the other pipelined kernels.

// Warps per CTA (tile width) and CTAs per SM of the pipelined fold.
constexpr int kFoldWarps = 4;
constexpr int kFoldMinBlocks = 4;

struct FoldMeta {
    int hu, c, slot, rs;  // c == 0: nothing to do
};

template <int USL>
__device__ __forceinline__ FoldMeta fold_meta(const FoldParams &p, long long u, int nunits) {
    FoldMeta m{};
    if (u >= nunits) return m;
    const int ui = (int)u;
    const int b = ui / USL / p.nv;
    m.hu = ui - b * p.nv * USL;
    m.c = p.counts[b];
    m.slot = p.slot_idx[b];
    m.rs = p.ring_slot[b];
    return m;
}

__device__ __forceinline__ bool fold_active(const FoldParams &p, const FoldMeta &m) {
    return m.c >= 1 && m.c <= p.ring_len && m.slot >= 0 && m.slot < p.max_slots && m.rs >= 0 &&
           m.rs < p.ring_rows;
}

template <typename ST, int K> struct FoldPipeShape {
    using P = PipeShape<ST, K, kFoldWarps>;
    static constexpr int RQ = K / 4 + P::CW / 4 + 1;  // 16-byte chunks per staged record
};

template <typename ST, int K>
__device__ __forceinline__ void fold_issue(const FoldParams &p, const FoldMeta &m, uint4 *stage) {
    using P = PipeShape<ST, K, kFoldWarps>;
    using F = FoldPipeShape<ST, K>;
    if (fold_active(p, m)) {
        const int h = m.hu / P::USL, us = m.hu % P::USL;
        tile_issue<ST, K, PipeShape<ST, K, kFoldWarps>::NT, kFoldWarps>(reinterpret_cast<const ST *>(p.state) + (long long)m.slot * p.st_slot +
                              (long long)h * p.st_head + us * P::CW,
                          p.st_k, stage);
        const int hk = h / p.r, jr = h % p.r;
        const float *rrow = p.ring + ((long long)m.rs * p.nk + hk) * p.ring_len * p.stride;
        uint4 *recs = stage + P::S_STATE;
        constexpr int RV = K / 4 + P::CW / 4;  // vector chunks per record
        for (int ch = threadIdx.x; ch < m.c * RV; ch += P::NT) {
            const int t = ch / RV, r = ch - t * RV;
            const float *rec = rrow + (long long)t * p.stride;
            const float *g = r < K / 4 ? rec + 4 * r : rec + p.u_off + jr * K + us * P::CW + 4 * (r - K / 4);
            cp_async16(recs + t * F::RQ + r, g);
        }
        for (int t = threadIdx.x; t < m.c; t += P::NT)
            cp_async4(recs + t * F::RQ + RV, rrow + (long long)t * p.stride + p.alpha_off + jr);
    }
    cp_async_commit();
}

template <typename ST, int K>
__device__ __forceinline__ bool fold_compute(const FoldParams &p, const FoldMeta &m, uint4 *stage) {
    using P = PipeShape<ST, K, kFoldWarps>;
    using F = FoldPipeShape<ST, K>;
    constexpr int LK = P::LK, C = P::C, CPR = P::CPR;
    using VT = typename Pack<ST, C>::VT;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const bool leader = tid == 0 && m.hu == 0;
    if (m.c == 0 || m.slot == -1 || m.c > p.ring_len) return false;
    if (m.c < 0) {
        if (leader) flag(p.status, GDR_STATUS_BAD_COUNT);
        return false;
    }
    if (m.slot < 0 || m.slot >= p.max_slots) {
        if (leader) flag(p.status, GDR_STATUS_BAD_SLOT);
        return false;
    }
    if (m.rs < 0 || m.rs >= p.ring_rows) {
        if (leader) flag(p.status, GDR_STATUS_BAD_RING_SLOT);
        return false;
    }
    const int kl = lane % LK, vl = lane / LK;
    const int col = warp * P::WC + vl * C;
    uint4 *mine = tile_lane_base<ST, K, kFoldWarps>(stage, kl, col);
    float s[8][C];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        Pack<ST, C> x;
        x.u.v = *reinterpret_cast<const VT *>(mine + i * CPR);
#pragma unroll
        for (int cc = 0; cc < C; ++cc) s[i][cc] = x.get(cc);
    }
    const float *recs = reinterpret_cast<const float *>(stage + P::S_STATE);
    for (int t = 0; t < m.c; ++t) {
        const float *rec = recs + t * F::RQ * 4;
        const float alpha = rec[K + P::CW];
        float kh[8], u[C];
#pragma unroll
        for (int i = 0; i < 8; i += 4) {
            const float4 a4 = *reinterpret_cast<const float4 *>(rec + kl * 8 + i);
            kh[i] = a4.x; kh[i + 1] = a4.y; kh[i + 2] = a4.z; kh[i + 3] = a4.w;
        }
#pragma unroll
        for (int cc = 0; cc < C; cc += 4) {
            const float4 b4 = *reinterpret_cast<const float4 *>(rec + K + col + cc);
            u[cc] = b4.x; u[cc + 1] = b4.y; u[cc + 2] = b4.z; u[cc + 3] = b4.w;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) advance_cols<C>(s[i], kh[i], u, alpha);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) pack_store<ST, C>(mine + i * CPR, s[i]);
    return true;
}

template <typename ST, int K>
__global__ void __launch_bounds__(PipeShape<ST, K, kFoldWarps>::NT, kFoldMinBlocks) k_fold_pipe(const FoldParams p, const int nunits) {
    using P = PipeShape<ST, K, kFoldWarps>;
    extern __shared__ uint4 smem_fold[];
    const int SC = P::S_STATE + p.ring_len * FoldPipeShape<ST, K>::RQ;
    uint4 *stage0 = smem_fold, *stage1 = smem_fold + SC;
    const long long G = gridDim.x;
    FoldMeta cur = fold_meta<P::USL>(p, blockIdx.x, nunits);
    fold_issue<ST, K>(p, cur, stage0);
    FoldMeta nxt = fold_meta<P::USL>(p, (long long)blockIdx.x + G, nunits);
    int sel = 0;
    for (long long u = blockIdx.x; u < nunits; u += G) {
        uint4 *s_cur = sel ? stage1 : stage0;
        uint4 *s_nxt = sel ? stage0 : stage1;
        fold_issue<ST, K>(p, nxt, s_nxt);
        const FoldMeta later = fold_meta<P::USL>(p, u + 2 * G, nunits);
        cp_async_wait<1>();
        __syncthreads();
        const bool done = fold_compute<ST, K>(p, cur, s_cur);
        __syncthreads();
        if (done) {
            const int h = cur.hu / P::USL, us = cur.hu % P::USL;
            tile_store<ST, K, PipeShape<ST, K, kFoldWarps>::NT, kFoldWarps>(reinterpret_cast<ST *>(p.state) + (long long)cur.slot * p.st_slot +
                                  (long long)h * p.st_head + us * P::CW,
                              p.st_k, s_cur);
        }
        __syncthreads();
        cur = nxt;
        nxt = later;
        sel ^= 1;
    }
    cp_async_wait<0>();
}

template <typename ST, int K> static cudaError_t launch_fold_pipe_t(const FoldParams &p, cudaStream_t st) {
    using P = PipeShape<ST, K, kFoldWarps>;
    const int smem = 2 * (P::S_STATE + p.ring_len * FoldPipeShape<ST, K>::RQ) * 16;
    static int sms[64] = {0};
    static int occ[64][33] = {{0}};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!occ[dev][p.ring_len]) {
        e = cudaFuncSetAttribute(k_fold_pipe<ST, K>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 2 * (P::S_STATE + 32 * FoldPipeShape<ST, K>::RQ) * 16);
        if (e != cudaSuccess) return e;
        e = cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        int o = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, k_fold_pipe<ST, K>, P::NT, smem);
        if (e != cudaSuccess) return e;
        occ[dev][p.ring_len] = o < 1 ? 1 : o;
    }
    const long long nunits = (long long)p.batch * p.nv * P::USL;
    long long grid = (long long)sms[dev] * occ[dev][p.ring_len];
    if (grid > nunits) grid = nunits;
    if (grid > 0) k_fold_pipe<ST, K><<<(unsigned)grid, P::NT, smem, st>>>(p, (int)nunits);
    return cudaGetLastError();
}

template <typename ST, int K> static cudaError_t launch_fold_t(const FoldParams &p, cudaStream_t st) {
    const long long blocks = (long long)p.batch * p.nv * FoldShape<ST, K>::BLOCKS;
    const size_t smem = (size_t)p.ring_len * (2 * K + 1) * sizeof(float);  // <= 32 x 257 x 4 bytes
    if (blocks > 0) k_fold<ST, K><<<(unsigned)blocks, kFoldThreads, smem, st>>>(p);
    return cudaGetLastError();
}

template <typename ST, int K> static cudaError_t launch_rollback_t(const RollbackParams &p, cudaStream_t st) {
    const long long blocks = (long long)p.batch * p.nv * FoldShape<ST, K>::BLOCKS;
    if (blocks > 0) k_rollback<ST, K><<<(unsigned)blocks, kFoldThreads, 0, st>>>(p);
    return cudaGetLastError();
}

template <typename ST, int K> static cudaError_t launch_fold_any(const FoldParams &p, cudaStream_t s) {
    if constexpr (PipeShape<ST, K, kFoldWarps>::OK) {
        const bool aligned = (reinterpret_cast<uintptr_t>(p.ring) & 15u) == 0 && p.stride % 4 == 0 &&
                             p.u_off % 4 == 0;
        if (aligned && (long long)p.batch * p.nv * PipeShape<ST, K, kFoldWarps>::USL < (1ll << 31))
            return launch_fold_pipe_t<ST, K>(p, s);
    }
    return launch_fold_t<ST, K>(p, s);
}

cudaError_t launch_fold(const FoldParams &p, int K, bool bf16, cudaStream_t s) {
#define GDR_CASE(KK)                                                                        \
    case KK:                                                                                \
        return bf16 ? launch_fold_any<uint16_t, KK>(p, s) : launch_fold_any<float, KK>(p, s);
    switch (K) {
        GDR_CASE(16)
        GDR_CASE(32)
        GDR_CASE(64)
        GDR_CASE(128)
    }
#undef GDR_CASE
    return cudaErrorInvalidValue;
}

cudaError_t launch_rollback(const RollbackParams &p, int K, bool bf16, cudaStream_t s) {
#define GDR_CASE(KK)                                                                            \
    case KK:                                                                                    \
        return bf16 ? launch_rollback_t<uint16_t, KK>(p, s) : launch_rollback_t<float, KK>(p, s);
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
