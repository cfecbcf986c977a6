// Fold (commit the accepted prefix of a verify window) and rollback (restore a
// snapshot) kernels.  Both are pure streams over the state: no reductions, so
// threads are laid out for 16-byte coalesced access along the value dimension.
//
// Fold ("gated_delta_recurrence_verify_ring_gpu", summary): for a live row
// with 0 < count <= ring_len, S <- k^_t u_t^T + alpha_t S for t < count, using
// the records the verify pass wrote, then the state is written back once.  The
// advance is the same float32 operation the forward pass applies, so with a
// float32 ring the result is the forward pass over the accepted prefix, bit for
// bit; a bfloat16 ring (records rounded once by the verify pass) is widened
// exactly.  Both kernels are templated on the ring's element type RT.
//
// Rollback ("core.ssm.ops.gdp.fused_recurrent", intermediate_states): a copy of
// the accepted draft's snapshot over the live state.
#include "gdr_pipe.cuh"

namespace gdr {

constexpr int kFoldThreads = 256;

template <typename ST, int K, int VV = K> struct FoldShape {
    static constexpr int V = VV;
    static constexpr int CF = cmin(16 / (int)sizeof(ST), V);  // columns per thread (16 B)
    static constexpr int LVF = V / CF;                         // threads along a row
    static constexpr int RPP = kFoldThreads / LVF;             // rows per pass of the CTA
    static constexpr int RF0 = K / RPP;
    static constexpr int RF = RF0 < 1 ? 1 : (RF0 > 4 ? 4 : RF0);  // rows per thread
    static constexpr int RB = RPP * RF;                           // rows per CTA
    static constexpr int BLOCKS = K / RB < 1 ? 1 : K / RB;         // CTAs per (row, head)
};

// Ring element i widened to float32.
template <typename RT> __device__ __forceinline__ float ring_get(const void *ring, long long i) {
    return to_f32(reinterpret_cast<const RT *>(ring)[i]);
}

// N consecutive ring elements from shared memory (p 16-byte aligned when N % 4 == 0), widened.
template <typename RT, int N>
__device__ __forceinline__ void ring_vec(const RT *p, float (&o)[N]) {
    if constexpr (N % 4 == 0 && sizeof(RT) == 4) {
#pragma unroll
        for (int i = 0; i < N; i += 4) {
            const float4 a = *reinterpret_cast<const float4 *>(p + i);
            o[i] = a.x; o[i + 1] = a.y; o[i + 2] = a.z; o[i + 3] = a.w;
        }
    } else if constexpr (N % 4 == 0 && sizeof(RT) == 2) {
#pragma unroll
        for (int i = 0; i < N; i += 4) {
            const uint2 a = *reinterpret_cast<const uint2 *>(p + i);
            o[i] = __uint_as_float(a.x << 16);
            o[i + 1] = __uint_as_float(a.x & 0xffff0000u);
            o[i + 2] = __uint_as_float(a.y << 16);
            o[i + 3] = __uint_as_float(a.y & 0xffff0000u);
        }
    } else {
#pragma unroll
        for (int i = 0; i < N; ++i) o[i] = to_f32(p[i]);
    }
}

template <typename ST, int K, typename RT>
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
    const long long rrow = ((long long)rs * p.nk + hk) * p.ring_len * p.stride;
    for (int idx = tid; idx < c * K; idx += kFoldThreads) {
        const int t = idx / K, i = idx - t * K;
        kh_s[t][i] = ring_get<RT>(p.ring, rrow + (long long)t * p.stride + i);
    }
    for (int idx = tid; idx < c * V; idx += kFoldThreads) {
        const int t = idx / V, j = idx - t * V;
        u_s[t][j] = ring_get<RT>(p.ring, rrow + (long long)t * p.stride + p.u_off + jr * V + j);
    }
    for (int t = tid; t < c; t += kFoldThreads)
        a_s[t] = ring_get<RT>(p.ring, rrow + (long long)t * p.stride + p.alpha_off + jr);
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

template <typename ST, int K, int VV>
__global__ void __launch_bounds__(kFoldThreads) k_rollback(const RollbackParams p) {
    using Sh = FoldShape<ST, K, VV>;
    constexpr int V = VV, CF = Sh::CF, LVF = Sh::LVF, RPP = Sh::RPP, RB = Sh::RB, BLOCKS = Sh::BLOCKS;
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
// Fold for the common layouts.  The advance has no reduction, so a unit is
// (row, head, KT-row slice): KT consecutive state rows with all V columns, one
// contiguous block of memory (16 KiB at K = V = 128).  Thread t owns R rows x
// C columns (one 16-byte vector per row): rows (t / LV) * R .. + R - 1,
// columns (t % LV) * C .. + C - 1, so a warp's loads and stores cover whole
// rows.

template <typename ST, int K, int NTT, typename RT = float> struct FoldTile {
    static constexpr int V = K;
    static constexpr int NT = NTT;                                  // threads per CTA
    static constexpr int C = 16 / (int)sizeof(ST);                  // columns per thread
    static constexpr int LV = V / C;                                // threads along a row
    static constexpr int LKR = NT / LV;                             // threads along K
    static constexpr int KT = cmin(K, 16384 / (V * (int)sizeof(ST)));  // rows per unit
    static constexpr int R = KT / LKR;                              // rows per thread
    static constexpr int KS = K / KT;                               // units per (row, head)
    static constexpr int EPR = 16 / (int)sizeof(RT);                // ring elements per 16-byte chunk
    static constexpr int RK = KT / EPR, RU = V / EPR;               // chunks of the k^ slice and of u
    static constexpr int RQ = RK + RU + 1;                          // + the chunk holding alpha
    static constexpr bool OK = LV <= NT && R >= 1 && K % KT == 0;
};

// One CTA per unit: the CTA's rows go straight to registers (its R 16-byte
// loads per thread issued first), the unit's first `count` records (the
// slice's k^, the head's u, alpha) to shared memory with cp.async meanwhile;
// after one barrier every thread advances its rows and stores them.  Many CTAs
// per SM keep enough loads in flight without a software pipeline.
constexpr int kFoldDirectThreads = 256;

template <typename ST, int K, typename RT>
__global__ void __launch_bounds__(kFoldDirectThreads) k_fold_direct(const FoldParams p) {
    using F = FoldTile<ST, K, kFoldDirectThreads, RT>;
    constexpr int C = F::C, R = F::R;
    using VT = typename Pack<ST, C>::VT;
    extern __shared__ uint4 smem_fd[];
    const long long u = blockIdx.x;
    const long long bq = u / F::KS;
    const int b = (int)(bq / p.nv);
    const int hs = (int)(u - (long long)b * p.nv * F::KS);  // h * KS + ks
    const int h = hs / F::KS, ks = hs % F::KS;
    const int c = p.counts[b], slot = p.slot_idx[b], rs = p.ring_slot[b];
    const int tid = threadIdx.x;
    const bool leader = tid == 0 && hs == 0;
    if (c == 0 || slot == -1 || c > p.ring_len) return;
    if (c < 0) {
        if (leader) flag(p.status, GDR_STATUS_BAD_COUNT);
        return;
    }
    if (slot < 0 || slot >= p.max_slots) {
        if (leader) flag(p.status, GDR_STATUS_BAD_SLOT);
        return;
    }
    if (rs < 0 || rs >= p.ring_rows) {
        if (leader) flag(p.status, GDR_STATUS_BAD_RING_SLOT);
        return;
    }
    const int cg = tid % F::LV, r0 = (tid / F::LV) * R;
    ST *rows = reinterpret_cast<ST *>(p.state) + (long long)slot * p.st_slot + (long long)h * p.st_head +
               (long long)(ks * F::KT + r0) * p.st_k + cg * C;
    VT raw[R];
#pragma unroll
    for (int i = 0; i < R; ++i) raw[i] = *reinterpret_cast<const VT *>(rows + (long long)i * p.st_k);
    // records -> shared memory: per record RQ chunks [k^ slice | u | the chunk holding alpha]
    const int jr = h % p.r;
    {
        const int hk = h / p.r;
        const RT *rrow = reinterpret_cast<const RT *>(p.ring) + ((long long)rs * p.nk + hk) * p.ring_len * p.stride;
        const int a0 = p.alpha_off + (jr / F::EPR) * F::EPR;  // alpha_off is a multiple of 8
        for (int ch = tid; ch < c * F::RQ; ch += F::NT) {
            const int t = ch / F::RQ, r = ch - t * F::RQ;
            const RT *rec = rrow + (long long)t * p.stride;
            const RT *g = r < F::RK ? rec + ks * F::KT + F::EPR * r
                                    : (r < F::RK + F::RU ? rec + p.u_off + jr * K + F::EPR * (r - F::RK) : rec + a0);
            cp_async16(smem_fd + ch, g);
        }
        cp_async_commit();
        cp_async_wait<0>();
        __syncthreads();
    }
    float s[R][C];
#pragma unroll
    for (int i = 0; i < R; ++i) {
        Pack<ST, C> x;
        x.u.v = raw[i];
#pragma unroll
        for (int cc = 0; cc < C; ++cc) s[i][cc] = x.get(cc);
    }
    const RT *recs = reinterpret_cast<const RT *>(smem_fd);
    for (int t = 0; t < c; ++t) {
        const RT *rec = recs + t * F::RQ * F::EPR;
        const float alpha = to_f32(rec[(F::RK + F::RU) * F::EPR + jr % F::EPR]);
        float kh[R], uu[C];
        ring_vec<RT, R>(rec + r0, kh);
        ring_vec<RT, C>(rec + F::KT + cg * C, uu);
#pragma unroll
        for (int i = 0; i < R; ++i) advance_cols<C>(s[i], kh[i], uu, alpha);
    }
#pragma unroll
    for (int i = 0; i < R; ++i) pack_store<ST, C>(reinterpret_cast<uint4 *>(rows + (long long)i * p.st_k), s[i]);
}

// Two neighbouring slices per CTA (the whole head at K = V = 128 in bf16):
// both slices' state loads are issued before the records are copied, so a CTA
// keeps twice the bytes in flight; the records of the two slices share u and
// alpha.  Measured 41.2 us against 45.1 us for one slice per CTA on the verify
// workload's fold.
template <typename ST, int K, typename RT>
__global__ void __launch_bounds__(kFoldDirectThreads) k_fold_pair(const FoldParams p) {
    using F = FoldTile<ST, K, kFoldDirectThreads, RT>;
    constexpr int C = F::C, R = F::R, KP = F::KS / 2, RQ2 = 2 * F::RK + F::RU + 1;
    using VT = typename Pack<ST, C>::VT;
    extern __shared__ uint4 smem_fd[];
    const long long u = blockIdx.x;
    const long long bq = u / KP;
    const int b = (int)(bq / p.nv);
    const int hp = (int)(u - (long long)b * p.nv * KP);
    const int h = hp / KP, kp = hp % KP;
    const int c = p.counts[b], slot = p.slot_idx[b], rs = p.ring_slot[b];
    const int tid = threadIdx.x;
    const bool leader = tid == 0 && hp == 0;
    if (c == 0 || slot == -1 || c > p.ring_len) return;
    if (c < 0) {
        if (leader) flag(p.status, GDR_STATUS_BAD_COUNT);
        return;
    }
    if (slot < 0 || slot >= p.max_slots) {
        if (leader) flag(p.status, GDR_STATUS_BAD_SLOT);
        return;
    }
    if (rs < 0 || rs >= p.ring_rows) {
        if (leader) flag(p.status, GDR_STATUS_BAD_RING_SLOT);
        return;
    }
    const int cg = tid % F::LV, r0 = (tid / F::LV) * R;
    ST *rows0 = reinterpret_cast<ST *>(p.state) + (long long)slot * p.st_slot + (long long)h * p.st_head +
                (long long)(2 * kp * F::KT + r0) * p.st_k + cg * C;
    ST *rows1 = rows0 + (long long)F::KT * p.st_k;
    VT raw0[R], raw1[R];
#pragma unroll
    for (int i = 0; i < R; ++i) raw0[i] = *reinterpret_cast<const VT *>(rows0 + (long long)i * p.st_k);
#pragma unroll
    for (int i = 0; i < R; ++i) raw1[i] = *reinterpret_cast<const VT *>(rows1 + (long long)i * p.st_k);
    // records -> shared memory: per record RQ2 chunks [k^ of both slices | u | the chunk holding alpha]
    const int jr = h % p.r;
    {
        const int hk = h / p.r;
        const RT *rrow = reinterpret_cast<const RT *>(p.ring) + ((long long)rs * p.nk + hk) * p.ring_len * p.stride;
        const int a0 = p.alpha_off + (jr / F::EPR) * F::EPR;
        for (int ch = tid; ch < c * RQ2; ch += F::NT) {
            const int t = ch / RQ2, r = ch - t * RQ2;
            const RT *rec = rrow + (long long)t * p.stride;
            const RT *g = r < 2 * F::RK ? rec + 2 * kp * F::KT + F::EPR * r
                                        : (r < 2 * F::RK + F::RU ? rec + p.u_off + jr * K + F::EPR * (r - 2 * F::RK) : rec + a0);
            cp_async16(smem_fd + ch, g);
        }
        cp_async_commit();
        cp_async_wait<0>();
        __syncthreads();
    }
    const RT *recs = reinterpret_cast<const RT *>(smem_fd);
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        float s[R][C];
#pragma unroll
        for (int i = 0; i < R; ++i) {
            Pack<ST, C> x;
            x.u.v = half ? raw1[i] : raw0[i];
#pragma unroll
            for (int cc = 0; cc < C; ++cc) s[i][cc] = x.get(cc);
        }
        for (int t = 0; t < c; ++t) {
            const RT *rec = recs + t * RQ2 * F::EPR;
            const float alpha = to_f32(rec[(2 * F::RK + F::RU) * F::EPR + jr % F::EPR]);
            float kh[R], uu[C];
            ring_vec<RT, R>(rec + half * F::KT + r0, kh);
            ring_vec<RT, C>(rec + 2 * F::KT + cg * C, uu);
#pragma unroll
            for (int i = 0; i < R; ++i) advance_cols<C>(s[i], kh[i], uu, alpha);
        }
        ST *rows = half ? rows1 : rows0;
#pragma unroll
        for (int i = 0; i < R; ++i) pack_store<ST, C>(reinterpret_cast<uint4 *>(rows + (long long)i * p.st_k), s[i]);
    }
}

template <typename ST, int K, typename RT> static cudaError_t launch_fold_direct_t(const FoldParams &p, cudaStream_t st) {
    using F = FoldTile<ST, K, kFoldDirectThreads, RT>;
    if constexpr (F::KS % 2 == 0) {
        const int smem2 = p.ring_len * (2 * F::RK + F::RU + 1) * 16;
        const long long blocks2 = (long long)p.batch * p.nv * (F::KS / 2);
        if (blocks2 > 0) k_fold_pair<ST, K, RT><<<(unsigned)blocks2, F::NT, smem2, st>>>(p);
        return cudaGetLastError();
    }
    const int smem = p.ring_len * F::RQ * 16;
    const long long blocks = (long long)p.batch * p.nv * F::KS;
    if (blocks > 0) k_fold_direct<ST, K, RT><<<(unsigned)blocks, F::NT, smem, st>>>(p);
    return cudaGetLastError();
}

template <typename ST, int K, typename RT> static cudaError_t launch_fold_t(const FoldParams &p, cudaStream_t st) {
    const long long blocks = (long long)p.batch * p.nv * FoldShape<ST, K>::BLOCKS;
    const size_t smem = (size_t)p.ring_len * (2 * K + 1) * sizeof(float);  // <= 32 x 257 x 4 bytes
    if (blocks > 0) k_fold<ST, K, RT><<<(unsigned)blocks, kFoldThreads, smem, st>>>(p);
    return cudaGetLastError();
}

template <typename ST, int K, int V> static cudaError_t launch_rollback_t(const RollbackParams &p, cudaStream_t st) {
    const long long blocks = (long long)p.batch * p.nv * FoldShape<ST, K, V>::BLOCKS;
    if (blocks > 0) k_rollback<ST, K, V><<<(unsigned)blocks, kFoldThreads, 0, st>>>(p);
    return cudaGetLastError();
}

template <typename ST, int K, typename RT> static cudaError_t launch_fold_rt(const FoldParams &p, cudaStream_t s) {
    using F = FoldTile<ST, K, kFoldDirectThreads, RT>;
    const bool aligned = (reinterpret_cast<uintptr_t>(p.ring) & 15u) == 0 && p.stride % F::EPR == 0 &&
                         p.u_off % F::EPR == 0 && p.alpha_off % 8 == 0;
    if constexpr (F::OK) {
        if (aligned && (long long)p.batch * p.nv * F::KS < (1ll << 31)) return launch_fold_direct_t<ST, K, RT>(p, s);
    }
    return launch_fold_t<ST, K, RT>(p, s);
}

template <typename ST, int K> static cudaError_t launch_fold_any(const FoldParams &p, cudaStream_t s) {
    return p.ring_bf16 ? launch_fold_rt<ST, K, uint16_t>(p, s) : launch_fold_rt<ST, K, float>(p, s);
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

// V = K, V = 2K, and V = K/2 for K >= 32.
template <typename ST, int K> static cudaError_t rollback_v(const RollbackParams &p, int V, cudaStream_t s) {
    if (V == K) return launch_rollback_t<ST, K, K>(p, s);
    if (V == 2 * K) return launch_rollback_t<ST, K, 2 * K>(p, s);
    if constexpr (K >= 32) {
        if (2 * V == K) return launch_rollback_t<ST, K, K / 2>(p, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_rollback(const RollbackParams &p, int K, int V, bool bf16, cudaStream_t s) {
#define GDR_CASE(KK) \
    case KK: return bf16 ? rollback_v<uint16_t, KK>(p, V, s) : rollback_v<float, KK>(p, V, s);
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
