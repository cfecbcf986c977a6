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
#include "gdr_device.cuh"

namespace gdr {

constexpr int kFoldThreads = 256;
constexpr int kMaxRingLen = 32;

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
    __shared__ __align__(16) float kh_s[kMaxRingLen][K];
    __shared__ __align__(16) float u_s[kMaxRingLen][V];
    __shared__ float a_s[kMaxRingLen];

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
            if (rows[i] < K) {
                const float kh = kh_s[t][rows[i]];
#pragma unroll
                for (int cc = 0; cc < CF; ++cc) s[i][cc] = gdr_advance(s[i][cc], kh, u[cc], alpha);
            }
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

template <typename ST, int K> static cudaError_t launch_fold_t(const FoldParams &p, cudaStream_t st) {
    const long long blocks = (long long)p.batch * p.nv * FoldShape<ST, K>::BLOCKS;
    if (blocks > 0) k_fold<ST, K><<<(unsigned)blocks, kFoldThreads, 0, st>>>(p);
    return cudaGetLastError();
}

template <typename ST, int K> static cudaError_t launch_rollback_t(const RollbackParams &p, cudaStream_t st) {
    const long long blocks = (long long)p.batch * p.nv * FoldShape<ST, K>::BLOCKS;
    if (blocks > 0) k_rollback<ST, K><<<(unsigned)blocks, kFoldThreads, 0, st>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_fold(const FoldParams &p, int K, bool bf16, cudaStream_t s) {
#define GDR_CASE(KK)                                                                    \
    case KK:                                                                            \
        return bf16 ? launch_fold_t<uint16_t, KK>(p, s) : launch_fold_t<float, KK>(p, s);
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
