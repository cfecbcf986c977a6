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

template <typename ST, int K> static cudaError_t launch_decode_t(const StepParams &p, cudaStream_t st) {
    const long long nunits = (long long)p.batch * p.nv * DecodeShape<ST, K>::SLICES;
    const long long blocks = (nunits + kDecodeThreads / 32 - 1) / (kDecodeThreads / 32);
    if (blocks > 0) k_decode<ST, K><<<(unsigned)blocks, kDecodeThreads, 0, st>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_decode(const StepParams &p, int K, bool bf16, cudaStream_t s) {
#define GDR_CASE(KK)                                                                        \
    case KK:                                                                                \
        return bf16 ? launch_decode_t<uint16_t, KK>(p, s) : launch_decode_t<float, KK>(p, s);
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
