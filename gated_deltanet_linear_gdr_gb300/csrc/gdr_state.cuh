// A lane's block of the float32 state and the per-token sweeps over it, for
// the multi-token kernels (general and short-row).
//
// A lane holds ROWS = 8*RG consecutive rows (RG consecutive 8-row groups) x C
// consecutive columns.  Two register forms:
//
//   * row-pair form (RG even): x[gp][i][c] = {S[16gp + i][c], S[16gp + 8 + i][c]}.
//     A packed f32x2 instruction then advances the chains of two groups at
//     once, and its per-row operands {k^_{16gp+i}, k^_{16gp+8+i}} come from
//     adjacent floats of the staged vector, which is stored pair-interleaved
//     (vpos), so no operand has to be duplicated into both halves.
//   * column form (RG odd): y[r][c], packed over column pairs when C is even.
//
// Both forms evaluate exactly the fixed operation sequence of gdr_device.cuh
// (8-row chains in ascending row order started by a multiply, pairwise tree),
// so the results are identical bit for bit whatever the form.
#pragma once

#include "gdr_device.cuh"

namespace gdr {

// Shared-memory position of row j of a staged q / k vector: rows pair-
// interleaved within 16-row blocks in the row-pair form, 4 spare floats after
// every run of PADROWS rows (keeps the LK distinct 16-byte reads of one warp
// instruction in different banks).
template <bool RPAIR, int PADROWS>
__host__ __device__ constexpr int vpos(int j) {
    return (RPAIR ? (j & ~15) + 2 * (j & 7) + ((j >> 3) & 1) : j) + (j / PADROWS) * 4;
}

template <int RG, int C, bool RPAIR = RG % 2 == 0> struct LaneState;

// ---- row-pair form ----------------------------------------------------------
template <int RG, int C> struct LaneState<RG, C, true> {
    static constexpr int NP = RG / 2;
    float2 x[NP][8][C];

    __device__ __forceinline__ float get(int r, int c) const {
        return (r & 8) ? x[r >> 4][r & 7][c].y : x[r >> 4][r & 7][c].x;
    }
    __device__ __forceinline__ void set(int r, int c, float v) {
        if (r & 8)
            x[r >> 4][r & 7][c].y = v;
        else
            x[r >> 4][r & 7][c].x = v;
    }

    // Row pairs i = 2m and 2m + 1 of group pair gp from the lane's staged vector v.
    static __device__ __forceinline__ void pair2(const float *v, int gp, int m, float2 &a, float2 &b) {
        const float4 t = *reinterpret_cast<const float4 *>(v + gp * 16 + 4 * m);
        a = make_float2(t.x, t.y);
        b = make_float2(t.z, t.w);
    }

    // Eight row pairs of group pair gp from the lane's staged vector v.
    static __device__ __forceinline__ void pairs(const float *v, int gp, float2 (&o)[8]) {
#pragma unroll
        for (int m = 0; m < 4; ++m) pair2(v, gp, m, o[2 * m], o[2 * m + 1]);
    }

    static __device__ __forceinline__ void fold_tree(const float2 (&pa)[NP][C], const float2 (&pb)[NP][C],
                                                     float (&a)[C], float (&b)[C]) {
#pragma unroll
        for (int c = 0; c < C; ++c) {
            float ac[RG], bc[RG];
#pragma unroll
            for (int gp = 0; gp < NP; ++gp) {
                ac[2 * gp] = pa[gp][c].x;
                ac[2 * gp + 1] = pa[gp][c].y;
                bc[2 * gp] = pb[gp][c].x;
                bc[2 * gp + 1] = pb[gp][c].y;
            }
            a[c] = tree<RG>(ac);
            b[c] = tree<RG>(bc);
        }
    }

    // In-thread part of a = S^T kv and b = S^T qv: the lane's group chains
    // combined by the first log2(RG) tree levels.  Rows advance in the outer
    // loop so that every step issues the 2 NP C independent chains together.
    __device__ __forceinline__ void partials(const float *kv, const float *qv, float (&a)[C], float (&b)[C]) const {
        float2 pa[NP][C], pb[NP][C];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            float2 kp[NP][2], qp[NP][2];
#pragma unroll
            for (int gp = 0; gp < NP; ++gp) {
                pair2(kv, gp, m, kp[gp][0], kp[gp][1]);
                pair2(qv, gp, m, qp[gp][0], qp[gp][1]);
            }
#pragma unroll
            for (int ii = 0; ii < 2; ++ii) {
                const int i = 2 * m + ii;
#pragma unroll
                for (int gp = 0; gp < NP; ++gp) {
#pragma unroll
                    for (int c = 0; c < C; ++c) {
                        if (i == 0) {
                            pa[gp][c] = __fmul2_rn(x[gp][0][c], kp[gp][0]);
                            pb[gp][c] = __fmul2_rn(x[gp][0][c], qp[gp][0]);
                        } else {
                            pa[gp][c] = __ffma2_rn(x[gp][i][c], kp[gp][ii], pa[gp][c]);
                            pb[gp][c] = __ffma2_rn(x[gp][i][c], qp[gp][ii], pb[gp][c]);
                        }
                    }
                }
            }
        }
        fold_tree(pa, pb, a, b);
    }

    // The two halves of advance: S <- alpha S, then S <- k^ u^T + S (the same
    // roundings; the decay can then run while the reductions are reduced).
    __device__ __forceinline__ void scale(float alpha) {
        const float2 aa = make_float2(alpha, alpha);
#pragma unroll
        for (int gp = 0; gp < NP; ++gp)
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int c = 0; c < C; ++c) x[gp][i][c] = __fmul2_rn(aa, x[gp][i][c]);
    }
    __device__ __forceinline__ void add_outer(const float *kv, const float (&u)[C]) {
        float2 uu[C];
#pragma unroll
        for (int c = 0; c < C; ++c) uu[c] = make_float2(u[c], u[c]);
#pragma unroll
        for (int gp = 0; gp < NP; ++gp) {
            float2 kp[8];
            pairs(kv, gp, kp);
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int c = 0; c < C; ++c) x[gp][i][c] = __ffma2_rn(kp[i], uu[c], x[gp][i][c]);
        }
    }

    // advance with kc, then partials of the next token (kn, qn) on the new state,
    // in one sweep.
    __device__ __forceinline__ void advance_partials(const float *kc, const float *kn, const float *qn,
                                                     const float (&u)[C], float alpha, float (&a)[C],
                                                     float (&b)[C]) {
        const float2 aa = make_float2(alpha, alpha);
        float2 uu[C];
#pragma unroll
        for (int c = 0; c < C; ++c) uu[c] = make_float2(u[c], u[c]);
        float2 pa[NP][C], pb[NP][C];
#pragma unroll
        for (int gp = 0; gp < NP; ++gp) {
            float2 kp[8], knp[8], qnp[8];
            pairs(kc, gp, kp);
            pairs(kn, gp, knp);
            pairs(qn, gp, qnp);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
#pragma unroll
                for (int c = 0; c < C; ++c) {
                    x[gp][i][c] = __ffma2_rn(kp[i], uu[c], __fmul2_rn(aa, x[gp][i][c]));
                    if (i == 0) {
                        pa[gp][c] = __fmul2_rn(x[gp][0][c], knp[0]);
                        pb[gp][c] = __fmul2_rn(x[gp][0][c], qnp[0]);
                    } else {
                        pa[gp][c] = __ffma2_rn(x[gp][i][c], knp[i], pa[gp][c]);
                        pb[gp][c] = __ffma2_rn(x[gp][i][c], qnp[i], pb[gp][c]);
                    }
                }
            }
        }
        fold_tree(pa, pb, a, b);
    }
};

// ---- column form --------------------------------------------------------------
template <int RG, int C> struct LaneState<RG, C, false> {
    static constexpr int ROWS = 8 * RG;
    float y[ROWS][C];

    __device__ __forceinline__ float get(int r, int c) const { return y[r][c]; }
    __device__ __forceinline__ void set(int r, int c, float v) { y[r][c] = v; }

    static __device__ __forceinline__ void rows8(const float *v, int g, float (&o)[8]) {
#pragma unroll
        for (int m = 0; m < 2; ++m) {
            const float4 t = *reinterpret_cast<const float4 *>(v + g * 8 + 4 * m);
            o[4 * m] = t.x;
            o[4 * m + 1] = t.y;
            o[4 * m + 2] = t.z;
            o[4 * m + 3] = t.w;
        }
    }

    static __device__ __forceinline__ void fold_tree(const float (&pa)[RG][C], const float (&pb)[RG][C],
                                                     float (&a)[C], float (&b)[C]) {
#pragma unroll
        for (int c = 0; c < C; ++c) {
            float ac[RG], bc[RG];
#pragma unroll
            for (int g = 0; g < RG; ++g) {
                ac[g] = pa[g][c];
                bc[g] = pb[g][c];
            }
            a[c] = tree<RG>(ac);
            b[c] = tree<RG>(bc);
        }
    }

    __device__ __forceinline__ void partials(const float *kv, const float *qv, float (&a)[C], float (&b)[C]) const {
        float pa[RG][C], pb[RG][C];
#pragma unroll
        for (int g = 0; g < RG; ++g) {
            float k8[8], q8[8];
            rows8(kv, g, k8);
            rows8(qv, g, q8);
            chain_first_cols<C>(y[g * 8], k8[0], pa[g]);
            chain_first_cols<C>(y[g * 8], q8[0], pb[g]);
#pragma unroll
            for (int i = 1; i < 8; ++i) {
                chain_next_cols<C>(y[g * 8 + i], k8[i], pa[g]);
                chain_next_cols<C>(y[g * 8 + i], q8[i], pb[g]);
            }
        }
        fold_tree(pa, pb, a, b);
    }

    __device__ __forceinline__ void scale(float alpha) {
#pragma unroll
        for (int r = 0; r < ROWS; ++r)
#pragma unroll
            for (int c = 0; c < C; ++c) y[r][c] = __fmul_rn(alpha, y[r][c]);
    }
    // advance_cols with alpha = 1 adds k^ u^T with the same rounding (1 * S == S)
    __device__ __forceinline__ void add_outer(const float *kv, const float (&u)[C]) { advance(kv, u, 1.0f); }

    __device__ __forceinline__ void advance(const float *kv, const float (&u)[C], float alpha) {
#pragma unroll
        for (int g = 0; g < RG; ++g) {
            float k8[8];
            rows8(kv, g, k8);
#pragma unroll
            for (int i = 0; i < 8; ++i) advance_cols<C>(y[g * 8 + i], k8[i], u, alpha);
        }
    }

    __device__ __forceinline__ void advance_partials(const float *kc, const float *kn, const float *qn,
                                                     const float (&u)[C], float alpha, float (&a)[C],
                                                     float (&b)[C]) {
        float pa[RG][C], pb[RG][C];
#pragma unroll
        for (int g = 0; g < RG; ++g) {
            float kc8[8], kn8[8], qn8[8];
            rows8(kc, g, kc8);
            rows8(kn, g, kn8);
            rows8(qn, g, qn8);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                advance_cols<C>(y[g * 8 + i], kc8[i], u, alpha);
                if (i == 0) {
                    chain_first_cols<C>(y[g * 8], kn8[0], pa[g]);
                    chain_first_cols<C>(y[g * 8], qn8[0], pb[g]);
                } else {
                    chain_next_cols<C>(y[g * 8 + i], kn8[i], pa[g]);
                    chain_next_cols<C>(y[g * 8 + i], qn8[i], pb[g]);
                }
            }
        }
        fold_tree(pa, pb, a, b);
    }
};

// One lane's share of normalising one staged token in place.  The token's
// raw q and k (rows in natural order, padded every PADROWS rows) are split
// over NL = K / (8 GPL) lanes, an aligned run of the warp; lane gl owns GPL
// consecutive 8-row groups (2 in the row-pair form, so that it can write its
// rows back pair-interleaved).  Every lane of the warp must call this
// together (shuffles); lanes with act == false contribute zeros and write
// nothing.  Writes k^ = k * inv_k and q~ = q * inv_q * scale in vpos order,
// and, from lane gl == 0, *kq_out = k^ . q~.  When ring is not null, k^ is
// also written in natural order to elements ring_k .. ring_k + K - 1 of the
// ring (float32, or bfloat16 when ring_bf16).
template <int K, bool RPAIR, int PADROWS>
__device__ __forceinline__ void norm_token(float *q, float *k, float *kq_out, int gl, bool act, const StepParams &p,
                                           void *ring, int ring_bf16, long long ring_k) {
    constexpr int GPL = RPAIR ? 2 : 1, NL = K / 8 / GPL, NR = 8 * GPL;
    static_assert(PADROWS % NR == 0, "a lane's rows must not straddle padding");
    const int r0 = gl * NR;
    const int o = vpos<false, PADROWS>(r0);  // raw rows r0 .. r0+NR-1 are contiguous here
    float qv[NR], kv[NR];
#pragma unroll
    for (int m = 0; m < NR; m += 4) {
        float4 a4 = make_float4(0.f, 0.f, 0.f, 0.f), b4 = a4;
        if (act) {
            a4 = *reinterpret_cast<const float4 *>(q + o + m);
            b4 = *reinterpret_cast<const float4 *>(k + o + m);
        }
        qv[m] = a4.x; qv[m + 1] = a4.y; qv[m + 2] = a4.z; qv[m + 3] = a4.w;
        kv[m] = b4.x; kv[m + 1] = b4.y; kv[m + 2] = b4.z; kv[m + 3] = b4.w;
    }
    float sq[GPL], sk[GPL], kr[GPL];
#pragma unroll
    for (int g = 0; g < GPL; ++g) {
        sq[g] = chain_first(qv[8 * g], qv[8 * g]);
        sk[g] = chain_first(kv[8 * g], kv[8 * g]);
        kr[g] = chain_first(kv[8 * g], qv[8 * g]);
#pragma unroll
        for (int i = 1; i < 8; ++i) {
            sq[g] = chain_next(qv[8 * g + i], qv[8 * g + i], sq[g]);
            sk[g] = chain_next(kv[8 * g + i], kv[8 * g + i], sk[g]);
            kr[g] = chain_next(kv[8 * g + i], qv[8 * g + i], kr[g]);
        }
    }
    const float ssq = tree_lanes<NL>(tree<GPL>(sq));
    const float ssk = tree_lanes<NL>(tree<GPL>(sk));
    const float kqr = tree_lanes<NL>(tree<GPL>(kr));
    if (!act) return;
    float inv_k, qsc, kq;
    gdr_norm_scalars(ssq, ssk, kqr, p.l2norm, p.scale, p.eps, inv_k, qsc, kq);
    float kn[NR], qn[NR];
#pragma unroll
    for (int j = 0; j < NR; ++j) {
        kn[j] = __fmul_rn(kv[j], inv_k);
        qn[j] = __fmul_rn(qv[j], qsc);
    }
    // write back in vpos order: position m of the lane's run holds row rowof(m)
#pragma unroll
    for (int m = 0; m < NR; m += 4) {
        int rr[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) rr[e] = RPAIR ? ((m + e) >> 1) + 8 * ((m + e) & 1) : m + e;
        *reinterpret_cast<float4 *>(k + o + m) = make_float4(kn[rr[0]], kn[rr[1]], kn[rr[2]], kn[rr[3]]);
        *reinterpret_cast<float4 *>(q + o + m) = make_float4(qn[rr[0]], qn[rr[1]], qn[rr[2]], qn[rr[3]]);
    }
    if (ring) {
#pragma unroll
        for (int m = 0; m < NR; m += 4)
            ring_put4(ring, ring_bf16, ring_k + r0 + m, make_float4(kn[m], kn[m + 1], kn[m + 2], kn[m + 3]));
    }
    if (gl == 0) *kq_out = kq;
}

}  // namespace gdr
