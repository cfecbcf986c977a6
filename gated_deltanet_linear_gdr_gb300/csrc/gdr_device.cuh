// Device-side building blocks shared by every GDR kernel.
//
// All kernels compute each token with ONE fixed sequence of float32 operations,
// written here with explicit round-to-nearest intrinsics so the compiler cannot
// contract or reorder them differently in different kernels:
//
//   * K-reductions (S^T k^, S^T q~, |q|^2, |k|^2, k.q) split the K rows into
//     groups of 8 consecutive rows; a group's partial is a multiply followed by
//     seven fused multiply-adds in ascending row order; group partials are
//     combined by a pairwise tree whose first level adds groups (0,1),(2,3),...,
//     the next ((0,1),(2,3)), and so on.  Any thread layout that gives a thread
//     a run of consecutive groups and puts the remaining levels on lanes reached
//     with xor-shuffles of increasing distance produces exactly this tree.
//   * Per token, with S the state before the token's decay:
//       a_j = sum_i S_ij k^_i,  b_j = sum_i S_ij q~_i   (q~ = q^ * scale)
//       u_j = beta * (v_j - alpha * a_j)
//       o_j = alpha * b_j + (k^ . q~) * u_j            (= scale * S_new^T q^)
//       S_ij <- k^_i * u_j + alpha * S_ij
//     which is the gated delta rule of "gated_delta_recurrence_fwd_gpu" and
//     "core.ssm.ops.gdp.fused_recurrent" with the readout of the new state
//     expanded, so one sweep over S serves both reductions.
//
// Because fwd, verify, fold and snapshots all apply the same advance
// S <- fma(k^, u, alpha*S) with the same u, verify+fold over a prefix and the
// forward pass over that prefix give identical bits.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "gdr_internal.h"

namespace gdr {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ void flag(unsigned *status, unsigned bit) {
    if (status) atomicOr(status, bit);
}

// ---- storage types ---------------------------------------------------------
// bfloat16 is carried as its raw 16-bit pattern (uint16_t).
__device__ __forceinline__ float to_f32(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }
__device__ __forceinline__ float to_f32(float x) { return x; }

template <typename ST> __device__ __forceinline__ ST from_f32(float x);
template <> __device__ __forceinline__ uint16_t from_f32<uint16_t>(float x) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }

template <int BYTES> struct VecT;
template <> struct VecT<16> { using T = uint4; };
template <> struct VecT<8> { using T = uint2; };
template <> struct VecT<4> { using T = uint32_t; };
template <> struct VecT<2> { using T = uint16_t; };

// C consecutive elements of storage type ST moved as one vector access.
template <typename ST, int C> struct Pack {
    static constexpr int BYTES = C * (int)sizeof(ST);
    using VT = typename VecT<BYTES>::T;
    union {
        VT v;
        ST e[C];
    } u;
    __device__ __forceinline__ float get(int i) const { return to_f32(u.e[i]); }
    __device__ __forceinline__ void set(int i, float x) { u.e[i] = from_f32<ST>(x); }
    __device__ __forceinline__ void load(const ST *p) { u.v = *reinterpret_cast<const VT *>(p); }
    __device__ __forceinline__ void store(ST *p) const { *reinterpret_cast<VT *>(p) = u.v; }
};

// N floats from p[0], p[stride], ...; one vector load when allowed.
template <int N>
__device__ __forceinline__ void load_f32(const float *p, long long stride, bool vec, float (&x)[N]) {
    if (vec) {
        if constexpr (N % 4 == 0) {
#pragma unroll
            for (int i = 0; i < N; i += 4) {
                float4 t = *reinterpret_cast<const float4 *>(p + i);
                x[i] = t.x; x[i + 1] = t.y; x[i + 2] = t.z; x[i + 3] = t.w;
            }
            return;
        } else if constexpr (N == 2) {
            float2 t = *reinterpret_cast<const float2 *>(p);
            x[0] = t.x; x[1] = t.y;
            return;
        }
    }
#pragma unroll
    for (int i = 0; i < N; ++i) x[i] = p[i * stride];
}

template <int N>
__device__ __forceinline__ void store_f32(float *p, long long stride, bool vec, const float (&x)[N]) {
    if (vec) {
        if constexpr (N % 4 == 0) {
#pragma unroll
            for (int i = 0; i < N; i += 4)
                *reinterpret_cast<float4 *>(p + i) = make_float4(x[i], x[i + 1], x[i + 2], x[i + 3]);
            return;
        } else if constexpr (N == 2) {
            *reinterpret_cast<float2 *>(p) = make_float2(x[0], x[1]);
            return;
        }
    }
#pragma unroll
    for (int i = 0; i < N; ++i) p[i * stride] = x[i];
}

// Zeroes C output columns of n consecutive tokens starting at row pointer o
// (rows p.out_ss apart): the output of a skipped (row, head).
template <int C>
__device__ __forceinline__ void zero_rows(float *o, int n, const StepParams &p) {
    float z[C];
#pragma unroll
    for (int c = 0; c < C; ++c) z[c] = 0.0f;
    for (int t = 0; t < n; ++t) store_f32<C>(o + (long long)t * p.out_ss, p.out_vs, p.out_vec, z);
}

// ---- ring records: float32, or bfloat16 rounded to nearest-even once --------
// i is an element index into the ring; i2 is even, i4 a multiple of 4 (the
// ring base is 16-byte aligned and record strides keep the alignment).
__device__ __forceinline__ void ring_put1(void *ring, int bf16, long long i, float v) {
    if (bf16)
        reinterpret_cast<uint16_t *>(ring)[i] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
    else
        reinterpret_cast<float *>(ring)[i] = v;
}
__device__ __forceinline__ void ring_put2(void *ring, int bf16, long long i2, float a, float b) {
    if (bf16)
        *reinterpret_cast<__nv_bfloat162 *>(reinterpret_cast<uint16_t *>(ring) + i2) = __floats2bfloat162_rn(a, b);
    else
        *reinterpret_cast<float2 *>(reinterpret_cast<float *>(ring) + i2) = make_float2(a, b);
}
__device__ __forceinline__ void ring_put4(void *ring, int bf16, long long i4, float4 v) {
    if (bf16) {
        const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
        uint2 w;
        w.x = *reinterpret_cast<const uint32_t *>(&lo);
        w.y = *reinterpret_cast<const uint32_t *>(&hi);
        *reinterpret_cast<uint2 *>(reinterpret_cast<uint16_t *>(ring) + i4) = w;
    } else {
        *reinterpret_cast<float4 *>(reinterpret_cast<float *>(ring) + i4) = v;
    }
}

// ---- the fixed per-token arithmetic ----------------------------------------

__device__ __forceinline__ float chain_first(float x, float y) { return __fmul_rn(x, y); }
__device__ __forceinline__ float chain_next(float x, float y, float p) { return __fmaf_rn(x, y, p); }

// Pairwise tree over a thread's RG consecutive group partials (level 1 first).
template <int N>
__device__ __forceinline__ float tree(const float *p) {
    if constexpr (N == 1) {
        return p[0];
    } else {
        return __fadd_rn(tree<N / 2>(p), tree<N / 2>(p + N / 2));
    }
}

// Remaining tree levels across the LK lanes that share a column (kl = lane % LK).
template <int LK>
__device__ __forceinline__ float tree_lanes(float x) {
#pragma unroll
    for (int m = 1; m < LK; m <<= 1) x = __fadd_rn(x, __shfl_xor_sync(kFull, x, m));
    return x;
}

__device__ __forceinline__ float gdr_alpha(float g, int is_log) { return is_log ? expf(g) : g; }

// From the reduced |q|^2, |k|^2 and raw k.q: the factors that turn raw q, k into
// q~ = q * qs (scale folded in) and k^ = k * inv_k, and k^ . q~.
__device__ __forceinline__ void gdr_norm_scalars(float ssq, float ssk, float kq_raw, int l2,
                                                 float scale, float eps, float &inv_k, float &qs,
                                                 float &kq) {
    float inv_q = 1.0f;
    inv_k = 1.0f;
    if (l2) {
        inv_q = rsqrtf(__fadd_rn(ssq, eps));
        inv_k = rsqrtf(__fadd_rn(ssk, eps));
    }
    qs = __fmul_rn(inv_q, scale);
    kq = __fmul_rn(kq_raw, __fmul_rn(inv_k, qs));
}

__device__ __forceinline__ float gdr_u(float beta, float alpha, float a, float v) {
    return __fmul_rn(beta, __fmaf_rn(-alpha, a, v));
}
__device__ __forceinline__ float gdr_o(float alpha, float b, float kq, float u) {
    return __fmaf_rn(alpha, b, __fmul_rn(kq, u));
}
__device__ __forceinline__ float gdr_advance(float s, float kh, float u, float alpha) {
    return __fmaf_rn(kh, u, __fmul_rn(alpha, s));
}

__host__ __device__ constexpr int cmin(int a, int b) { return a < b ? a : b; }

// ---- the same operations on pairs of columns --------------------------------
// Blackwell's packed f32x2 FMA / MUL round each element exactly like the
// scalar instruction, so these are bit-identical to the scalar helpers above
// and issue half as many instructions.  x[] holds C consecutive columns.
template <int C>
__device__ __forceinline__ void chain_first_cols(const float (&s)[C], float k, float (&p)[C]) {
    if constexpr (C % 2 == 0) {
        const float2 kk = make_float2(k, k);
#pragma unroll
        for (int j = 0; j < C; j += 2) {
            const float2 r = __fmul2_rn(make_float2(s[j], s[j + 1]), kk);
            p[j] = r.x;
            p[j + 1] = r.y;
        }
    } else {
#pragma unroll
        for (int j = 0; j < C; ++j) p[j] = chain_first(s[j], k);
    }
}

template <int C>
__device__ __forceinline__ void chain_next_cols(const float (&s)[C], float k, float (&p)[C]) {
    if constexpr (C % 2 == 0) {
        const float2 kk = make_float2(k, k);
#pragma unroll
        for (int j = 0; j < C; j += 2) {
            const float2 r = __ffma2_rn(make_float2(s[j], s[j + 1]), kk, make_float2(p[j], p[j + 1]));
            p[j] = r.x;
            p[j + 1] = r.y;
        }
    } else {
#pragma unroll
        for (int j = 0; j < C; ++j) p[j] = chain_next(s[j], k, p[j]);
    }
}

// s[j] <- kh * u[j] + alpha * s[j] for C columns (gdr_advance on each).
template <int C>
__device__ __forceinline__ void advance_cols(float (&s)[C], float kh, const float (&u)[C], float alpha) {
    if constexpr (C % 2 == 0) {
        const float2 kk = make_float2(kh, kh), aa = make_float2(alpha, alpha);
#pragma unroll
        for (int j = 0; j < C; j += 2) {
            const float2 r =
                __ffma2_rn(kk, make_float2(u[j], u[j + 1]), __fmul2_rn(aa, make_float2(s[j], s[j + 1])));
            s[j] = r.x;
            s[j + 1] = r.y;
        }
    } else {
#pragma unroll
        for (int j = 0; j < C; ++j) s[j] = gdr_advance(s[j], kh, u[j], alpha);
    }
}

}  // namespace gdr

namespace gdr {

// ---- cp.async (LDGSTS): asynchronous global -> shared copies ---------------
// Completion is awaited with cp.async.wait_group, a hardware wait (no spin loop).
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
}
// The same with the destination given as a shared-window address.
__device__ __forceinline__ void cp_async16_s(unsigned saddr, const void *gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(saddr), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async4(void *smem, const void *gmem) {
    const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N> __device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

}  // namespace gdr
