// Diagnostic kernels: how fast one SM sub-partition runs packed f32x2
// arithmetic of a given register-operand pattern, every operand already in
// registers (no memory traffic, no shuffles).  They bound what the recurrence
// kernels can reach on the FP32 pipe with their fixed operation order:
//
//   pattern 0: the per-element sequence of the recurrence sweep
//              (gdr_state.cuh, LaneState::advance_partials) on a lane of
//              64 rows x 2 columns: t = alpha*x; x = k^ u + t; a += x k';
//              b += x q' (8-row chains, 4 group pairs, 2 columns), then a
//              short dependent tail that turns the partials into the next
//              iteration's u;
//   pattern 1: independent packed FMA chains whose multiplier and addend are
//              the same registers in every instruction (reusable operands);
//   pattern 2: independent packed FMA chains with three distinct operand
//              register pairs per instruction.
#include "gdr_internal.h"

namespace gdr {

constexpr int kProbeNP = 4, kProbeC = 2, kProbeChains = 8;

__global__ void k_probe_sweep(float *sink, int iters, float s) {
    constexpr int NP = kProbeNP, C = kProbeC;
    float2 x[NP][8][C], kp[NP][8], kn[NP][8], qn[NP][8];
#pragma unroll
    for (int g = 0; g < NP; ++g)
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            kp[g][i] = make_float2(1e-3f * (i + 1), 2e-3f * (g + 1));
            kn[g][i] = make_float2(s * 1e-3f * i, 1e-3f);
            qn[g][i] = make_float2(2e-3f, s * 1e-3f * (i + g));
#pragma unroll
            for (int c = 0; c < C; ++c) x[g][i][c] = make_float2(threadIdx.x * 1e-6f + i, c + g * 1e-2f);
        }
    float2 uu[C];
#pragma unroll
    for (int c = 0; c < C; ++c) uu[c] = make_float2(1e-4f * c, 1e-4f * c);
    const float2 aa = make_float2(s, s);
    for (int it = 0; it < iters; ++it) {
        float2 pa[NP][C], pb[NP][C];
#pragma unroll
        for (int g = 0; g < NP; ++g)
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int c = 0; c < C; ++c) {
                    x[g][i][c] = __ffma2_rn(kp[g][i], uu[c], __fmul2_rn(aa, x[g][i][c]));
                    if (i == 0) {
                        pa[g][c] = __fmul2_rn(x[g][0][c], kn[g][0]);
                        pb[g][c] = __fmul2_rn(x[g][0][c], qn[g][0]);
                    } else {
                        pa[g][c] = __ffma2_rn(x[g][i][c], kn[g][i], pa[g][c]);
                        pb[g][c] = __ffma2_rn(x[g][i][c], qn[g][i], pb[g][c]);
                    }
                }
#pragma unroll
        for (int c = 0; c < C; ++c) {
            float a = 0.f, b = 0.f;
#pragma unroll
            for (int g = 0; g < NP; ++g) {
                a += pa[g][c].x + pa[g][c].y;
                b += pb[g][c].x + pb[g][c].y;
            }
            const float u = 1e-6f * (a - b);
            uu[c] = make_float2(u, u);
        }
    }
    float t = 0.f;
#pragma unroll
    for (int g = 0; g < NP; ++g)
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int c = 0; c < C; ++c) t += x[g][i][c].x + x[g][i][c].y;
    sink[blockIdx.x * blockDim.x + threadIdx.x] = t;
}

template <bool SHARED>
__global__ void k_probe_chains(float *sink, int iters, float s) {
    constexpr int CH = kProbeChains;
    float2 acc[CH], a[CH], b[CH];
#pragma unroll
    for (int c = 0; c < CH; ++c) {
        acc[c] = make_float2(threadIdx.x * 1e-3f + c, c * 0.5f);
        a[c] = make_float2(s + c * 1e-4f, s - c * 1e-4f);
        b[c] = make_float2(1e-3f * (c + 1), -1e-3f * (c + 1));
    }
    const float2 aa = make_float2(s, s), bb = make_float2(1e-3f, 2e-3f);
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int c = 0; c < CH; ++c) acc[c] = SHARED ? __ffma2_rn(acc[c], aa, bb) : __ffma2_rn(a[c], b[c], acc[c]);
    }
    float t = 0.f;
#pragma unroll
    for (int c = 0; c < CH; ++c) t += acc[c].x + acc[c].y + a[c].x + b[c].y;
    sink[blockIdx.x * blockDim.x + threadIdx.x] = t;
}

cudaError_t launch_probe_fma(int pattern, int warps, int iters, float *sink, cudaStream_t st, int *blocks_out) {
    int dev = 0, sms = 0, regs_sm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev);
    if (e != cudaSuccess) return e;
    const void *fn = pattern == 0   ? reinterpret_cast<const void *>(k_probe_sweep)
                     : pattern == 1 ? reinterpret_cast<const void *>(k_probe_chains<true>)
                                    : reinterpret_cast<const void *>(k_probe_chains<false>);
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, fn);
    if (e != cudaSuccess) return e;
    const int threads = 128 * warps;
    // one CTA per SM: it must fit the SM's registers
    if (threads > fa.maxThreadsPerBlock || (long long)fa.numRegs * threads > regs_sm) return cudaErrorInvalidConfiguration;
    *blocks_out = sms;
    if (pattern == 0)
        k_probe_sweep<<<sms, threads, 0, st>>>(sink, iters, 0.999f);
    else if (pattern == 1)
        k_probe_chains<true><<<sms, threads, 0, st>>>(sink, iters, 0.999f);
    else
        k_probe_chains<false><<<sms, threads, 0, st>>>(sink, iters, 0.999f);
    return cudaGetLastError();
}

}  // namespace gdr
