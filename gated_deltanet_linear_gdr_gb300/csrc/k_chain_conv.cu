// The forward pass with the Pass-1 convolution ("gated_delta_recurrence_fwd_gpu",
// Args: qkv_conv_output is the "Conv1d output from Pass 1") fused into the
// general kernel's operand staging, and the conv-state update that follows it.
#include "k_chain.cuh"

namespace gdr {

// Conv-state update: for every live row b and channel c, the new state is the
// last width-1 entries of (old state, the row's raw inputs).  One thread per
// (row, channel) reads every value it needs before writing, so the update is
// in place.  Rows the forward kernel skipped (bad offsets or slot, longer
// than the caller's bound) and empty rows keep their state.  Runs after the
// forward kernel on the same stream, which has read the old state.
__global__ void __launch_bounds__(256) k_conv_state(const StepParams p, const ConvParams cv, long long max_len) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (long long)p.batch * cv.channels) return;
    const int b = (int)(i / cv.channels), c = (int)(i - (long long)b * cv.channels);
    const int slot = p.slot_idx[b];
    if (slot < 0 || slot >= p.max_slots) return;
    const int t0 = p.offsets[b], t1 = p.offsets[b + 1];
    if (t0 < 0 || t1 < t0 || t1 > p.T) return;
    const int L = t1 - t0;
    if (L == 0 || (max_len > 0 && L > max_len)) return;
    const int w1 = cv.width - 1;  // 1 .. 3
    float *st = cv.state + (long long)slot * cv.cs_slot + (long long)c * cv.cs_chan;
    float nv[3];
#pragma unroll
    for (int j = 0; j < 3; ++j) {
        if (j < w1) {
            const int idx = L + j;  // into (old state, inputs)
            nv[j] = idx < w1 ? st[idx * cv.cs_tap] : p.qkv[(long long)(t0 + idx - w1) * p.qkv_ss + (long long)c * p.qkv_cs];
        }
    }
#pragma unroll
    for (int j = 0; j < 3; ++j)
        if (j < w1) st[j * cv.cs_tap] = nv[j];
}

template <typename ST, int K>
static cudaError_t conv_t(const StepParams &p, const ConvParams &cv, long long max_len, cudaStream_t st) {
    const RingParams rp{};
    const SnapParams sp{};
    // the forward pass's chunk sizes: 8 tokens for rows bounded at 8, else kChainLongTC
    if (max_len >= 1 && max_len <= 8)
        return launch_chain_k<ST, K, K, Mode::Fwd, false, 8, true>(p, rp, sp, max_len, st, cv);
    return launch_chain_k<ST, K, K, Mode::Fwd, false, kChainLongTC, true>(p, rp, sp, max_len, st, cv);
}

cudaError_t launch_chain_conv(const StepParams &p, const ConvParams &cv, int K, bool bf16, long long max_row_len,
                              cudaStream_t s) {
    cudaError_t e = cudaErrorInvalidValue;
#define GDR_CASE(KK) \
    case KK: e = bf16 ? conv_t<uint16_t, KK>(p, cv, max_row_len, s) : conv_t<float, KK>(p, cv, max_row_len, s); break;
    switch (K) {
        GDR_CASE(16)
        GDR_CASE(32)
        GDR_CASE(64)
        GDR_CASE(128)
    }
#undef GDR_CASE
    if (e != cudaSuccess) return e;
    if (cv.width > 1 && p.batch > 0) {
        const long long n = (long long)p.batch * cv.channels;
        k_conv_state<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(p, cv, max_row_len);
    }
    return cudaGetLastError();
}

}  // namespace gdr
