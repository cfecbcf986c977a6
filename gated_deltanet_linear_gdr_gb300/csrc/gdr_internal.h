// Internal launch parameters shared by the host API (api.cu) and the kernels.
// Host code validates gdr_step_args and lowers it into these plain structs,
// which travel to the kernels by value.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "../../include/gdr.h"

namespace gdr {

// One recurrence call, after validation.  Strides in elements.
struct StepParams {
    int batch, nv, nk, r;  // r = nv / nk (GQA ratio)
    int decay_is_log, l2norm;
    long long T;
    const float *qkv;
    long long qkv_ss, qkv_cs;
    const float *decay, *beta;
    long long tok_ss, tok_hs;
    float scale, eps;
    float *out;
    long long out_ss, out_vs;
    void *state;
    long long st_slot, st_head, st_k;  // value-dim stride is 1
    long long max_slots;
    const int *slot_idx, *offsets;
    // general kernel: rows read state_in (zeros if null) and commit to state_out
    // (nothing if null); both equal `state` except in the dense mode, where
    // row b uses slot b and every row is live (dense != 0)
    const void *state_in;
    void *state_out;
    int dense;
    int bpv;      // beta per value element: element (t, h, j) at t*beta_ss + h*beta_hs + j*beta_vs
    long long beta_ss, beta_hs, beta_vs;
    int beta_vec; // per-element beta rows may be read with 16-byte vector loads
    int qkv_vec;  // Q/K/V rows may be read with 16-byte vector loads
    int out_vec;  // output rows may be written with 16-byte vector stores
    unsigned *status;
};

// Verify ring ("gated_delta_recurrence_verify_ring_gpu", ring / ring_slot_idx /
// ring_dtype): float32 records, or bfloat16 (bf16 != 0).
struct RingParams {
    void *ring;        // 16-byte aligned
    int bf16;
    long long rows;
    int len;
    long long stride;  // elements per record
    const int *ring_slot;
    int alpha_off;     // = K
    int u_off;         // = K + 8*ceil(r/8)
};

// Snapshots ("core.ssm.ops.gdp.fused_recurrent", intermediate_states).
struct SnapParams {
    void *inter;
    long long s_slot, s_tok, s_head;
    int n_inter;
    int spt;
};

struct FoldParams {
    int batch, nv, nk, r;
    void *state;
    long long st_slot, st_head, st_k;
    long long max_slots;
    const int *slot_idx;
    const void *ring;
    int ring_bf16;
    long long ring_rows;
    int ring_len;
    long long stride;
    const int *ring_slot;
    const int *counts;
    int alpha_off, u_off;
    unsigned *status;
};

struct RollbackParams {
    int batch, nv;
    void *state;
    long long st_slot, st_head, st_k;
    long long max_slots;
    const int *slot_idx;
    const void *inter;
    long long s_slot, s_tok, s_head;
    int n_inter;
    const int *accepted;
    unsigned *status;
};

// Pass-1 convolution of the forward pass (gdr_fwd_conv): causal depthwise over
// the conv_dim channels of the raw input staged from StepParams::qkv.
struct ConvParams {
    int width, silu;
    const float *w;
    long long w_cs, w_ts;
    const float *bias;  // or null
    float *state;       // [max_slots, conv_dim, width-1] float32 (null when width == 1)
    long long cs_slot, cs_chan, cs_tap;
    int channels;       // conv_dim
};

enum class Mode : int { Fwd = 0, Verify = 1, Snap = 2 };

// Unsigned division by a divisor fixed at launch, as a multiply-high, an add
// and a shift (Granlund and Montgomery, "Division by Invariant Integers using
// Multiplication", 1994): with l = ceil(log2 d) and m = floor(2^32 (2^l - d) / d) + 1,
// n / d = (mulhi(n, m) + n) >> l for every 32-bit n (the add is done in 64 bits).
struct FastDiv {
    unsigned d, m, l;
    FastDiv() = default;
    __host__ explicit FastDiv(unsigned dd) : d(dd ? dd : 1u), m(0), l(0) {
        while ((1ull << l) < d) ++l;
        m = (unsigned)(((1ull << 32) * ((1ull << l) - d)) / d + 1);
    }
#ifdef __CUDACC__
    __device__ __forceinline__ unsigned div(unsigned n) const {
        return (unsigned)(((unsigned long long)__umulhi(n, m) + n) >> l);
    }
#endif
};

// Per-device facts a launcher looks up once: the SM count and what its init
// callback fills in (resident CTAs per SM; the callback also opts the kernel
// into its dynamic shared memory).  The first caller on a device fills them in
// under the mutex and publishes them with a release store; later callers, on
// any thread, read `ready` with acquire and so see complete values.  A failed
// init publishes nothing and is retried by the next call.
constexpr int kMaxDevices = 64;
struct LaunchInfo {
    int sms, occ;
};
struct LaunchCache {
    std::atomic<int> ready[kMaxDevices];  // zero-initialised: instances are static
    LaunchInfo info[kMaxDevices];
    std::mutex mu;
};

template <typename Init>
inline cudaError_t launch_info(LaunchCache &c, LaunchInfo *out, Init &&init) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (!c.ready[dev].load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lk(c.mu);
        if (!c.ready[dev].load(std::memory_order_relaxed)) {
            LaunchInfo li{0, 1};
            e = cudaDeviceGetAttribute(&li.sms, cudaDevAttrMultiProcessorCount, dev);
            if (e == cudaSuccess) e = init(li);
            if (e != cudaSuccess) return e;
            if (li.sms < 1) li.sms = 1;
            if (li.occ < 1) li.occ = 1;
            c.info[dev] = li;
            c.ready[dev].store(1, std::memory_order_release);
        }
    }
    *out = c.info[dev];
    return cudaSuccess;
}

// Launchers (defined next to their kernels).  Return cudaGetLastError().
cudaError_t launch_decode(const StepParams &p, int K, bool bf16, cudaStream_t s);
cudaError_t launch_chain(const StepParams &p, int K, int V, bool bf16, Mode mode, const RingParams &rp,
                         const SnapParams &sp, long long max_row_len, cudaStream_t s);
// Pipelined short-row kernel; sets *used = false (launching nothing) when the
// layout does not allow it, so the caller falls back to launch_chain.
cudaError_t launch_short(const StepParams &p, int K, bool bf16, Mode mode, const RingParams &rp,
                         const SnapParams &sp, long long max_row_len, cudaStream_t s, bool *used);
cudaError_t launch_fold(const FoldParams &p, int K, bool bf16, cudaStream_t s);
cudaError_t launch_rollback(const RollbackParams &p, int K, int V, bool bf16, cudaStream_t s);
// The forward pass with the Pass-1 convolution fused into operand staging,
// then the conv-state update (two launches on s).
cudaError_t launch_chain_conv(const StepParams &p, const ConvParams &cp, int K, bool bf16, long long max_row_len,
                              cudaStream_t s);

// Diagnostic packed-FMA probes (k_probe.cu): one CTA of 128 * warps threads per
// SM; *blocks_out receives the CTA count.
cudaError_t launch_probe_fma(int pattern, int warps, int iters, float *sink, cudaStream_t st, int *blocks_out);

}  // namespace gdr
