// Snapshot pass of the general kernel: instantiations and launcher.
#include "k_chain.cuh"

namespace gdr {

template <typename ST, int K, int V>
static cudaError_t snap_t(const StepParams &p, const SnapParams &sp, long long max_len, cudaStream_t st) {
    const RingParams rp{};
    if (p.bpv) return launch_chain_k<ST, K, V, Mode::Snap, true, 8>(p, rp, sp, max_len, st);
    if (max_len >= 1 && max_len <= 8) return launch_chain_k<ST, K, V, Mode::Snap, false, 8>(p, rp, sp, max_len, st);
    return launch_chain_k<ST, K, V, Mode::Snap, false, 16>(p, rp, sp, max_len, st);
}

// V = K, V = 2K, and V = K/2 for K >= 32.
template <typename ST, int K>
static cudaError_t snap_v(const StepParams &p, int V, const SnapParams &sp, long long max_len, cudaStream_t st) {
    if (V == K) return snap_t<ST, K, K>(p, sp, max_len, st);
    if (V == 2 * K) return snap_t<ST, K, 2 * K>(p, sp, max_len, st);
    if constexpr (K >= 32) {
        if (2 * V == K) return snap_t<ST, K, K / 2>(p, sp, max_len, st);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_chain_snap(const StepParams &p, int K, int V, bool bf16, const SnapParams &sp, long long max_len,
                              cudaStream_t st) {
#define GDR_CASE(KK) \
    case KK: return bf16 ? snap_v<uint16_t, KK>(p, V, sp, max_len, st) : snap_v<float, KK>(p, V, sp, max_len, st);
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
