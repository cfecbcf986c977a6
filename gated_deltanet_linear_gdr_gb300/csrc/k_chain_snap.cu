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

cudaError_t launch_chain_snap(const StepParams &p, int K, int V, bool bf16, const SnapParams &sp, long long max_len,
                              cudaStream_t st) {
#define GDR_CASE(KK)                                                                                        \
    case KK:                                                                                                \
        if (V == KK) return bf16 ? snap_t<uint16_t, KK, KK>(p, sp, max_len, st) : snap_t<float, KK, KK>(p, sp, max_len, st); \
        if (V == 2 * KK)                                                                                    \
            return bf16 ? snap_t<uint16_t, KK, 2 * KK>(p, sp, max_len, st) : snap_t<float, KK, 2 * KK>(p, sp, max_len, st); \
        return cudaErrorInvalidValue;
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
