// Forward pass of the general kernel: instantiations and launcher.
#include "k_chain.cuh"

namespace gdr {

template <typename ST, int K, int V>
static cudaError_t fwd_t(const StepParams &p, long long max_len, cudaStream_t st) {
    const RingParams rp{};
    const SnapParams sp{};
    // chunk tokens: rows bounded at 8 or 16 tokens get chunks of that size (a
    // smaller stage, more L1); longer or unbounded rows take kChainLongTC
    // (fewer chunk barriers and normalisation passes per token)
    if (p.bpv) return launch_chain_k<ST, K, V, Mode::Fwd, true, 8>(p, rp, sp, max_len, st);
    if (max_len >= 1 && max_len <= 8) return launch_chain_k<ST, K, V, Mode::Fwd, false, 8>(p, rp, sp, max_len, st);
    if (max_len >= 1 && max_len <= 16)
        return launch_chain_k<ST, K, V, Mode::Fwd, false, 16>(p, rp, sp, max_len, st);
    return launch_chain_k<ST, K, V, Mode::Fwd, false, kChainLongTC>(p, rp, sp, max_len, st);
}

cudaError_t launch_chain_fwd(const StepParams &p, int K, int V, bool bf16, long long max_len, cudaStream_t st) {
#define GDR_CASE(KK)                                                                                     \
    case KK:                                                                                             \
        if (V == KK) return bf16 ? fwd_t<uint16_t, KK, KK>(p, max_len, st) : fwd_t<float, KK, KK>(p, max_len, st); \
        if (V == 2 * KK)                                                                                 \
            return bf16 ? fwd_t<uint16_t, KK, 2 * KK>(p, max_len, st) : fwd_t<float, KK, 2 * KK>(p, max_len, st); \
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
