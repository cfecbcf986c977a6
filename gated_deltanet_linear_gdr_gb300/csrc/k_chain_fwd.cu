// Forward pass of the general kernel: instantiations and launcher.
#include "k_chain.cuh"

namespace gdr {

// Value head size V = K here; other ratios in k_chain_fwd_kv.cu.
template <typename ST, int K>
static cudaError_t fwd_t(const StepParams &p, long long max_len, cudaStream_t st) {
    return launch_chain_fwd_t<ST, K, K>(p, max_len, st);
}

cudaError_t launch_chain_fwd(const StepParams &p, int K, int V, bool bf16, long long max_len, cudaStream_t st) {
    if (V != K) return launch_chain_fwd_kv(p, K, V, bf16, max_len, st);
#define GDR_CASE(KK) \
    case KK: return bf16 ? fwd_t<uint16_t, KK>(p, max_len, st) : fwd_t<float, KK>(p, max_len, st);
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
