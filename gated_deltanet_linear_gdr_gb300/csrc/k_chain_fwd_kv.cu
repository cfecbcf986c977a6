// Forward pass of the general kernel with a value head size other than the
// key head size ("core.ssm.ops.gdp.fused_recurrent" sizes K and V
// separately): V = 2K, and V = K/2 for K >= 32.  Instantiations and launcher.
#include "k_chain.cuh"

namespace gdr {

template <typename ST, int K>
static cudaError_t fwd_kv_t(const StepParams &p, int V, long long max_len, cudaStream_t st) {
    if (V == 2 * K) return launch_chain_fwd_t<ST, K, 2 * K>(p, max_len, st);
    if constexpr (K >= 32) {
        if (2 * V == K) return launch_chain_fwd_t<ST, K, K / 2>(p, max_len, st);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_chain_fwd_kv(const StepParams &p, int K, int V, bool bf16, long long max_len, cudaStream_t st) {
#define GDR_CASE(KK) \
    case KK: return bf16 ? fwd_kv_t<uint16_t, KK>(p, V, max_len, st) : fwd_kv_t<float, KK>(p, V, max_len, st);
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
