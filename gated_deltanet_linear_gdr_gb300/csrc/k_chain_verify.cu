// Verify pass of the general kernel (V = K, head-wise beta): instantiations and launcher.
#include "k_chain.cuh"

namespace gdr {

template <typename ST, int K>
static cudaError_t verify_t(const StepParams &p, const RingParams &rp, long long max_len, cudaStream_t st) {
    if (p.bpv) return cudaErrorInvalidValue;
    return launch_chain_k<ST, K, K, Mode::Verify, false, 16>(p, rp, SnapParams{}, max_len, st);
}

cudaError_t launch_chain_verify(const StepParams &p, int K, bool bf16, const RingParams &rp, long long max_len,
                                cudaStream_t st) {
#define GDR_CASE(KK) \
    case KK: return bf16 ? verify_t<uint16_t, KK>(p, rp, max_len, st) : verify_t<float, KK>(p, rp, max_len, st);
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
