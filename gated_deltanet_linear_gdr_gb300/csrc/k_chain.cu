// The general kernel's entry: dispatch by pass to the per-pass launchers
// (k_chain_fwd.cu, k_chain_verify.cu, k_chain_snap.cu).
#include "k_chain.cuh"

namespace gdr {

cudaError_t launch_chain(const StepParams &p, int K, int V, bool bf16, Mode mode, const RingParams &rp,
                         const SnapParams &sp, long long max_row_len, cudaStream_t s) {
    switch (mode) {
        case Mode::Fwd: return launch_chain_fwd(p, K, V, bf16, max_row_len, s);
        case Mode::Verify: return V == K ? launch_chain_verify(p, K, bf16, rp, max_row_len, s) : cudaErrorInvalidValue;
        case Mode::Snap: return launch_chain_snap(p, K, V, bf16, sp, max_row_len, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace gdr
