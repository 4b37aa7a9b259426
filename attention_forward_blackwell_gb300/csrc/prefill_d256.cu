// Prefill kernels for head_dim = 256 (non-causal and causal instantiations).
#include "prefill.cuh"

namespace fa {
cudaError_t launch_prefill_d256(const PrefillLaunch& p, cudaStream_t s) {
    return launch_prefill_impl<256>(p, s);
}
}  // namespace fa
