// Prefill kernels for head_dim = 96 (non-causal and causal instantiations).
#include "prefill.cuh"

namespace fa {
cudaError_t launch_prefill_d96(const PrefillLaunch& p, cudaStream_t s) {
    return launch_prefill_impl<96>(p, s);
}
}  // namespace fa
