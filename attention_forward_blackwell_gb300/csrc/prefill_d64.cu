// Prefill kernels for head_dim = 64 (non-causal and causal instantiations).
#include "prefill.cuh"

namespace fa {
cudaError_t launch_prefill_d64(const PrefillLaunch& p, cudaStream_t s) {
    return launch_prefill_impl<64>(p, s);
}
}  // namespace fa
