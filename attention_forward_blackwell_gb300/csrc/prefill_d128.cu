// Prefill kernels for head_dim = 128 (non-causal and causal instantiations).
#include "prefill.cuh"

namespace fa {
cudaError_t launch_prefill_d128(const PrefillLaunch& p, cudaStream_t s) {
    return launch_prefill_impl<128>(p, s);
}
}  // namespace fa
