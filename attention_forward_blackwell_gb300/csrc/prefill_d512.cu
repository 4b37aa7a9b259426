// Prefill kernels for head_dim = 512 (two CTAs per Q tile, each computing
// one 256-column half of O).
#include "prefill.cuh"

namespace fa {
cudaError_t launch_prefill_d512(const PrefillLaunch& p, cudaStream_t s) {
    return launch_prefill_impl<512>(p, s);
}
}  // namespace fa
