// Backward main kernel (key/value stationary), sm_103a.
#include "fa_device.cuh"
#include "fa_kernels.h"

namespace fa {

cudaError_t launch_bwd_main(const BwdParams& p, int d, cudaStream_t stream) {
  (void)p; (void)d; (void)stream;
  return cudaErrorNotSupported;
}

}  // namespace fa
