// Backward pass (kernels not yet built: fa_bwd reports FA_ERR_UNSUPPORTED).
#include <cuda_runtime.h>

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace bwd {
__device__ DeviceError g_err;
}

fa_status launch_bwd(const BwdLaunch&, cudaStream_t) { return FA_ERR_UNSUPPORTED; }

fa_status bwd_take_device_error() {
  DeviceError e{0, 0};
  if (cudaMemcpyFromSymbol(&e, bwd::g_err, sizeof(e)) != cudaSuccess) return FA_ERR_CUDA;
  if (e.status != 0) {
    const DeviceError z{0, 0};
    if (cudaMemcpyToSymbol(bwd::g_err, &z, sizeof(z)) != cudaSuccess) return FA_ERR_CUDA;
  }
  return static_cast<fa_status>(e.status);
}

}  // namespace fa
