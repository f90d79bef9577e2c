// Self-check kernels behind include/fa_diag.h: the two exp2 paths of the
// softmax evaluated side by side, and a pipeline wait that is made to run out.
#include <cuda_runtime.h>

#include "fa_internal.h"
#include "ptx.cuh"
#include "softmax_math.cuh"

namespace fa {
namespace diag {

__device__ DeviceError g_err;

__global__ void exp2_kernel(const float* __restrict__ x, float* __restrict__ y_emu, float* __restrict__ y_hw,
                            long long n) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    const float v = x[i];
    y_emu[i] = exp2_fma(v);
    y_hw[i] = ex2_mufu(v);
  }
}

// One barrier expecting one arrival that never comes; thread 0 waits on it
// with the production bounded wait.
__global__ void wait_kernel(unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait_bounded(smem_u32(&bar), 0, smem_u32(&abort_flag), &g_err, 1, limit_ns);
  __syncthreads();
}

}  // namespace diag

fa_status launch_diag_exp2(const float* x, float* y_emu, float* y_hw, long long n, cudaStream_t stream) {
  long long blocks = (n + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  diag::exp2_kernel<<<(unsigned)blocks, 256, 0, stream>>>(x, y_emu, y_hw, n);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status launch_diag_wait(unsigned long long limit_ns, cudaStream_t stream) {
  diag::wait_kernel<<<1, 32, 0, stream>>>(limit_ns);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status diag_take_device_error() {
  DeviceError e{0, 0};
  if (cudaMemcpyFromSymbol(&e, diag::g_err, sizeof(e)) != cudaSuccess) return FA_ERR_CUDA;
  if (e.status != 0) {
    const DeviceError z{0, 0};
    if (cudaMemcpyToSymbol(diag::g_err, &z, sizeof(z)) != cudaSuccess) return FA_ERR_CUDA;
  }
  return static_cast<fa_status>(e.status);
}

}  // namespace fa
