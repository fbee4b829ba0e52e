// selftest.cu -- exercises the kernels' bounded-wait failure path without any
// fault: one warp waits on an mbarrier that nothing ever arrives on, with the
// same bounded wait the GEMM kernels use, gives up after the requested time,
// records GEMM_ERR_TIMEOUT in the device error word and returns normally.
#include <cstdint>

#include <cuda_runtime.h>

#include "../../include/dense_gemm_row.h"
#include "launch.h"
#include "ptx.cuh"

namespace dgr {
namespace {

__global__ void wait_timeout_kernel(uint64_t limit_ns, uint32_t *err_word) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);  // one arrival expected; none will come
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncwarp();
  if (threadIdx.x == 0)
    mbar_wait_bounded(smem_u32(&bar), 0, &abort_flag, err_word, kWaitTest, limit_ns);
  __syncwarp();
}

}  // namespace
}  // namespace dgr

extern "C" gemm_status_t gemm_selftest_wait_timeout(uint32_t limit_us, cudaStream_t stream) {
  if (limit_us == 0 || limit_us > 1000000u) return GEMM_ERR_INVALID_VALUE;
  const dgr::DeviceInfo *dev = nullptr;
  int st = dgr::abi_current_device(&dev);
  if (st != GEMM_OK) return static_cast<gemm_status_t>(st);
  dgr::wait_timeout_kernel<<<1, 32, 0, stream>>>(uint64_t(limit_us) * 1000u, dev->err_word);
  return static_cast<gemm_status_t>(dgr::abi_from_cuda(cudaGetLastError()));
}
