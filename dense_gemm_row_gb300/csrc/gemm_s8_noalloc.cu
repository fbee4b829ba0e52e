// gemm_s8_noalloc.cu -- gemm_s8 for callers that must not allocate device memory.
//
// gemm_s8 takes the scratch for its fp16-widened copies of A and B from a
// library-owned stream-ordered pool. Callers whose device memory is reserved
// in full by another allocator, latency-critical loops that must stay out of
// the driver's allocation path, and deployments that forbid allocation after
// start-up cannot accept that. This file gives them gemm_s8_noalloc: the same
// computation on a fixed scratch array that lives in the library's own device
// memory, so no call allocates or frees anything.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/dense_gemm_row.h"
#include "launch.h"

namespace dgr {
namespace {

// 64 MiB: enough for the widened operands of M = N = K = 4096.
constexpr size_t kScratchBytes = size_t(64) << 20;
// After the operands: 4 KiB of flags for the kernel's split-k tail (zeroed by
// each call before use).
constexpr size_t kFlagBytes = 4096;

// The scratch array. Every GPU that loads this module keeps it until the
// process exits. All calls on a device share it.
static __device__ __align__(256) unsigned char g_s8_scratch[kScratchBytes + kFlagBytes];

constexpr int kMaxDevices = 64;

struct ScratchSlot {
  std::once_flag once;
  cudaError_t err = cudaSuccess;
  void *ptr = nullptr;
};
ScratchSlot g_scratch[kMaxDevices];

// Device address of the array on device `dev`, which must be current. The
// host-side name of a __device__ array is only a stand-in, so the address is
// looked up once per device and checked.
cudaError_t scratch_address(int dev, void **out) {
  ScratchSlot &slot = g_scratch[dev];
  std::call_once(slot.once, [&] {
    void *p = nullptr;
    slot.err = cudaGetSymbolAddress(&p, g_s8_scratch);
    if (slot.err == cudaSuccess && p == nullptr) slot.err = cudaErrorInvalidSymbol;
    slot.ptr = p;
  });
  *out = slot.ptr;
  return slot.err;
}

}  // namespace
}  // namespace dgr

extern "C" gemm_status_t gemm_s8_noalloc(int64_t M, int64_t N, int64_t K, int32_t alpha,
                                         const int8_t *A, int64_t lda, const int8_t *B,
                                         int64_t ldb, int32_t beta, int32_t *C, int64_t ldc,
                                         cudaStream_t stream) {
  bool skip = false;
  int st = dgr::abi_check_args(M, N, K, A, lda, B, ldb, C, ldc, &skip);
  if (st != GEMM_OK || skip) return static_cast<gemm_status_t>(st);
  if (K > 0 && dgr::s8_scratch_bytes(int(M), int(N), int(K)) > dgr::kScratchBytes)
    return GEMM_ERR_TOO_LARGE;
  const dgr::DeviceInfo *dev = nullptr;
  if ((st = dgr::abi_current_device(&dev)) != GEMM_OK) return static_cast<gemm_status_t>(st);
  if (K == 0)  // C = beta*C needs no scratch
    return static_cast<gemm_status_t>(
        dgr::abi_from_cuda(dgr::launch_scale_s32(int(M), int(N), beta, C, ldc, stream)));
  void *scratch = nullptr;
  if (dgr::scratch_address(dev->device, &scratch) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_DEVICE;
  }
  uint32_t *flags =
      reinterpret_cast<uint32_t *>(static_cast<unsigned char *>(scratch) + dgr::kScratchBytes);
  return static_cast<gemm_status_t>(dgr::abi_from_cuda(
      dgr::launch_gemm_s8_scratch(*dev, int(M), int(N), int(K), alpha, A, lda, B, ldb, beta, C,
                                  ldc, scratch, flags, dgr::kFlagBytes / 4, stream)));
}
