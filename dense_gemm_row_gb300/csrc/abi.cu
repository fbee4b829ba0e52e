// abi.cu -- the C entry points of libdense_gemm_row.so (include/dense_gemm_row.h).
//
// Host-side argument checks, per-device set-up, the K == 0 path (C = beta*C)
// and dispatch to the kernels. Nothing here allocates or frees user memory,
// prints, or aborts.
#include <cstdint>
#include <map>
#include <mutex>
#include <type_traits>
#include <utility>

#include <cuda_runtime.h>

#include "../../include/dense_gemm_row.h"
#include "launch.h"

namespace dgr {
namespace {

constexpr int kMaxDevices = 64;
constexpr int kVersion = 100;  // 0.1.0

// One error word per device (see gemm_check_device_error).
__device__ uint32_t g_error_word;

struct DeviceSlot {
  std::once_flag once;
  cudaError_t init_error = cudaSuccess;
  DeviceInfo info;
};
DeviceSlot g_devices[kMaxDevices];

cudaError_t init_device(int dev, DeviceInfo &info) {
  cudaDeviceProp prop;
  cudaError_t e = cudaGetDeviceProperties(&prop, dev);
  if (e != cudaSuccess) return e;
  if (prop.major != 10 || prop.minor != 3) return cudaErrorNoKernelImageForDevice;
  info.device = dev;
  info.sm_count = prop.multiProcessorCount;
  void *p = nullptr;
  e = cudaGetSymbolAddress(&p, g_error_word);
  if (e != cudaSuccess) return e;
  info.err_word = static_cast<uint32_t *>(p);
  return cudaSuccess;
}

// The current device's info, set up once per device.
gemm_status_t current_device(const DeviceInfo **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return GEMM_ERR_DEVICE;
  }
  DeviceSlot &slot = g_devices[dev];
  std::call_once(slot.once, [&] { slot.init_error = init_device(dev, slot.info); });
  if (slot.init_error != cudaSuccess) return GEMM_ERR_DEVICE;
  *out = &slot.info;
  return GEMM_OK;
}

constexpr int64_t kMaxDim = 0x7fffffffLL;

// Shared argument checks. Returns GEMM_OK when the call should proceed; sets
// *nothing_to_do when the output is empty.
gemm_status_t check_args(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda,
                         const void *B, int64_t ldb, const void *C, int64_t ldc,
                         bool *nothing_to_do) {
  *nothing_to_do = false;
  if (M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_VALUE;
  if (M > kMaxDim || N > kMaxDim || K > kMaxDim) return GEMM_ERR_INVALID_VALUE;
  if (M == 0 || N == 0) {
    *nothing_to_do = true;
    return GEMM_OK;
  }
  if (ldc < N || C == nullptr) return GEMM_ERR_INVALID_VALUE;
  if (K > 0) {
    if (lda < K || A == nullptr) return GEMM_ERR_INVALID_VALUE;
    if (ldb < N || B == nullptr) return GEMM_ERR_INVALID_VALUE;
  }
  return GEMM_OK;
}

gemm_status_t from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return GEMM_OK;
  cudaGetLastError();  // clear a sticky launch error so later calls are not blamed
  return GEMM_ERR_LAUNCH;
}

// ------------------------------------------------------------ K == 0 kernels

template <typename T>
__global__ void scale_kernel(int M, int N, T beta, T *C, int64_t ldc) {
  const int64_t total = static_cast<int64_t>(M) * N;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = i / N, c = i - r * N;
    T *p = C + r * ldc + c;
    if (beta == T(0)) {
      *p = T(0);
    } else if constexpr (std::is_integral<T>::value) {  // int32 wrap-around
      *p = static_cast<T>(static_cast<uint32_t>(beta) * static_cast<uint32_t>(*p));
    } else {
      *p = beta * *p;
    }
  }
}

template <typename T>
cudaError_t launch_scale(int M, int N, T beta, T *C, int64_t ldc, cudaStream_t stream) {
  const int64_t total = static_cast<int64_t>(M) * N;
  int64_t blocks = (total + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  scale_kernel<T><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(M, N, beta, C, ldc);
  return cudaGetLastError();
}

}  // namespace

cudaError_t set_max_dynamic_smem(const void *kernel, int bytes, int device) {
  static std::mutex mu;
  static std::map<std::pair<const void *, int>, int> done;  // -> bytes already set
  std::lock_guard<std::mutex> lock(mu);
  auto key = std::make_pair(kernel, device);
  auto it = done.find(key);
  if (it != done.end() && it->second >= bytes) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done[key] = bytes;
  return e;
}

int abi_check_args(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda, const void *B,
                   int64_t ldb, const void *C, int64_t ldc, bool *nothing_to_do) {
  return check_args(M, N, K, A, lda, B, ldb, C, ldc, nothing_to_do);
}

int abi_current_device(const DeviceInfo **out) { return current_device(out); }

int abi_from_cuda(cudaError_t e) { return from_cuda(e); }

cudaError_t launch_scale_f32(int M, int N, float beta, float *C, int64_t ldc,
                             cudaStream_t stream) {
  return launch_scale<float>(M, N, beta, C, ldc, stream);
}

cudaError_t launch_scale_s32(int M, int N, int32_t beta, int32_t *C, int64_t ldc,
                             cudaStream_t stream) {
  return launch_scale<int32_t>(M, N, beta, C, ldc, stream);
}

}  // namespace dgr

using dgr::check_args;
using dgr::current_device;
using dgr::DeviceInfo;
using dgr::from_cuda;

extern "C" {

gemm_status_t gemm_f32(int64_t M, int64_t N, int64_t K, float alpha, const float *A, int64_t lda,
                       const float *B, int64_t ldb, float beta, float *C, int64_t ldc,
                       cudaStream_t stream) {
  bool skip = false;
  gemm_status_t st = check_args(M, N, K, A, lda, B, ldb, C, ldc, &skip);
  if (st != GEMM_OK || skip) return st;
  const DeviceInfo *dev = nullptr;
  if ((st = current_device(&dev)) != GEMM_OK) return st;
  if (K == 0) return from_cuda(dgr::launch_scale_f32(int(M), int(N), beta, C, ldc, stream));
  if (dgr::small_m_supported(int(M), A, lda, B, ldb, 4))  // few rows: stream B once
    return from_cuda(dgr::launch_small_m_f32(*dev, int(M), int(N), int(K), alpha, A, lda, B, ldb,
                                             beta, C, ldc, stream));
  return from_cuda(dgr::launch_sgemm_simt(*dev, int(M), int(N), int(K), alpha, A, lda, B, ldb,
                                          beta, C, ldc, stream));
}

static gemm_status_t gemm_half(bool is_bf16, int64_t M, int64_t N, int64_t K, float alpha,
                               const uint16_t *A, int64_t lda, const uint16_t *B, int64_t ldb,
                               float beta, float *C, int64_t ldc, cudaStream_t stream) {
  bool skip = false;
  gemm_status_t st = check_args(M, N, K, A, lda, B, ldb, C, ldc, &skip);
  if (st != GEMM_OK || skip) return st;
  if (K > 0) {
    // TMA: 16-byte aligned bases and row strides.
    if ((reinterpret_cast<uintptr_t>(A) & 15u) || (reinterpret_cast<uintptr_t>(B) & 15u) ||
        (lda % 8) || (ldb % 8))
      return GEMM_ERR_UNSUPPORTED_LAYOUT;
  }
  const DeviceInfo *dev = nullptr;
  if ((st = current_device(&dev)) != GEMM_OK) return st;
  if (K == 0) return from_cuda(dgr::launch_scale_f32(int(M), int(N), beta, C, ldc, stream));
  return from_cuda(dgr::launch_gemm_tc_f16(*dev, is_bf16, int(M), int(N), int(K), alpha, A, lda,
                                           B, ldb, beta, C, ldc, stream));
}

gemm_status_t gemm_bf16(int64_t M, int64_t N, int64_t K, float alpha, const gemm_bf16_t *A,
                        int64_t lda, const gemm_bf16_t *B, int64_t ldb, float beta, float *C,
                        int64_t ldc, cudaStream_t stream) {
  return gemm_half(true, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream);
}

gemm_status_t gemm_f16(int64_t M, int64_t N, int64_t K, float alpha, const gemm_f16_t *A,
                       int64_t lda, const gemm_f16_t *B, int64_t ldb, float beta, float *C,
                       int64_t ldc, cudaStream_t stream) {
  return gemm_half(false, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream);
}

gemm_status_t gemm_s8(int64_t M, int64_t N, int64_t K, int32_t alpha, const int8_t *A,
                      int64_t lda, const int8_t *B, int64_t ldb, int32_t beta, int32_t *C,
                      int64_t ldc, cudaStream_t stream) {
  bool skip = false;
  gemm_status_t st = check_args(M, N, K, A, lda, B, ldb, C, ldc, &skip);
  if (st != GEMM_OK || skip) return st;
  const DeviceInfo *dev = nullptr;
  if ((st = current_device(&dev)) != GEMM_OK) return st;
  if (K == 0) return from_cuda(dgr::launch_scale_s32(int(M), int(N), beta, C, ldc, stream));
  if (dgr::small_m_supported(int(M), A, lda, B, ldb, 1))  // few rows: int8 B read once, dp4a
    return from_cuda(dgr::launch_small_m_s8(*dev, int(M), int(N), int(K), alpha, A, lda, B, ldb,
                                            beta, C, ldc, stream));
  return from_cuda(dgr::launch_gemm_s8(*dev, int(M), int(N), int(K), alpha, A, lda, B, ldb, beta,
                                       C, ldc, stream));
}

const char *gemm_status_string(gemm_status_t status) {
  switch (status) {
    case GEMM_OK: return "GEMM_OK";
    case GEMM_ERR_INVALID_VALUE: return "GEMM_ERR_INVALID_VALUE";
    case GEMM_ERR_UNSUPPORTED_LAYOUT: return "GEMM_ERR_UNSUPPORTED_LAYOUT";
    case GEMM_ERR_LAUNCH: return "GEMM_ERR_LAUNCH";
    case GEMM_ERR_DEVICE: return "GEMM_ERR_DEVICE";
    case GEMM_ERR_TIMEOUT: return "GEMM_ERR_TIMEOUT";
    case GEMM_ERR_TOO_LARGE: return "GEMM_ERR_TOO_LARGE";
  }
  return "GEMM_ERR_UNKNOWN";
}

gemm_status_t gemm_check_device_error(uint32_t *word) {
  const DeviceInfo *dev = nullptr;
  gemm_status_t st = current_device(&dev);
  if (st != GEMM_OK) return st;
  uint32_t w = 0;
  if (cudaMemcpy(&w, dev->err_word, sizeof w, cudaMemcpyDeviceToHost) != cudaSuccess)
    return from_cuda(cudaErrorUnknown);
  const uint32_t zero = 0;
  if (cudaMemcpy(dev->err_word, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
    return from_cuda(cudaErrorUnknown);
  if (word) *word = w;
  return (w & dgr::kErrTimeoutBit) ? GEMM_ERR_TIMEOUT : GEMM_OK;
}

int gemm_version(void) { return dgr::kVersion; }

}  // extern "C"
