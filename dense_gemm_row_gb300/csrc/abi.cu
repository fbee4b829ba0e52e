// abi.cu -- the C entry points of libdense_gemm_row.so (include/dense_gemm_row.h).
//
// Host-side argument checks, per-device set-up, the K == 0 path (C = beta*C)
// and dispatch to the kernels. Nothing here allocates or frees user memory,
// prints, or aborts.
#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <type_traits>
#include <utility>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
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

// The CUDA error behind this thread's last GEMM_ERR_LAUNCH (gemm_last_launch_error).
thread_local cudaError_t g_last_launch_error = cudaSuccess;

gemm_status_t from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return GEMM_OK;
  g_last_launch_error = e;
  cudaGetLastError();  // clear a sticky launch error so later calls are not blamed
  return GEMM_ERR_LAUNCH;
}

// ------------------------------------------------------------ K == 0 kernels

template <typename T>
__global__ void scale_kernel(int M, int N, T beta, T *C, int64_t ldc, int batch,
                             int64_t stride) {
  const int64_t per = static_cast<int64_t>(M) * N;
  const int64_t total = per * batch;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t b = i / per, j = i - b * per;
    const int64_t r = j / N, c = j - r * N;
    T *p = C + b * stride + r * ldc + c;
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
cudaError_t launch_scale(int M, int N, T beta, T *C, int64_t ldc, cudaStream_t stream,
                         int batch = 1, int64_t stride = 0) {
  const int64_t total = static_cast<int64_t>(M) * N * batch;
  int64_t blocks = (total + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  scale_kernel<T><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(M, N, beta, C, ldc, batch,
                                                                     stride);
  return cudaGetLastError();
}

// 16-bit C: C = round16(beta * C), 0 when beta == 0.
template <bool kBf16>
__global__ void scale16_kernel(int M, int N, float beta, uint16_t *C, int64_t ldc) {
  const int64_t total = static_cast<int64_t>(M) * N;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = i / N, c = i - r * N;
    uint16_t *p = C + r * ldc + c;
    if (kBf16) {
      const float v = beta == 0.f ? 0.f : beta * __bfloat162float(__ushort_as_bfloat16(*p));
      *p = __bfloat16_as_ushort(__float2bfloat16_rn(v));
    } else {
      const float v = beta == 0.f ? 0.f : beta * __half2float(__ushort_as_half(*p));
      *p = __half_as_ushort(__float2half_rn(v));
    }
  }
}

// Argument checks of the extended entry points: operand forms, sizes, the
// stored operands' row strides, batch count and strides. Returns GEMM_OK when
// the call should proceed; sets *nothing_to_do when there is no output.
gemm_status_t check_ex(gemm_op_t opA, gemm_op_t opB, int64_t M, int64_t N, int64_t K,
                       const void *A, int64_t lda, int64_t strideA, const void *B, int64_t ldb,
                       int64_t strideB, const void *C, int64_t ldc, int64_t strideC,
                       int64_t batch, bool *nothing_to_do) {
  *nothing_to_do = false;
  if ((opA != GEMM_OP_N && opA != GEMM_OP_T) || (opB != GEMM_OP_N && opB != GEMM_OP_T))
    return GEMM_ERR_INVALID_VALUE;
  if (batch < 0 || batch > kMaxDim) return GEMM_ERR_INVALID_VALUE;
  if (strideA < 0 || strideB < 0 || strideC < 0) return GEMM_ERR_INVALID_VALUE;
  // Stored row lengths: A's rows hold K (op N) or M (op T) values, B's N or K.
  const int64_t a_row = opA == GEMM_OP_N ? K : M;
  const int64_t b_row = opB == GEMM_OP_N ? N : K;
  if (M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_VALUE;
  if (M > kMaxDim || N > kMaxDim || K > kMaxDim) return GEMM_ERR_INVALID_VALUE;
  if (batch == 0 || M == 0 || N == 0) {
    *nothing_to_do = true;
    return GEMM_OK;
  }
  if (ldc < N || C == nullptr) return GEMM_ERR_INVALID_VALUE;
  if (K > 0) {
    if (lda < a_row || A == nullptr) return GEMM_ERR_INVALID_VALUE;
    if (ldb < b_row || B == nullptr) return GEMM_ERR_INVALID_VALUE;
  }
  if (batch > 1) {
    // The C matrices must not overlap: strideC >= (M - 1) * ldc + N.
    if (M > 1 && ldc > (INT64_MAX - N) / (M - 1)) return GEMM_ERR_INVALID_VALUE;
    if (strideC < (M - 1) * ldc + N) return GEMM_ERR_INVALID_VALUE;
  }
  return GEMM_OK;
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

// Library-owned stream-ordered memory pool of a device (scratch for the 8-bit
// paths, the tf32 operand copies and split-k workspaces); freed blocks stay
// mapped for reuse.
std::mutex g_pool_mu;
cudaMemPool_t g_pools[kMaxDevices] = {};

cudaError_t device_pool(const DeviceInfo &dev, cudaMemPool_t *out) {
  std::lock_guard<std::mutex> lock(g_pool_mu);
  cudaMemPool_t *pools = g_pools;
  if (dev.device < 0 || dev.device >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!pools[dev.device]) {
    cudaMemPoolProps props;
    std::memset(&props, 0, sizeof props);
    props.allocType = cudaMemAllocationTypePinned;
    props.handleTypes = cudaMemHandleTypeNone;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev.device;
    cudaMemPool_t pl;
    cudaError_t e = cudaMemPoolCreate(&pl, &props);
    if (e != cudaSuccess) return e;
    uint64_t keep = ~0ull;  // keep freed memory mapped for the next call
    cudaMemPoolSetAttribute(pl, cudaMemPoolAttrReleaseThreshold, &keep);
    pools[dev.device] = pl;
  }
  *out = pools[dev.device];
  return cudaSuccess;
}

cudaError_t launch_scale_batched_f32(int M, int N, float beta, float *C, int64_t ldc, int batch,
                                     int64_t stride, cudaStream_t stream) {
  return launch_scale<float>(M, N, beta, C, ldc, stream, batch, stride);
}
cudaError_t launch_scale_batched_s32(int M, int N, int32_t beta, int32_t *C, int64_t ldc,
                                     int batch, int64_t stride, cudaStream_t stream) {
  return launch_scale<int32_t>(M, N, beta, C, ldc, stream, batch, stride);
}

int abi_check_args(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda, const void *B,
                   int64_t ldb, const void *C, int64_t ldc, bool *nothing_to_do) {
  return check_args(M, N, K, A, lda, B, ldb, C, ldc, nothing_to_do);
}

int abi_current_device(const DeviceInfo **out) { return current_device(out); }

int abi_from_cuda(cudaError_t e) { return from_cuda(e); }

cudaError_t launch_scale_f64(int M, int N, double beta, double *C, int64_t ldc,
                             cudaStream_t stream) {
  return launch_scale<double>(M, N, beta, C, ldc, stream);
}

cudaError_t launch_scale_out16(bool is_bf16, int M, int N, float beta, uint16_t *C, int64_t ldc,
                               cudaStream_t stream) {
  const int64_t total = static_cast<int64_t>(M) * N;
  int64_t blocks = (total + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  if (is_bf16) {
    scale16_kernel<true><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(M, N, beta, C, ldc);
  } else {
    scale16_kernel<false><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(M, N, beta, C, ldc);
  }
  return cudaGetLastError();
}

cudaError_t launch_scale_f32(int M, int N, float beta, float *C, int64_t ldc,
                             cudaStream_t stream) {
  return launch_scale<float>(M, N, beta, C, ldc, stream);
}

cudaError_t launch_scale_s32(int M, int N, int32_t beta, int32_t *C, int64_t ldc,
                             cudaStream_t stream) {
  return launch_scale<int32_t>(M, N, beta, C, ldc, stream);
}

}  // namespace dgr

using dgr::BatchOps;
using dgr::check_args;
using dgr::check_ex;
using dgr::current_device;
using dgr::DeviceInfo;
using dgr::from_cuda;

extern "C" {

gemm_status_t gemm_pool_usage(int64_t *used_high_bytes, int64_t *reserved_bytes, int reset_high) {
  int device = -1;
  if (cudaGetDevice(&device) != cudaSuccess || device < 0 || device >= dgr::kMaxDevices) {
    cudaGetLastError();
    return GEMM_ERR_DEVICE;
  }
  uint64_t used_high = 0, reserved = 0;
  std::lock_guard<std::mutex> lock(dgr::g_pool_mu);
  cudaMemPool_t pl = dgr::g_pools[device];
  if (pl != nullptr) {  // no pool yet: nothing was ever taken from it
    if (cudaMemPoolGetAttribute(pl, cudaMemPoolAttrUsedMemHigh, &used_high) != cudaSuccess ||
        cudaMemPoolGetAttribute(pl, cudaMemPoolAttrReservedMemCurrent, &reserved) !=
            cudaSuccess) {
      cudaGetLastError();
      return GEMM_ERR_LAUNCH;
    }
    if (reset_high) {
      uint64_t zero = 0;
      if (cudaMemPoolSetAttribute(pl, cudaMemPoolAttrUsedMemHigh, &zero) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
      }
    }
  }
  if (used_high_bytes) *used_high_bytes = static_cast<int64_t>(used_high);
  if (reserved_bytes) *reserved_bytes = static_cast<int64_t>(reserved);
  return GEMM_OK;
}

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
  // 33..64 rows: two streaming passes (32 rows, then the rest) beat one
  // 128-row tile, half of whose rows would be empty (measured on GB300 at
  // N = K = 8192: M = 64 in 2 x 139 us against 362 us).
  if (M <= 2 * dgr::kSkinnyMaxM && dgr::small_m_supported(dgr::kSkinnyMaxM, A, lda, B, ldb, 4)) {
    const int m1 = dgr::kSkinnyMaxM, m2 = int(M) - m1;
    cudaError_t e = dgr::launch_small_m_f32(*dev, m1, int(N), int(K), alpha, A, lda, B, ldb,
                                            beta, C, ldc, stream);
    if (e == cudaSuccess)
      e = dgr::launch_small_m_f32(*dev, m2, int(N), int(K), alpha, A + int64_t(m1) * lda, lda,
                                  B, ldb, beta, C + int64_t(m1) * ldc, ldc, stream);
    return from_cuda(e);
  }
  if (dgr::small_n_supported(int(M), int(N), A, lda, 4))  // few columns: stream A once
    return from_cuda(dgr::launch_small_n_f32(int(M), int(N), int(K), alpha, A, lda, B, ldb, beta,
                                             C, ldc, stream));
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
  if (dgr::small_n_supported(int(M), int(N), A, lda, 2))  // few columns: stream A once
    return from_cuda(dgr::launch_small_n_half(is_bf16, int(M), int(N), int(K), alpha, A, lda, B,
                                              ldb, beta, C, ldc, stream));
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
  // Short and wide with at least 16 column blocks of 128: the tensor-core
  // kernel that reads int8 B once, as stored.
  if (N >= 16 * 128 && dgr::tc_skinny_i8_supported(int(M), B, ldb) &&
      (M >= dgr::kI8RawMinM ||
       (M >= dgr::kI8ClusterMinM && dgr::tc_skinny_s8_supported(int(M), A, lda, B, ldb))))
    return from_cuda(dgr::launch_gemm_s8_skinny_raw(*dev, int(M), int(N), int(K), alpha, A, lda,
                                                    B, ldb, beta, C, ldc, stream));
  if (dgr::small_m_supported(int(M), A, lda, B, ldb, 1))  // few rows: int8 B read once, dp4a
    return from_cuda(dgr::launch_small_m_s8(*dev, int(M), int(N), int(K), alpha, A, lda, B, ldb,
                                            beta, C, ldc, stream));
  if (dgr::small_n_supported(int(M), int(N), A, lda, 1))  // few columns: stream A once
    return from_cuda(dgr::launch_small_n_s8(int(M), int(N), int(K), alpha, A, lda, B, ldb, beta,
                                            C, ldc, stream));
  return from_cuda(dgr::launch_gemm_s8(*dev, int(M), int(N), int(K), alpha, A, lda, B, ldb, beta,
                                       C, ldc, stream));
}

gemm_status_t gemm_u8(int64_t M, int64_t N, int64_t K, int32_t alpha, const uint8_t *A,
                      int64_t lda, const uint8_t *B, int64_t ldb, int32_t beta, int32_t *C,
                      int64_t ldc, cudaStream_t stream) {
  bool skip = false;
  gemm_status_t st = check_args(M, N, K, A, lda, B, ldb, C, ldc, &skip);
  if (st != GEMM_OK || skip) return st;
  const DeviceInfo *dev = nullptr;
  if ((st = current_device(&dev)) != GEMM_OK) return st;
  if (K == 0) return from_cuda(dgr::launch_scale_s32(int(M), int(N), beta, C, ldc, stream));
  return from_cuda(dgr::launch_gemm_u8(*dev, int(M), int(N), int(K), alpha, A, lda, B, ldb, beta,
                                       C, ldc, stream));
}

static gemm_status_t gemm_out16(bool is_bf16, int64_t M, int64_t N, int64_t K, float alpha,
                                const uint16_t *A, int64_t lda, const uint16_t *B, int64_t ldb,
                                float beta, uint16_t *C, int64_t ldc, cudaStream_t stream) {
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
  if (K == 0)
    return from_cuda(dgr::launch_scale_out16(is_bf16, int(M), int(N), beta, C, ldc, stream));
  return from_cuda(dgr::launch_gemm_tc_out16(*dev, is_bf16, int(M), int(N), int(K), alpha, A, lda,
                                             B, ldb, beta, C, ldc, stream));
}

gemm_status_t gemm_f16_f16(int64_t M, int64_t N, int64_t K, float alpha, const gemm_f16_t *A,
                           int64_t lda, const gemm_f16_t *B, int64_t ldb, float beta,
                           gemm_f16_t *C, int64_t ldc, cudaStream_t stream) {
  return gemm_out16(false, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream);
}

gemm_status_t gemm_bf16_bf16(int64_t M, int64_t N, int64_t K, float alpha, const gemm_bf16_t *A,
                             int64_t lda, const gemm_bf16_t *B, int64_t ldb, float beta,
                             gemm_bf16_t *C, int64_t ldc, cudaStream_t stream) {
  return gemm_out16(true, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream);
}

gemm_status_t gemm_tf32(int64_t M, int64_t N, int64_t K, float alpha, const float *A,
                        int64_t lda, const float *B, int64_t ldb, float beta, float *C,
                        int64_t ldc, cudaStream_t stream) {
  bool skip = false;
  gemm_status_t st = check_args(M, N, K, A, lda, B, ldb, C, ldc, &skip);
  if (st != GEMM_OK || skip) return st;
  if (K > 0 && (reinterpret_cast<uintptr_t>(A) & 3u || reinterpret_cast<uintptr_t>(B) & 3u))
    return GEMM_ERR_UNSUPPORTED_LAYOUT;  // fp32 elements must be 4-byte aligned
  const DeviceInfo *dev = nullptr;
  if ((st = current_device(&dev)) != GEMM_OK) return st;
  if (K == 0) return from_cuda(dgr::launch_scale_f32(int(M), int(N), beta, C, ldc, stream));
  return from_cuda(dgr::launch_gemm_tf32(*dev, int(M), int(N), int(K), alpha, A, lda, B, ldb,
                                         beta, C, ldc, stream));
}

gemm_status_t gemm_f64(int64_t M, int64_t N, int64_t K, double alpha, const double *A,
                       int64_t lda, const double *B, int64_t ldb, double beta, double *C,
                       int64_t ldc, cudaStream_t stream) {
  bool skip = false;
  gemm_status_t st = check_args(M, N, K, A, lda, B, ldb, C, ldc, &skip);
  if (st != GEMM_OK || skip) return st;
  const DeviceInfo *dev = nullptr;
  if ((st = current_device(&dev)) != GEMM_OK) return st;
  if (K == 0) return from_cuda(dgr::launch_scale_f64(int(M), int(N), beta, C, ldc, stream));
  return from_cuda(dgr::launch_dgemm(*dev, int(M), int(N), int(K), alpha, A, lda, B, ldb, beta, C,
                                     ldc, stream));
}

static BatchOps make_ops(gemm_op_t opA, gemm_op_t opB, int64_t strideA, int64_t strideB,
                         int64_t strideC, int64_t batch) {
  BatchOps ops;
  ops.a_t = opA == GEMM_OP_T;
  ops.b_t = opB == GEMM_OP_T;
  ops.batch = static_cast<int>(batch);
  ops.stride_a = strideA;
  ops.stride_b = strideB;
  ops.stride_c = strideC;
  return ops;
}

gemm_status_t gemm_f32_ex(gemm_op_t opA, gemm_op_t opB, int64_t M, int64_t N, int64_t K,
                          float alpha, const float *A, int64_t lda, int64_t strideA,
                          const float *B, int64_t ldb, int64_t strideB, float beta, float *C,
                          int64_t ldc, int64_t strideC, int64_t batch, cudaStream_t stream) {
  bool skip = false;
  gemm_status_t st = check_ex(opA, opB, M, N, K, A, lda, strideA, B, ldb, strideB, C, ldc,
                              strideC, batch, &skip);
  if (st != GEMM_OK || skip) return st;
  const BatchOps ops = make_ops(opA, opB, strideA, strideB, strideC, batch);
  if (ops.plain()) return gemm_f32(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream);
  const DeviceInfo *dev = nullptr;
  if ((st = current_device(&dev)) != GEMM_OK) return st;
  if (K == 0)
    return from_cuda(dgr::launch_scale_batched_f32(int(M), int(N), beta, C, ldc, ops.batch,
                                                   strideC, stream));
  return from_cuda(dgr::launch_sgemm_simt_ex(*dev, ops, int(M), int(N), int(K), alpha, A, lda, B,
                                             ldb, beta, C, ldc, stream));
}

static gemm_status_t gemm_half_ex(bool is_bf16, gemm_op_t opA, gemm_op_t opB, int64_t M,
                                  int64_t N, int64_t K, float alpha, const uint16_t *A,
                                  int64_t lda, int64_t strideA, const uint16_t *B, int64_t ldb,
                                  int64_t strideB, float beta, float *C, int64_t ldc,
                                  int64_t strideC, int64_t batch, cudaStream_t stream) {
  bool skip = false;
  gemm_status_t st = check_ex(opA, opB, M, N, K, A, lda, strideA, B, ldb, strideB, C, ldc,
                              strideC, batch, &skip);
  if (st != GEMM_OK || skip) return st;
  const BatchOps ops = make_ops(opA, opB, strideA, strideB, strideC, batch);
  if (ops.plain()) return gemm_half(is_bf16, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream);
  if (K > 0) {
    // TMA: 16-byte aligned bases, row strides and matrix strides.
    if ((reinterpret_cast<uintptr_t>(A) & 15u) || (reinterpret_cast<uintptr_t>(B) & 15u) ||
        (lda % 8) || (ldb % 8))
      return GEMM_ERR_UNSUPPORTED_LAYOUT;
    if (batch > 1 && ((strideA % 8) || (strideB % 8))) return GEMM_ERR_UNSUPPORTED_LAYOUT;
  }
  const DeviceInfo *dev = nullptr;
  if ((st = current_device(&dev)) != GEMM_OK) return st;
  if (K == 0)
    return from_cuda(dgr::launch_scale_batched_f32(int(M), int(N), beta, C, ldc, ops.batch,
                                                   strideC, stream));
  return from_cuda(dgr::launch_gemm_tc_f16_ex(*dev, is_bf16, ops, int(M), int(N), int(K), alpha,
                                              A, lda, B, ldb, beta, C, ldc, stream));
}

gemm_status_t gemm_bf16_ex(gemm_op_t opA, gemm_op_t opB, int64_t M, int64_t N, int64_t K,
                           float alpha, const gemm_bf16_t *A, int64_t lda, int64_t strideA,
                           const gemm_bf16_t *B, int64_t ldb, int64_t strideB, float beta,
                           float *C, int64_t ldc, int64_t strideC, int64_t batch,
                           cudaStream_t stream) {
  return gemm_half_ex(true, opA, opB, M, N, K, alpha, A, lda, strideA, B, ldb, strideB, beta, C,
                      ldc, strideC, batch, stream);
}

gemm_status_t gemm_f16_ex(gemm_op_t opA, gemm_op_t opB, int64_t M, int64_t N, int64_t K,
                          float alpha, const gemm_f16_t *A, int64_t lda, int64_t strideA,
                          const gemm_f16_t *B, int64_t ldb, int64_t strideB, float beta,
                          float *C, int64_t ldc, int64_t strideC, int64_t batch,
                          cudaStream_t stream) {
  return gemm_half_ex(false, opA, opB, M, N, K, alpha, A, lda, strideA, B, ldb, strideB, beta, C,
                      ldc, strideC, batch, stream);
}

gemm_status_t gemm_s8_ex(gemm_op_t opA, gemm_op_t opB, int64_t M, int64_t N, int64_t K,
                         int32_t alpha, const int8_t *A, int64_t lda, int64_t strideA,
                         const int8_t *B, int64_t ldb, int64_t strideB, int32_t beta, int32_t *C,
                         int64_t ldc, int64_t strideC, int64_t batch, cudaStream_t stream) {
  bool skip = false;
  gemm_status_t st = check_ex(opA, opB, M, N, K, A, lda, strideA, B, ldb, strideB, C, ldc,
                              strideC, batch, &skip);
  if (st != GEMM_OK || skip) return st;
  const BatchOps ops = make_ops(opA, opB, strideA, strideB, strideC, batch);
  if (ops.plain()) return gemm_s8(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream);
  const DeviceInfo *dev = nullptr;
  if ((st = current_device(&dev)) != GEMM_OK) return st;
  if (K == 0)
    return from_cuda(dgr::launch_scale_batched_s32(int(M), int(N), beta, C, ldc, ops.batch,
                                                   strideC, stream));
  return from_cuda(dgr::launch_gemm_s8_ex(*dev, ops, int(M), int(N), int(K), alpha, A, lda, B,
                                          ldb, beta, C, ldc, stream));
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

const char *gemm_last_launch_error(void) {
  return cudaGetErrorName(dgr::g_last_launch_error);
}

int gemm_version(void) { return dgr::kVersion; }

}  // extern "C"
