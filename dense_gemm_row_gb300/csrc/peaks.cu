// peaks.cu -- peak-rate microbenchmarks for the two pipes that bound the GEMM
// kernels: the FP32 FMA pipe (the exact-fp32 SIMT GEMM) and the tensor pipe
// with tcgen05 kind::f16 (the bf16 / fp16 / exact-int8 GEMM). They give the
// measured denominators that the roofline fractions are cross-checked against.
// Neither touches user data; the tensor-core one holds TMEM only while it runs
// and its single wait is bounded like the GEMM kernels' waits.
#include <cstdint>

#include <cuda_runtime.h>

#include "../../include/dense_gemm_row.h"
#include "launch.h"
#include "ptx.cuh"

namespace dgr {
namespace {

// (c0, c1) = (a * b0 + c0, a * b1 + c1) with one packed fp32 FMA.
__device__ __forceinline__ void ffma2(float &c0, float &c1, float a, float b0, float b1) {
  asm("{\n .reg .b64 ra, rb, rc;\n mov.b64 ra, {%2, %2};\n mov.b64 rb, {%3, %4};\n"
      " mov.b64 rc, {%0, %1};\n fma.rn.f32x2 rc, ra, rb, rc;\n mov.b64 {%0, %1}, rc;\n}\n"
      : "+f"(c0), "+f"(c1)
      : "f"(a), "f"(b0), "f"(b1));
}

constexpr int kFfmaThreads = 256;
constexpr int kFfmaBlocksPerSm = 4;
constexpr int kFfmaChains = 32;  // independent accumulators per thread (16 packed pairs)

// Every thread: `iters` rounds of 16 independent packed FMAs. The values stay
// normal and bounded (each round adds about 1e-4 to every accumulator).
__global__ void __launch_bounds__(kFfmaThreads) ffma_peak_kernel(int iters, float *sink) {
  const float a = 1.0f + static_cast<float>(threadIdx.x) * 1e-7f;
  const float b0 = 1e-4f, b1 = 2e-4f;
  float acc[kFfmaChains];
#pragma unroll
  for (int j = 0; j < kFfmaChains; ++j) acc[j] = static_cast<float>(j) * 1e-3f;
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int j = 0; j < kFfmaChains; j += 2) ffma2(acc[j], acc[j + 1], a, b0, b1);
  }
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < kFfmaChains; ++j) s += acc[j];
  if (s == -1.0f) *sink = s;  // never true for these values; keeps the sums live
}

// Tensor pipe: one CTA per SM; operands (A: 128 x 64 bf16, B: 256 x 64 bf16,
// both K-major with the 128-byte swizzle, as the GEMM kernel stages A) are
// filled once; one thread issues iters x 4 MMAs (M = 128, N = 256, K = 16)
// into a 256-column TMEM accumulator, then waits for the last one.
constexpr int kTcThreads = 128;
constexpr uint32_t kTcABytes = 128 * 128;  // 128 rows x 128 bytes
constexpr uint32_t kTcBBytes = 256 * 128;  // 256 rows x 128 bytes
constexpr uint32_t kTcSmem = kTcABytes + kTcBBytes + 1024;  // + alignment slack
constexpr uint32_t kTcCols = 256;

__global__ void __launch_bounds__(kTcThreads, 1)
    tc_peak_kernel(int iters, uint32_t idesc, uint32_t *err_word) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t done_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const int warp = threadIdx.x >> 5;

  // Operand values: every bf16 element 1/64 (0x3C80), so the sums stay finite.
  for (uint32_t off = threadIdx.x * 16u; off < kTcABytes + kTcBBytes; off += kTcThreads * 16u)
    st_shared_v4(base + off, 0x3C803C80u, 0x3C803C80u, 0x3C803C80u, 0x3C803C80u);
  fence_proxy_async_shared();  // the MMA reads shared memory through the async proxy
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&done_bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&tmem_base_sh), kTcCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = tmem_base_sh;

  if (threadIdx.x == 0) {
    const uint32_t a_addr = base, b_addr = base + kTcABytes;
    for (int it = 0; it < iters; ++it) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t adesc = smem_desc(a_addr + kk * 32, 16, 1024, 2u);
        const uint64_t bdesc = smem_desc(b_addr + kk * 32, 16, 1024, 2u);
        tc_mma_f16(tmem_base, adesc, bdesc, idesc, (it > 0 || kk > 0) ? 1u : 0u);
      }
    }
    tc_commit(smem_u32(&done_bar));
    mbar_wait_bounded(smem_u32(&done_bar), 0, &abort_flag, err_word, kWaitDrain);
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, kTcCols);
  }
}

}  // namespace
}  // namespace dgr

extern "C" gemm_status_t gemm_peak_ffma(int32_t iters, float *sink, double *flops,
                                        cudaStream_t stream) {
  if (iters < 1 || iters > (1 << 24) || sink == nullptr) return GEMM_ERR_INVALID_VALUE;
  const dgr::DeviceInfo *dev = nullptr;
  int st = dgr::abi_current_device(&dev);
  if (st != GEMM_OK) return static_cast<gemm_status_t>(st);
  const int blocks = dev->sm_count * dgr::kFfmaBlocksPerSm;
  dgr::ffma_peak_kernel<<<blocks, dgr::kFfmaThreads, 0, stream>>>(iters, sink);
  if (flops)
    *flops = static_cast<double>(blocks) * dgr::kFfmaThreads * iters * dgr::kFfmaChains * 2.0;
  return static_cast<gemm_status_t>(dgr::abi_from_cuda(cudaGetLastError()));
}

extern "C" gemm_status_t gemm_peak_tc_f16(int32_t iters, double *flops, cudaStream_t stream) {
  // At most 2^20 rounds (about 0.3 s of MMAs), far inside the 2 s bound on the
  // kernel's one wait, so TMEM is never freed under MMAs still running.
  if (iters < 1 || iters > (1 << 20)) return GEMM_ERR_INVALID_VALUE;
  const dgr::DeviceInfo *dev = nullptr;
  int st = dgr::abi_current_device(&dev);
  if (st != GEMM_OK) return static_cast<gemm_status_t>(st);
  cudaError_t e = dgr::set_max_dynamic_smem(reinterpret_cast<const void *>(dgr::tc_peak_kernel),
                                            static_cast<int>(dgr::kTcSmem), dev->device);
  if (e != cudaSuccess) return static_cast<gemm_status_t>(dgr::abi_from_cuda(e));
  const uint32_t idesc = dgr::idesc_mma(dgr::kFmtBF16, false, false, 128, 256);
  dgr::tc_peak_kernel<<<dev->sm_count, dgr::kTcThreads, dgr::kTcSmem, stream>>>(iters, idesc,
                                                                             dev->err_word);
  if (flops) *flops = static_cast<double>(dev->sm_count) * iters * 4 * 2.0 * 128 * 256 * 16;
  return static_cast<gemm_status_t>(dgr::abi_from_cuda(cudaGetLastError()));
}
