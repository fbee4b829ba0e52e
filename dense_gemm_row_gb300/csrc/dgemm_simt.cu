// dgemm_simt.cu -- fp64 GEMM on the SIMT FP64 pipe (the warp-matrix-function
// type table's double row: double inputs, double accumulate), row-major:
//
//     C = alpha * A * B + beta * C
//
// GB300's FP64 rate is a small fraction of its FP32 rate, so the FP64 pipe is
// the bound at any useful tile size and the kernel is kept plain: one CTA of
// 256 threads per 64 x 64 tile of C, k-steps of 16 staged in shared memory (A
// transposed, so a thread's four A values for one k are one row of the tile),
// each thread 4 x 4 outputs at a stride of 16 rows and 16 columns (a warp's
// shared loads of B are 16 consecutive doubles, its loads of A two broadcast
// addresses). Many CTAs per SM hide the load latency. Out-of-range tile cells
// are zero and the epilogue's stores are guarded ("使用CUDA和瓦片算法计算矩阵
// 乘法": residual tile cells zeroed, guarded store). C is not read when
// beta == 0. Products and sums use the hardware fused multiply-add (fma).
#include <cstdint>

#include <cuda_runtime.h>

#include "launch.h"

namespace dgr {
namespace {

constexpr int kDT = 64;       // tile rows and columns
constexpr int kDK = 16;       // k per step
constexpr int kDThreads = 256;

struct DArgs {
  int M, N, K;
  double alpha, beta;
  const double *A;
  int64_t lda;
  const double *B;
  int64_t ldb;
  double *C;
  int64_t ldc;
};

__global__ void __launch_bounds__(kDThreads) dgemm_kernel(const DArgs p) {
  __shared__ double as[kDK][kDT + 1];  // A tile, transposed: as[k][m]
  __shared__ double bs[kDK][kDT];      // B tile: bs[k][n]
  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
  const int64_t m0 = static_cast<int64_t>(blockIdx.y) * kDT;
  const int64_t n0 = static_cast<int64_t>(blockIdx.x) * kDT;
  double acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.0;

  for (int k0 = 0; k0 < p.K; k0 += kDK) {
#pragma unroll
    for (int i = 0; i < kDT * kDK / kDThreads; ++i) {
      const int e = tid + i * kDThreads;
      // A: 64 rows x 16 k, 16 consecutive k per row (one 128-byte segment)
      const int ar = e / kDK, ak = e % kDK;
      const int64_t gm = m0 + ar;
      const int gk = k0 + ak;
      as[ak][ar] = (gm < p.M && gk < p.K) ? p.A[gm * p.lda + gk] : 0.0;
      // B: 16 k x 64 columns
      const int bk = e / kDT, bc = e % kDT;
      const int gkb = k0 + bk;
      const int64_t gn = n0 + bc;
      bs[bk][bc] = (gkb < p.K && gn < p.N) ? p.B[static_cast<int64_t>(gkb) * p.ldb + gn] : 0.0;
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kDK; ++k) {
      double a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = as[k][ty + 16 * i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = bs[k][tx + 16 * j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fma(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t row = m0 + ty + 16 * i;
    if (row >= p.M) continue;
    double *crow = p.C + row * p.ldc;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t col = n0 + tx + 16 * j;
      if (col < p.N) {
        const double r = p.alpha * acc[i][j];
        crow[col] = (p.beta != 0.0) ? r + p.beta * crow[col] : r;
      }
    }
  }
}

}  // namespace

cudaError_t launch_dgemm(const DeviceInfo &dev, int M, int N, int K, double alpha,
                         const double *A, int64_t lda, const double *B, int64_t ldb, double beta,
                         double *C, int64_t ldc, cudaStream_t stream) {
  (void)dev;
  DArgs a{M, N, K, alpha, beta, A, lda, B, ldb, C, ldc};
  const int64_t gy = (static_cast<int64_t>(M) + kDT - 1) / kDT;
  const int64_t gx = (static_cast<int64_t>(N) + kDT - 1) / kDT;
  if (gy > 65535 || gx > 0x7fffffffLL) return cudaErrorInvalidValue;
  dgemm_kernel<<<dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy)), kDThreads, 0,
                 stream>>>(a);
  return cudaGetLastError();
}

}  // namespace dgr
