// gemm_small_n.cu -- GEMM for tall, narrow problems (N <= 16), including the
// matrix-vector product (N = 1):
//
//     C = alpha * A * B + beta * C       A: M x K, B: K x N, C: M x N, row-major
//
// With a handful of columns of B the work is bound by reading A (M x K) once,
// and a tile 128 or 256 columns wide would multiply mostly zeros. Here each
// warp owns kRows rows of A and streams them with 16-byte loads (a warp reads
// 512 contiguous bytes of a row per step); every lane keeps kRows x NP partial
// sums over its own slice of k. B is small: each CTA stages it in shared
// memory chunk by chunk, transposed so that the values of one column are
// contiguous in k (a lane reads its k-slice of a column with 16-byte loads,
// and the 32 lanes of a warp read 512 contiguous bytes). At the end the lanes'
// partial sums are added by a fixed butterfly of shuffles, so every element is
// summed in the same order on every run, and alpha * sum + beta * C is written.
//
// Element types: fp32 (fp32 FMAs, each rounded once), bf16 / fp16 (products of
// two 16-bit values are exact in fp32; fp32 accumulation), int8 (dp4a into
// int32, wrap-around like the other int8 paths).
//
// Sources: C = alpha*A*B + beta*C, row-major ("Sgemm [128,128,8]", the
// kernel's header comment and host_gemm); the type table of the C++ warp
// matrix function page (half / bfloat16 x half / bfloat16 -> float, signed
// char -> int). The pages have no narrow-N kernel; this is a layout choice for
// the same computation.
#include <cstdint>
#include <type_traits>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "launch.h"
#include "ptx.cuh"

namespace dgr {
namespace {

constexpr int kSnThreads = 256;
constexpr int kSnWarps = kSnThreads / 32;
constexpr int kRows = 4;                   // rows of A per warp
constexpr int kSnRowsPerCta = kSnWarps * kRows;
constexpr int kMaxNP = 16;

template <typename In>
struct SnType {
  // values of k per 16-byte load of A
  static constexpr int kVec = 16 / static_cast<int>(sizeof(In));
  static constexpr bool kInt = std::is_same<In, int8_t>::value;
  using Acc = typename std::conditional<kInt, int32_t, float>::type;
  using Bt = typename std::conditional<kInt, int8_t, float>::type;  // staged B element
};

// Per column count: KC values of k per staged chunk of B (at most 32 staged
// values per thread, so that all loads of a chunk are in flight at once: 512
// for 16 columns), S the staged row (one column of B) stride, with 16 bytes
// of padding so that the transposing stores of one k spread over the banks,
// and G the steps of A loaded ahead (kRows x NP accumulators and G x kRows
// 16-byte loads per lane must fit the 128 registers of two CTAs per SM).
template <typename In, int NP>
struct SnShape {
  using Bt = typename SnType<In>::Bt;
  static constexpr int KC = NP * 1024 > 32 * kSnThreads ? 512 : 1024;
  static constexpr int S = KC + 16 / static_cast<int>(sizeof(Bt));
  static constexpr int kSteps = KC / (32 * SnType<In>::kVec);
  static constexpr int G = (NP >= 16 ? 2 : 4) < kSteps ? (NP >= 16 ? 2 : 4) : kSteps;
};

__device__ __forceinline__ float to_float(float x) { return x; }
__device__ __forceinline__ float to_float(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float to_float(__half x) { return __half2float(x); }

__device__ __forceinline__ float sn_axpby(float a, float x, float b, float c, bool use_c) {
  return use_c ? a * x + b * c : a * x;
}
__device__ __forceinline__ int32_t sn_axpby(int32_t a, int32_t x, int32_t b, int32_t c,
                                            bool use_c) {
  uint32_t r = static_cast<uint32_t>(a) * static_cast<uint32_t>(x);
  if (use_c) r += static_cast<uint32_t>(b) * static_cast<uint32_t>(c);
  return static_cast<int32_t>(r);
}

template <typename In>
struct SnArgs {
  using Acc = typename SnType<In>::Acc;
  int M, N, K;
  Acc alpha, beta;
  const In *A;
  int64_t lda;
  const In *B;
  int64_t ldb;
  Acc *C;
  int64_t ldc;
  int b_vec;  // B 16-byte aligned (fp32) / 4-byte aligned (int8), row stride a multiple of 4
};

// One lane's k-slice of kRows rows (kVec values of A each, packed in a[r])
// times the same k-slice of every staged column of B, each column's slice read
// once for all rows: acc[r][n] += sum_k a_rk * B[k][n].
template <typename In, int NP>
__device__ __forceinline__ void sn_step(const uint4 (&a)[kRows],
                                        const typename SnType<In>::Bt *bt, int kk,
                                        typename SnType<In>::Acc (&acc)[kRows][NP]) {
  constexpr int S = SnShape<In, NP>::S;
  if constexpr (std::is_same<In, int8_t>::value) {
#pragma unroll
    for (int n = 0; n < NP; ++n) {
      const int4 b = *reinterpret_cast<const int4 *>(bt + n * S + kk);
#pragma unroll
      for (int r = 0; r < kRows; ++r) {
        acc[r][n] = __dp4a(static_cast<int>(a[r].x), b.x, acc[r][n]);
        acc[r][n] = __dp4a(static_cast<int>(a[r].y), b.y, acc[r][n]);
        acc[r][n] = __dp4a(static_cast<int>(a[r].z), b.z, acc[r][n]);
        acc[r][n] = __dp4a(static_cast<int>(a[r].w), b.w, acc[r][n]);
      }
    }
  } else if constexpr (std::is_same<In, float>::value) {
#pragma unroll
    for (int n = 0; n < NP; ++n) {
      const float4 b = *reinterpret_cast<const float4 *>(bt + n * S + kk);
#pragma unroll
      for (int r = 0; r < kRows; ++r) {
        acc[r][n] = fmaf(__uint_as_float(a[r].x), b.x, acc[r][n]);
        acc[r][n] = fmaf(__uint_as_float(a[r].y), b.y, acc[r][n]);
        acc[r][n] = fmaf(__uint_as_float(a[r].z), b.z, acc[r][n]);
        acc[r][n] = fmaf(__uint_as_float(a[r].w), b.w, acc[r][n]);
      }
    }
  } else {
    float x[kRows][8];
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
      const In *h = reinterpret_cast<const In *>(&a[r]);
#pragma unroll
      for (int j = 0; j < 8; ++j) x[r][j] = to_float(h[j]);
    }
#pragma unroll
    for (int n = 0; n < NP; ++n) {
      const float4 b0 = *reinterpret_cast<const float4 *>(bt + n * S + kk);
      const float4 b1 = *reinterpret_cast<const float4 *>(bt + n * S + kk + 4);
#pragma unroll
      for (int r = 0; r < kRows; ++r) {
        acc[r][n] = fmaf(x[r][0], b0.x, acc[r][n]);
        acc[r][n] = fmaf(x[r][1], b0.y, acc[r][n]);
        acc[r][n] = fmaf(x[r][2], b0.z, acc[r][n]);
        acc[r][n] = fmaf(x[r][3], b0.w, acc[r][n]);
        acc[r][n] = fmaf(x[r][4], b1.x, acc[r][n]);
        acc[r][n] = fmaf(x[r][5], b1.y, acc[r][n]);
        acc[r][n] = fmaf(x[r][6], b1.z, acc[r][n]);
        acc[r][n] = fmaf(x[r][7], b1.w, acc[r][n]);
      }
    }
  }
}

// kVec values of row `row` of A from k = gk: one 16-byte load when they are
// all inside the matrix, element loads with zeros beyond K otherwise.
template <typename In>
__device__ __forceinline__ uint4 sn_load_a(const SnArgs<In> &p, int row, int gk) {
  constexpr int V = SnType<In>::kVec;
  const In *src = p.A + static_cast<int64_t>(row) * p.lda + gk;
  if (gk + V <= p.K) return __ldcs(reinterpret_cast<const uint4 *>(src));
  uint4 out = make_uint4(0u, 0u, 0u, 0u);
  In *o = reinterpret_cast<In *>(&out);
#pragma unroll
  for (int j = 0; j < V; ++j)
    if (gk + j < p.K) o[j] = src[j];
  return out;
}

// 16 bytes of A, read once (evict-first); volatile so that a group of these
// stays together ahead of the arithmetic that uses them.
__device__ __forceinline__ uint4 ld_stream_v4(const void *src) {
  uint4 v;
  asm volatile("ld.global.cs.v4.u32 {%0, %1, %2, %3}, [%4];\n"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(src));
  return v;
}

__device__ __forceinline__ float sn_add(float a, float b) { return a + b; }
__device__ __forceinline__ int32_t sn_add(int32_t a, int32_t b) {
  return static_cast<int32_t>(static_cast<uint32_t>(a) + static_cast<uint32_t>(b));
}

// Staging of one chunk of B[kc0 .. kc0 + KC) x NP into bt (transposed: bt[n *
// S + k] = B[kc0 + k][n], zeros beyond K and N). Every load of the chunk is
// issued before the first store, so staging a chunk costs one round trip to
// L2. Three forms: element by element (any B); fp32 with 16-byte loads of 4
// columns (b_vec); int8 in blocks of 4 rows x 4 columns, one 4-byte load per
// row and a byte transpose into 4 words of 4 consecutive k of one column
// (b_vec).
template <typename In, int NP>
__device__ __forceinline__ void sn_stage_b(const SnArgs<In> &p, int kc0,
                                           typename SnType<In>::Bt *bt) {
  using T = SnType<In>;
  using Bt = typename T::Bt;
  constexpr int S = SnShape<In, NP>::S;
  constexpr int KC = SnShape<In, NP>::KC;
  const int tid = static_cast<int>(threadIdx.x);
  if constexpr (std::is_same<In, float>::value && NP >= 4) {
    if (p.b_vec) {
      constexpr int kQ = NP / 4;  // 4-column groups per row of B
      constexpr int kIt = KC * kQ / kSnThreads;
      constexpr int kRound = kIt < 4 ? kIt : 4;  // 16-byte loads in flight per thread
      static_assert(kIt * kSnThreads == KC * kQ && kIt % kRound == 0,
                    "whole 4-column groups per thread");
#pragma unroll 1
      for (int u0 = 0; u0 < kIt; u0 += kRound) {
        float4 v[kRound];
#pragma unroll
        for (int u = 0; u < kRound; ++u) {
          const int idx = (u0 + u) * kSnThreads + tid;
          const int gk = kc0 + idx / kQ, n0 = (idx % kQ) * 4;
          v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (gk < p.K && n0 < p.N) {
            const float *src = p.B + static_cast<int64_t>(gk) * p.ldb + n0;
            if (n0 + 4 <= p.N) {
              v[u] = *reinterpret_cast<const float4 *>(src);
            } else {  // the last columns of a row: nothing past its end is read
              v[u].x = src[0];
              if (n0 + 1 < p.N) v[u].y = src[1];
              if (n0 + 2 < p.N) v[u].z = src[2];
            }
          }
        }
#pragma unroll
        for (int u = 0; u < kRound; ++u) {
          const int idx = (u0 + u) * kSnThreads + tid;
          const int k = idx / kQ, n0 = (idx % kQ) * 4;
          bt[(n0 + 0) * S + k] = v[u].x;
          bt[(n0 + 1) * S + k] = v[u].y;
          bt[(n0 + 2) * S + k] = v[u].z;
          bt[(n0 + 3) * S + k] = v[u].w;
        }
      }
      return;
    }
  }
  if constexpr (T::kInt && NP >= 4) {
    if (p.b_vec) {
      constexpr int kQ = NP / 4;  // 4-column groups per row of B
      constexpr int kIt = KC / 4 * kQ / kSnThreads;  // 4 x 4 blocks per thread
      static_assert(kIt * kSnThreads == KC / 4 * kQ, "whole 4 x 4 blocks per thread");
      uint32_t w[kIt][4];
#pragma unroll
      for (int u = 0; u < kIt; ++u) {
        const int idx = u * kSnThreads + tid;
        const int gk = kc0 + (idx / kQ) * 4, n0 = (idx % kQ) * 4;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          w[u][r] = 0u;
          if (gk + r < p.K && n0 < p.N) {
            const int8_t *src = p.B + static_cast<int64_t>(gk + r) * p.ldb + n0;
            if (n0 + 4 <= p.N) {
              w[u][r] = *reinterpret_cast<const uint32_t *>(src);
            } else {  // the last columns of a row: nothing past its end is read
              uint32_t x = static_cast<uint8_t>(src[0]);
              if (n0 + 1 < p.N) x |= static_cast<uint32_t>(static_cast<uint8_t>(src[1])) << 8;
              if (n0 + 2 < p.N) x |= static_cast<uint32_t>(static_cast<uint8_t>(src[2])) << 16;
              w[u][r] = x;
            }
          }
        }
      }
#pragma unroll
      for (int u = 0; u < kIt; ++u) {
        const int idx = u * kSnThreads + tid;
        const int k = (idx / kQ) * 4, n0 = (idx % kQ) * 4;
        // w[r] holds columns n0 .. n0+3 of row k + r; o[j] gets column n0 + j
        // of rows k .. k+3 (byte r = row k + r).
        const uint32_t t0 = __byte_perm(w[u][0], w[u][1], 0x5140);
        const uint32_t t1 = __byte_perm(w[u][0], w[u][1], 0x7362);
        const uint32_t t2 = __byte_perm(w[u][2], w[u][3], 0x5140);
        const uint32_t t3 = __byte_perm(w[u][2], w[u][3], 0x7362);
        *reinterpret_cast<uint32_t *>(bt + (n0 + 0) * S + k) = __byte_perm(t0, t2, 0x5410);
        *reinterpret_cast<uint32_t *>(bt + (n0 + 1) * S + k) = __byte_perm(t0, t2, 0x7632);
        *reinterpret_cast<uint32_t *>(bt + (n0 + 2) * S + k) = __byte_perm(t1, t3, 0x5410);
        *reinterpret_cast<uint32_t *>(bt + (n0 + 3) * S + k) = __byte_perm(t1, t3, 0x7632);
      }
      return;
    }
  }
  // Element by element, at most 16 values in flight per thread (the 64
  // accumulators of 16 columns leave no room for more).
  constexpr int kIters = KC * NP / kSnThreads;
  constexpr int kRound = kIters < 16 ? kIters : 16;
  static_assert(kIters * kSnThreads == KC * NP && kIters % kRound == 0, "staged values per thread");
#pragma unroll 1
  for (int u0 = 0; u0 < kIters; u0 += kRound) {
    Bt v[kRound];
#pragma unroll
    for (int u = 0; u < kRound; ++u) {
      const int idx = (u0 + u) * kSnThreads + tid;
      const int gk = kc0 + idx / NP, n = idx % NP;
      v[u] = Bt(0);
      if (gk < p.K && n < p.N) {
        if constexpr (T::kInt) {
          v[u] = p.B[static_cast<int64_t>(gk) * p.ldb + n];
        } else {
          v[u] = to_float(p.B[static_cast<int64_t>(gk) * p.ldb + n]);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kRound; ++u) {
      const int idx = (u0 + u) * kSnThreads + tid;
      bt[(idx % NP) * S + idx / NP] = v[u];
    }
  }
}

// NP: N rounded up to 1, 2, 4, 8 or 16 (every per-column loop runs NP times).
template <typename In, int NP>
__global__ void __launch_bounds__(kSnThreads, 2)
    gemm_small_n_kernel(const SnArgs<In> p) {
  using T = SnType<In>;
  using Acc = typename T::Acc;
  using Bt = typename T::Bt;
  using Sh = SnShape<In, NP>;
  constexpr int S = Sh::S;
  constexpr int KC = Sh::KC;
  constexpr int V = T::kVec;
  __shared__ __align__(16) Bt bt[NP * S];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int row0 = static_cast<int>(blockIdx.x) * kSnRowsPerCta + warp * kRows;

  // Launched as a programmatic dependent of the previous kernel on the
  // stream: nothing in global memory is read before it has completed.
  grid_dependency_wait();
  grid_launch_dependents();

  Acc acc[kRows][NP];
#pragma unroll
  for (int r = 0; r < kRows; ++r)
#pragma unroll
    for (int n = 0; n < NP; ++n) acc[r][n] = Acc(0);

  for (int kc0 = 0; kc0 < p.K; kc0 += KC) {
    sn_stage_b<In, NP>(p, kc0, bt);
    __syncthreads();
    // kG steps of 32 * kVec values of k at a time: all their loads of A are
    // issued before the first multiply, so kG * kRows 16-byte loads per lane
    // are in flight.
    constexpr int kSteps = Sh::kSteps;
    constexpr int kG = Sh::G;
    const bool rows_full = row0 + kRows <= p.M;  // the same for the whole warp
#pragma unroll 1
    for (int s0 = 0; s0 < kSteps; s0 += kG) {
      uint4 a[kG][kRows];
      if (rows_full && kc0 + (s0 + kG) * 32 * V <= p.K) {
        // Every load of the group is inside A: no guards, all issued at once.
        const In *base = p.A + static_cast<int64_t>(row0) * p.lda + kc0 + s0 * 32 * V + lane * V;
#pragma unroll
        for (int u = 0; u < kG; ++u)
#pragma unroll
          for (int r = 0; r < kRows; ++r)
            a[u][r] = ld_stream_v4(base + static_cast<int64_t>(r) * p.lda + u * 32 * V);
      } else {
#pragma unroll
        for (int u = 0; u < kG; ++u) {
          const int gk = kc0 + (s0 + u) * 32 * V + lane * V;
#pragma unroll
          for (int r = 0; r < kRows; ++r)
            a[u][r] = (gk < p.K && row0 + r < p.M) ? sn_load_a<In>(p, row0 + r, gk)
                                                    : make_uint4(0u, 0u, 0u, 0u);
        }
      }
#pragma unroll
      for (int u = 0; u < kG; ++u) sn_step<In, NP>(a[u], bt, (s0 + u) * 32 * V + lane * V, acc);
    }
    __syncthreads();  // the next chunk overwrites bt
  }

  // The lanes' partial sums: one fixed butterfly per element, after which
  // every lane holds every total; lane (r * NP + n) mod 32 writes element
  // (r, n) (one element per lane up to 8 columns, two for 16).
#pragma unroll
  for (int r = 0; r < kRows; ++r)
#pragma unroll
    for (int n = 0; n < NP; ++n)
#pragma unroll
      for (int off = 16; off > 0; off >>= 1)
        acc[r][n] = sn_add(acc[r][n], __shfl_xor_sync(0xffffffffu, acc[r][n], off));
  const bool use_c = p.beta != Acc(0);
#pragma unroll
  for (int r = 0; r < kRows; ++r)
#pragma unroll
    for (int n = 0; n < NP; ++n)
      if (lane == ((r * NP + n) & 31) && row0 + r < p.M && n < p.N) {
        Acc *cp = p.C + static_cast<int64_t>(row0 + r) * p.ldc + n;
        *cp = sn_axpby(p.alpha, acc[r][n], p.beta, use_c ? *cp : Acc(0), use_c);
      }
}
static_assert(kRows * kMaxNP <= 64, "at most two output elements per lane");
static_assert(SnShape<float, 16>::KC % (32 * 4) == 0 && SnShape<int8_t, 16>::KC % (32 * 16) == 0 &&
                  SnShape<__nv_bfloat16, 2>::KC % (32 * 8) == 0,
              "whole steps of every element type in a chunk");
static_assert(SnShape<float, 16>::kSteps % SnShape<float, 16>::G == 0 &&
                  SnShape<float, 8>::kSteps % SnShape<float, 8>::G == 0 &&
                  SnShape<int8_t, 16>::kSteps % SnShape<int8_t, 16>::G == 0 &&
                  SnShape<int8_t, 1>::kSteps % SnShape<int8_t, 1>::G == 0,
              "whole groups of steps in a chunk");
static_assert(SnShape<float, 16>::S * 16 * 4 <= 48 * 1024, "staged B within static shared memory");

template <typename In, int NP>
cudaError_t sn_launch(const SnArgs<In> &p, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((p.M + kSnRowsPerCta - 1) / kSnRowsPerCta), 1, 1);
  cfg.blockDim = dim3(kSnThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, gemm_small_n_kernel<In, NP>, p);
  return e == cudaSuccess ? cudaGetLastError() : e;
}

template <typename In>
cudaError_t sn_dispatch(int M, int N, int K, typename SnType<In>::Acc alpha, const In *A,
                        int64_t lda, const In *B, int64_t ldb, typename SnType<In>::Acc beta,
                        typename SnType<In>::Acc *C, int64_t ldc, cudaStream_t stream) {
  if (M < 1 || N < 1 || N > kMaxNP || K < 1) return cudaErrorInvalidValue;
  if (static_cast<int64_t>(M) + kSnRowsPerCta > 0x7fffffffLL) return cudaErrorInvalidValue;
  SnArgs<In> p;
  p.M = M;
  p.N = N;
  p.K = K;
  p.alpha = alpha;
  p.beta = beta;
  p.A = A;
  p.lda = lda;
  p.B = B;
  p.ldb = ldb;
  p.C = C;
  p.ldc = ldc;
  p.b_vec = (sizeof(In) == 4 && reinterpret_cast<uintptr_t>(B) % 16 == 0 && ldb % 4 == 0) ||
            (sizeof(In) == 1 && reinterpret_cast<uintptr_t>(B) % 4 == 0 && ldb % 4 == 0);
  if (N <= 1) return sn_launch<In, 1>(p, stream);
  if (N <= 2) return sn_launch<In, 2>(p, stream);
  if constexpr (sizeof(In) == 2) {
    return cudaErrorInvalidValue;  // 16-bit inputs: up to 2 columns here
  } else {
    if (N <= 4) return sn_launch<In, 4>(p, stream);
    if (N <= 8) return sn_launch<In, 8>(p, stream);
    return sn_launch<In, 16>(p, stream);
  }
}

}  // namespace

bool small_n_supported(int M, int N, const void *A, int64_t lda, int esize) {
  // 16-bit inputs: up to 2 columns. Measured on GB300 at M = K = 8192 (bf16):
  // N = 1 / 2 / 4 / 8 in 26.9 / 27.4 / 38.4 / 62.5 us here, about 38 us on the
  // tiled tensor-core kernel: from 4 columns the fp32 arithmetic per 16-bit
  // element of A catches up with the stream.
  const int max_n = esize == 2 ? 2 : kMaxNP;
  return N >= 1 && N <= max_n && M >= kSmallNMinM && reinterpret_cast<uintptr_t>(A) % 16 == 0 &&
         (lda * esize) % 16 == 0;
}

cudaError_t launch_small_n_f32(int M, int N, int K, float alpha, const float *A, int64_t lda,
                               const float *B, int64_t ldb, float beta, float *C, int64_t ldc,
                               cudaStream_t stream) {
  return sn_dispatch<float>(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream);
}

cudaError_t launch_small_n_half(bool is_bf16, int M, int N, int K, float alpha, const void *A,
                                int64_t lda, const void *B, int64_t ldb, float beta, float *C,
                                int64_t ldc, cudaStream_t stream) {
  if (is_bf16)
    return sn_dispatch<__nv_bfloat16>(M, N, K, alpha, static_cast<const __nv_bfloat16 *>(A), lda,
                                      static_cast<const __nv_bfloat16 *>(B), ldb, beta, C, ldc,
                                      stream);
  return sn_dispatch<__half>(M, N, K, alpha, static_cast<const __half *>(A), lda,
                             static_cast<const __half *>(B), ldb, beta, C, ldc, stream);
}

cudaError_t launch_small_n_s8(int M, int N, int K, int32_t alpha, const int8_t *A, int64_t lda,
                              const int8_t *B, int64_t ldb, int32_t beta, int32_t *C, int64_t ldc,
                              cudaStream_t stream) {
  return sn_dispatch<int8_t>(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream);
}

}  // namespace dgr
