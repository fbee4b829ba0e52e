// gemm_tc_int.cu -- exact 8-bit integer GEMM on the fp16 tensor pipe (int8 and
// uint8 inputs, int32 C with wrap-around): each operand is widened to fp16 in
// stream-ordered scratch memory (exact), then the tensor-core kernel
// (gemm_tc_kernel.cuh) runs in exact-integer mode, restarting its fp32
// accumulator every 1024 values of k so that every partial sum is an integer
// of at most 2^24 in magnitude.
//
// uint8 runs on the same int8 kernel: with a = sa + 128 and b = sb + 128
// (sa, sb in [-128, 127], exact in fp16 and the int8 kernel's range),
//     sum_k a_ik b_kj = sum_k sa_ik sb_kj + 128 rowsum(A)_i + 128 colsum(B)_j
//                       - 16384 K,
// so the operands are widened as x - 128 and the epilogue adds
// row_corr[i] + col_corr[j] + corr_const with row_corr[i] = 128 rowsum(A)_i,
// col_corr[j] = 128 colsum(B)_j and corr_const = -16384 K (all modulo 2^32,
// like the result). A direct uint8 kernel would need
// 256-value chunks (256 * 255^2 < 2^24 < 1024 * 255^2), four times as many
// accumulator hand-offs to the epilogue.
#include "gemm_tc_kernel.cuh"

namespace dgr {
namespace {

// 8-bit -> fp16, exact, for a stack of `count` rows x cols matrices (source
// matrix stride src_stride; destination matrices packed at rows * ldd). dst has
// row stride ldd (multiple of 8) and its padding columns [cols, ldd) are
// written with zeros. Each thread widens 16 consecutive elements of a row: one
// 16-byte load when the source row is 16-byte aligned and the chunk is inside
// the matrix, byte loads otherwise, and one or two 16-byte stores.
// kOffset: uint8 values are stored as x - 128.
template <typename T8, int kOffset = 0>
__global__ void widen8_kernel(const T8 *__restrict__ src, int64_t lds, int64_t src_stride,
                              __half *dst, int64_t ldd, int rows, int cols, int count,
                              int vec_ok) {
  const int64_t chunks_per_row = (ldd + 15) / 16;
  const int64_t total = static_cast<int64_t>(rows) * count * chunks_per_row;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = i / chunks_per_row;  // row of the whole stack
    const int c0 = static_cast<int>((i - r * chunks_per_row) * 16);
    const int64_t m = r / rows;            // matrix of the stack
    const T8 *s = src + m * src_stride + (r - m * rows) * lds;
    __align__(16) __half h[16];
    if (vec_ok && c0 + 16 <= cols) {
      const int4 v = *reinterpret_cast<const int4 *>(s + c0);
      const int w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 16; ++j)
        h[j] = __int2half_rn(
            static_cast<int>(static_cast<T8>(static_cast<uint32_t>(w[j >> 2]) >> (8 * (j & 3)))) -
            kOffset);
    } else {
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int c = c0 + j;
        h[j] = __int2half_rn(c < cols ? static_cast<int>(s[c]) - kOffset : 0);
      }
    }
    uint4 *d = reinterpret_cast<uint4 *>(dst + r * ldd + c0);
    d[0] = *reinterpret_cast<const uint4 *>(h);
    if (c0 + 16 <= ldd) d[1] = *reinterpret_cast<const uint4 *>(h + 8);
  }
}

template <typename T8, int kOffset = 0>
cudaError_t widen8(const DeviceInfo &dev, const T8 *src, int64_t lds, __half *dst, int64_t ldd,
                   int rows, int cols, cudaStream_t stream, int count = 1,
                   int64_t src_stride = 0) {
  const int64_t total = static_cast<int64_t>(rows) * count * ((ldd + 15) / 16);
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  const int64_t cap = static_cast<int64_t>(dev.sm_count) * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  const int vec_ok = (reinterpret_cast<uintptr_t>(src) % 16 == 0) && (lds % 16 == 0) &&
                     (count == 1 || src_stride % 16 == 0);
  widen8_kernel<T8, kOffset><<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
      src, lds, src_stride, dst, ldd, rows, cols, count, vec_ok);
  return cudaGetLastError();
}

// Both operands of one GEMM in a single launch (one grid-stride loop over A's
// chunks, then B's), which also zeroes `nflags` words of split-k tail flags
// for the tensor-core kernel that follows; it lets that kernel start as a
// programmatic dependent once every thread here is done.
struct WidenJob {
  const void *src;
  int64_t lds, src_stride;
  __half *dst;
  int64_t ldd;
  int rows, cols, count;
  int vec_ok;
};
template <typename T8, int kOffset = 0>
__device__ __forceinline__ void widen_chunk(const WidenJob &j, int64_t i) {
  const int64_t chunks_per_row = (j.ldd + 15) / 16;
  const int64_t r = i / chunks_per_row;
  const int c0 = static_cast<int>((i - r * chunks_per_row) * 16);
  const int64_t m = r / j.rows;
  const T8 *s = static_cast<const T8 *>(j.src) + m * j.src_stride + (r - m * j.rows) * j.lds;
  __align__(16) __half h[16];
  if (j.vec_ok && c0 + 16 <= j.cols) {
    const int4 v = *reinterpret_cast<const int4 *>(s + c0);
    const int w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 16; ++q)
      h[q] = __int2half_rn(
          static_cast<int>(static_cast<T8>(static_cast<uint32_t>(w[q >> 2]) >> (8 * (q & 3)))) -
          kOffset);
  } else {
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      const int c = c0 + q;
      h[q] = __int2half_rn(c < j.cols ? static_cast<int>(s[c]) - kOffset : 0);
    }
  }
  uint4 *d = reinterpret_cast<uint4 *>(j.dst + r * j.ldd + c0);
  d[0] = *reinterpret_cast<const uint4 *>(h);
  if (c0 + 16 <= j.ldd) d[1] = *reinterpret_cast<const uint4 *>(h + 8);
}
template <typename T8>
__global__ void widen8x2_kernel(WidenJob a, WidenJob b, uint32_t *flags, int nflags) {
  const int64_t tid = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = tid; i < nflags; i += step) flags[i] = 0;
  const int64_t ta = static_cast<int64_t>(a.rows) * a.count * ((a.ldd + 15) / 16);
  const int64_t tb = static_cast<int64_t>(b.rows) * b.count * ((b.ldd + 15) / 16);
  for (int64_t i = tid; i < ta + tb; i += step) {
    if (i < ta) {
      widen_chunk<T8>(a, i);
    } else {
      widen_chunk<T8>(b, i - ta);
    }
  }
  grid_launch_dependents();
}

template <typename T8>
cudaError_t widen8x2(const DeviceInfo &dev, const WidenJob &a, const WidenJob &b,
                     uint32_t *flags, int nflags, cudaStream_t stream) {
  const int64_t total = static_cast<int64_t>(a.rows) * a.count * ((a.ldd + 15) / 16) +
                        static_cast<int64_t>(b.rows) * b.count * ((b.ldd + 15) / 16);
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  const int64_t cap = static_cast<int64_t>(dev.sm_count) * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  widen8x2_kernel<T8><<<static_cast<unsigned>(blocks), threads, 0, stream>>>(a, b, flags, nflags);
  return cudaGetLastError();
}

// The widened operands of an 8-bit GEMM in one scratch block: A's copies at
// offset 0, B's at b_off (256-byte aligned); each copy packed (row stride
// rounded up to 8 values, matrices back to back).
struct WideLayout {
  int a_rows, a_cols, b_rows, b_cols;  // stored shapes
  int na, nb;                          // matrices widened per operand
  int64_t lda16, ldb16, a_mat, b_mat;  // row and matrix strides of the copies (elements)
  size_t b_off, total;                 // bytes

  WideLayout(const BatchOps &ops, int M, int N, int K) {
    a_rows = ops.a_t ? K : M;
    a_cols = ops.a_t ? M : K;
    b_rows = ops.b_t ? N : K;
    b_cols = ops.b_t ? K : N;
    na = (ops.batch > 1 && ops.stride_a != 0) ? ops.batch : 1;
    nb = (ops.batch > 1 && ops.stride_b != 0) ? ops.batch : 1;
    lda16 = (static_cast<int64_t>(a_cols) + 7) / 8 * 8;
    ldb16 = (static_cast<int64_t>(b_cols) + 7) / 8 * 8;
    a_mat = a_rows * lda16;
    b_mat = b_rows * ldb16;
    b_off = (static_cast<size_t>(na) * a_mat * 2 + 255) / 256 * 256;
    total = b_off + static_cast<size_t>(nb) * b_mat * 2;
  }
};

// Widens A and B into `scratch` and runs the exact-integer kernel of kind
// kKind (kAllForms: built with every operand form).
template <int kKind, bool kAllForms, typename T8>
cudaError_t run_int(const DeviceInfo &dev, const BatchOps &ops, int M, int N, int K,
                    int32_t alpha, const T8 *A, int64_t lda, const T8 *B, int64_t ldb,
                    int32_t beta, int32_t *C, int64_t ldc, void *scratch, uint32_t *flags,
                    size_t flags_words, cudaStream_t stream, bool caller_flags) {
  const WideLayout w(ops, M, N, K);
  __half *a16 = static_cast<__half *>(scratch);
  __half *b16 = reinterpret_cast<__half *>(static_cast<uint8_t *>(scratch) + w.b_off);
  auto job = [](const T8 *src, int64_t ld, int64_t stride, __half *dst, int64_t ldd, int rows,
                int cols, int count) {
    WidenJob j;
    j.src = src;
    j.lds = ld;
    j.src_stride = stride;
    j.dst = dst;
    j.ldd = ldd;
    j.rows = rows;
    j.cols = cols;
    j.count = count;
    j.vec_ok = (reinterpret_cast<uintptr_t>(src) % 16 == 0) && (ld % 16 == 0) &&
               (count == 1 || stride % 16 == 0);
    return j;
  };
  // The flags for the tensor-core kernel's split-k tail are zeroed by the
  // same launch (at most kTailFlagWords of them are ever used).
  const int nflags = flags != nullptr ? static_cast<int>(flags_words < kTailFlagWords
                                                             ? flags_words
                                                             : kTailFlagWords)
                                      : 0;
  cudaError_t e = widen8x2<T8>(dev,
                               job(A, lda, ops.stride_a, a16, w.lda16, w.a_rows, w.a_cols, w.na),
                               job(B, ldb, ops.stride_b, b16, w.ldb16, w.b_rows, w.b_cols, w.nb),
                               flags, nflags, stream);
  if (e != cudaSuccess) return e;
  // Short, wide int8 problems: the transposed-role kernel (1024-k chunks).
  if (kKind == kKindS8 && tc_skinny_route(M, N, dev.sm_count) && ops.plain())
    return launch_tc_skinny_int(dev, M, N, K, alpha, a16, w.lda16, b16, w.ldb16, beta, C, ldc,
                                stream, caller_flags ? flags : nullptr, flags_words);
  BatchOps wide = ops;
  wide.stride_a = w.na > 1 ? w.a_mat : 0;
  wide.stride_b = w.nb > 1 ? w.b_mat : 0;
  return launch_tc<kKind, kAllForms>(dev, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, kFmtF16,
                                     CU_TENSOR_MAP_DATA_TYPE_FLOAT16, wide, M, N, K, alpha, a16,
                                     w.lda16, b16, w.ldb16, beta, C, ldc, stream, flags,
                                     static_cast<size_t>(nflags), nullptr, nullptr, 0,
                                     /*flags_zeroed=*/true);
}

// The same on scratch drawn from the library's stream-ordered pool and
// returned to it on the same stream.
template <int kKind, bool kAllForms, typename T8>
cudaError_t run_int_pooled(const DeviceInfo &dev, const BatchOps &ops, int M, int N, int K,
                           int32_t alpha, const T8 *A, int64_t lda, const T8 *B, int64_t ldb,
                           int32_t beta, int32_t *C, int64_t ldc, cudaStream_t stream) {
  const WideLayout w(ops, M, N, K);
  cudaMemPool_t pool = nullptr;
  cudaError_t e = device_pool(dev, &pool);
  if (e != cudaSuccess) return e;
  void *scratch = nullptr;
  const size_t flags_off = (w.total + 255) / 256 * 256;
  e = cudaMallocFromPoolAsync(&scratch, flags_off + kTailFlagWords * 4, pool, stream);
  if (e != cudaSuccess) return e;
  uint32_t *flags =
      reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(scratch) + flags_off);
  e = run_int<kKind, kAllForms, T8>(dev, ops, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
                                    scratch, flags, kTailFlagWords, stream, false);
  cudaError_t f = cudaFreeAsync(scratch, stream);
  return e != cudaSuccess ? e : f;
}

}  // namespace

// Short, wide int8 GEMM with B read as stored: A (M x K, a few rows) is
// widened to fp16 in pool scratch; B goes straight to the transposed-role
// kernel, whose converter warps widen each tile in shared memory.
cudaError_t launch_gemm_s8_skinny_raw(const DeviceInfo &dev, int M, int N, int K, int32_t alpha,
                                      const int8_t *A, int64_t lda, const int8_t *B, int64_t ldb,
                                      int32_t beta, int32_t *C, int64_t ldc,
                                      cudaStream_t stream) {
  // A read as stored too when its rows are whole 16-byte units: one launch.
  if (tc_skinny_s8_supported(M, A, lda, B, ldb))
    return launch_tc_skinny_s8(dev, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream);
  const int64_t lda16 = (static_cast<int64_t>(K) + 7) / 8 * 8;
  cudaMemPool_t pool = nullptr;
  cudaError_t e = device_pool(dev, &pool);
  if (e != cudaSuccess) return e;
  void *scratch = nullptr;
  e = cudaMallocFromPoolAsync(&scratch, static_cast<size_t>(M) * lda16 * 2, pool, stream);
  if (e != cudaSuccess) return e;
  __half *a16 = static_cast<__half *>(scratch);
  e = widen8<int8_t>(dev, A, lda, a16, lda16, M, K, stream);
  if (e == cudaSuccess)
    e = launch_tc_skinny_i8(dev, M, N, K, alpha, a16, lda16, B, ldb, beta, C, ldc, stream);
  cudaError_t f = cudaFreeAsync(scratch, stream);
  return e != cudaSuccess ? e : f;
}

namespace {

// row_corr[i] = 128 * sum_k A[i, k] (mod 2^32): one warp per row, lanes along
// k, 16 bytes per lane per step when rows are 16-byte aligned (byte sums by
// dp4a against 0x01010101), a shuffle reduction at the end.
__global__ void u8_row_corr_kernel(const uint8_t *__restrict__ A, int64_t lda, int rows, int K,
                                   int vec, int32_t *row_corr) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t r = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5; r < rows;
       r += warps) {
    const uint8_t *row = A + r * lda;
    uint32_t s = 0;
    int k0 = 0;
    if (vec) {
      const int kv = K / 16 * 16;
      for (int k = lane * 16; k < kv; k += 32 * 16) {
        const uint4 w = *reinterpret_cast<const uint4 *>(row + k);
        s = __dp4a(w.x, 0x01010101u, s);
        s = __dp4a(w.y, 0x01010101u, s);
        s = __dp4a(w.z, 0x01010101u, s);
        s = __dp4a(w.w, 0x01010101u, s);
      }
      k0 = kv;
    }
    for (int k = k0 + lane; k < K; k += 32) s += row[k];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) row_corr[r] = static_cast<int32_t>(128u * s);
  }
}

// col_corr[j] += 128 * sum over this block's rows of B[k, j] (mod 2^32);
// col_corr starts at zero. A block covers 512 columns x kColRows rows: lane l
// of every warp owns columns 16 l .. 16 l + 15 (one 16-byte load per row when
// rows are 16-byte aligned, so a warp reads 512 contiguous bytes), warp w owns
// every 8th row of the block's range; the 8 warps' sums meet in shared memory
// and one atomic per column leaves the block.
constexpr int kColRows = 256;
__global__ void __launch_bounds__(256)
    u8_col_corr_kernel(const uint8_t *__restrict__ B, int64_t ldb, int K, int N, int vec,
                       int32_t *col_corr) {
  __shared__ uint32_t part[8][512];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t c0 = static_cast<int64_t>(blockIdx.x) * 512 + lane * 16;
  const int64_t k0 = static_cast<int64_t>(blockIdx.y) * kColRows;
  const int64_t k1 = k0 + kColRows < K ? k0 + kColRows : K;
  uint32_t s[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) s[j] = 0;
  if (vec && c0 + 15 < N) {
#pragma unroll 4
    for (int64_t k = k0 + warp; k < k1; k += 8) {
      const uint4 w = *reinterpret_cast<const uint4 *>(B + k * ldb + c0);
      const uint32_t q[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int j = 0; j < 16; ++j) s[j] += (q[j >> 2] >> (8 * (j & 3))) & 0xffu;
    }
  } else {
    for (int64_t k = k0 + warp; k < k1; k += 8)
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (c0 + j < N) s[j] += B[k * ldb + c0 + j];
  }
#pragma unroll
  for (int j = 0; j < 16; ++j) part[warp][lane * 16 + j] = s[j];
  __syncthreads();
  for (int c = threadIdx.x; c < 512; c += 256) {
    const int64_t col = static_cast<int64_t>(blockIdx.x) * 512 + c;
    if (col >= N) continue;
    uint32_t t = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) t += part[w][c];
    atomicAdd(reinterpret_cast<unsigned int *>(col_corr + col), 128u * t);
  }
}

}  // namespace

cudaError_t launch_gemm_s8(const DeviceInfo &dev, int M, int N, int K, int32_t alpha,
                           const int8_t *A, int64_t lda, const int8_t *B, int64_t ldb,
                           int32_t beta, int32_t *C, int64_t ldc, cudaStream_t stream) {
  return run_int_pooled<kKindS8, true, int8_t>(dev, BatchOps(), M, N, K, alpha, A, lda, B, ldb,
                                                beta, C, ldc, stream);
}

cudaError_t launch_gemm_s8_ex(const DeviceInfo &dev, const BatchOps &ops, int M, int N, int K,
                              int32_t alpha, const int8_t *A, int64_t lda, const int8_t *B,
                              int64_t ldb, int32_t beta, int32_t *C, int64_t ldc,
                              cudaStream_t stream) {
  return run_int_pooled<kKindS8, true, int8_t>(dev, ops, M, N, K, alpha, A, lda, B, ldb, beta, C,
                                                ldc, stream);
}

cudaError_t launch_gemm_u8(const DeviceInfo &dev, int M, int N, int K, int32_t alpha,
                           const uint8_t *A, int64_t lda, const uint8_t *B, int64_t ldb,
                           int32_t beta, int32_t *C, int64_t ldc, cudaStream_t stream) {
  const WideLayout w(BatchOps(), M, N, K);
  const size_t corr_off = (w.total + 255) / 256 * 256;
  const size_t total = corr_off + (static_cast<size_t>(M) + N) * 4;
  cudaMemPool_t pool = nullptr;
  cudaError_t e = device_pool(dev, &pool);
  if (e != cudaSuccess) return e;
  void *scratch = nullptr;
  e = cudaMallocFromPoolAsync(&scratch, total, pool, stream);
  if (e != cudaSuccess) return e;
  __half *a16 = static_cast<__half *>(scratch);
  __half *b16 = reinterpret_cast<__half *>(static_cast<uint8_t *>(scratch) + w.b_off);
  int32_t *row_corr = reinterpret_cast<int32_t *>(static_cast<uint8_t *>(scratch) + corr_off);
  int32_t *col_corr = row_corr + M;
  e = widen8<uint8_t, 128>(dev, A, lda, a16, w.lda16, M, K, stream);
  if (e == cudaSuccess) e = widen8<uint8_t, 128>(dev, B, ldb, b16, w.ldb16, K, N, stream);
  if (e == cudaSuccess) {
    int64_t blocks = (static_cast<int64_t>(M) * 32 + 255) / 256;
    if (blocks > dev.sm_count * 8) blocks = dev.sm_count * 8;
    const int vec = (reinterpret_cast<uintptr_t>(A) % 16 == 0) && (lda % 16 == 0);
    u8_row_corr_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(A, lda, M, K, vec,
                                                                          row_corr);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) e = cudaMemsetAsync(col_corr, 0, static_cast<size_t>(N) * 4, stream);
  if (e == cudaSuccess) {
    const int64_t gy = (static_cast<int64_t>(K) + kColRows - 1) / kColRows;
    if (gy > 65535) e = cudaErrorInvalidValue;  // K beyond 16.7 million
    const dim3 grid(static_cast<unsigned>((N + 511) / 512), static_cast<unsigned>(gy));
    const int vec = (reinterpret_cast<uintptr_t>(B) % 16 == 0) && (ldb % 16 == 0);
    if (e == cudaSuccess) {
      u8_col_corr_kernel<<<grid, 256, 0, stream>>>(B, ldb, K, N, vec, col_corr);
      e = cudaGetLastError();
    }
  }
  if (e == cudaSuccess)
    e = launch_tc<kKindS8, true>(dev, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, kFmtF16,
                                 CU_TENSOR_MAP_DATA_TYPE_FLOAT16, BatchOps(), M, N, K, alpha, a16,
                                 w.lda16, b16, w.ldb16, beta, C, ldc, stream, nullptr, 0,
                                 row_corr, col_corr, static_cast<int32_t>(0u - 16384u *
                                                                          static_cast<uint32_t>(K)));
  cudaError_t f = cudaFreeAsync(scratch, stream);
  return e != cudaSuccess ? e : f;
}

// The int8 path with scratch memory supplied by the caller instead of drawn
// from the library's pool: widen A and B into `scratch` (which must hold
// s8_scratch_bytes(M, N, K) bytes, 256-byte aligned) and run the tensor-core
// kernel in exact-integer mode. Allocates nothing.
size_t s8_scratch_bytes(int M, int N, int K) { return WideLayout(BatchOps(), M, N, K).total; }

cudaError_t launch_gemm_s8_scratch(const DeviceInfo &dev, int M, int N, int K, int32_t alpha,
                                   const int8_t *A, int64_t lda, const int8_t *B, int64_t ldb,
                                   int32_t beta, int32_t *C, int64_t ldc, void *scratch,
                                   uint32_t *flags, size_t flags_words, cudaStream_t stream) {
  return run_int<kKindS8, true, int8_t>(dev, BatchOps(), M, N, K, alpha, A, lda, B, ldb, beta, C,
                                         ldc, scratch, flags, flags_words, stream, true);
}

}  // namespace dgr
