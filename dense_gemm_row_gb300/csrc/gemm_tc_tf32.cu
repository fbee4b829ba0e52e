// gemm_tc_tf32.cu -- fp32 inputs used at tf32 precision on the tensor cores
// (tcgen05 kind::tf32; the warp-matrix-function type table's precision::tf32
// row: tf32 inputs, float accumulate), fp32 C. Opt-in: gemm_f32 stays exact
// fp32 on the SIMT pipe.
//
// Both operands are staged K-major, the layout every tcgen05 operand kind
// accepts: A (row-major M x K) is K-major as it stands; B (row-major K x N) is
// N-major, so a K-major copy (N x K) is made first by a shared-memory tiled
// transpose. A whose base or row stride is not in whole 16-byte units (which
// TMA needs) is first repacked into an aligned copy. The kernel is in
// gemm_tc_kernel.cuh.
#include "gemm_tc_kernel.cuh"

namespace dgr {
namespace {

// dst (cols x rows, row stride ldd) = transpose of src (rows x cols, row
// stride lds), through 32 x 32 tiles in shared memory (the extra column keeps
// the transposed reads free of bank conflicts). Reads and writes are both
// coalesced along rows. Blocks of 32 x 8 threads walk the tiles grid-stride.
__global__ void transpose_f32_kernel(const float *__restrict__ src, int64_t lds,
                                     float *__restrict__ dst, int64_t ldd, int rows, int cols) {
  __shared__ float tile[32][33];
  const int64_t tiles_c = (cols + 31) / 32;
  const int64_t tiles = (static_cast<int64_t>(rows) + 31) / 32 * tiles_c;
  for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
    const int64_t r0 = t / tiles_c * 32, c0 = t % tiles_c * 32;
    for (int i = threadIdx.y; i < 32; i += 8) {
      const int64_t r = r0 + i, c = c0 + threadIdx.x;
      if (r < rows && c < cols) tile[i][threadIdx.x] = src[r * lds + c];
    }
    __syncthreads();
    for (int i = threadIdx.y; i < 32; i += 8) {
      const int64_t c = c0 + i, r = r0 + threadIdx.x;  // dst row c, column r
      if (c < cols && r < rows) dst[c * ldd + r] = tile[threadIdx.x][i];
    }
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_gemm_tf32(const DeviceInfo &dev, int M, int N, int K, float alpha,
                             const float *A, int64_t lda, const float *B, int64_t ldb, float beta,
                             float *C, int64_t ldc, cudaStream_t stream) {
  const int64_t ldk = (static_cast<int64_t>(K) + 3) / 4 * 4;  // K-major copies: 16-byte rows
  const bool a_ok = (reinterpret_cast<uintptr_t>(A) % 16 == 0) && (lda % 4 == 0);
  const size_t bt_bytes = static_cast<size_t>(N) * ldk * 4;
  const size_t a_off = (bt_bytes + 255) / 256 * 256;
  const size_t total = a_off + (a_ok ? 0 : static_cast<size_t>(M) * ldk * 4);
  cudaMemPool_t pool = nullptr;
  cudaError_t e = device_pool(dev, &pool);
  if (e != cudaSuccess) return e;
  void *scratch = nullptr;
  e = cudaMallocFromPoolAsync(&scratch, total, pool, stream);
  if (e != cudaSuccess) return e;
  float *bt = static_cast<float *>(scratch);
  const float *a = A;
  int64_t lda_used = lda;
  if (!a_ok) {
    float *a_copy = reinterpret_cast<float *>(static_cast<uint8_t *>(scratch) + a_off);
    e = cudaMemcpy2DAsync(a_copy, ldk * 4, A, lda * 4, static_cast<size_t>(K) * 4, M,
                          cudaMemcpyDeviceToDevice, stream);
    a = a_copy;
    lda_used = ldk;
  }
  if (e == cudaSuccess) {
    const int64_t tiles = (static_cast<int64_t>(K) + 31) / 32 * ((N + 31) / 32);
    int64_t blocks = tiles < static_cast<int64_t>(dev.sm_count) * 16 ? tiles
                                                                      : dev.sm_count * 16;
    transpose_f32_kernel<<<static_cast<unsigned>(blocks), dim3(32, 8), 0, stream>>>(B, ldb, bt,
                                                                                   ldk, K, N);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) {
    BatchOps ops;
    ops.b_t = true;  // B is now the N x K copy
    e = launch_tc<kKindTF32, false>(dev, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, kFmtTF32,
                                    CU_TENSOR_MAP_DATA_TYPE_FLOAT32, ops, M, N, K, alpha, a,
                                    lda_used, bt, ldk, beta, C, ldc, stream, nullptr, 0);
  }
  cudaError_t f = cudaFreeAsync(scratch, stream);
  return e != cudaSuccess ? e : f;
}

}  // namespace dgr
