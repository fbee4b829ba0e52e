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
// stride lds), through 64 x 64 tiles in shared memory (row stride 65: the
// column reads of the write phase fall in distinct banks). Each of the 256
// threads moves 16 values per phase: 16-byte loads along src rows when the
// source allows them (vec_src) and 16-byte stores along dst rows when dst
// does (vec_dst), element accesses otherwise. Blocks walk the tiles
// grid-stride.
__global__ void __launch_bounds__(256)
    transpose_f32_kernel(const float *__restrict__ src, int64_t lds, float *__restrict__ dst,
                         int64_t ldd, int rows, int cols, int vec_src, int vec_dst) {
  __shared__ float tile[64][65];
  const int tid = threadIdx.x;
  const int64_t tiles_c = (cols + 63) / 64;
  const int64_t tiles = (static_cast<int64_t>(rows) + 63) / 64 * tiles_c;
  for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
    const int64_t r0 = t / tiles_c * 64, c0 = t % tiles_c * 64;
    // Read phase: 64 rows x 16 chunks of 4 columns; thread -> (row, chunk).
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e = tid + 256 * i;
      const int r = e >> 4, q = (e & 15) * 4;
      const int64_t gr = r0 + r, gc = c0 + q;
      float v[4];
      if (vec_src && gr < rows && gc + 3 < cols) {
        const float4 f = *reinterpret_cast<const float4 *>(src + gr * lds + gc);
        v[0] = f.x, v[1] = f.y, v[2] = f.z, v[3] = f.w;
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) v[j] = (gr < rows && gc + j < cols) ? src[gr * lds + gc + j] : 0.f;
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) tile[r][q + j] = v[j];
    }
    __syncthreads();
    // Write phase: dst rows c0 .. c0+63 (src columns), 16 chunks of 4 src rows.
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e = tid + 256 * i;
      const int c = e >> 4, q = (e & 15) * 4;
      const int64_t gc = c0 + c, gr = r0 + q;  // dst row gc, columns gr .. gr+3
      if (gc >= cols) continue;
      const float v0 = tile[q][c], v1 = tile[q + 1][c], v2 = tile[q + 2][c], v3 = tile[q + 3][c];
      if (vec_dst && gr + 3 < rows) {
        *reinterpret_cast<float4 *>(dst + gc * ldd + gr) = make_float4(v0, v1, v2, v3);
      } else {
        const float v[4] = {v0, v1, v2, v3};
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (gr + j < rows) dst[gc * ldd + gr + j] = v[j];
      }
    }
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_transpose_f32(const DeviceInfo &dev, const float *src, int64_t lds, int rows,
                                 int cols, float *dst, int64_t ldd, cudaStream_t stream) {
  const int64_t tiles = (static_cast<int64_t>(rows) + 63) / 64 * ((cols + 63) / 64);
  const int64_t blocks = tiles < static_cast<int64_t>(dev.sm_count) * 8 ? tiles : dev.sm_count * 8;
  const int vec_src = (reinterpret_cast<uintptr_t>(src) % 16 == 0) && (lds % 4 == 0);
  const int vec_dst = (reinterpret_cast<uintptr_t>(dst) % 16 == 0) && (ldd % 4 == 0);
  if (blocks < 1) return cudaSuccess;
  transpose_f32_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(src, lds, dst, ldd, rows,
                                                                         cols, vec_src, vec_dst);
  return cudaGetLastError();
}

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
  if (e == cudaSuccess) e = launch_transpose_f32(dev, B, ldb, K, N, bt, ldk, stream);
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
