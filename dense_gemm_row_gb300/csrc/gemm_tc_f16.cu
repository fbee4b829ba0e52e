// gemm_tc_f16.cu -- bf16 / fp16 inputs, fp32 C on the tensor cores (every
// operand form and strided batches); the kernel is in gemm_tc_kernel.cuh.
#include "gemm_tc_kernel.cuh"

namespace dgr {

cudaError_t launch_gemm_tc_f16_ex(const DeviceInfo &dev, bool is_bf16, const BatchOps &ops, int M,
                                  int N, int K, float alpha, const void *A, int64_t lda,
                                  const void *B, int64_t ldb, float beta, float *C, int64_t ldc,
                                  cudaStream_t stream) {
  // Short, wide problems: the transposed-role kernel streams B at HBM speed
  // instead of multiplying a mostly-zero 256-row tile.
  if (tc_skinny_route(M, N, dev.sm_count) && ops.plain())
    return launch_tc_skinny_float(dev, is_bf16, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
                                  stream);
  const CUtensorMapDataType dt =
      is_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  return launch_tc<kKindF32, true>(dev, dt, is_bf16 ? kFmtBF16 : kFmtF16, dt, ops, M, N, K, alpha,
                                   A, lda, B, ldb, beta, C, ldc, stream, nullptr, 0);
}

cudaError_t launch_gemm_tc_f16(const DeviceInfo &dev, bool is_bf16, int M, int N, int K,
                               float alpha, const void *A, int64_t lda, const void *B,
                               int64_t ldb, float beta, float *C, int64_t ldc,
                               cudaStream_t stream) {
  return launch_gemm_tc_f16_ex(dev, is_bf16, BatchOps(), M, N, K, alpha, A, lda, B, ldb, beta, C,
                               ldc, stream);
}

}  // namespace dgr
