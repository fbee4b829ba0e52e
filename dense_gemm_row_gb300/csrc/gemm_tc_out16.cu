// gemm_tc_out16.cu -- 16-bit inputs with a C of the same 16-bit format on the
// tensor cores (the warp-matrix-function type table's half -> half row, and
// its bf16 analogue): fp32 accumulation in TMEM, alpha/beta in fp32, one
// round-to-nearest-even to 16 bits when C is written. The kernel is in
// gemm_tc_kernel.cuh.
#include "gemm_tc_kernel.cuh"

namespace dgr {

cudaError_t launch_gemm_tc_out16(const DeviceInfo &dev, bool is_bf16, int M, int N, int K,
                                 float alpha, const void *A, int64_t lda, const void *B,
                                 int64_t ldb, float beta, uint16_t *C, int64_t ldc,
                                 cudaStream_t stream) {
  const CUtensorMapDataType dt =
      is_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  if (is_bf16)
    return launch_tc<kKindBF16Out, false>(dev, dt, kFmtBF16, dt, BatchOps(), M, N, K, alpha, A,
                                          lda, B, ldb, beta, C, ldc, stream, nullptr, 0);
  return launch_tc<kKindF16Out, false>(dev, dt, kFmtF16, dt, BatchOps(), M, N, K, alpha, A, lda,
                                       B, ldb, beta, C, ldc, stream, nullptr, 0);
}

}  // namespace dgr
