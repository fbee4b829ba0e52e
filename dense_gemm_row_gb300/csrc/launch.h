// launch.h -- internal interface between the C-ABI layer (abi.cu) and the
// kernel translation units. Not installed; not part of the public ABI.
#pragma once

#include <cstdint>

#include <cuda_runtime_api.h>

namespace dgr {

// Layout of the per-device error word (read and cleared by
// gemm_check_device_error): bit 0 = a bounded wait gave up; bits 8..15 = the
// code of the first wait that gave up.
constexpr uint32_t kErrTimeoutBit = 1u;
constexpr uint32_t kWaitFull = 1, kWaitEmpty = 2, kWaitTmemFull = 3, kWaitTmemEmpty = 4,
                   kWaitDrain = 5, kWaitFlag = 6, kWaitTest = 7;

// Per-device facts gathered once by the ABI layer.
struct DeviceInfo {
  int device = -1;
  int sm_count = 0;
  uint32_t *err_word = nullptr;  // device address of this device's error word
};

// Operand forms and batching of the extended entry points (gemm_*_ex):
// C_b = alpha * op(A_b) * op(B_b) + beta * C_b for b < batch, X_b = X + b *
// stride_x elements. A stride of 0 (or batch == 1) means one shared matrix.
struct BatchOps {
  bool a_t = false;  // A stored K x M (row-major), used transposed
  bool b_t = false;  // B stored N x K (row-major), used transposed
  int batch = 1;
  int64_t stride_a = 0, stride_b = 0, stride_c = 0;  // elements
  bool plain() const { return !a_t && !b_t && batch == 1; }
};

// All sizes are already validated: M, N >= 1, K >= 1, each < 2^31, ld >= row length.
cudaError_t launch_sgemm_simt(const DeviceInfo &dev, int M, int N, int K, float alpha,
                              const float *A, int64_t lda, const float *B, int64_t ldb,
                              float beta, float *C, int64_t ldc, cudaStream_t stream);

// 16-bit inputs (is_bf16 selects bf16 or fp16), fp32 output. Layout already
// checked: A, B 16-byte aligned, lda and ldb multiples of 8.
cudaError_t launch_gemm_tc_f16(const DeviceInfo &dev, bool is_bf16, int M, int N, int K,
                               float alpha, const void *A, int64_t lda, const void *B,
                               int64_t ldb, float beta, float *C, int64_t ldc,
                               cudaStream_t stream);

// The same with transposed operands and batches (A and B stored as BatchOps
// says; the layout rule above applies to the stored matrices, and non-zero
// strides of A and B are multiples of 8 elements).
cudaError_t launch_gemm_tc_f16_ex(const DeviceInfo &dev, bool is_bf16, const BatchOps &ops, int M,
                                  int N, int K, float alpha, const void *A, int64_t lda,
                                  const void *B, int64_t ldb, float beta, float *C, int64_t ldc,
                                  cudaStream_t stream);
cudaError_t launch_gemm_s8_ex(const DeviceInfo &dev, const BatchOps &ops, int M, int N, int K,
                              int32_t alpha, const int8_t *A, int64_t lda, const int8_t *B,
                              int64_t ldb, int32_t beta, int32_t *C, int64_t ldc,
                              cudaStream_t stream);
cudaError_t launch_sgemm_simt_ex(const DeviceInfo &dev, const BatchOps &ops, int M, int N, int K,
                                 float alpha, const float *A, int64_t lda, const float *B,
                                 int64_t ldb, float beta, float *C, int64_t ldc,
                                 cudaStream_t stream);

cudaError_t launch_gemm_s8(const DeviceInfo &dev, int M, int N, int K, int32_t alpha,
                           const int8_t *A, int64_t lda, const int8_t *B, int64_t ldb,
                           int32_t beta, int32_t *C, int64_t ldc, cudaStream_t stream);

// uint8 inputs, exact int32 C (wrap-around) on the fp16 tensor pipe.
cudaError_t launch_gemm_u8(const DeviceInfo &dev, int M, int N, int K, int32_t alpha,
                           const uint8_t *A, int64_t lda, const uint8_t *B, int64_t ldb,
                           int32_t beta, int32_t *C, int64_t ldc, cudaStream_t stream);

// 16-bit inputs and a 16-bit C of the same format (is_bf16), fp32 accumulation,
// one round-to-nearest-even. Layout rule of launch_gemm_tc_f16 for A and B.
cudaError_t launch_gemm_tc_out16(const DeviceInfo &dev, bool is_bf16, int M, int N, int K,
                                 float alpha, const void *A, int64_t lda, const void *B,
                                 int64_t ldb, float beta, uint16_t *C, int64_t ldc,
                                 cudaStream_t stream);

// fp32 inputs at tf32 precision on the tensor cores, fp32 C. Any layout.
cudaError_t launch_gemm_tf32(const DeviceInfo &dev, int M, int N, int K, float alpha,
                             const float *A, int64_t lda, const float *B, int64_t ldb, float beta,
                             float *C, int64_t ldc, cudaStream_t stream);

// fp64 on the SIMT pipe (dgemm_simt.cu).
cudaError_t launch_dgemm(const DeviceInfo &dev, int M, int N, int K, double alpha,
                         const double *A, int64_t lda, const double *B, int64_t ldb, double beta,
                         double *C, int64_t ldc, cudaStream_t stream);

// Bytes of scratch the int8 path needs, and the int8 path on caller-provided
// scratch (256-byte aligned, at least s8_scratch_bytes(M, N, K) bytes) and
// caller-provided split-k tail flags (flags_words 32-bit words, zeroed by the
// call with cudaMemsetAsync; a buffer too small for the split turns it off).
size_t s8_scratch_bytes(int M, int N, int K);
cudaError_t launch_gemm_s8_scratch(const DeviceInfo &dev, int M, int N, int K, int32_t alpha,
                                   const int8_t *A, int64_t lda, const int8_t *B, int64_t ldb,
                                   int32_t beta, int32_t *C, int64_t ldc, void *scratch,
                                   uint32_t *flags, size_t flags_words, cudaStream_t stream);

// Short, wide problems on the tensor cores, computed as C^T = B^T A^T so that N
// fills the MMA rows (gemm_tc_skinny.cu, up to 64 rows; which problems take it:
// tc_skinny_route). 16-bit inputs with the same layout rule as
// launch_gemm_tc_f16; the int version takes the fp16-widened operands of the
// int8 path and optional caller-provided flags. kSkinnyMaxM is also the row
// limit of the small-M SIMT kernel (gemm_small_m.cu).
constexpr int kSkinnyMaxM = 32;
// Whether the 16-bit / int8 tensor-core paths take the transposed-role kernel
// for an M x N problem: up to 32 rows always; 33..64 rows when its k range is
// split across a cluster (16..sm_count-1 column blocks of 128). Measured on
// GB300 at 64 rows against the 256-row pair tiles: bf16 N = K = 8192 29.2 vs
// 38.5 us, 64 x 4096 x 4096 12.6 vs 31.3 us.
bool tc_skinny_route(int M, int N, int sm_count);
cudaError_t launch_tc_skinny_float(const DeviceInfo &dev, bool is_bf16, int M, int N, int K,
                                   float alpha, const void *A, int64_t lda, const void *B,
                                   int64_t ldb, float beta, float *C, int64_t ldc,
                                   cudaStream_t stream);
cudaError_t launch_tc_skinny_int(const DeviceInfo &dev, int M, int N, int K, int32_t alpha,
                                 const void *A16, int64_t lda, const void *B16, int64_t ldb,
                                 int32_t beta, int32_t *C, int64_t ldc, cudaStream_t stream,
                                 uint32_t *flags, size_t flags_words);
// The transposed-role kernel with int8 B read as stored (converted to fp16 in
// shared memory; A already widened to fp16): M <= 64, B 16-byte aligned with
// a row stride in whole 16-byte units (tc_skinny_i8_supported).
bool tc_skinny_i8_supported(int M, const void *B, int64_t ldb);
// gemm_s8 for short, wide problems through that kernel (gemm_tc_int.cu).
cudaError_t launch_gemm_s8_skinny_raw(const DeviceInfo &dev, int M, int N, int K, int32_t alpha,
                                      const int8_t *A, int64_t lda, const int8_t *B, int64_t ldb,
                                      int32_t beta, int32_t *C, int64_t ldc, cudaStream_t stream);
// Rows from which gemm_s8 prefers it over the dp4a small-M kernel: with A and
// B read as stored (the cluster form) from 5 rows, with a widened A from 10.
// Measured on GB300 at N = K = 8192: dp4a 19.1 us at 4 rows and 26.3 us at 6;
// the cluster form about 19.5 us for any row count up to 16; the widened-A
// form tied with dp4a at 10 rows.
#ifndef DGR_I8RAW_MIN_M
#define DGR_I8RAW_MIN_M 10
#endif
constexpr int kI8RawMinM = DGR_I8RAW_MIN_M;
constexpr int kI8ClusterMinM = 5;
// int8 A and B read as stored by the cluster form of the transposed-role
// kernel (gemm_tc_skinny.cu; up to 64 rows): both operands 16-byte aligned
// with row strides in whole 16-byte units (tc_skinny_s8_supported).
bool tc_skinny_s8_supported(int M, const void *A, int64_t lda, const void *B, int64_t ldb);
cudaError_t launch_tc_skinny_s8(const DeviceInfo &dev, int M, int N, int K, int32_t alpha,
                                const int8_t *A, int64_t lda, const int8_t *B, int64_t ldb,
                                int32_t beta, int32_t *C, int64_t ldc, cudaStream_t stream);
cudaError_t launch_tc_skinny_i8(const DeviceInfo &dev, int M, int N, int K, int32_t alpha,
                                const void *A16, int64_t lda, const int8_t *B, int64_t ldb,
                                int32_t beta, int32_t *C, int64_t ldc, cudaStream_t stream);

// dst (cols x rows, row stride ldd) = transpose of the row-major rows x cols
// fp32 matrix src (row stride lds): 64 x 64 tiles through shared memory
// (gemm_tc_tf32.cu).
cudaError_t launch_transpose_f32(const DeviceInfo &dev, const float *src, int64_t lds, int rows,
                                 int cols, float *dst, int64_t ldd, cudaStream_t stream);

// Raises a kernel's dynamic shared-memory limit on the current device, once
// per (kernel, device); later calls only look the pair up.
cudaError_t set_max_dynamic_smem(const void *kernel, int bytes, int device);

// Tall, narrow problems (gemm_small_n.cu): N <= 16 columns (16-bit inputs:
// N <= 2) and at least
// kSmallNMinM rows; A read once with 16-byte loads (A 16-byte aligned, rows a
// whole number of 16-byte units: small_n_supported), B staged in shared
// memory. fp32, bf16 / fp16 (fp32 accumulation, fp32 C) and int8 (int32 C).
constexpr int kSmallNMinM = 512;
bool small_n_supported(int M, int N, const void *A, int64_t lda, int esize);
cudaError_t launch_small_n_f32(int M, int N, int K, float alpha, const float *A, int64_t lda,
                               const float *B, int64_t ldb, float beta, float *C, int64_t ldc,
                               cudaStream_t stream);
cudaError_t launch_small_n_half(bool is_bf16, int M, int N, int K, float alpha, const void *A,
                                int64_t lda, const void *B, int64_t ldb, float beta, float *C,
                                int64_t ldc, cudaStream_t stream);
cudaError_t launch_small_n_s8(int M, int N, int K, int32_t alpha, const int8_t *A, int64_t lda,
                              const int8_t *B, int64_t ldb, int32_t beta, int32_t *C, int64_t ldc,
                              cudaStream_t stream);

// fp32 and int8 GEMM for M <= 32 (gemm_small_m.cu): streams B once with TMA,
// 4 columns x all rows per thread (packed fp32 FMA / dp4a). Usable when
// small_m_supported(): A and B 16-byte aligned with row strides that are whole
// multiples of 16 bytes (esize = element size in bytes).
bool small_m_supported(int M, const void *A, int64_t lda, const void *B, int64_t ldb,
                       int esize);
cudaError_t launch_small_m_f32(const DeviceInfo &dev, int M, int N, int K, float alpha,
                               const float *A, int64_t lda, const float *B, int64_t ldb,
                               float beta, float *C, int64_t ldc, cudaStream_t stream);
cudaError_t launch_small_m_s8(const DeviceInfo &dev, int M, int N, int K, int32_t alpha,
                              const int8_t *A, int64_t lda, const int8_t *B, int64_t ldb,
                              int32_t beta, int32_t *C, int64_t ldc, cudaStream_t stream);

// The library's stream-ordered memory pool on a device (created on first use;
// freed blocks stay mapped for reuse).
cudaError_t device_pool(const DeviceInfo &dev, cudaMemPool_t *out);

// K == 0: C = beta * C (C = 0 when beta == 0), M x N window only.
cudaError_t launch_scale_f32(int M, int N, float beta, float *C, int64_t ldc,
                             cudaStream_t stream);
cudaError_t launch_scale_s32(int M, int N, int32_t beta, int32_t *C, int64_t ldc,
                             cudaStream_t stream);
// K == 0 for the other C types: C = beta * C (16-bit: decoded, scaled in fp32,
// rounded to nearest even).
cudaError_t launch_scale_f64(int M, int N, double beta, double *C, int64_t ldc,
                             cudaStream_t stream);
cudaError_t launch_scale_out16(bool is_bf16, int M, int N, float beta, uint16_t *C, int64_t ldc,
                               cudaStream_t stream);
// The same over a stack of `batch` C matrices, `stride` elements apart.
cudaError_t launch_scale_batched_f32(int M, int N, float beta, float *C, int64_t ldc, int batch,
                                     int64_t stride, cudaStream_t stream);
cudaError_t launch_scale_batched_s32(int M, int N, int32_t beta, int32_t *C, int64_t ldc,
                                     int batch, int64_t stride, cudaStream_t stream);

// Accessors to the ABI layer's shared host logic (defined in abi.cu). The
// status values are those of gemm_status_t.
int abi_check_args(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda, const void *B,
                   int64_t ldb, const void *C, int64_t ldc, bool *nothing_to_do);
int abi_current_device(const DeviceInfo **out);
int abi_from_cuda(cudaError_t e);

}  // namespace dgr
