/*
 * dense_gemm_row.h -- C ABI of the GB300 (sm_103a) row-major dense GEMM library
 * (libdense_gemm_row.so).
 *
 * Every entry point computes
 *
 *     C = alpha * A * B + beta * C
 *
 * with A an M x K matrix, B a K x N matrix and C an M x N matrix, all stored
 * row-major with a leading dimension (row stride, in elements):
 *
 *     A(i,k) = A[i*lda + k],  B(k,j) = B[k*ldb + j],  C(i,j) = C[i*ldc + j]
 *
 * Sources for the operation: "Sgemm [128,128,8]" (jianshu page) defines
 * gemm as C = alpha*A*B + beta*C with all matrices row-major and indexes them
 * through the A(i,j) / B(i,j) / C(i,j) macros with lda, ldb, ldc; its host
 * reference routine host_gemm is the same loop nest. "使用CUDA和瓦片算法计算
 * 矩阵乘法" (the tiled-multiply page) requires shapes that are not multiples of
 * the tile to give correct results (residual tile cells act as zeros). The C++
 * warp-matrix-function page's type table fixes the precisions: half and
 * bfloat16 inputs accumulate in float, signed char inputs accumulate in int.
 *
 * Common contract of gemm_f32 / gemm_bf16 / gemm_f16 / gemm_s8:
 *
 *   Sizes   M, N, K >= 0 and each < 2^31. When M > 0 and K > 0, lda >= K; when
 *           K > 0 and N > 0, ldb >= N; when M > 0 and N > 0, ldc >= N.
 *   Memory  A, B and C are device pointers (or pointers the device can access)
 *           owned by the caller; the library neither allocates nor frees them.
 *           A pointer may be NULL only when its matrix is empty. Only the
 *           M x K, K x N and M x N windows are read or written; row padding
 *           beyond the row length is never touched. C must not overlap A or B.
 *   beta    When beta == 0, C is write-only: its old contents (even NaN/Inf)
 *           are never read. When alpha == 0 the product is still formed and
 *           scaled by zero.
 *   K == 0  C = beta * C (C = 0 when beta == 0).
 *   M or N == 0  Nothing is launched; GEMM_OK is returned.
 *   Stream  The call only enqueues work on `stream` (0 = the legacy default
 *           stream) and returns; results are ready when the stream is.
 *           Calls on different streams may overlap on the GPU. The
 *           tensor-core kernel, and the SIMT SGEMM on grids of under two
 *           waves, split the k range of their last wave's tiles across CTAs,
 *           size their grids to be resident all at once, and a later part
 *           waits for the one before. When another stream's work
 *           holds part of the GPU for longer than that wait's bound (2 s),
 *           the call gives up, like any other bounded wait: its C is
 *           incomplete and gemm_check_device_error() returns
 *           GEMM_ERR_TIMEOUT. Two such calls can do this to each other.
 *           Order calls that must not fail this way on one stream. (The
 *           short-wide SIMT kernel, whose split parts also wait for one
 *           another, is launched cooperatively and so is always resident
 *           in full.)
 *   Device  The current CUDA device must be an sm_103 (GB300) GPU.
 *   Errors  Never aborts and never prints. Argument checks run on the host
 *           before anything is enqueued; a failed check returns a status and
 *           launches nothing. A kernel that waits on its own pipeline gives up
 *           after a bounded time, records the fact in a device error word and
 *           returns; gemm_check_device_error() reads and clears that word.
 *
 * Thread safety: the entry points may be called from several host threads;
 * per-device set-up (kernel attributes, device properties) is done once under
 * a lock.
 */
#ifndef DENSE_GEMM_ROW_H
#define DENSE_GEMM_ROW_H

#include <stdint.h>

#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define GEMM_API __attribute__((visibility("default")))
#else
#define GEMM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_VALUE = 1,      /* negative size, ld < row length, NULL operand */
    GEMM_ERR_UNSUPPORTED_LAYOUT = 2, /* tensor-core path: base or row stride not 16-byte aligned */
    GEMM_ERR_LAUNCH = 3,             /* a CUDA call or kernel launch failed */
    GEMM_ERR_DEVICE = 4,             /* no current device, or it is not an sm_103 GPU */
    GEMM_ERR_TIMEOUT = 5,            /* a kernel's bounded pipeline wait gave up */
    GEMM_ERR_TOO_LARGE = 6           /* gemm_s8_noalloc: problem needs more than its fixed scratch */
} gemm_status_t;

/* Bit patterns of 16-bit floats, as stored in memory. */
typedef uint16_t gemm_bf16_t; /* bfloat16: the upper half of an IEEE binary32 */
typedef uint16_t gemm_f16_t;  /* IEEE binary16 */

/*
 * gemm_f32 -- exact-fp32 SGEMM on the SIMT FP32 pipe (no TF32).
 * A, B, C: float. Each output is one fp32 sum of the K products in some order,
 * then alpha*acc + beta*C in fp32. Any alignment and any ld are accepted.
 * Sources: "Sgemm [128,128,8]" (the 128x128x8 tiled kernel with 8x8 per-thread
 * register blocks); "CUDA学习之路[11]：矩阵乘法计算详解", sections V1 2D Thread,
 * V2 Tile and V3 双缓冲 (register tiling, float4 loads, double buffering).
 */
GEMM_API gemm_status_t gemm_f32(int64_t M, int64_t N, int64_t K, float alpha,
                       const float *A, int64_t lda, const float *B, int64_t ldb,
                       float beta, float *C, int64_t ldc, cudaStream_t stream);

/*
 * gemm_bf16 / gemm_f16 -- tensor-core GEMM: 16-bit inputs, fp32 accumulation,
 * fp32 output C. Each product of two 16-bit values is exact in fp32; sums are
 * accumulated in fp32 in the tensor core's order.
 * Layout rule (the same one the WMMA page states for ldm, and the one the
 * tensor-memory copy engine requires): A and B must start on a 16-byte boundary
 * and lda, ldb must be multiples of 8 elements; otherwise
 * GEMM_ERR_UNSUPPORTED_LAYOUT is returned and nothing is launched. C has no
 * alignment requirement.
 * Source: C++ warp-matrix-function page, section mma_sync and the type table
 * rows __half x __half -> float and __nv_bfloat16 x __nv_bfloat16 -> float.
 */
GEMM_API gemm_status_t gemm_bf16(int64_t M, int64_t N, int64_t K, float alpha,
                        const gemm_bf16_t *A, int64_t lda, const gemm_bf16_t *B,
                        int64_t ldb, float beta, float *C, int64_t ldc,
                        cudaStream_t stream);

GEMM_API gemm_status_t gemm_f16(int64_t M, int64_t N, int64_t K, float alpha,
                       const gemm_f16_t *A, int64_t lda, const gemm_f16_t *B,
                       int64_t ldb, float beta, float *C, int64_t ldc,
                       cudaStream_t stream);

/*
 * gemm_s8 -- int8 inputs, exact int32 accumulation, int32 output C.
 * C = alpha*acc + beta*C in int32 two's-complement wrap-around arithmetic: the
 * result is the exact integer value modulo 2^32.
 * Source: C++ warp-matrix-function page, type table row signed char x signed
 * char -> int.
 */
GEMM_API gemm_status_t gemm_s8(int64_t M, int64_t N, int64_t K, int32_t alpha,
                      const int8_t *A, int64_t lda, const int8_t *B, int64_t ldb,
                      int32_t beta, int32_t *C, int64_t ldc, cudaStream_t stream);

/*
 * Further rows of the warp-matrix-function page's type table (C++ warp matrix
 * functions, the matrix_a / matrix_b / accumulator type table). Same call
 * shape, row-major layout, statuses, K == 0 and beta == 0 rules as the entry
 * points above.
 *
 * gemm_u8 -- unsigned char -> int row: uint8 A and B, int32 C and int32
 *   alpha/beta, exact (the product accumulated in 64-bit integers, the update
 *   alpha*acc + beta*C taken modulo 2^32). Any layout.
 *
 * gemm_f16_f16, gemm_bf16_bf16 -- half -> half row (and its bf16 analogue):
 *   16-bit A, B and C of one format. The result is accumulated in fp32, the
 *   update alpha*acc + beta*C is evaluated in fp32 and rounded once to the
 *   16-bit format (round-to-nearest-even) when C is written. A and B follow the
 *   layout rule of gemm_bf16 (16-byte aligned bases, lda and ldb multiples of
 *   8, else GEMM_ERR_UNSUPPORTED_LAYOUT); C may have any layout.
 *
 * gemm_tf32 -- precision::tf32 -> float row: fp32 A, B, C; the tensor cores
 *   use A and B at tf32 precision (8 exponent bits, 10 fraction bits: the low
 *   13 fraction bits of each input are not used), accumulate in fp32. Opt-in:
 *   gemm_f32 stays exact fp32. Any layout with 4-byte aligned elements. The
 *   call allocates and frees stream-ordered scratch for a K-major copy of B.
 *
 * gemm_f64 -- double -> double row: fp64 A, B, C, alpha, beta, fp64 fused
 *   multiply-adds. Any layout; M up to 4194240 (65535 tiles of 64 rows).
 */
GEMM_API gemm_status_t gemm_u8(int64_t M, int64_t N, int64_t K, int32_t alpha,
                               const uint8_t *A, int64_t lda, const uint8_t *B, int64_t ldb,
                               int32_t beta, int32_t *C, int64_t ldc, cudaStream_t stream);
GEMM_API gemm_status_t gemm_f16_f16(int64_t M, int64_t N, int64_t K, float alpha,
                                    const gemm_f16_t *A, int64_t lda, const gemm_f16_t *B,
                                    int64_t ldb, float beta, gemm_f16_t *C, int64_t ldc,
                                    cudaStream_t stream);
GEMM_API gemm_status_t gemm_bf16_bf16(int64_t M, int64_t N, int64_t K, float alpha,
                                      const gemm_bf16_t *A, int64_t lda, const gemm_bf16_t *B,
                                      int64_t ldb, float beta, gemm_bf16_t *C, int64_t ldc,
                                      cudaStream_t stream);
GEMM_API gemm_status_t gemm_tf32(int64_t M, int64_t N, int64_t K, float alpha, const float *A,
                                 int64_t lda, const float *B, int64_t ldb, float beta, float *C,
                                 int64_t ldc, cudaStream_t stream);
GEMM_API gemm_status_t gemm_f64(int64_t M, int64_t N, int64_t K, double alpha, const double *A,
                                int64_t lda, const double *B, int64_t ldb, double beta, double *C,
                                int64_t ldc, cudaStream_t stream);

/* Operand forms for the extended entry points. */
typedef enum {
    GEMM_OP_N = 0, /* the operand as stored (row-major) */
    GEMM_OP_T = 1  /* the transpose of the stored row-major matrix */
} gemm_op_t;

/*
 * Extended entry points: strided-batched GEMM with transposed operands.
 *
 *   for b in [0, batch):
 *     C_b = alpha * op(A_b) * op(B_b) + beta * C_b
 *   A_b = A + b*strideA, B_b = B + b*strideB, C_b = C + b*strideC (elements)
 *
 * op(A_b) is M x K: with GEMM_OP_N, A_b is stored M x K row-major (lda >= K);
 * with GEMM_OP_T, A_b is stored K x M row-major (lda >= M) and transposed.
 * op(B_b) is K x N: GEMM_OP_N stores K x N (ldb >= N); GEMM_OP_T stores N x K
 * (ldb >= K). C_b is M x N row-major (ldc >= N). batch >= 1 (batch = 0 does
 * nothing). The C_b must not overlap each other or any input: when batch > 1,
 * strideC >= (M - 1) * ldc + N (else GEMM_ERR_INVALID_VALUE). Input strides
 * may be any value >= 0, including 0 (one matrix shared by every batch entry);
 * gemm_bf16_ex and gemm_f16_ex need them to be multiples of 8 elements (16
 * bytes) when batch > 1 (else GEMM_ERR_UNSUPPORTED_LAYOUT).
 * Everything else -- beta == 0 never reads C, K == 0, alignment rules, status
 * codes, streams -- is as for the plain entry points, and a call with
 * GEMM_OP_N, GEMM_OP_N and batch == 1 computes exactly what the plain call does.
 * Sources: the plain entry points' definition applied to each batch entry; the
 * batched (bmm) and transposed forms are the dlog page's PyTorch matmul
 * survey (section 矩阵相乘的若干写法: mm, bmm, einsum) and the WMMA page's
 * row_major / col_major operand layouts.
 */
GEMM_API gemm_status_t gemm_f32_ex(gemm_op_t opA, gemm_op_t opB, int64_t M, int64_t N, int64_t K,
                                   float alpha, const float *A, int64_t lda, int64_t strideA,
                                   const float *B, int64_t ldb, int64_t strideB, float beta,
                                   float *C, int64_t ldc, int64_t strideC, int64_t batch,
                                   cudaStream_t stream);
GEMM_API gemm_status_t gemm_bf16_ex(gemm_op_t opA, gemm_op_t opB, int64_t M, int64_t N,
                                    int64_t K, float alpha, const gemm_bf16_t *A, int64_t lda,
                                    int64_t strideA, const gemm_bf16_t *B, int64_t ldb,
                                    int64_t strideB, float beta, float *C, int64_t ldc,
                                    int64_t strideC, int64_t batch, cudaStream_t stream);
GEMM_API gemm_status_t gemm_f16_ex(gemm_op_t opA, gemm_op_t opB, int64_t M, int64_t N, int64_t K,
                                   float alpha, const gemm_f16_t *A, int64_t lda,
                                   int64_t strideA, const gemm_f16_t *B, int64_t ldb,
                                   int64_t strideB, float beta, float *C, int64_t ldc,
                                   int64_t strideC, int64_t batch, cudaStream_t stream);
GEMM_API gemm_status_t gemm_s8_ex(gemm_op_t opA, gemm_op_t opB, int64_t M, int64_t N, int64_t K,
                                  int32_t alpha, const int8_t *A, int64_t lda, int64_t strideA,
                                  const int8_t *B, int64_t ldb, int64_t strideB, int32_t beta,
                                  int32_t *C, int64_t ldc, int64_t strideC, int64_t batch,
                                  cudaStream_t stream);

/*
 * gemm_s8_noalloc -- gemm_s8 for callers that must not allocate device memory.
 * The pages have no counterpart of this entry point; it is part of this
 * library's interface only.
 *
 * gemm_s8 widens A and B to fp16 in scratch memory that it takes from a
 * library-owned stream-ordered pool. Some callers cannot allow that: a process
 * whose device memory is entirely reserved up front by another allocator (so
 * any extra allocation can fail or fragment it), a latency-critical loop that
 * must never enter the driver's allocation path, or a deployment that forbids
 * allocation after start-up. This variant computes exactly what gemm_s8
 * computes (same arguments, same bit-exact result) but calls no cudaMalloc,
 * cudaFree or allocating library routine: its scratch is a fixed 64 MiB array
 * in the library's device memory, which every GPU that loads this part of the
 * library keeps until the process exits. The caller still provides A, B and C.
 *
 * Limit: 2 * (M * ceil8(K) + K * ceil8(N)) bytes, with the A part rounded up
 * to 256 bytes, must not exceed 64 MiB (for example M = N = K = 4096 fits);
 * larger problems return GEMM_ERR_TOO_LARGE and launch nothing. Argument
 * checks are those of gemm_s8.
 * Set-up: the first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call before
 * any stream capture begins. A failed look-up returns GEMM_ERR_DEVICE, clears
 * the CUDA runtime's last-error state of the calling thread (including an
 * error an earlier asynchronous launch may have left there), and is
 * remembered: every later call on that device returns GEMM_ERR_DEVICE too,
 * for the life of the process (the look-up is not retried).
 * Concurrency: all calls on a device share the one array, and each call
 * overwrites every scratch element it later reads, so no state carries over
 * from the previous call; but calls that can overlap on the GPU (different
 * streams without ordering between them) race on the array and give wrong
 * results. Order them on one stream, or use gemm_s8.
 */
GEMM_API gemm_status_t gemm_s8_noalloc(int64_t M, int64_t N, int64_t K, int32_t alpha,
                                       const int8_t *A, int64_t lda, const int8_t *B,
                                       int64_t ldb, int32_t beta, int32_t *C, int64_t ldc,
                                       cudaStream_t stream);

/* A constant, human-readable name for a status. Never NULL. */
GEMM_API const char *gemm_status_string(gemm_status_t status);

/*
 * Reads and clears the current device's error word. Synchronises the device.
 * Returns GEMM_ERR_TIMEOUT if a kernel gave up a bounded wait since the last
 * call, GEMM_OK otherwise (or GEMM_ERR_DEVICE / GEMM_ERR_LAUNCH when the device
 * cannot be queried). Optionally stores the raw word in *word (may be NULL):
 * bit 0 = a wait timed out, bits 8..15 = the code of the first wait that did.
 */
GEMM_API gemm_status_t gemm_check_device_error(uint32_t *word);

/*
 * Diagnostic of the failure path: enqueues one warp that waits, with the same
 * bounded mbarrier wait as the GEMM kernels, on a barrier nothing arrives on.
 * After limit_us microseconds (1 .. 1000000) the wait gives up, records a
 * timeout (wait code 7) in the device error word and the kernel returns; the
 * context stays usable and gemm_check_device_error() then reports
 * GEMM_ERR_TIMEOUT. Nothing faults, traps or hangs. Returns
 * GEMM_ERR_INVALID_VALUE for a limit outside the range, else the launch status.
 * Source: none on the pages (their error handling aborts the process); this is
 * the library's own failure detection.
 */
GEMM_API gemm_status_t gemm_selftest_wait_timeout(uint32_t limit_us, cudaStream_t stream);

/*
 * Peak-rate microbenchmarks: the measured denominators that the GEMM kernels'
 * roofline fractions are cross-checked against. Neither reads or writes
 * user data beyond `sink`; both are asynchronous on `stream` (time them with
 * events around the call). *flops (a host pointer, may be NULL) receives the
 * floating-point operations the launch performs (a multiply-add counts 2).
 *
 * gemm_peak_ffma: every SM runs 4 blocks of 256 threads; each thread issues
 * `iters` rounds of 16 independent packed fp32 FMAs (fma.rn.f32x2, 32 lanes'
 * worth of multiply-adds), the instruction the exact-fp32 GEMM uses. `sink` is
 * a device float that is written only if the accumulated values happen to
 * equal a fixed sentinel (never, in practice; it keeps the work observable).
 * flops = SMs * 1024 * iters * 64.
 *
 * gemm_peak_tc_f16: one CTA per SM issues `iters` rounds of four
 * tcgen05.mma.cta_group::1.kind::f16 (bf16 in, fp32 accumulate; M = 128,
 * N = 256, K = 16) on operands held in shared memory, accumulating in TMEM;
 * one thread issues, as in the GEMM kernel. flops = SMs * iters * 4 *
 * 2 * 128 * 256 * 16. Its one wait (for the last MMA) is bounded like the
 * GEMM kernels' waits.
 *
 * Both return GEMM_ERR_INVALID_VALUE for iters outside 1 .. 2^24 (gemm_peak_ffma;
 * also for a NULL sink) or 1 .. 2^20 (gemm_peak_tc_f16: at most about 0.3 s of
 * MMAs, well inside the bound on its wait), else the launch status. Source: the rooflines are
 * bounded by these two pipes ("Sgemm [128,128,8]": FFMA-bound inner loop; the
 * C++ warp-matrix-function page: tensor-core matrix multiply-accumulate).
 */
GEMM_API gemm_status_t gemm_peak_ffma(int32_t iters, float *sink, double *flops,
                                      cudaStream_t stream);
GEMM_API gemm_status_t gemm_peak_tc_f16(int32_t iters, double *flops, cudaStream_t stream);

/*
 * The CUDA runtime's name for the error behind the calling thread's most
 * recent GEMM_ERR_LAUNCH (e.g. "cudaErrorLaunchOutOfResources"), or
 * "cudaSuccess" if there was none. A static string; never NULL.
 */
GEMM_API const char *gemm_last_launch_error(void);

/*
 * Usage of the library's own stream-ordered memory pool on the current device
 * (the pool that gemm_s8, gemm_u8, gemm_tf32, the fp32 transposing paths and
 * the split-k workspaces draw their scratch from). *used_high_bytes receives
 * the most memory in use at one time since the pool was created or the mark
 * was last reset; *reserved_bytes the device memory the pool holds now (freed
 * blocks stay reserved for reuse). Either pointer may be NULL. reset_high != 0
 * resets the high-water mark to zero after reading it. Before the first call
 * that needs the pool, both values are 0. Host-only: nothing is enqueued.
 * Returns GEMM_ERR_DEVICE when no device is current, GEMM_ERR_LAUNCH when the
 * pool cannot be queried, else GEMM_OK. Source: none on the pages; a
 * diagnostic of this library's memory use (it lets a test show that
 * gemm_s8_noalloc takes nothing from the pool).
 */
GEMM_API gemm_status_t gemm_pool_usage(int64_t *used_high_bytes, int64_t *reserved_bytes,
                                       int reset_high);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
GEMM_API int gemm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DENSE_GEMM_ROW_H */
