// gemm_tc_skinny.cu -- tensor-core GEMM for short, wide problems (M <= 32).
//
//     C = alpha * A * B + beta * C       A: M x K, B: K x N, C: M x N, row-major
//
// With few rows of A a 128- or 256-row MMA tile would mostly multiply zeros;
// such a GEMM is bound by streaming B (K x N) from HBM. This kernel computes
// the transposed product instead, C^T = B^T * A^T, so that N fills the MMA's
// 128-row dimension and M (rounded up to a multiple of 16) is the MMA's N:
//   * the MMA's A operand is a 64(k) x 128(n) tile of B, read N-major straight
//     from row-major B (two 64 x 64 TMA boxes, 128-byte swizzle);
//   * the MMA's B operand is the 64(k) x Mp tile of A, read K-major straight
//     from row-major A (one TMA box, 128-byte swizzle);
//   * the accumulator is 128 TMEM lanes (columns of C) x Mp columns (rows of C),
//     so each epilogue warp stores 32 consecutive columns of one row of C at a
//     time: full 128-byte segments.
// Every CTA computes one slice of work: a 128-column block of C over one part
// of the k range. When there are fewer column blocks than SMs, k is split into
// `split` parts: every part stores its partial sums in a workspace and counts
// itself done on its column block; the part that finishes last adds the
// partials in part order and writes alpha * sum + beta * C. The result is
// deterministic (and exact in the int8 mode, whose split points fall on
// 1024-k chunks), and no part waits for another.
//
// Sources: as gemm_tc_kernel.cuh (C = alpha*A*B + beta*C, "Sgemm [128,128,8]"; half /
// bfloat16 x half / bfloat16 -> float and signed char -> int, C++ warp matrix
// function page, type table). The pages have no skinny-shape kernel; this is a
// layout choice for the same computation.
#include <cstdint>
#include <cstring>
#include <mutex>
#include <type_traits>

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "launch.h"
#include "ptx.cuh"

namespace dgr {
namespace {

constexpr int kBN = 128;       // columns of C per CTA (the MMA's M)
constexpr int kBK = 64;        // k-block: one 128-byte swizzle row of 16-bit values
constexpr int kMaxM = 64;      // largest M the kernel supports (Mp <= 64)
constexpr int kStages = 8;
constexpr int kEpiWarps = 4;
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kChunkKB = 1024 / kBK;  // int mode: exact fp32 chunks of 1024 k
constexpr uint32_t kBufCols = 64;               // one accumulator: up to 64 columns
constexpr uint32_t kTmemCols = 2 * kBufCols;     // two buffers (int mode alternates)
constexpr uint32_t kBBox = 64 * kBK * 2;          // one 64(n) x 64(k) box: 8 KiB
constexpr uint32_t kBBytes = kBK * kBN * 2;       // 16 KiB
constexpr uint32_t kABytes = kMaxM * kBK * 2;     // 8 KiB (room for 64 rows)
constexpr int kMaxSplit = 16;

struct __align__(1024) SkSmem {
  uint8_t b[kStages][kBBytes];  // B tile, N-major: the MMA's A operand
  uint8_t a[kStages][kABytes];  // A tile, K-major: the MMA's B operand
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t tmem_full[2];
  uint64_t tmem_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

template <bool kInt>
struct SkArgs {
  using Out = typename std::conditional<kInt, int32_t, float>::type;
  int M, N, K;
  int mp;  // M rounded up to a multiple of 16 (the MMA's N)
  Out alpha, beta;
  Out *C;
  int64_t ldc;
  int split;           // parts of k per column block
  uint32_t *counters;  // parts done, one per column block (split > 1), zero at launch
  Out *ws;             // partial sums [split][M][ws_ld] (split > 1)
  int64_t ws_ld;       // column blocks * 128
  uint32_t idesc;
  uint32_t *err_word;
};

__device__ __forceinline__ bool drain_wait(uint32_t bar, uint32_t parity, uint32_t *err_word) {
  volatile int never = 0;
  return mbar_wait_bounded(bar, parity, &never, err_word, kWaitDrain);
}

__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%16];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void epilogue_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(32 * kEpiWarps) : "memory");
}

__device__ __forceinline__ float axpby(float a, float x, float b, float c, bool use_c) {
  return use_c ? a * x + b * c : a * x;
}
__device__ __forceinline__ int32_t axpby(int32_t a, int32_t x, int32_t b, int32_t c,
                                         bool use_c) {
  uint32_t r = static_cast<uint32_t>(a) * static_cast<uint32_t>(x);
  if (use_c) r += static_cast<uint32_t>(b) * static_cast<uint32_t>(c);
  return static_cast<int32_t>(r);
}

template <bool kInt>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_skinny_kernel(const __grid_constant__ CUtensorMap tmA,
                          const __grid_constant__ CUtensorMap tmB, const SkArgs<kInt> p) {
  using Out = typename SkArgs<kInt>::Out;
  extern __shared__ uint8_t smem_raw[];
  SkSmem &sm = *reinterpret_cast<SkSmem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int *abort = &sm.abort;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&sm.full[s]), 1);
      mbar_init(smem_u32(&sm.empty[s]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&sm.tmem_full[i]), 1);
      mbar_init(smem_u32(&sm.tmem_empty[i]), kEpiWarps);
    }
    mbar_init(smem_u32(&sm.drain), 1);
    sm.abort = 0;
    fence_mbar_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&sm.tmem_base), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = sm.tmem_base;

  // This CTA's slice: column block `blk`, part `part` of the k range.
  const int blk = static_cast<int>(blockIdx.x) / p.split;
  const int part = static_cast<int>(blockIdx.x) % p.split;
  const int n0 = blk * kBN;
  const int KB = (p.K + kBK - 1) / kBK;
  const int kb_unit = kInt ? kChunkKB : 1;
  const int nunits = (KB + kb_unit - 1) / kb_unit;
  const int kb0 = min(KB, (part * nunits / p.split) * kb_unit);
  const int kb1 = min(KB, ((part + 1) * nunits / p.split) * kb_unit);
  const int chunk_kb = kInt ? kChunkKB : KB;
  const uint32_t a_bytes = static_cast<uint32_t>(p.mp) * kBK * 2;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, issued = 0, issued_parity = 0;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait_bounded(smem_u32(&sm.empty[stage]), phase ^ 1u, abort, p.err_word,
                               kWaitEmpty))
          break;
        const uint32_t full_bar = smem_u32(&sm.full[stage]);
        mbar_arrive_expect_tx(full_bar, kBBytes + a_bytes);
        tma_load_2d(smem_u32(sm.b[stage]), &tmB, full_bar, n0, kb * kBK);
        tma_load_2d(smem_u32(sm.b[stage] + kBBox), &tmB, full_bar, n0 + 64, kb * kBK);
        tma_load_2d(smem_u32(sm.a[stage]), &tmA, full_bar, kb * kBK, 0);
        issued |= 1u << stage;
        issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      for (int s = 0; s < kStages; ++s)
        if (issued & (1u << s))
          drain_wait(smem_u32(&sm.full[s]), (issued_parity >> s) & 1u, p.err_word);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, chunk = 0;
      bool ok = true, any = false;
      for (int c0 = kb0; ok && c0 < kb1; c0 += chunk_kb) {
        const int c1 = min(kb1, c0 + chunk_kb);
        const uint32_t buf = chunk & 1u, use = (chunk >> 1) & 1u;
        ++chunk;
        if (!mbar_wait_bounded(smem_u32(&sm.tmem_empty[buf]), use ^ 1u, abort, p.err_word,
                               kWaitTmemEmpty))
          break;
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + buf * kBufCols;
        for (int kb = c0; kb < c1; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&sm.full[stage]), phase, abort, p.err_word,
                                 kWaitFull)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t b_addr = smem_u32(sm.b[stage]);
          const uint32_t a_addr = smem_u32(sm.a[stage]);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            // MMA A operand = B tile, N-major: LBO = one 64-column box, SBO = 1 KiB
            // between groups of 8 k-rows; 16 k = 16 rows of 128 B further.
            const uint64_t adesc = smem_desc(b_addr + kk * 2048, kBBox, 1024, 2u);
            // MMA B operand = A tile, K-major: SBO = 8 rows of 128 B; 16 k = 32 B.
            const uint64_t bdesc = smem_desc(a_addr + kk * 32, 16, 1024, 2u);
            tc_mma_f16(d_tmem, adesc, bdesc, p.idesc, (kb > c0 || kk > 0) ? 1u : 0u);
          }
          any = true;
          tc_commit(smem_u32(&sm.empty[stage]));
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(smem_u32(&sm.tmem_full[buf]));
      }
      if (any) {
        tc_commit(smem_u32(&sm.drain));
        drain_wait(smem_u32(&sm.drain), 0, p.err_word);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    // Lanes are columns of C: lane -> column n0 + 32 * quarter + lane.
    const int quarter = warp & 3;
    const int n = n0 + quarter * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    uint32_t acc[kInt ? kMaxM : 1];
    if constexpr (kInt) {
#pragma unroll
      for (int j = 0; j < kMaxM; ++j) acc[j] = 0;
    }
    float facc[kInt ? 1 : kMaxM];
    uint32_t chunk = 0;
    for (int c0 = kb0; c0 < kb1; c0 += chunk_kb) {
      const uint32_t buf = chunk & 1u, use = (chunk >> 1) & 1u;
      ++chunk;
      int got = 0;
      if (lane == 0)
        got = mbar_wait_bounded(smem_u32(&sm.tmem_full[buf]), use, abort, p.err_word,
                                kWaitTmemFull);
      got = __shfl_sync(0xffffffffu, got, 0);
      if (!got) break;
      tc_fence_after_sync();
      const uint32_t taddr = tmem_base + lane_base + buf * 64;
#pragma unroll
      for (int c = 0; c < kMaxM; c += 16) {
        if (c < p.mp) {
          uint32_t r[16];
          tmem_ld_32x32b_x16(taddr + c, r);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            if constexpr (kInt) {
              acc[c + j] += static_cast<uint32_t>(__float2int_rn(__uint_as_float(r[j])));
            } else {
              facc[c + j] = __uint_as_float(r[j]);
            }
          }
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.tmem_empty[buf]));
    }
    auto value = [&](int m) -> Out {
      if constexpr (kInt) {
        return static_cast<int32_t>(acc[m]);
      } else {
        return facc[m];
      }
    };
    const bool use_c = p.beta != Out(0);
    if (p.split == 1) {
      if (n < p.N && !*abort && kb1 > kb0) {
#pragma unroll
        for (int m = 0; m < kMaxM; ++m)
          if (m < p.M) {
            Out *cp = p.C + static_cast<int64_t>(m) * p.ldc + n;
            *cp = axpby(p.alpha, value(m), p.beta, use_c ? *cp : Out(0), use_c);
          }
      }
    } else {
      // Store this part's partial sums, count the part done; the last part of
      // the column block adds all parts in order.
#pragma unroll
      for (int m = 0; m < kMaxM; ++m)
        if (m < p.M) p.ws[(static_cast<int64_t>(part) * p.M + m) * p.ws_ld + n] = value(m);
      __threadfence();
      epilogue_sync();
      __shared__ int last;
      if (warp == 2 && lane == 0)
        last = (atomicAdd(p.counters + blk, 1u) == static_cast<uint32_t>(p.split - 1));
      epilogue_sync();
      if (last) {
        __threadfence();
        if (n < p.N) {
#pragma unroll 1
          for (int m = 0; m < p.M; ++m) {
            Out sum = Out(0);
            for (int q = 0; q < p.split; ++q) {
              const Out v = __ldcg(p.ws + (static_cast<int64_t>(q) * p.M + m) * p.ws_ld + n);
              if constexpr (kInt) {
                sum = static_cast<int32_t>(static_cast<uint32_t>(sum) + static_cast<uint32_t>(v));
              } else {
                sum += v;
              }
            }
            Out *cp = p.C + static_cast<int64_t>(m) * p.ldc + n;
            *cp = axpby(p.alpha, sum, p.beta, use_c ? *cp : Out(0), use_c);
          }
        }
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void *q = nullptr;
    cudaDriverEntryPointQueryResult r;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &q, 12000, cudaEnableDefault,
                                         &r) == cudaSuccess &&
        r == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(q);
  });
  return fn;
}

// Row-major rows x cols 16-bit matrix, boxes of box_rows x 64 elements, 128-byte swizzle.
bool tmap16(CUtensorMap *tm, CUtensorMapDataType dt, const void *base, int64_t rows,
            int64_t cols, int64_t ld, uint32_t box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(tm, dt, 2, const_cast<void *>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

template <bool kInt>
cudaError_t launch(const DeviceInfo &dev, CUtensorMapDataType dt, bool is_bf16, int M, int N,
                   int K, typename SkArgs<kInt>::Out alpha, const void *A, int64_t lda,
                   const void *B, int64_t ldb, typename SkArgs<kInt>::Out beta,
                   typename SkArgs<kInt>::Out *C, int64_t ldc, cudaStream_t stream,
                   uint32_t *flags_ws, size_t flags_words) {
  if (M < 1 || M > kMaxM) return cudaErrorInvalidValue;
  SkArgs<kInt> p;
  p.M = M;
  p.N = N;
  p.K = K;
  p.mp = (M + 15) / 16 * 16;
  p.alpha = alpha;
  p.beta = beta;
  p.C = C;
  p.ldc = ldc;
  p.idesc = idesc_f16(is_bf16, /*a_mn_major=*/true, /*b_mn_major=*/false, kBN, p.mp);
  p.err_word = dev.err_word;
  CUtensorMap tmA, tmB;
  if (!tmap16(&tmA, dt, A, M, K, lda, static_cast<uint32_t>(p.mp))) return cudaErrorInvalidValue;
  if (!tmap16(&tmB, dt, B, K, N, ldb, kBK)) return cudaErrorInvalidValue;

  // One slice per CTA: column blocks times parts of k, at most one CTA per SM
  // when k is split.
  const int blocks = (N + kBN - 1) / kBN;
  const int KB = (K + kBK - 1) / kBK;
  const int nunits = kInt ? (KB + kChunkKB - 1) / kChunkKB : KB;
  int split = blocks < dev.sm_count ? dev.sm_count / blocks : 1;
  if (split > kMaxSplit) split = kMaxSplit;
  if (split > nunits) split = nunits;
  if (split < 1) split = 1;

  // split > 1 needs a workspace for the partial sums (from the pool); a caller
  // that provides its own memory gets whole column blocks instead.
  if (flags_ws != nullptr) split = 1;
  (void)flags_words;
  void *pool_ws = nullptr;
  p.counters = nullptr;
  p.ws = nullptr;
  p.ws_ld = static_cast<int64_t>(blocks) * kBN;
  if (split > 1) {
    cudaMemPool_t pool;
    cudaError_t e = device_pool(dev, &pool);
    if (e != cudaSuccess) return e;
    const size_t ws_bytes =
        static_cast<size_t>(split) * M * p.ws_ld * sizeof(typename SkArgs<kInt>::Out);
    const size_t cnt_off = (ws_bytes + 255) / 256 * 256;
    e = cudaMallocFromPoolAsync(&pool_ws, cnt_off + static_cast<size_t>(blocks) * 4, pool,
                                stream);
    if (e != cudaSuccess) return e;
    p.ws = static_cast<typename SkArgs<kInt>::Out *>(pool_ws);
    p.counters = reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(pool_ws) + cnt_off);
    e = cudaMemsetAsync(p.counters, 0, static_cast<size_t>(blocks) * 4, stream);
    if (e != cudaSuccess) {
      cudaFreeAsync(pool_ws, stream);
      return e;
    }
  }
  p.split = split;

  const size_t smem = sizeof(SkSmem) + 1024;
  static_assert(sizeof(SkSmem) + 1024 <= 232448, "skinny kernel shared memory");
  auto kern = gemm_tc_skinny_kernel<kInt>;
  cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void *>(kern),
                                       static_cast<int>(smem), dev.device);
  if (e == cudaSuccess) {
    kern<<<static_cast<unsigned>(blocks * split), kThreads, smem, stream>>>(tmA, tmB, p);
    e = cudaGetLastError();
  }
  if (pool_ws) {
    cudaError_t f = cudaFreeAsync(pool_ws, stream);
    if (e == cudaSuccess) e = f;
  }
  return e;
}

}  // namespace

cudaError_t launch_tc_skinny_float(const DeviceInfo &dev, bool is_bf16, int M, int N, int K,
                                   float alpha, const void *A, int64_t lda, const void *B,
                                   int64_t ldb, float beta, float *C, int64_t ldc,
                                   cudaStream_t stream) {
  return launch<false>(dev,
                       is_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                       is_bf16, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream, nullptr, 0);
}

cudaError_t launch_tc_skinny_int(const DeviceInfo &dev, int M, int N, int K, int32_t alpha,
                                 const void *A16, int64_t lda, const void *B16, int64_t ldb,
                                 int32_t beta, int32_t *C, int64_t ldc, cudaStream_t stream,
                                 uint32_t *flags, size_t flags_words) {
  return launch<true>(dev, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, false, M, N, K, alpha, A16, lda, B16,
                      ldb, beta, C, ldc, stream, flags, flags_words);
}

}  // namespace dgr
