// gemm_tc.cu -- tensor-core GEMM for sm_103a: tcgen05.mma with the
// accumulator in tensor memory (TMEM), operands staged by TMA.
//
//     C = alpha * op(A) * op(B) + beta * C      op(A): M x K, op(B): K x N,
//                                                C: M x N, all row-major
//
// op(X) is X as stored or its transpose, and the problem may be a stack of
// `batch` such GEMMs at fixed element strides (strided-batched GEMM). Neither
// costs anything on this path: a transposed operand is staged by TMA in the
// other major order and the MMA's descriptors say so; the batch index is the
// third coordinate of every tensor map and one more dimension of the tile
// list.
//
// 16-bit inputs (bf16 or fp16), fp32 accumulation, and either
//   * fp32 output (gemm_bf16 / gemm_f16), or
//   * exact int32 output from integer-valued fp16 operands (the int8 path: an
//     int8 value is exact in fp16, a product of two is at most 2^14 in
//     magnitude, and a sum of at most 1024 such products is an integer of at
//     most 2^24 in magnitude, which fp32 represents exactly. The kernel
//     therefore restarts the fp32 accumulator every 1024 values of k, and the
//     epilogue adds each finished partial sum into int32 registers).
//
// Sources: C++ warp-matrix-function page (D = A*B + C on tensor cores; type
// table: half / bfloat16 inputs with float accumulate, signed char inputs with
// int accumulate); "Sgemm [128,128,8]" (C = alpha*A*B + beta*C, row-major, the
// alpha/beta epilogue); "使用CUDA和瓦片算法计算矩阵乘法" (residual tiles act as
// zeros: here the TMA unit fills out-of-range elements with zeros).
//
// Structure (one CTA per SM, persistent):
//   warp 0      one thread issues TMA loads of A (128 x 64, K-major, 128-byte
//               swizzle) and B (64 x 256 as four 64 x 64 boxes, N-major,
//               128-byte swizzle) into a kStages-deep ring guarded by
//               full/empty mbarriers. A stored transposed (K x M) arrives as
//               two 64(M) x 64(K) M-major boxes; B stored transposed (N x K)
//               as one 256(N) x 64(K) K-major box. Every layout fills the same
//               bytes per stage.
//   warp 1      allocates 512 TMEM columns; one thread issues
//               tcgen05.mma.cta_group::1.kind::f16 (M=128, N=256, K=16) into
//               one of two 256-column accumulators and commits each stage's
//               completion to that stage's empty barrier.
//   warps 2..9  epilogue: tcgen05.ld of the finished accumulator (each warp
//               reads its 32-lane quarter and one 128-column half), then
//               alpha/beta and guarded stores to C. The two accumulators let
//               the epilogue of one tile overlap the main loop of the next.
// Tiles are visited in groups of kGroupM tile rows so that the CTAs resident
// at one time share A rows and B columns in L2.
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

#ifndef DGR_TC_BK
#define DGR_TC_BK 64
#endif
#ifndef DGR_TC_STAGES
#define DGR_TC_STAGES 4
#endif
#ifndef DGR_TC_STAGES_PAIR
#define DGR_TC_STAGES_PAIR 6
#endif
#ifndef DGR_TC_GROUP_M
#define DGR_TC_GROUP_M 16
#endif
#ifndef DGR_TC_GROUP_M_PAIR
#define DGR_TC_GROUP_M_PAIR 8
#endif
#ifndef DGR_TC_PAIR
#define DGR_TC_PAIR 1
#endif

// k-block: 64 16-bit values (one 128-byte swizzle row of A) or 32 (64-byte rows).
constexpr int kBK = DGR_TC_BK;
static_assert(kBK == 64 || kBK == 32, "k-block of 32 or 64 values");
constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + 32 * kEpiWarps;
// int mode: k-blocks per exact fp32 chunk (1024 values of k)
constexpr int kChunkKB = 1024 / kBK;
constexpr uint32_t kTmemCols = 512;  // two 256-column fp32 accumulators
constexpr int kBN = 256;             // tile columns (MMA N)
constexpr int kBM = 128;             // tile rows held by one CTA (TMEM lanes)

// A rows are kBK * 2 bytes long: 128-byte swizzle for 64 values, 64-byte for 32.
constexpr uint32_t kARowBytes = kBK * 2;
constexpr uint32_t kASwizzleMode = kBK == 64 ? 2u : 4u;   // descriptor encoding
constexpr uint32_t kAAtomBytes = 8 * kARowBytes;          // 8-row swizzle atom
constexpr uint32_t kMNBoxBytes = 64 * kBK * 2;            // any 64(M or N) x kBK MN-major box

// Single CTA: 128 x 256 tile, the CTA stages all 256 columns of B.
// CTA pair:   256 x 256 tile, each CTA stages its 128 rows of A and its 128
//             columns of B; the leader's MMA (M = 256) reads both CTAs.
template <bool kPair>
struct Cfg {
  static constexpr int kTileM = kPair ? 256 : 128;
  static constexpr int kBNLoad = kPair ? 128 : 256;   // B columns staged per CTA
  static constexpr int kStages = kPair ? DGR_TC_STAGES_PAIR : DGR_TC_STAGES;
  // Tiles are visited in groups of kGroupM tile rows so that the CTAs resident
  // at one time share A rows and B columns in L2.
  static constexpr int kGroupM = kPair ? DGR_TC_GROUP_M_PAIR : DGR_TC_GROUP_M;
  static constexpr uint32_t kABytes = kBM * kBK * 2;
  static constexpr uint32_t kBBytes = kBK * kBNLoad * 2;
  static constexpr uint32_t kStageBytes = kABytes + kBBytes;           // per CTA
  static constexpr uint32_t kTxBytes = kStageBytes * (kPair ? 2 : 1);  // per full phase
};

// Epilogue staging: one 32 x 32 x 4-byte block of C per epilogue warp, in the
// 128-byte-swizzled layout of the C tensor map's box.
constexpr uint32_t kStageCBytes = 32 * 128;

template <bool kPair>
struct __align__(1024) TcSmem {
  uint8_t a[Cfg<kPair>::kStages][Cfg<kPair>::kABytes];
  uint8_t b[Cfg<kPair>::kStages][Cfg<kPair>::kBBytes];
  uint8_t stage_c[kEpiWarps][kStageCBytes];
  uint64_t full[Cfg<kPair>::kStages];
  uint64_t empty[Cfg<kPair>::kStages];
  uint64_t tmem_full[2];
  uint64_t tmem_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

template <bool kInt>
struct TcArgs {
  using Out = typename std::conditional<kInt, int32_t, float>::type;
  int M, N, K;
  Out alpha, beta;
  Out *C;
  int64_t ldc;
  int tiles_m, tiles_n;
  int tiles_per_batch;   // tiles_m * tiles_n; tile t is tile t % this of matrix t / this
  int a_batched, b_batched;  // the operand's tensor map has one matrix per batch entry
  int64_t stride_c;      // elements between consecutive C matrices
  int c_vec_ok;  // C 16-byte aligned and ldc % 4 == 0
  int c_tma;     // the epilogue writes C through the C tensor map (needs c_vec_ok)
  uint32_t idesc;
  uint32_t *err_word;
  // Work split: the first dp_tiles tiles (a multiple of the number of units)
  // are computed whole, round-robin; each of the remaining tail_tiles tiles
  // is split along k into `split` parts, one per unit. Part j > 0 adds its
  // partial product into C after part j - 1 has stored (tail flags, one per
  // tail tile and CTA of a pair, zero at launch).
  int dp_tiles, tail_tiles, split;
  uint32_t *tail_flags;
};

// One item of a unit's work list: a tile and a range of its k-blocks.
struct WorkItem {
  int tile, kb0, kb1, part, parts;
};

// Item n of unit u's work list (false past its end). kb_unit is the k
// granularity of split points: 1 k-block, or one exact 1024-k chunk in int
// mode.
__device__ __forceinline__ bool get_work(int u, int n, int units, int dp_tiles, int tail_tiles,
                                         int split, int KB, int kb_unit, WorkItem &w) {
  const int dp_per_unit = dp_tiles / units;
  if (n < dp_per_unit) {
    w.tile = u + n * units;
    w.kb0 = 0;
    w.kb1 = KB;
    w.part = 0;
    w.parts = 1;
    return true;
  }
  if (n == dp_per_unit && u < tail_tiles * split) {
    w.tile = dp_tiles + u / split;
    w.part = u % split;
    w.parts = split;
    const int nunits = (KB + kb_unit - 1) / kb_unit;
    w.kb0 = min(KB, (w.part * nunits / split) * kb_unit);
    w.kb1 = min(KB, ((w.part + 1) * nunits / split) * kb_unit);
    return true;
  }
  return false;
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t *p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_gpu(uint32_t *p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Bounded wait until *flag >= value (another unit's part has been stored).
__device__ __forceinline__ bool wait_flag(const uint32_t *flag, uint32_t value,
                                          volatile int *abort, uint32_t *err_word) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 0;; ++it) {
    if (ld_acquire_gpu(flag) >= value) return true;
    __nanosleep(128);  // keep the polling off the L2 the other units are streaming from
    if ((it & 63u) == 63u) {
      if (*abort) return false;
      if (global_timer_ns() - t0 > kWaitLimitNs || it >= kWaitMaxPolls) {
        *abort = 1;
        record_timeout(err_word, kWaitFlag);
        return false;
      }
    }
  }
}

// Barrier among the epilogue warps only (named barrier 1).
__device__ __forceinline__ void epilogue_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(32 * kEpiWarps) : "memory");
}

template <int kGroupM>
__device__ __forceinline__ void tile_coords(int t, int tiles_m, int tiles_n, int &tm, int &tn) {
  const int per_group = kGroupM * tiles_n;
  const int g = t / per_group;
  const int first = g * kGroupM;
  const int rows = min(tiles_m - first, kGroupM);
  const int r = t - g * per_group;
  tm = first + r % rows;
  tn = r / rows;
}

// Tile t of a batched problem: batch entry bt, tile (tm, tn) within it. The
// tiles of one matrix are contiguous in t, so the resident CTAs work on one or
// two matrices at a time and the grouped raster's L2 reuse holds within each.
template <int kGroupM, bool kInt>
__device__ __forceinline__ void batch_tile_coords(int t, const TcArgs<kInt> &p, int &bt, int &tm,
                                                  int &tn) {
  bt = t / p.tiles_per_batch;
  tile_coords<kGroupM>(t - bt * p.tiles_per_batch, p.tiles_m, p.tiles_n, tm, tn);
}

// Waits without looking at the abort flag (used to drain in-flight work).
__device__ __forceinline__ bool drain_wait(uint32_t bar, uint32_t parity, uint32_t *err_word) {
  volatile int never = 0;
  return mbar_wait_bounded(bar, parity, &never, err_word, kWaitDrain);
}

// alpha*acc + beta*c (the c term only when use_c). fp32: two roundings, or one
// when the compiler fuses them. int32: wrap-around, computed in unsigned
// arithmetic so that overflow is defined.
__device__ __forceinline__ float scale_add(float alpha, float acc, float beta, float c,
                                           bool use_c) {
  return use_c ? alpha * acc + beta * c : alpha * acc;
}
__device__ __forceinline__ int32_t scale_add(int32_t alpha, int32_t acc, int32_t beta, int32_t c,
                                             bool use_c) {
  uint32_t r = static_cast<uint32_t>(alpha) * static_cast<uint32_t>(acc);
  if (use_c) r += static_cast<uint32_t>(beta) * static_cast<uint32_t>(c);
  return static_cast<int32_t>(r);
}

// C[row, col .. col+31] = alpha * v + beta * C (the C term only when use_c).
// C is read through L2 (another SM may have just written it).
template <bool kInt>
__device__ __forceinline__ void store_row_chunk(const TcArgs<kInt> &p,
                                                typename TcArgs<kInt>::Out *C, int row, int col,
                                                const typename TcArgs<kInt>::Out (&v)[32],
                                                typename TcArgs<kInt>::Out beta, bool use_c) {
  using Out = typename TcArgs<kInt>::Out;
  Out *crow = C + static_cast<int64_t>(row) * p.ldc;
  const Out alpha = p.alpha;
  if (p.c_vec_ok && col + 31 < p.N) {
    using Vec = typename std::conditional<kInt, int4, float4>::type;
#pragma unroll
    for (int j = 0; j < 32; j += 4) {
      Vec c = {};
      if (use_c) c = __ldcg(reinterpret_cast<const Vec *>(crow + col + j));
      Vec o;
      o.x = scale_add(alpha, v[j], beta, c.x, use_c);
      o.y = scale_add(alpha, v[j + 1], beta, c.y, use_c);
      o.z = scale_add(alpha, v[j + 2], beta, c.z, use_c);
      o.w = scale_add(alpha, v[j + 3], beta, c.w, use_c);
      *reinterpret_cast<Vec *>(crow + col + j) = o;
    }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      if (col + j < p.N) {
        const Out c = use_c ? __ldcg(crow + col + j) : Out(0);
        crow[col + j] = scale_add(alpha, v[j], beta, c, use_c);
      }
    }
  }
}

// Writes one 32 x 32 block of C matrix z (rows y .. y+31, columns x .. x+31;
// the lane's row is y + lane) from registers: stages it in the warp's swizzled
// buffer and issues one TMA store, or one TMA reduce-add when `addto`
// (C += block). Elements outside C are dropped by the tensor map's bounds.
__device__ __forceinline__ void tma_write_block(uint32_t stage, const void *tmC, int x, int y,
                                                int z, int M, int N, const uint32_t (&w)[32],
                                                bool addto, int lane) {
  if (lane == 0) bulk_wait_read_all();  // the previous block has left the buffer
  __syncwarp();
  const uint32_t row = stage + static_cast<uint32_t>(lane) * 128u;
#pragma unroll
  for (int j = 0; j < 8; ++j)
    st_shared_v4(row + ((static_cast<uint32_t>(j) ^ (lane & 7u)) << 4), w[4 * j], w[4 * j + 1],
                 w[4 * j + 2], w[4 * j + 3]);
  fence_proxy_async_shared();
  __syncwarp();
  if (lane == 0 && x < N && y < M) {  // a block wholly outside C issues nothing
    if (addto) {
      tma_reduce_add_3d(tmC, x, y, z, stage);
    } else {
      tma_store_3d(tmC, x, y, z, stage);
    }
    bulk_commit();
  }
}

// kAT / kBT: A stored K x M / B stored N x K (used transposed).
template <bool kInt, bool kPair, bool kAT, bool kBT>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const TcArgs<kInt> p) {
  using Cf = Cfg<kPair>;
  using Out = typename TcArgs<kInt>::Out;
  constexpr int kStages = Cf::kStages;
  extern __shared__ uint8_t smem_raw[];
  // Swizzled TMA destinations need 1024-byte alignment. The offset is the same
  // in both CTAs of a pair, which the pair MMA relies on.
  TcSmem<kPair> &sm = *reinterpret_cast<TcSmem<kPair> *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int *abort = &sm.abort;

  uint32_t rank = 0;  // rank within the CTA pair; rank 0 issues the MMAs
  if constexpr (kPair) rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int unit = kPair ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int units = kPair ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&sm.full[s]), 1);
      mbar_init(smem_u32(&sm.empty[s]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&sm.tmem_full[i]), 1);
      mbar_init(smem_u32(&sm.tmem_empty[i]), kEpiWarps * (kPair ? 2 : 1));
    }
    mbar_init(smem_u32(&sm.drain), 1);
    sm.abort = 0;
    fence_mbar_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    if (p.c_tma) prefetch_tmap(&tmC);
  }
  if (warp == 1) {
    if constexpr (kPair) {
      tmem_alloc_pair(smem_u32(&sm.tmem_base), kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(&sm.tmem_base), kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before_sync();
  if constexpr (kPair) {
    cluster_sync();  // the leader's barriers exist before the peer signals them
  } else {
    __syncthreads();
  }
  tc_fence_after_sync();
  const uint32_t tmem_base = sm.tmem_base;

  const int KB = (p.K + kBK - 1) / kBK;
  // int mode: exact fp32 chunks of 1024 k; float mode: one chunk per item
  const int chunk_kb = kInt ? kChunkKB : KB;
  const int kb_unit = kInt ? kChunkKB : 1;
  WorkItem wi;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      uint32_t issued = 0;         // stages with a load issued
      uint32_t issued_parity = 0;  // parity of the last load issued per stage
      bool ok = true;
      for (int n = 0; ok && get_work(unit, n, units, p.dp_tiles, p.tail_tiles, p.split, KB,
                                     kb_unit, wi);
           ++n) {
        int bt, tm, tn;
        batch_tile_coords<Cf::kGroupM>(wi.tile, p, bt, tm, tn);
        const int m0 = tm * Cf::kTileM + static_cast<int>(rank) * kBM;
        const int nb = tn * kBN + static_cast<int>(rank) * Cf::kBNLoad;
        const int za = p.a_batched ? bt : 0, zb = p.b_batched ? bt : 0;
        for (int kb = wi.kb0; kb < wi.kb1; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&sm.empty[stage]), phase ^ 1u, abort, p.err_word,
                                 kWaitEmpty)) {
            ok = false;
            break;
          }
          const uint32_t full_bar = smem_u32(&sm.full[stage]);
          if (leader) mbar_arrive_expect_tx(full_bar, Cf::kTxBytes);
          // A pair's loads signal the leader's barrier; a single CTA's its own.
          const uint32_t bar = kPair ? mapa_shared(full_bar, 0) : full_bar;
          auto load = [&](uint32_t dst, const CUtensorMap *tm, int x, int y, int z) {
            if constexpr (kPair) {
              tma_load_3d_pair(dst, tm, bar, x, y, z);
            } else {
              tma_load_3d(dst, tm, bar, x, y, z);
            }
          };
          const int k0 = kb * kBK;
          if constexpr (!kAT) {
            load(smem_u32(sm.a[stage]), &tmA, k0, m0, za);  // 128 rows x kBK, K-major
          } else {
#pragma unroll
            for (int j = 0; j < kBM / 64; ++j)  // kBK rows of k x 64 values of m, twice
              load(smem_u32(sm.a[stage] + j * kMNBoxBytes), &tmA, m0 + 64 * j, k0, za);
          }
          if constexpr (!kBT) {
#pragma unroll
            for (int j = 0; j < Cf::kBNLoad / 64; ++j)  // kBK rows of k x 64 values of n
              load(smem_u32(sm.b[stage] + j * kMNBoxBytes), &tmB, nb + 64 * j, k0, zb);
          } else {
            load(smem_u32(sm.b[stage]), &tmB, k0, nb, zb);  // kBNLoad rows x kBK, K-major
          }
          issued |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Never leave with a copy still writing into shared memory. The leader's
      // full barriers count both CTAs' bytes; the peer CTA is held at the final
      // cluster barrier until the leader has drained.
      if (leader)
        for (int s = 0; s < kStages; ++s)
          if (issued & (1u << s))
            drain_wait(smem_u32(&sm.full[s]), (issued_parity >> s) & 1u, p.err_word);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0 && leader) {
      uint32_t stage = 0, phase = 0, chunk = 0;
      bool ok = true;
      bool any = false;
      for (int n = 0; ok && get_work(unit, n, units, p.dp_tiles, p.tail_tiles, p.split, KB,
                                     kb_unit, wi);
           ++n) {
        for (int kb0 = wi.kb0; ok && kb0 < wi.kb1; kb0 += chunk_kb) {
          const int kb1 = min(wi.kb1, kb0 + chunk_kb);
          const uint32_t buf = chunk & 1u, use = (chunk >> 1) & 1u;
          ++chunk;
          bool got;
          if constexpr (kPair) {
            got = mbar_wait_bounded_cluster(smem_u32(&sm.tmem_empty[buf]), use ^ 1u, abort,
                                            p.err_word, kWaitTmemEmpty);
          } else {
            got = mbar_wait_bounded(smem_u32(&sm.tmem_empty[buf]), use ^ 1u, abort, p.err_word,
                                    kWaitTmemEmpty);
          }
          if (!got) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t d_tmem = tmem_base + buf * kBN;
          for (int kb = kb0; kb < kb1; ++kb) {
            if (!mbar_wait_bounded(smem_u32(&sm.full[stage]), phase, abort, p.err_word,
                                   kWaitFull)) {
              ok = false;
              break;
            }
            tc_fence_after_sync();
            const uint32_t a_addr = smem_u32(sm.a[stage]);
            const uint32_t b_addr = smem_u32(sm.b[stage]);
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk) {
              // K-major operand: swizzled rows of kBK values; 16 values of k =
              // 32 B further along the row; SBO = one 8-row swizzle atom.
              // MN-major operand: 128-byte swizzled rows of 64 values of m or n,
              // one row per k; 16 values of k = 16 * 128 B further; LBO = one
              // 64-value box, SBO = 1 KiB between groups of 8 k-rows.
              const uint64_t adesc =
                  kAT ? smem_desc(a_addr + kk * 2048, kMNBoxBytes, 1024, 2u)
                      : smem_desc(a_addr + kk * 32, 16, kAAtomBytes, kASwizzleMode);
              const uint64_t bdesc =
                  kBT ? smem_desc(b_addr + kk * 32, 16, kAAtomBytes, kASwizzleMode)
                      : smem_desc(b_addr + kk * 2048, kMNBoxBytes, 1024, 2u);
              const uint32_t acc = (kb > kb0 || kk > 0) ? 1u : 0u;
              if constexpr (kPair) {
                tc_mma_f16_pair(d_tmem, adesc, bdesc, p.idesc, acc);
              } else {
                tc_mma_f16(d_tmem, adesc, bdesc, p.idesc, acc);
              }
            }
            any = true;
            // This stage's shared memory is free again in both CTAs.
            if constexpr (kPair) {
              tc_commit_pair_mc(smem_u32(&sm.empty[stage]), 0x3);
            } else {
              tc_commit(smem_u32(&sm.empty[stage]));
            }
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          if constexpr (kPair) {
            tc_commit_pair_mc(smem_u32(&sm.tmem_full[buf]), 0x3);
          } else {
            tc_commit(smem_u32(&sm.tmem_full[buf]));
          }
        }
      }
      // Never leave with an MMA still reading shared memory or writing TMEM.
      if (any) {
        if constexpr (kPair) {
          tc_commit_pair_mc(smem_u32(&sm.drain), 0x1);
        } else {
          tc_commit(smem_u32(&sm.drain));
        }
        drain_wait(smem_u32(&sm.drain), 0, p.err_word);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    // Every epilogue warp walks the same work list and meets the same named
    // barriers, whatever happens to its waits, so none can be left behind.
    const int e = warp - 2;
    const int quarter = warp & 3;  // TMEM lanes this warp may access
    const int col_half = e >> 2;   // which 128 columns of the tile
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const bool flag_thread = (e == 0 && lane == 0);
    uint32_t chunk = 0;
    for (int n = 0;
         get_work(unit, n, units, p.dp_tiles, p.tail_tiles, p.split, KB, kb_unit, wi); ++n) {
      int bt, tm, tn;
      batch_tile_coords<Cf::kGroupM>(wi.tile, p, bt, tm, tn);
      Out *const Cb = p.C + static_cast<int64_t>(bt) * p.stride_c;
      const int row = tm * Cf::kTileM + static_cast<int>(rank) * kBM + quarter * 32 + lane;
      const int col0 = tn * kBN + col_half * 128;
      // Part 0 (or a whole tile) applies beta to the old C; a later part adds
      // its partial product to what the previous part stored.
      const bool addto = wi.part > 0;
      const Out beta = addto ? Out(1) : p.beta;
      const bool use_c = addto || p.beta != Out(0);
      uint32_t *flag = nullptr;
      if (wi.parts > 1)
        flag = p.tail_flags + (wi.tile - p.dp_tiles) * 2 + static_cast<int>(rank);
      if (addto) {
        if (flag_thread) wait_flag(flag, static_cast<uint32_t>(wi.part), abort, p.err_word);
        epilogue_sync();
      }
      uint32_t acc[kInt ? 128 : 1];  // int mode: running int32 sums (wrap-around)
      if constexpr (kInt) {
#pragma unroll
        for (int j = 0; j < 128; ++j) acc[j] = 0;
      }
      for (int kb0 = wi.kb0; kb0 < wi.kb1; kb0 += chunk_kb) {
        const uint32_t buf = chunk & 1u, use = (chunk >> 1) & 1u;
        ++chunk;
        int got = 0;
        if (lane == 0)
          got = mbar_wait_bounded(smem_u32(&sm.tmem_full[buf]), use, abort, p.err_word,
                                  kWaitTmemFull);
        got = __shfl_sync(0xffffffffu, got, 0);
        if (!got) break;
        tc_fence_after_sync();
        const uint32_t taddr = tmem_base + lane_base + buf * kBN + col_half * 128;
#pragma unroll
        for (int c = 0; c < 128; c += 32) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(taddr + c, r);
          tmem_ld_wait();
          if constexpr (kInt) {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              acc[c + j] += static_cast<uint32_t>(__float2int_rn(__uint_as_float(r[j])));
          } else if (p.c_tma) {
            if (!*abort) {
              uint32_t w[32];
              const bool read_c = use_c && !addto && row < p.M;
              const float *crow = Cb + static_cast<int64_t>(row) * p.ldc + col0 + c;
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                const float c0 = (read_c && col0 + c + j < p.N) ? __ldcg(crow + j) : 0.f;
                w[j] = __float_as_uint(
                    scale_add(p.alpha, __uint_as_float(r[j]), beta, c0, read_c));
              }
              tma_write_block(smem_u32(sm.stage_c[e]), &tmC, col0 + c, row - lane, bt, p.M, p.N,
                              w, addto, lane);
            }
          } else {
            if (row < p.M && !*abort) {
              float v[32];
#pragma unroll
              for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
              store_row_chunk<kInt>(p, Cb, row, col0 + c, v, beta, use_c);
            }
          }
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) {
          if constexpr (kPair) {
            mbar_arrive_cluster(mapa_shared(smem_u32(&sm.tmem_empty[buf]), 0));
          } else {
            mbar_arrive(smem_u32(&sm.tmem_empty[buf]));
          }
        }
      }
      if constexpr (kInt) {
        if (p.c_tma) {
          if (!*abort) {
            const bool read_c = use_c && !addto && row < p.M;
            const int32_t *crow = Cb + static_cast<int64_t>(row) * p.ldc + col0;
#pragma unroll
            for (int c = 0; c < 128; c += 32) {
              uint32_t w[32];
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                const int32_t c0 = (read_c && col0 + c + j < p.N) ? __ldcg(crow + c + j) : 0;
                w[j] = static_cast<uint32_t>(
                    scale_add(p.alpha, static_cast<int32_t>(acc[c + j]), beta, c0, read_c));
              }
              tma_write_block(smem_u32(sm.stage_c[e]), &tmC, col0 + c, row - lane, bt, p.M, p.N,
                              w, addto, lane);
            }
          }
        } else if (row < p.M && !*abort) {
#pragma unroll
          for (int c = 0; c < 128; c += 32) {
            int32_t v[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = static_cast<int32_t>(acc[c + j]);
            store_row_chunk<kInt>(p, Cb, row, col0 + c, v, beta, use_c);
          }
        }
      }
      if (flag) {
        // Publish this part: every epilogue warp's stores complete, then the flag.
        if (p.c_tma && lane == 0) bulk_wait_all();
        __syncwarp();
        epilogue_sync();
        if (flag_thread && !*abort) {
          __threadfence();
          st_release_gpu(flag, static_cast<uint32_t>(wi.part + 1));
        }
      }
    }
    // Never leave with a TMA store still reading the staging buffer.
    if (p.c_tma && lane == 0) bulk_wait_all();
    __syncwarp();
  }

  tc_fence_before_sync();
  if constexpr (kPair) {
    cluster_sync();  // both CTAs done: no MMA, copy or arrival targets either CTA
  } else {
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after_sync();
    if constexpr (kPair) {
      tmem_dealloc_pair(tmem_base, kTmemCols);
    } else {
      tmem_dealloc(tmem_base, kTmemCols);
    }
  }
}

// ------------------------------------------------------------------ host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// Stride in bytes between the matrices of a stack: the caller's stride, or,
// for a single matrix, any legal value (the third coordinate is always 0).
cuuint64_t matrix_stride_bytes(int64_t count, int64_t stride, int64_t rows, int64_t ld,
                               int esize) {
  if (count > 1) return static_cast<cuuint64_t>(stride) * esize;
  return (static_cast<cuuint64_t>(rows) * ld * esize + 15) / 16 * 16;
}

// A stack of `count` row-major rows x cols matrices of 16-bit elements, row
// stride ld and matrix stride `stride` (elements), in boxes of box_rows x
// box_cols elements; the swizzle spans one box row (box_cols * 2 bytes: 128
// or 64).
bool make_tmap(CUtensorMap *tm, CUtensorMapDataType dt, const void *base, int64_t rows,
               int64_t cols, int64_t ld, int64_t count, int64_t stride, uint32_t box_rows,
               uint32_t box_cols) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(count)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld) * 2,
                           matrix_stride_bytes(count, stride, rows, ld, 2)};
  cuuint32_t box[3] = {box_cols, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(tm, dt, 3, const_cast<void *>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE,
                   box_cols == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// C (a stack of `count` row-major rows x cols matrices, 4-byte elements, row
// stride ld, matrix stride `stride`) in boxes of 32 x 32 elements with 128-byte
// swizzle, for the epilogue's TMA stores and reduces.
bool make_tmap_c(CUtensorMap *tm, bool is_int, const void *base, int64_t rows, int64_t cols,
                 int64_t ld, int64_t count, int64_t stride) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(count)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld) * 4,
                           matrix_stride_bytes(count, stride, rows, ld, 4)};
  cuuint32_t box[3] = {32, 32, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(tm, is_int ? CU_TENSOR_MAP_DATA_TYPE_INT32 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                   3, const_cast<void *>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// The kernel for an operand form.
template <bool kInt, bool kPair>
auto tc_kernel_for(bool a_t, bool b_t) -> decltype(&gemm_tc_kernel<kInt, kPair, false, false>) {
  if (a_t)
    return b_t ? gemm_tc_kernel<kInt, kPair, true, true> : gemm_tc_kernel<kInt, kPair, true, false>;
  return b_t ? gemm_tc_kernel<kInt, kPair, false, true>
             : gemm_tc_kernel<kInt, kPair, false, false>;
}

// Co-resident CTA pairs for a pair kernel on this device (0 if pairs are not
// available), queried once per device and kernel.
template <bool kInt>
int pair_capacity(const DeviceInfo &dev, size_t smem) {
  static std::mutex mu;
  static int cache[64];
  static bool known[64] = {};
  std::lock_guard<std::mutex> lock(mu);
  if (dev.device < 0 || dev.device >= 64) return 0;
  if (known[dev.device]) return cache[dev.device];
  auto kern = gemm_tc_kernel<kInt, true, false, false>;
  int n = 0;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * static_cast<unsigned>(dev.sm_count / 2), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
  }
  cudaGetLastError();
  cache[dev.device] = n;
  known[dev.device] = true;
  return n;
}

}  // namespace

// Library-owned stream-ordered memory pool of a device (scratch for the int8
// path and the split-k tail flags); freed blocks stay mapped for reuse.
cudaError_t device_pool(const DeviceInfo &dev, cudaMemPool_t *out) {
  static std::mutex mu;
  static cudaMemPool_t pools[64] = {};
  std::lock_guard<std::mutex> lock(mu);
  if (dev.device < 0 || dev.device >= 64) return cudaErrorInvalidDevice;
  if (!pools[dev.device]) {
    cudaMemPoolProps props;
    std::memset(&props, 0, sizeof props);
    props.allocType = cudaMemAllocationTypePinned;
    props.handleTypes = cudaMemHandleTypeNone;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev.device;
    cudaMemPool_t pl;
    cudaError_t e = cudaMemPoolCreate(&pl, &props);
    if (e != cudaSuccess) return e;
    uint64_t keep = ~0ull;  // keep freed memory mapped for the next call
    cudaMemPoolSetAttribute(pl, cudaMemPoolAttrReleaseThreshold, &keep);
    pools[dev.device] = pl;
  }
  *out = pools[dev.device];
  return cudaSuccess;
}

namespace {

#ifndef DGR_TC_MAX_SPLIT
#define DGR_TC_MAX_SPLIT 4
#endif
constexpr int kMaxSplit = DGR_TC_MAX_SPLIT;  // parts per tail tile (each adds one pass over C)

// Splits T tiles of KB k-blocks over at most `cap` units: whole tiles
// round-robin, then the leftover tiles split along k (at most max_split
// parts, in steps of kb_unit k-blocks) so that every unit gets one part (see
// TcArgs).
void plan_work(int64_t T, int KB, int kb_unit, int cap, int max_split, int &units, int &dp_tiles,
               int &tail_tiles, int &split) {
  const int nunits = (KB + kb_unit - 1) / kb_unit;
  int U = cap;
  int64_t W = T / U, R = T - W * U;
  int S = 1;
  if (R > 0) {
    S = static_cast<int>(U / R);
    if (S > max_split) S = max_split;
    if (S > nunits) S = nunits;
    if (S < 1) S = 1;
  }
  if (S == 1) {
    if (T < U) U = static_cast<int>(T);
    W = T / U;
    R = T - W * U;
  }
  units = U;
  dp_tiles = static_cast<int>(W * U);
  tail_tiles = static_cast<int>(R);
  split = S;
}

template <bool kInt>
cudaError_t launch_tc(const DeviceInfo &dev, CUtensorMapDataType dt, bool is_bf16,
                      const BatchOps &ops, int M, int N, int K,
                      typename TcArgs<kInt>::Out alpha, const void *A, int64_t lda,
                      const void *B, int64_t ldb, typename TcArgs<kInt>::Out beta,
                      typename TcArgs<kInt>::Out *C, int64_t ldc, cudaStream_t stream,
                      uint32_t *flags_ws, size_t flags_words) {
  // Short, wide problems: the transposed-role kernel streams B at HBM speed
  // instead of multiplying a mostly-zero 256-row tile.
  if (M <= kSkinnyMaxM && ops.plain()) {
    if constexpr (kInt) {
      return launch_tc_skinny_int(dev, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream,
                                  flags_ws, flags_words);
    } else {
      return launch_tc_skinny_float(dev, is_bf16, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
                                    stream);
    }
  }
  static_assert(sizeof(TcSmem<true>) + 1024 <= 232448, "pair kernel shared memory");
  static_assert(sizeof(TcSmem<false>) + 1024 <= 232448, "single-CTA kernel shared memory");
  const size_t smem_pair = sizeof(TcSmem<true>) + 1024;
  const int pairs = DGR_TC_PAIR ? pair_capacity<kInt>(dev, smem_pair) : 0;
  const bool use_pairs = pairs > 0;
  const int tile_m = use_pairs ? Cfg<true>::kTileM : Cfg<false>::kTileM;
  const uint32_t bn_load = use_pairs ? Cfg<true>::kBNLoad : Cfg<false>::kBNLoad;

  // Operand tensor maps: one matrix, or one per batch entry.
  const int64_t batch = ops.batch;
  const int64_t na = (batch > 1 && ops.stride_a != 0) ? batch : 1;
  const int64_t nb = (batch > 1 && ops.stride_b != 0) ? batch : 1;
  CUtensorMap tmA, tmB;
  const bool maps_ok =
      (ops.a_t ? make_tmap(&tmA, dt, A, K, M, lda, na, ops.stride_a, kBK, 64)
               : make_tmap(&tmA, dt, A, M, K, lda, na, ops.stride_a, kBM, kBK)) &&
      (ops.b_t ? make_tmap(&tmB, dt, B, N, K, ldb, nb, ops.stride_b, bn_load, kBK)
               : make_tmap(&tmB, dt, B, K, N, ldb, nb, ops.stride_b, kBK, 64));
  if (!maps_ok) {
    if (na == 1 && nb == 1) return cudaErrorInvalidValue;
    // A stride the tensor-map encoder does not take (matrices that overlap):
    // one launch per batch entry, each on a single matrix.
    BatchOps one = ops;
    one.batch = 1;
    for (int64_t b = 0; b < batch; ++b) {
      const void *Ab = static_cast<const uint16_t *>(A) + b * ops.stride_a;
      const void *Bb = static_cast<const uint16_t *>(B) + b * ops.stride_b;
      cudaError_t e = launch_tc<kInt>(dev, dt, is_bf16, one, M, N, K, alpha, Ab, lda, Bb, ldb,
                                      beta, C + b * ops.stride_c, ldc, stream, nullptr, 0);
      if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
  }
  TcArgs<kInt> p;
  p.M = M;
  p.N = N;
  p.K = K;
  p.alpha = alpha;
  p.beta = beta;
  p.C = C;
  p.ldc = ldc;
  p.tiles_m = (M + tile_m - 1) / tile_m;
  p.tiles_n = (N + kBN - 1) / kBN;
  p.tiles_per_batch = p.tiles_m * p.tiles_n;
  p.a_batched = na > 1;
  p.b_batched = nb > 1;
  p.stride_c = batch > 1 ? ops.stride_c : 0;
  p.c_vec_ok = (reinterpret_cast<uintptr_t>(C) % 16 == 0) && (ldc % 4 == 0);
  p.err_word = dev.err_word;
  p.tail_flags = nullptr;
  // TMA stores of C need a 16-byte aligned base and row stride, and rows whose
  // length is a whole number of 16-byte units: a store box is clipped at the
  // right edge of C only in 16-byte units, so with N % 4 != 0 it would also
  // write the first columns of the row padding. A stack of C matrices also
  // needs a matrix stride of whole 16-byte units. Otherwise the epilogue
  // writes C with plain guarded stores.
  CUtensorMap tmC;
  std::memset(&tmC, 0, sizeof tmC);
  p.c_tma = p.c_vec_ok && (N % 4 == 0) && (batch == 1 || ops.stride_c % 4 == 0) &&
            make_tmap_c(&tmC, kInt, C, M, N, ldc, batch, ops.stride_c);
  p.idesc = idesc_f16(is_bf16, ops.a_t, !ops.b_t, tile_m, kBN);
  const int64_t tiles = static_cast<int64_t>(p.tiles_per_batch) * batch;
  if (static_cast<int64_t>(p.tiles_m) * p.tiles_n > 0x7fffffffLL || tiles > 0x7fffffffLL)
    return cudaErrorInvalidValue;
  const int KB = (K + kBK - 1) / kBK;
  const int cap = use_pairs ? pairs : dev.sm_count;
  const int kb_unit = kInt ? kChunkKB : 1;
  int units = 0;
  plan_work(tiles, KB, kb_unit, cap, kMaxSplit, units, p.dp_tiles, p.tail_tiles, p.split);

  // Tail flags: zeroed per call; from the caller's buffer or the pool.
  void *pool_flags = nullptr;
  if (p.split > 1) {
    const size_t need = static_cast<size_t>(p.tail_tiles) * 2;
    if (flags_ws != nullptr) {
      if (flags_words >= need) {
        p.tail_flags = flags_ws;
      } else {  // the caller's buffer is too small: whole tiles only
        plan_work(tiles, KB, kb_unit, cap, 1, units, p.dp_tiles, p.tail_tiles, p.split);
      }
    } else {
      cudaMemPool_t pool;
      cudaError_t e = device_pool(dev, &pool);
      if (e != cudaSuccess) return e;
      e = cudaMallocFromPoolAsync(&pool_flags, need * 4, pool, stream);
      if (e != cudaSuccess) return e;
      p.tail_flags = static_cast<uint32_t *>(pool_flags);
    }
    if (p.split > 1) {
      cudaError_t e = cudaMemsetAsync(p.tail_flags, 0, need * 4, stream);
      if (e != cudaSuccess) {
        if (pool_flags) cudaFreeAsync(pool_flags, stream);
        return e;
      }
    }
  }

  cudaError_t e;
  if (use_pairs) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * static_cast<unsigned>(units), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem_pair;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    auto kern = tc_kernel_for<kInt, true>(ops.a_t, ops.b_t);
    // Every form has the same shared memory; raise the limit for this one.
    e = set_max_dynamic_smem(reinterpret_cast<const void *>(kern), static_cast<int>(smem_pair),
                             dev.device);
    if (e == cudaSuccess) e = cudaLaunchKernelEx(&cfg, kern, tmA, tmB, tmC, p);
    if (e == cudaSuccess) e = cudaGetLastError();
  } else {
    const size_t smem = sizeof(TcSmem<false>) + 1024;
    auto kern = tc_kernel_for<kInt, false>(ops.a_t, ops.b_t);
    e = set_max_dynamic_smem(reinterpret_cast<const void *>(kern), static_cast<int>(smem),
                             dev.device);
    if (e == cudaSuccess) {
      kern<<<units, kThreads, smem, stream>>>(tmA, tmB, tmC, p);
      e = cudaGetLastError();
    }
  }
  if (pool_flags) {
    cudaError_t f = cudaFreeAsync(pool_flags, stream);
    if (e == cudaSuccess) e = f;
  }
  return e;
}

// int8 -> fp16, exact (|x| <= 128), for a stack of `count` rows x cols
// matrices (source matrix stride src_stride; destination matrices packed at
// rows * ldd). dst has row stride ldd (multiple of 8) and its padding columns
// [cols, ldd) are written with zeros. Each thread widens 16 consecutive
// elements of a row: one 16-byte load when the source row is 16-byte aligned
// and the chunk is inside the matrix, byte loads otherwise, and one or two
// 16-byte stores.
__global__ void widen_s8_kernel(const int8_t *__restrict__ src, int64_t lds, int64_t src_stride,
                                __half *dst, int64_t ldd, int rows, int cols, int count,
                                int vec_ok) {
  const int64_t chunks_per_row = (ldd + 15) / 16;
  const int64_t total = static_cast<int64_t>(rows) * count * chunks_per_row;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = i / chunks_per_row;  // row of the whole stack
    const int c0 = static_cast<int>((i - r * chunks_per_row) * 16);
    const int64_t m = r / rows;            // matrix of the stack
    const int8_t *s = src + m * src_stride + (r - m * rows) * lds;
    __align__(16) __half h[16];
    if (vec_ok && c0 + 16 <= cols) {
      const int4 v = *reinterpret_cast<const int4 *>(s + c0);
      const int w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 16; ++j)
        h[j] = __int2half_rn(static_cast<int8_t>(static_cast<uint32_t>(w[j >> 2]) >> (8 * (j & 3))));
    } else {
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int c = c0 + j;
        h[j] = __int2half_rn(c < cols ? static_cast<int>(s[c]) : 0);
      }
    }
    uint4 *d = reinterpret_cast<uint4 *>(dst + r * ldd + c0);
    d[0] = *reinterpret_cast<const uint4 *>(h);
    if (c0 + 16 <= ldd) d[1] = *reinterpret_cast<const uint4 *>(h + 8);
  }
}

cudaError_t widen_s8(const DeviceInfo &dev, const int8_t *src, int64_t lds, __half *dst,
                     int64_t ldd, int rows, int cols, cudaStream_t stream, int count = 1,
                     int64_t src_stride = 0) {
  const int64_t total = static_cast<int64_t>(rows) * count * ((ldd + 15) / 16);
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  const int64_t cap = static_cast<int64_t>(dev.sm_count) * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  const int vec_ok = (reinterpret_cast<uintptr_t>(src) % 16 == 0) && (lds % 16 == 0) &&
                     (count == 1 || src_stride % 16 == 0);
  widen_s8_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
      src, lds, src_stride, dst, ldd, rows, cols, count, vec_ok);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm_tc_f16(const DeviceInfo &dev, bool is_bf16, int M, int N, int K,
                               float alpha, const void *A, int64_t lda, const void *B,
                               int64_t ldb, float beta, float *C, int64_t ldc,
                               cudaStream_t stream) {
  const CUtensorMapDataType dt =
      is_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  return launch_tc<false>(dev, dt, is_bf16, BatchOps(), M, N, K, alpha, A, lda, B, ldb, beta, C,
                          ldc, stream, nullptr, 0);
}

cudaError_t launch_gemm_tc_f16_ex(const DeviceInfo &dev, bool is_bf16, const BatchOps &ops, int M,
                                  int N, int K, float alpha, const void *A, int64_t lda,
                                  const void *B, int64_t ldb, float beta, float *C, int64_t ldc,
                                  cudaStream_t stream) {
  const CUtensorMapDataType dt =
      is_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  return launch_tc<false>(dev, dt, is_bf16, ops, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
                          stream, nullptr, 0);
}

// The int8 path widens A and B to fp16 in stream-ordered scratch memory from a
// library-owned pool, runs the tensor-core kernel in exact-integer mode and
// returns the scratch to the pool on the same stream.
cudaError_t launch_gemm_s8(const DeviceInfo &dev, int M, int N, int K, int32_t alpha,
                           const int8_t *A, int64_t lda, const int8_t *B, int64_t ldb,
                           int32_t beta, int32_t *C, int64_t ldc, cudaStream_t stream) {
  const int64_t lda16 = (static_cast<int64_t>(K) + 7) / 8 * 8;
  const int64_t ldb16 = (static_cast<int64_t>(N) + 7) / 8 * 8;
  const size_t a_bytes = static_cast<size_t>(M) * lda16 * 2;
  const size_t a_off = (a_bytes + 255) / 256 * 256;
  const size_t total = a_off + static_cast<size_t>(K) * ldb16 * 2;

  cudaMemPool_t pool = nullptr;
  {
    cudaError_t e = device_pool(dev, &pool);
    if (e != cudaSuccess) return e;
  }
  void *scratch = nullptr;
  cudaError_t e = cudaMallocFromPoolAsync(&scratch, total, pool, stream);
  if (e != cudaSuccess) return e;
  __half *a16 = static_cast<__half *>(scratch);
  __half *b16 = reinterpret_cast<__half *>(static_cast<uint8_t *>(scratch) + a_off);
  e = widen_s8(dev, A, lda, a16, lda16, M, K, stream);
  if (e == cudaSuccess) e = widen_s8(dev, B, ldb, b16, ldb16, K, N, stream);
  if (e == cudaSuccess)
    e = launch_tc<true>(dev, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, false, BatchOps(), M, N, K, alpha,
                        a16, lda16, b16, ldb16, beta, C, ldc, stream, nullptr, 0);
  cudaError_t f = cudaFreeAsync(scratch, stream);
  return e != cudaSuccess ? e : f;
}

// Batched / transposed int8: each operand is widened in its stored layout
// (one matrix, or one per batch entry, packed), then the tensor-core kernel
// reads the fp16 copies with the same transposes and strides.
cudaError_t launch_gemm_s8_ex(const DeviceInfo &dev, const BatchOps &ops, int M, int N, int K,
                              int32_t alpha, const int8_t *A, int64_t lda, const int8_t *B,
                              int64_t ldb, int32_t beta, int32_t *C, int64_t ldc,
                              cudaStream_t stream) {
  // Stored shapes: A is M x K or K x M, B is K x N or N x K.
  const int a_rows = ops.a_t ? K : M, a_cols = ops.a_t ? M : K;
  const int b_rows = ops.b_t ? N : K, b_cols = ops.b_t ? K : N;
  const int na = (ops.batch > 1 && ops.stride_a != 0) ? ops.batch : 1;
  const int nb = (ops.batch > 1 && ops.stride_b != 0) ? ops.batch : 1;
  const int64_t lda16 = (static_cast<int64_t>(a_cols) + 7) / 8 * 8;
  const int64_t ldb16 = (static_cast<int64_t>(b_cols) + 7) / 8 * 8;
  const int64_t a_mat = a_rows * lda16, b_mat = b_rows * ldb16;  // packed strides (elements)
  const size_t a_bytes = static_cast<size_t>(na) * a_mat * 2;
  const size_t a_off = (a_bytes + 255) / 256 * 256;
  const size_t total = a_off + static_cast<size_t>(nb) * b_mat * 2;

  cudaMemPool_t pool = nullptr;
  {
    cudaError_t e = device_pool(dev, &pool);
    if (e != cudaSuccess) return e;
  }
  void *scratch = nullptr;
  cudaError_t e = cudaMallocFromPoolAsync(&scratch, total, pool, stream);
  if (e != cudaSuccess) return e;
  __half *a16 = static_cast<__half *>(scratch);
  __half *b16 = reinterpret_cast<__half *>(static_cast<uint8_t *>(scratch) + a_off);
  e = widen_s8(dev, A, lda, a16, lda16, a_rows, a_cols, stream, na, ops.stride_a);
  if (e == cudaSuccess)
    e = widen_s8(dev, B, ldb, b16, ldb16, b_rows, b_cols, stream, nb, ops.stride_b);
  if (e == cudaSuccess) {
    BatchOps wide = ops;
    wide.stride_a = na > 1 ? a_mat : 0;
    wide.stride_b = nb > 1 ? b_mat : 0;
    e = launch_tc<true>(dev, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, false, wide, M, N, K, alpha, a16,
                        lda16, b16, ldb16, beta, C, ldc, stream, nullptr, 0);
  }
  cudaError_t f = cudaFreeAsync(scratch, stream);
  return e != cudaSuccess ? e : f;
}

// The int8 path with scratch memory supplied by the caller instead of drawn
// from the library's pool: widen A and B into `scratch` (which must hold
// s8_scratch_bytes(M, N, K) bytes, 256-byte aligned) and run the tensor-core
// kernel in exact-integer mode. Allocates nothing.
size_t s8_scratch_bytes(int M, int N, int K) {
  const int64_t lda16 = (static_cast<int64_t>(K) + 7) / 8 * 8;
  const int64_t ldb16 = (static_cast<int64_t>(N) + 7) / 8 * 8;
  const size_t a_off = (static_cast<size_t>(M) * lda16 * 2 + 255) / 256 * 256;
  return a_off + static_cast<size_t>(K) * ldb16 * 2;
}

cudaError_t launch_gemm_s8_scratch(const DeviceInfo &dev, int M, int N, int K, int32_t alpha,
                                   const int8_t *A, int64_t lda, const int8_t *B, int64_t ldb,
                                   int32_t beta, int32_t *C, int64_t ldc, void *scratch,
                                   uint32_t *flags, size_t flags_words, cudaStream_t stream) {
  const int64_t lda16 = (static_cast<int64_t>(K) + 7) / 8 * 8;
  const int64_t ldb16 = (static_cast<int64_t>(N) + 7) / 8 * 8;
  const size_t a_off = (static_cast<size_t>(M) * lda16 * 2 + 255) / 256 * 256;
  __half *a16 = static_cast<__half *>(scratch);
  __half *b16 = reinterpret_cast<__half *>(static_cast<uint8_t *>(scratch) + a_off);
  cudaError_t e = widen_s8(dev, A, lda, a16, lda16, M, K, stream);
  if (e == cudaSuccess) e = widen_s8(dev, B, ldb, b16, ldb16, K, N, stream);
  if (e == cudaSuccess)
    e = launch_tc<true>(dev, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, false, BatchOps(), M, N, K, alpha,
                        a16, lda16, b16, ldb16, beta, C, ldc, stream, flags, flags_words);
  return e;
}

}  // namespace dgr
