// gemm_tc_kernel.cuh -- the tensor-core GEMM kernel for sm_103a and its host
// launcher, shared by the translation units that instantiate it (one per
// element kind, compiled in parallel):
//
//     C = alpha * op(A) * op(B) + beta * C      op(A): M x K, op(B): K x N,
//                                                C: M x N, all row-major
//
// tcgen05.mma with the accumulator in tensor memory (TMEM), operands staged by
// TMA. Element kinds (TcKind below):
//   * 16-bit inputs (bf16 or fp16), fp32 accumulation, fp32 C;
//   * the same with a 16-bit C of the inputs' format (fp32 accumulation, one
//     round-to-nearest-even at the end);
//   * exact int32 C from integer-valued fp16 operands (the int8 and uint8
//     paths). An int8 value is exact in fp16 and a product of two is exact in
//     fp32; a sum of at most 1024 such products (each at most 2^14 in
//     magnitude) is an integer of at most 2^24, which fp32 holds exactly. The
//     kernel therefore restarts the fp32 accumulator every 1024 values of k,
//     and the epilogue adds each finished partial sum into int32 registers
//     (wrap-around). uint8 operands arrive offset by -128 (int8 range), and
//     the epilogue adds the exact correction row_corr[i] + col_corr[j] +
//     corr_const once;
//   * fp32 inputs used at tf32 precision (kind::tf32), fp32 C; both operands
//     are staged K-major.
//
// op(X) is X as stored or its transpose, and the problem may be a stack of
// `batch` such GEMMs at fixed element strides (strided-batched GEMM). Neither
// costs anything on this path: a transposed operand is staged by TMA in the
// other major order and the MMA's descriptors say so (the form is a template
// parameter, so each loop is compiled for one layout); the batch index is the
// third coordinate of every tensor map and one more dimension of the tile list.
//
// Sources: C++ warp-matrix-function page (D = A*B + C on tensor cores; type
// table: half / bfloat16 inputs with float accumulate, half -> half, signed and
// unsigned char inputs with int accumulate, precision::tf32 with float
// accumulate); "Sgemm [128,128,8]" (C = alpha*A*B + beta*C, row-major, the
// alpha/beta epilogue); "使用CUDA和瓦片算法计算矩阵乘法" (residual tiles act as
// zeros: here the TMA unit fills out-of-range elements with zeros).
//
// Structure (one CTA per SM, or one CTA pair per two SMs, persistent):
//   warp 0      one thread issues TMA loads of A (128 rows x 128 bytes of k,
//               K-major, 128-byte swizzle) and B (128 bytes of k x 256 columns,
//               N-major, as boxes 128 bytes wide) into a kStages-deep ring
//               guarded by full/empty mbarriers. A stored transposed (K x M)
//               arrives as M-major boxes; B stored transposed (N x K) as one
//               256(n) x 128-byte(k) K-major box. Every layout and element size
//               fills the same bytes per stage.
//   warp 1      allocates 512 TMEM columns; one thread issues tcgen05.mma
//               (M = 128, or 256 on a CTA pair; N = 256) into one of two
//               256-column accumulators and commits each stage's completion to
//               that stage's empty barrier.
//   warps 2..9  epilogue: tcgen05.ld of the finished accumulator (each warp
//               reads its 32-lane quarter and one 128-column half), then
//               alpha/beta and TMA (or guarded plain) stores to C. The two
//               accumulators let the epilogue of one tile overlap the main loop
//               of the next.
// Tiles are visited in groups of kGroupM tile rows so that the CTAs resident
// at one time share A rows and B columns in L2.
#pragma once

#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <type_traits>
#include <utility>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "launch.h"
#include "ptx.cuh"
#include "work_split.cuh"

namespace dgr {
namespace {

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
#ifndef DGR_TC_MAX_SPLIT
#define DGR_TC_MAX_SPLIT 4
#endif
// L2 eviction hints on the TMA copies: A (reused across a group's tile
// columns) evict-last, C stores evict-first. Measured on GB300 at 8192^3:
// bf16 +0.5 %, int8 +0.9 % over no hints.
#ifndef DGR_TC_L2HINT
#define DGR_TC_L2HINT 1
#endif

// Element kinds of one instantiation.
constexpr int kKindF32 = 0;      // bf16 / fp16 in, fp32 C
constexpr int kKindS8 = 1;       // int8 (or offset uint8) widened to fp16, exact int32 C
constexpr int kKindF16Out = 3;   // fp16 in, fp16 C
constexpr int kKindBF16Out = 4;  // bf16 in, bf16 C
constexpr int kKindTF32 = 5;     // fp32 in at tf32 precision, fp32 C

template <int kKind>
struct TcKind {
  static constexpr int kInBytes = kKind == kKindTF32 ? 4 : 2;
  static constexpr bool kInt = kKind == kKindS8;
  static constexpr bool kOut16 = kKind == kKindF16Out || kKind == kKindBF16Out;
  // exact-int mode: values of k per fp32 chunk (sums stay within 2^24)
  static constexpr int kChunkK = kKind == kKindS8 ? 1024 : 0;
  using Out = typename std::conditional<
      kInt, int32_t, typename std::conditional<kOut16, uint16_t, float>::type>::type;
  using Scale = typename std::conditional<kInt, int32_t, float>::type;  // alpha, beta
  // k per stage: one 128-byte swizzle row of a K-major operand
  static constexpr int kBK = 128 / kInBytes;
  // k per MMA instruction: 32 bytes
  static constexpr int kMmaK = 32 / kInBytes;
  // values of m or n in one 128-byte row of an MN-major box
  static constexpr int kMNElems = 128 / kInBytes;
};

constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr uint32_t kTmemCols = 512;  // two 256-column fp32 accumulators
constexpr int kBN = 256;             // tile columns (MMA N)
constexpr int kBM = 128;             // tile rows held by one CTA (TMEM lanes)
constexpr uint32_t kRowBytes = 128;  // one swizzle row
constexpr uint32_t kAtomBytes = 8 * kRowBytes;  // 8-row swizzle atom (SBO)

// Single CTA: 128 x 256 tile, the CTA stages all 256 columns of B.
// CTA pair:   256 x 256 tile, each CTA stages its 128 rows of A and its 128
//             columns of B; the leader's MMA (M = 256) reads both CTAs.
template <bool kPair>
struct Cfg {
  static constexpr int kTileM = kPair ? 256 : 128;
  static constexpr int kBNLoad = kPair ? 128 : 256;   // B columns staged per CTA
  static constexpr int kStages = kPair ? DGR_TC_STAGES_PAIR : DGR_TC_STAGES;
  static constexpr int kGroupM = kPair ? DGR_TC_GROUP_M_PAIR : DGR_TC_GROUP_M;
  static constexpr uint32_t kABytes = kBM * kRowBytes;
  static constexpr uint32_t kBBytes = kBNLoad * kRowBytes;
  static constexpr uint32_t kStageBytes = kABytes + kBBytes;           // per CTA
  static constexpr uint32_t kTxBytes = kStageBytes * (kPair ? 2 : 1);  // per full phase
};

// Epilogue staging: one 32-row x 128-byte block of C per epilogue warp (32 x
// 32 fp32/int32 values or 32 x 64 16-bit values), in the 128-byte-swizzled
// layout of the C tensor map's box.
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

// Exact-int kinds only: optional exact per-row and per-column terms added to
// the product before alpha/beta (the uint8 path's offset correction). A base
// that is empty for the other kinds: the fp32 kernels' code generation is
// sensitive to the size of their argument block (two more pointers there
// cost them 35 registers and spills).
template <bool kInt>
struct TcCorr {};
template <>
struct TcCorr<true> {
  const int32_t *row_corr, *col_corr;
  int32_t corr_const;
};

template <int kKind>
struct TcArgs : TcCorr<TcKind<kKind>::kInt> {
  using Out = typename TcKind<kKind>::Out;
  using Scale = typename TcKind<kKind>::Scale;
  int M, N, K;
  Scale alpha, beta;
  Out *C;
  int64_t ldc;
  int tiles_m, tiles_n;
  int tiles_per_batch;       // tiles_m * tiles_n; tile t is tile t % this of matrix t / this
  int a_batched, b_batched;  // the operand's tensor map has one matrix per batch entry
  int64_t stride_c;          // elements between consecutive C matrices
  int c_vec_ok;  // C 16-byte aligned and rows a whole number of 16-byte units apart
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
template <int kGroupM, int kKind>
__device__ __forceinline__ void batch_tile_coords(int t, const TcArgs<kKind> &p, int &bt, int &tm,
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

// 16-bit C of kind kKind: the stored bits <-> float (exact widening; one
// round-to-nearest-even narrowing).
template <int kKind>
__device__ __forceinline__ float out16_to_float(uint16_t h) {
  if constexpr (kKind == kKindBF16Out) {
    return __bfloat162float(__ushort_as_bfloat16(h));
  } else {
    return __half2float(__ushort_as_half(h));
  }
}
template <int kKind>
__device__ __forceinline__ uint16_t float_to_out16(float v) {
  if constexpr (kKind == kKindBF16Out) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(v));
  } else {
    return __half_as_ushort(__float2half_rn(v));
  }
}

// C[row, col .. col+31] = alpha * v + beta * C (the C term only when use_c),
// fp32 or int32 C. C is read through L2 (another SM may have just written it).
template <int kKind>
__device__ __forceinline__ void store_row_chunk(const TcArgs<kKind> &p,
                                                typename TcArgs<kKind>::Out *C, int row, int col,
                                                const typename TcArgs<kKind>::Scale (&v)[32],
                                                typename TcArgs<kKind>::Scale beta, bool use_c) {
  using Out = typename TcArgs<kKind>::Out;
  constexpr bool kInt = TcKind<kKind>::kInt;
  Out *crow = C + static_cast<int64_t>(row) * p.ldc;
  const auto alpha = p.alpha;
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

// 16-bit C: already-final values h[0..31] for C[row, col .. col+31].
template <int kKind>
__device__ __forceinline__ void store_row_chunk16(const TcArgs<kKind> &p, uint16_t *C, int row,
                                                  int col, const uint32_t (&h)[16]) {
  uint16_t *crow = C + static_cast<int64_t>(row) * p.ldc;
  if (p.c_vec_ok && col + 31 < p.N) {
#pragma unroll
    for (int j = 0; j < 16; j += 4)
      *reinterpret_cast<uint4 *>(crow + col + 2 * j) = make_uint4(h[j], h[j + 1], h[j + 2], h[j + 3]);
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (col + j < p.N) crow[col + j] = static_cast<uint16_t>(h[j >> 1] >> (16 * (j & 1)));
  }
}

// Writes one 32-row x 128-byte block of C matrix z (rows y .. y+31, columns
// from x; the lane's row is y + lane) from registers: stages it in the warp's
// swizzled buffer and issues one TMA store, or one TMA reduce-add when `addto`
// (C += block). Elements outside C are dropped by the tensor map's bounds.
__device__ __forceinline__ void tma_write_block(uint32_t stage, const void *tmC, int x, int y,
                                                int z, int M, int N, const uint32_t (&w)[32],
                                                bool addto, int lane) {
  [[maybe_unused]] uint64_t pol_stream = 0;
  if constexpr (DGR_TC_L2HINT != 0) pol_stream = l2_policy_evict_first();
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
    } else if constexpr (DGR_TC_L2HINT != 0) {
      tma_store_3d_hint(tmC, x, y, z, stage, pol_stream);
    } else {
      tma_store_3d(tmC, x, y, z, stage);
    }
    bulk_commit();
  }
}

template <int kKind, bool kPair>
__device__ __forceinline__ void issue_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                          uint32_t acc) {
  if constexpr (kKind == kKindTF32) {
    if constexpr (kPair) {
      tc_mma_tf32_pair(d, a, b, idesc, acc);
    } else {
      tc_mma_tf32(d, a, b, idesc, acc);
    }
  } else {
    if constexpr (kPair) {
      tc_mma_f16_pair(d, a, b, idesc, acc);
    } else {
      tc_mma_f16(d, a, b, idesc, acc);
    }
  }
}

// The kernel body. kAT / kBT: A stored K x M / B stored N x K (used
// transposed). The tensor maps are the kernel's grid-constant parameters,
// passed by reference so that TMA reads them in parameter space.
template <int kKind, bool kPair, bool kAT, bool kBT>
__device__ __forceinline__ void gemm_tc_body(const CUtensorMap &tmA, const CUtensorMap &tmB,
                                             const CUtensorMap &tmC, const TcArgs<kKind> p) {
  using K_ = TcKind<kKind>;
  using Cf = Cfg<kPair>;
  using Out = typename K_::Out;
  using Scale = typename K_::Scale;
  constexpr bool kInt = K_::kInt;
  constexpr bool kOut16 = K_::kOut16;
  constexpr int kBK = K_::kBK;
  constexpr int kStages = Cf::kStages;
  // A box of kMNElems values of m or n by kBK rows of k (MN-major operands).
  constexpr uint32_t kMNBoxBytes = kRowBytes * kBK;
  // kMmaK rows of an MN-major operand: the step between MMAs along k.
  constexpr uint32_t kMNStep = kRowBytes * K_::kMmaK;
  static_assert(kKind != kKindTF32 || (!kAT && kBT), "tf32 operands are staged K-major");
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
  // Launched as a programmatic dependent of the previous kernel on the stream
  // (for instance the int8 path's widening pass): the set-up above overlaps
  // that kernel's tail; nothing in global memory is touched before it has
  // completed and its writes are visible.
  grid_dependency_wait();
  grid_launch_dependents();

  const int KB = (p.K + kBK - 1) / kBK;
  // int mode: exact fp32 chunks of kChunkK values of k; float mode: one chunk per item
  constexpr int kChunkKB = kInt ? K_::kChunkK / kBK : 1;
  const int chunk_kb = kInt ? kChunkKB : KB;
  const int kb_unit = kInt ? kChunkKB : 1;
  WorkItem wi;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      [[maybe_unused]] uint64_t pol_keep = 0;
      if constexpr (DGR_TC_L2HINT != 0) pol_keep = l2_policy_evict_last();
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
          auto load_keep = [&](uint32_t dst, const CUtensorMap *tm, int x, int y, int z) {
            if constexpr (DGR_TC_L2HINT != 0) {
              if constexpr (kPair) {
                tma_load_3d_pair_hint(dst, tm, bar, x, y, z, pol_keep);
              } else {
                tma_load_3d_hint(dst, tm, bar, x, y, z, pol_keep);
              }
            } else {
              load(dst, tm, x, y, z);
            }
          };
          const int k0 = kb * kBK;
          if constexpr (!kAT) {
            load_keep(smem_u32(sm.a[stage]), &tmA, k0, m0, za);  // 128 rows x kBK, K-major
          } else {
#pragma unroll
            for (int j = 0; j < kBM / K_::kMNElems; ++j)  // kBK rows of k x kMNElems of m
              load_keep(smem_u32(sm.a[stage] + j * kMNBoxBytes), &tmA, m0 + K_::kMNElems * j, k0,
                        za);
          }
          if constexpr (!kBT) {
#pragma unroll
            for (int j = 0; j < Cf::kBNLoad / K_::kMNElems; ++j)  // kBK rows of k x kMNElems of n
              load(smem_u32(sm.b[stage] + j * kMNBoxBytes), &tmB, nb + K_::kMNElems * j, k0, zb);
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
      // Descriptors of stage 0 (layouts below); a stage or a k-step only moves
      // the start address, the descriptor's low 14 bits (address / 16), so each
      // MMA's descriptors are one add away from these.
      const uint64_t adesc0 = kAT ? smem_desc(smem_u32(sm.a[0]), kMNBoxBytes, kAtomBytes, 2u)
                                  : smem_desc(smem_u32(sm.a[0]), 16, kAtomBytes, 2u);
      const uint64_t bdesc0 = kBT ? smem_desc(smem_u32(sm.b[0]), 16, kAtomBytes, 2u)
                                  : smem_desc(smem_u32(sm.b[0]), kMNBoxBytes, kAtomBytes, 2u);
      constexpr uint32_t kAStage = sizeof(sm.a[0]) >> 4, kBStage = sizeof(sm.b[0]) >> 4;
      constexpr uint32_t kAStepK = (kAT ? kMNStep : 32u) >> 4;  // one MMA's k, in 16 B
      constexpr uint32_t kBStepK = (kBT ? 32u : kMNStep) >> 4;
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
            const uint64_t ad = adesc0 + stage * kAStage, bd = bdesc0 + stage * kBStage;
            const uint32_t first = kb > kb0 ? 1u : 0u;
#pragma unroll
            for (int kk = 0; kk < kBK / K_::kMmaK; ++kk) {
              // K-major operand: 128-byte swizzled rows of k; one MMA's k is 32 B
              // further along the row; SBO = one 8-row swizzle atom.
              // MN-major operand: 128-byte swizzled rows of m or n, one row per
              // k; one MMA's k is kMmaK rows further; LBO = one box of
              // kMNElems values, SBO = 1 KiB between groups of 8 k-rows.
              issue_mma<kKind, kPair>(d_tmem, ad + kk * kAStepK, bd + kk * kBStepK, p.idesc,
                                      kk > 0 ? 1u : first);
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
      const Scale beta = addto ? Scale(1) : p.beta;
      const bool use_c = addto || p.beta != Scale(0);
      uint32_t *flag = nullptr;
      if (wi.parts > 1)
        flag = p.tail_flags + (wi.tile - p.dp_tiles) * 2 + static_cast<int>(rank);
      if (addto) {
        if (flag_thread) wait_flag(flag, static_cast<uint32_t>(wi.part), abort, p.err_word);
        epilogue_sync();
      }
      uint32_t acc[kInt ? 128 : 1];  // int mode: running int32 sums (wrap-around)
      if constexpr (kInt) {
        // The sums start at the offset correction row_corr + col_corr +
        // corr_const (part 0 of a tile only), else at zero.
        if (p.row_corr != nullptr && !addto && row < p.M) {
          const uint32_t rc = static_cast<uint32_t>(__ldg(p.row_corr + row)) +
                              static_cast<uint32_t>(p.corr_const);
#pragma unroll
          for (int j = 0; j < 128; ++j)
            acc[j] = col0 + j < p.N ? rc + static_cast<uint32_t>(__ldg(p.col_corr + col0 + j)) : 0u;
        } else {
#pragma unroll
          for (int j = 0; j < 128; ++j) acc[j] = 0;
        }
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
        [[maybe_unused]] uint32_t w16[32];  // 16-bit C: 64 packed values (one TMA block)
#pragma unroll
        for (int c = 0; c < 128; c += 32) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(taddr + c, r);
          tmem_ld_wait();
          if constexpr (kInt) {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              acc[c + j] += static_cast<uint32_t>(__float2int_rn(__uint_as_float(r[j])));
          } else if constexpr (kOut16) {
            // alpha * acc + beta * C in fp32, then one rounding to 16 bits
            if (!*abort) {
              const bool read_c = use_c && row < p.M;
              const uint16_t *crow = Cb + static_cast<int64_t>(row) * p.ldc + col0 + c;
              uint32_t h[16];
#pragma unroll
              for (int j = 0; j < 32; j += 2) {
                const float c0 = (read_c && col0 + c + j < p.N)
                                     ? out16_to_float<kKind>(__ldcg(crow + j)) : 0.f;
                const float c1 = (read_c && col0 + c + j + 1 < p.N)
                                     ? out16_to_float<kKind>(__ldcg(crow + j + 1)) : 0.f;
                const uint32_t lo = float_to_out16<kKind>(
                    scale_add(p.alpha, __uint_as_float(r[j]), beta, c0, read_c));
                const uint32_t hi = float_to_out16<kKind>(
                    scale_add(p.alpha, __uint_as_float(r[j + 1]), beta, c1, read_c));
                h[j >> 1] = lo | (hi << 16);
              }
              if (p.c_tma) {
#pragma unroll
                for (int j = 0; j < 16; ++j) w16[(c & 32) / 2 + j] = h[j];
                if (c & 32)
                  tma_write_block(smem_u32(sm.stage_c[e]), &tmC, col0 + c - 32, row - lane, bt,
                                  p.M, p.N, w16, false, lane);
              } else if (row < p.M) {
                store_row_chunk16<kKind>(p, Cb, row, col0 + c, h);
              }
            }
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
              store_row_chunk<kKind>(p, Cb, row, col0 + c, v, beta, use_c);
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
            store_row_chunk<kKind>(p, Cb, row, col0 + c, v, beta, use_c);
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

template <int kKind, bool kPair, bool kAT, bool kBT>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const TcArgs<kKind> p) {
  gemm_tc_body<kKind, kPair, kAT, kBT>(tmA, tmB, tmC, p);
}

// ------------------------------------------------------------------ host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn get_encode_fn() {
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
inline cuuint64_t matrix_stride_bytes(int64_t count, int64_t stride, int64_t rows, int64_t ld,
                                      int esize) {
  if (count > 1) return static_cast<cuuint64_t>(stride) * esize;
  return (static_cast<cuuint64_t>(rows) * ld * esize + 15) / 16 * 16;
}

// A stack of `count` row-major rows x cols matrices (element size esize, row
// stride ld and matrix stride `stride` in elements), in boxes of box_rows x
// box_cols elements with 128-byte swizzle (a box row is 128 bytes).
inline bool make_tmap(CUtensorMap *tm, CUtensorMapDataType dt, int esize, const void *base,
                      int64_t rows, int64_t cols, int64_t ld, int64_t count, int64_t stride,
                      uint32_t box_rows, uint32_t box_cols, bool l2_promote = true) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(count)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld) * esize,
                           matrix_stride_bytes(count, stride, rows, ld, esize)};
  cuuint32_t box[3] = {box_cols, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(tm, dt, 3, const_cast<void *>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   l2_promote ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B
                              : CU_TENSOR_MAP_L2_PROMOTION_NONE,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Co-resident CTA pairs for a pair kernel on this device (0 if pairs are not
// available), queried once per device and kernel.
inline int pair_capacity(const DeviceInfo &dev, const void *kern, size_t smem) {
  static std::mutex mu;
  static std::map<std::pair<const void *, int>, int> cache;
  std::lock_guard<std::mutex> lock(mu);
  const auto key = std::make_pair(kern, dev.device);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  int n = 0;
  if (set_max_dynamic_smem(kern, static_cast<int>(smem), dev.device) == cudaSuccess) {
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
  cache[key] = n;
  return n;
}

constexpr int kMaxSplit = DGR_TC_MAX_SPLIT;  // parts per tail tile (each adds one pass over C)
// Tail flags any one launch can need: two per split tile, and fewer tiles are
// split than there are units (at most one per SM).
constexpr size_t kTailFlagWords = 1024;

// The kernel for an operand form (only the forms a kind is built with).
template <int kKind, bool kPair, bool kAT, bool kBT>
constexpr auto tc_kernel() {
  return gemm_tc_kernel<kKind, kPair, kAT, kBT>;
}

// One tensor-core GEMM launch for element kind kKind. dt and ab_format are the
// inputs' TMA data type and MMA operand format, c_dt the 16-bit C's TMA data
// type (16-bit C only). Kinds built with every operand form take ops as given;
// the others must be called with the single form they are built with.
template <int kKind, bool kAllForms>
cudaError_t launch_tc(const DeviceInfo &dev, CUtensorMapDataType dt, uint32_t ab_format,
                      CUtensorMapDataType c_dt, const BatchOps &ops, int M, int N, int K,
                      typename TcKind<kKind>::Scale alpha, const void *A, int64_t lda,
                      const void *B, int64_t ldb, typename TcKind<kKind>::Scale beta,
                      typename TcKind<kKind>::Out *C, int64_t ldc, cudaStream_t stream,
                      uint32_t *flags_ws, size_t flags_words, const int32_t *row_corr = nullptr,
                      const int32_t *col_corr = nullptr, int32_t corr_const = 0,
                      bool flags_zeroed = false) {
  using K_ = TcKind<kKind>;
  constexpr int kEs = K_::kInBytes;
  constexpr int kBK = K_::kBK;
  static_assert(sizeof(TcSmem<true>) + 1024 <= 232448, "pair kernel shared memory");
  static_assert(sizeof(TcSmem<false>) + 1024 <= 232448, "single-CTA kernel shared memory");
  const size_t smem_pair = sizeof(TcSmem<true>) + 1024;
  const size_t smem_single = sizeof(TcSmem<false>) + 1024;

  // Kernel for this form.
  using Kern = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, TcArgs<kKind>);
  Kern kern_pair, kern_single;
  if constexpr (kAllForms) {
    if (ops.a_t) {
      kern_pair =
          ops.b_t ? tc_kernel<kKind, true, true, true>() : tc_kernel<kKind, true, true, false>();
      kern_single =
          ops.b_t ? tc_kernel<kKind, false, true, true>() : tc_kernel<kKind, false, true, false>();
    } else {
      kern_pair =
          ops.b_t ? tc_kernel<kKind, true, false, true>() : tc_kernel<kKind, true, false, false>();
      kern_single =
          ops.b_t ? tc_kernel<kKind, false, false, true>() : tc_kernel<kKind, false, false, false>();
    }
  } else if constexpr (kKind == kKindTF32) {
    if (ops.a_t || !ops.b_t) return cudaErrorInvalidValue;
    kern_pair = tc_kernel<kKind, true, false, true>();
    kern_single = tc_kernel<kKind, false, false, true>();
  } else {
    if (ops.a_t || ops.b_t) return cudaErrorInvalidValue;
    kern_pair = tc_kernel<kKind, true, false, false>();
    kern_single = tc_kernel<kKind, false, false, false>();
  }

  const int pairs =
      DGR_TC_PAIR ? pair_capacity(dev, reinterpret_cast<const void *>(kern_pair), smem_pair) : 0;
  const bool use_pairs = pairs > 0;
  const int tile_m = use_pairs ? Cfg<true>::kTileM : Cfg<false>::kTileM;
  const uint32_t bn_load = use_pairs ? Cfg<true>::kBNLoad : Cfg<false>::kBNLoad;

  // Operand tensor maps: one matrix, or one per batch entry.
  const int64_t batch = ops.batch;
  const int64_t na = (batch > 1 && ops.stride_a != 0) ? batch : 1;
  const int64_t nb = (batch > 1 && ops.stride_b != 0) ? batch : 1;
  CUtensorMap tmA, tmB;
  const bool maps_ok =
      (ops.a_t ? make_tmap(&tmA, dt, kEs, A, K, M, lda, na, ops.stride_a, kBK, K_::kMNElems)
               : make_tmap(&tmA, dt, kEs, A, M, K, lda, na, ops.stride_a, kBM, kBK)) &&
      (ops.b_t ? make_tmap(&tmB, dt, kEs, B, N, K, ldb, nb, ops.stride_b, bn_load, kBK)
               : make_tmap(&tmB, dt, kEs, B, K, N, ldb, nb, ops.stride_b, kBK, K_::kMNElems));
  if (!maps_ok) {
    if (na == 1 && nb == 1) return cudaErrorInvalidValue;
    // A stride the tensor-map encoder does not take (matrices that overlap):
    // one launch per batch entry, each on a single matrix.
    BatchOps one = ops;
    one.batch = 1;
    for (int64_t b = 0; b < batch; ++b) {
      const void *Ab = static_cast<const uint8_t *>(A) + b * ops.stride_a * kEs;
      const void *Bb = static_cast<const uint8_t *>(B) + b * ops.stride_b * kEs;
      cudaError_t e = launch_tc<kKind, kAllForms>(dev, dt, ab_format, c_dt, one, M, N, K, alpha,
                                                  Ab, lda, Bb, ldb, beta, C + b * ops.stride_c,
                                                  ldc, stream, nullptr, 0, row_corr, col_corr,
                                                  corr_const);
      if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
  }
  TcArgs<kKind> p;
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
  // C in whole 16-byte units: base, row stride and (for a stack) matrix stride.
  constexpr int kOutBytes = sizeof(typename K_::Out);
  constexpr int kPer16 = 16 / kOutBytes;
  p.c_vec_ok = (reinterpret_cast<uintptr_t>(C) % 16 == 0) && (ldc % kPer16 == 0);
  p.err_word = dev.err_word;
  p.tail_flags = nullptr;
  if constexpr (K_::kInt) {
    p.row_corr = row_corr;
    p.col_corr = col_corr;
    p.corr_const = corr_const;
  }
  // TMA stores of C need a 16-byte aligned base and row stride, and rows whose
  // length is a whole number of 16-byte units: a store box is clipped at the
  // right edge of C only in 16-byte units, so otherwise it would also write
  // the first columns of the row padding. A stack of C matrices also needs a
  // matrix stride of whole 16-byte units. Otherwise the epilogue writes C with
  // plain guarded stores.
  CUtensorMap tmC;
  std::memset(&tmC, 0, sizeof tmC);
  const CUtensorMapDataType cdt =
      K_::kOut16 ? c_dt
                 : (K_::kInt ? CU_TENSOR_MAP_DATA_TYPE_INT32 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32);
  p.c_tma = p.c_vec_ok && (N % kPer16 == 0) && (batch == 1 || ops.stride_c % kPer16 == 0) &&
            make_tmap(&tmC, cdt, kOutBytes, C, M, N, ldc, batch, ops.stride_c, 32,
                      128 / kOutBytes, false);
  p.idesc = idesc_mma(ab_format, ops.a_t, !ops.b_t, tile_m, kBN);
  const int64_t tiles = static_cast<int64_t>(p.tiles_per_batch) * batch;
  if (static_cast<int64_t>(p.tiles_m) * p.tiles_n > 0x7fffffffLL || tiles > 0x7fffffffLL)
    return cudaErrorInvalidValue;
  const int KB = (K + kBK - 1) / kBK;
  const int cap = use_pairs ? pairs : dev.sm_count;
  const int kb_unit = K_::kInt ? K_::kChunkK / kBK : 1;
  // 16-bit C: no k-split (partial sums would be rounded to 16 bits in between).
  const int max_split = K_::kOut16 ? 1 : kMaxSplit;
  int units = 0;
  plan_work(tiles, KB, kb_unit, cap, max_split, units, p.dp_tiles, p.tail_tiles, p.split);

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
    if (p.split > 1 && !(flags_zeroed && p.tail_flags == flags_ws)) {
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
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, kern_pair, tmA, tmB, tmC, p);
    if (e == cudaSuccess) e = cudaGetLastError();
  } else {
    e = set_max_dynamic_smem(reinterpret_cast<const void *>(kern_single),
                             static_cast<int>(smem_single), dev.device);
    if (e == cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(static_cast<unsigned>(units), 1, 1);
      cfg.blockDim = dim3(kThreads, 1, 1);
      cfg.dynamicSmemBytes = smem_single;
      cfg.stream = stream;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[0].val.programmaticStreamSerializationAllowed = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      e = cudaLaunchKernelEx(&cfg, kern_single, tmA, tmB, tmC, p);
      if (e == cudaSuccess) e = cudaGetLastError();
    }
  }
  if (pool_flags) {
    cudaError_t f = cudaFreeAsync(pool_flags, stream);
    if (e == cudaSuccess) e = f;
  }
  return e;
}

}  // namespace
}  // namespace dgr
