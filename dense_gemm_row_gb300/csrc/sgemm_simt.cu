// sgemm_simt.cu -- exact-fp32 SGEMM on the SIMT FP32 pipe, row-major.
//
//     C = alpha * A * B + beta * C
//
// Design (restated from the pages, rebuilt for sm_103a):
//  * One CTA computes a 128 x 128 tile of C; every thread owns 8 rows x TN
//    columns of it, in 4 x 4 blocks at row offsets {0, 64} and column offsets
//    128 / (TN / 4) apart, so that neighbouring threads touch neighbouring
//    16-byte chunks of C ("Sgemm [128,128,8]", the kernel's header comment:
//    256 threads, 128x128 tile, 8x8 per thread, cyclic distribution of C for
//    coalescing). Two shapes: TN = 8 (256 threads, the pages' shape) and
//    TN = 16 (128 threads, 8 x 16 per thread: half the shared loads per FMA),
//    both at two CTAs per SM.
//  * A is staged into shared memory transposed (k-major), so the eight A
//    values a thread needs for one k are two 16-byte shared loads ("Sgemm
//    [128,128,8]", the transposed smema buffer; "CUDA学习之路[11]", section
//    V3 双缓冲, the transposed A tile).
//  * Staging uses cp.async with an S-stage ring of BK-deep k tiles instead of
//    the pages' register prefetch plus two shared buffers: the same overlap of
//    the next tiles' loads with this tile's FMAs, without holding the prefetch
//    in registers. The transposing copy of A is 4 bytes per lane, arranged so
//    a warp's 32 stores hit 32 distinct banks.
//  * The FMAs of a thread are issued as packed fma.rn.f32x2 (two independent
//    fp32 FMAs, each rounded to nearest like fmaf), which halves the issue
//    slots the FP32 pipe needs on sm_103a.
//  * Residual tiles: out-of-range cells of the A and B tiles are filled with
//    zeros by the copy itself (cp.async with a zero source size) and the
//    epilogue's stores are guarded, so any M, N, K works ("使用CUDA和瓦片算法
//    计算矩阵乘法": residual tile cells must be zeroed; thread function's
//    guarded store).
//  * B is copied in 16-byte chunks when every chunk is either wholly inside or
//    wholly outside the matrix and 16-byte aligned (N % 4 == 0, ldb % 4 == 0,
//    aligned base); otherwise in 4-byte elements. The dlog page's float4
//    kernel (section V2 Tile) guards only the first element of each float4;
//    here a chunk is only used when that is safe.
//  * Epilogue: alpha*acc + beta*C with 16-byte accesses where aligned, scalar
//    guarded accesses at the edges. C is not read when beta == 0.
//  * Transposed operands and batches (the extended entry point): the shared
//    tiles keep their layouts (A k-major, B n-major), only the copies change.
//    A stored K x M is copied straight (16-byte chunks when aligned); B stored
//    N x K is copied with the same conflict-free transposing pattern as A
//    (its tile then also has a padded row stride of 132). The batch entry is
//    blockIdx.y.
//  * Grids of at least two waves of resident CTAs run TN = 16 with 8-deep k
//    tiles in a 6-stage ring (one CTA per tile); smaller single problems run
//    TN = 8 with 32-deep k tiles in a 2-stage ring on the persistent k-split
//    grid, where the extra warps per SM pay more than the wider thread tile.
#include <cstdint>

#include <cuda_runtime.h>

#include <map>
#include <mutex>
#include <tuple>
#include <type_traits>

#include "launch.h"
#include "ptx.cuh"
#include "work_split.cuh"

namespace dgr {
namespace {

#ifndef DGR_SIMT_FFMA2
#define DGR_SIMT_FFMA2 1
#endif

// (c0, c1) = (a * b0 + c0, a * b1 + c1) with one packed fp32 FMA.
__device__ __forceinline__ void ffma2(float &c0, float &c1, float a, float b0, float b1) {
  asm("{\n .reg .b64 ra, rb, rc;\n mov.b64 ra, {%2, %2};\n mov.b64 rb, {%3, %4};\n"
      " mov.b64 rc, {%0, %1};\n fma.rn.f32x2 rc, ra, rb, rc;\n mov.b64 {%0, %1}, rc;\n}\n"
      : "+f"(c0), "+f"(c1)
      : "f"(a), "f"(b0), "f"(b1));
}

constexpr int kBM = 128;
constexpr int kBN = 128;
constexpr int kGroupM = 8;  // tiles of M visited together (L2 reuse of B columns)

// Outputs per thread: 8 rows x TN columns (TN = 8: 256 threads; TN = 16: 128
// threads). Rows sit at offsets {0, 64}, columns in TN / 4 blocks of 4,
// 128 / (TN / 4) apart; lanes form a 4 x 8 grid, warps a grid of (64 / 16)
// rows x (block stride / 32) columns.
template <int TN>
struct SimtShape {
  static_assert(TN == 8 || TN == 16, "8 or 16 columns per thread");
  static constexpr int kThreads = kBM * kBN / (8 * TN);
  static constexpr int kColBlocks = TN / 4;
  static constexpr int kColStride = kBN / kColBlocks;  // 64 or 32
  static constexpr int kWarpsN = kColStride / 32;
};

struct SimtArgs {
  int M, N, K;
  float alpha, beta;
  const float *A;
  int64_t lda;
  const float *B;
  int64_t ldb;
  float *C;
  int64_t ldc;
  int64_t stride_a, stride_b, stride_c;  // elements between batch entries (blockIdx.y)
  int tiles_m, tiles_n;
  int c_vec_ok;  // C 16-byte aligned and ldc % 4 == 0
  // Persistent single-problem form: the work split (work_split.cuh) and the
  // tail flags (zero at launch), and the device error word for bounded waits.
  int dp_tiles, tail_tiles, split;
  uint32_t *tail_flags;
  uint32_t *err_word;
};

// Row stride of the transposed A tile: 132 = 128 + 4 floats. With it, the
// 4-byte copies of one warp (4 rows x 8 consecutive k) land in 32 distinct
// banks, and every 4-float group stays 16-byte aligned for the fragment loads.
constexpr int kAStride = kBM + 4;

template <int BK, int STAGES, int BStride>
struct SimtSmem {
  float a[STAGES][BK][kAStride];  // A tile, transposed: a[s][k][m]
  float b[STAGES][BK][BStride];   // B tile: b[s][k][n]
};

// Linear CTA index -> (tile_m, tile_n): groups of kGroupM tile rows are walked
// column by column, so CTAs resident together share B columns and A rows in L2.
__device__ __forceinline__ void tile_coords(int bid, int tiles_m, int tiles_n, int &tm, int &tn) {
  const int per_group = kGroupM * tiles_n;
  const int g = bid / per_group;
  const int first = g * kGroupM;
  const int rows = min(tiles_m - first, kGroupM);
  const int r = bid - g * per_group;
  tm = first + r % rows;
  tn = r / rows;
}

// Copies a 4 x 8 (rows x k) block per warp instruction from a row-major matrix
// whose rows run along k into the k-major tile dst[k][row] (row stride 132):
// lane = 8 * row + k, so one warp reads four 32-byte segments and its 32
// stores hit 32 distinct banks. rows_valid / k_valid bound the source. Each
// of the THREADS threads issues kCount copies; one() issues copy number c.
template <int BK, int THREADS>
struct TransposingCopy {
  static_assert(BK % 8 == 0, "transposing copies take k in groups of 8");
  static constexpr int kCount = 4 * BK / (THREADS / 32);
  __device__ static __forceinline__ void one(int c, const float *src, int64_t ld,
                                             float (*dst)[kAStride], int r0, int k0,
                                             int rows_valid, int k_valid, int tid) {
    constexpr int kGroupsK = BK / 8;
    const int warp = tid >> 5, lane = tid & 31;
    const int pair = warp * kCount + c;                // 0 .. 4*BK-1
    const int r = (pair / kGroupsK) * 4 + (lane >> 3);  // 32 groups of 4 rows
    const int k = (pair % kGroupsK) * 8 + (lane & 7);   // groups of 8 k
    const int gr = r0 + r, gk = k0 + k;
    const bool ok = gr < rows_valid && gk < k_valid;
    const float *p = ok ? src + static_cast<int64_t>(gr) * ld + gk : src;
    cp_async_4(smem_u32(&dst[k][r]), p, ok ? 4u : 0u);
  }
};

// Copies rows k0 .. k0+BK-1, columns c0 .. c0+127 of a row-major matrix whose
// rows run along k straight into dst[k][col]: 16-byte chunks when VEC (every
// chunk then lies wholly inside or outside the matrix), 4-byte elements
// otherwise. Each of the THREADS threads issues kCount copies.
template <int BK, bool VEC, int Stride, int THREADS>
struct StraightCopy {
  static constexpr int kCount = VEC ? BK * 128 / 4 / THREADS : BK * 128 / THREADS;
  __device__ static __forceinline__ void one(int c, const float *src, int64_t ld,
                                             float (*dst)[Stride], int k0, int c0, int k_valid,
                                             int c_valid, int tid) {
    const int e = tid + c * THREADS;
    const int row = VEC ? e >> 5 : e >> 7;
    const int col = VEC ? (e & 31) * 4 : e & 127;
    const int gk = k0 + row, gc = c0 + col;
    const bool ok = gk < k_valid && gc < c_valid;
    const float *p = ok ? src + static_cast<int64_t>(gk) * ld + gc : src;
    if constexpr (VEC)
      cp_async_16(smem_u32(&dst[row][col]), p, ok ? 16u : 0u);
    else
      cp_async_4(smem_u32(&dst[row][col]), p, ok ? 4u : 0u);
  }
};

// One BK-deep stage: the A tile (k-major, 128 rows of op(A)) and the B tile
// (k rows x 128 columns of op(B)). A_T / B_T: the operand is stored
// transposed; VEC_A / VEC_B: its straight copy may use 16-byte chunks.
template <int BK, int THREADS, bool A_T, bool VEC_A, bool B_T, bool VEC_B, int BStride>
__device__ __forceinline__ void load_tile(const SimtArgs &p, const float *A, const float *B,
                                          float (*sa)[kAStride], float (*sb)[BStride], int m0,
                                          int n0, int k0, int tid) {
  using CA = typename std::conditional<A_T, StraightCopy<BK, VEC_A, kAStride, THREADS>,
                                       TransposingCopy<BK, THREADS>>::type;
  using CB = typename std::conditional<B_T, TransposingCopy<BK, THREADS>,
                                       StraightCopy<BK, VEC_B, BStride, THREADS>>::type;
#pragma unroll
  for (int c = 0; c < CA::kCount; ++c) {
    if constexpr (A_T)
      CA::one(c, A, p.lda, sa, k0, m0, p.K, p.M, tid);  // stored K x M
    else
      CA::one(c, A, p.lda, sa, m0, k0, p.M, p.K, tid);  // stored M x K
  }
#pragma unroll
  for (int c = 0; c < CB::kCount; ++c) {
    if constexpr (B_T)
      CB::one(c, B, p.ldb, sb, n0, k0, p.N, p.K, tid);  // stored N x K
    else
      CB::one(c, B, p.ldb, sb, k0, n0, p.K, p.N, tid);  // stored K x N
  }
}

// The k-loop of one 128 x 128 tile at (m0, n0) over k-tiles [kt0, kt1):
// acc += op(A) op(B) over those k. Leaves shared memory free for the next
// tile (every copy waited for, every thread past its last read). The k-tile's
// loop is unrolled whole, so the compiler schedules each k's shared loads
// ahead of the previous k's FMAs.
template <int TN, int BK, int STAGES, bool A_T, bool VEC_A, bool B_T, bool VEC_B, int BStride>
__device__ __forceinline__ void tile_mainloop(const SimtArgs &p, const float *A, const float *B,
                                              SimtSmem<BK, STAGES, BStride> &sm, int m0, int n0,
                                              int kt0, int kt1, int tid, int rm, int cn,
                                              float (&acc)[8][TN]) {
  using Sh = SimtShape<TN>;
  const int KT = kt1 - kt0;
#pragma unroll
  for (int s = 0; s < STAGES - 1; ++s) {
    if (s < KT)
      load_tile<BK, Sh::kThreads, A_T, VEC_A, B_T, VEC_B, BStride>(p, A, B, sm.a[s], sm.b[s], m0,
                                                                  n0, (kt0 + s) * BK, tid);
    cp_async_commit();
  }
  for (int kt = 0; kt < KT; ++kt) {
    cp_async_wait<STAGES - 2>();
    __syncthreads();  // tile kt landed for everyone; tile kt-1 fully consumed
    {
      const int nt = kt + STAGES - 1;
      if (nt < KT) {
        const int s = nt % STAGES;
        load_tile<BK, Sh::kThreads, A_T, VEC_A, B_T, VEC_B, BStride>(
            p, A, B, sm.a[s], sm.b[s], m0, n0, (kt0 + nt) * BK, tid);
      }
      cp_async_commit();
    }
    const int s = kt % STAGES;
#pragma unroll
    for (int k = 0; k < BK; ++k) {
      const float4 a_lo = *reinterpret_cast<const float4 *>(&sm.a[s][k][rm]);
      const float4 a_hi = *reinterpret_cast<const float4 *>(&sm.a[s][k][rm + 64]);
      const float a[8] = {a_lo.x, a_lo.y, a_lo.z, a_lo.w, a_hi.x, a_hi.y, a_hi.z, a_hi.w};
      float b[TN];
#pragma unroll
      for (int q = 0; q < Sh::kColBlocks; ++q) {
        const float4 v = *reinterpret_cast<const float4 *>(&sm.b[s][k][cn + q * Sh::kColStride]);
        b[4 * q] = v.x;
        b[4 * q + 1] = v.y;
        b[4 * q + 2] = v.z;
        b[4 * q + 3] = v.w;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
#if DGR_SIMT_FFMA2
        // Two lanes of one row per instruction: (acc[i][j], acc[i][j+1]) +=
        // a[i] * (b[j], b[j+1]); one IEEE round-to-nearest per lane, as fmaf.
#pragma unroll
        for (int j = 0; j < TN; j += 2) ffma2(acc[i][j], acc[i][j + 1], a[i], b[j], b[j + 1]);
#else
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
#endif
      }
    }
  }
  cp_async_wait<0>();
  __syncthreads();  // no thread still reads the ring when the next tile's copies start
}

// C[tile] = alpha * acc + beta * C (the C term only when use_c; beta = 1 when
// a later k-part adds to what an earlier one stored). C is read through L2
// (another CTA may have just written it).
template <int TN>
__device__ __forceinline__ void tile_epilogue(const SimtArgs &p, float *C, int m0, int n0, int rm,
                                              int cn, const float (&acc)[8][TN], float beta,
                                              bool use_c) {
  using Sh = SimtShape<TN>;
  const float alpha = p.alpha;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int row = m0 + rm + (i & 3) + (i >> 2) * 64;
    if (row >= p.M) continue;
    float *crow = C + static_cast<int64_t>(row) * p.ldc;
#pragma unroll
    for (int h = 0; h < Sh::kColBlocks; ++h) {
      const int col = n0 + cn + h * Sh::kColStride;
      const float *v = &acc[i][h * 4];
      if (p.c_vec_ok && col + 3 < p.N) {
        float4 out;
        if (use_c) {
          const float4 c = __ldcg(reinterpret_cast<const float4 *>(crow + col));
          out = make_float4(alpha * v[0] + beta * c.x, alpha * v[1] + beta * c.y,
                            alpha * v[2] + beta * c.z, alpha * v[3] + beta * c.w);
        } else {
          out = make_float4(alpha * v[0], alpha * v[1], alpha * v[2], alpha * v[3]);
        }
        *reinterpret_cast<float4 *>(crow + col) = out;
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (col + j < p.N) {
            const float r = alpha * v[j];
            crow[col + j] = use_c ? r + beta * __ldcg(crow + col + j) : r;
          }
        }
      }
    }
  }
}

// Grid forms of the kernel.
constexpr int kModeTile = 0;     // one problem, one CTA per tile
constexpr int kModeBatch = 1;    // one CTA per tile, blockIdx.y = batch entry
constexpr int kModeSplit = 2;    // one problem, persistent CTAs over a k-split work list

// kModeSplit: a persistent grid of at most the co-resident CTAs walks the work
// list of work_split.cuh (whole tiles, then the last wave's leftover tiles
// split along k, parts added in order). For grids of fewer than two waves;
// with more, one CTA per tile measures faster (CTAs that start together stay
// in step, and their loads stop overlapping each other's arithmetic).
template <int TN, int BK, int STAGES, bool A_T, bool VEC_A, bool B_T, bool VEC_B, int MODE>
__global__ void __launch_bounds__(SimtShape<TN>::kThreads, 2)
    sgemm_simt_kernel(const SimtArgs p) {
  using Sh = SimtShape<TN>;
  constexpr int kBStride = B_T ? kAStride : kBN;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  auto &sm = *reinterpret_cast<SimtSmem<BK, STAGES, kBStride> *>(smem_raw);

  const int tid = threadIdx.x;
  // Thread -> 8 x TN outputs: rows rm..rm+3 and 64+rm..64+rm+3, columns
  // cn..cn+3 plus multiples of the column-block stride (SimtShape).
  const int warp = tid >> 5, lane = tid & 31;
  const int rm = (warp / Sh::kWarpsN) * 16 + (lane >> 3) * 4;
  const int cn = (warp % Sh::kWarpsN) * 32 + (lane & 7) * 4;
  const int KT = (p.K + BK - 1) / BK;
  float acc[8][TN];

  if constexpr (MODE != kModeSplit) {
    // The operand addresses of a single problem stay in the parameter bank.
    const float *A = MODE == kModeBatch ? p.A + blockIdx.y * p.stride_a : p.A;
    const float *B = MODE == kModeBatch ? p.B + blockIdx.y * p.stride_b : p.B;
    float *C = MODE == kModeBatch ? p.C + blockIdx.y * p.stride_c : p.C;
    int tm, tn;
    tile_coords(blockIdx.x, p.tiles_m, p.tiles_n, tm, tn);
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < TN; ++j) acc[i][j] = 0.f;
    tile_mainloop<TN, BK, STAGES, A_T, VEC_A, B_T, VEC_B, kBStride>(p, A, B, sm, tm * kBM,
                                                                    tn * kBN, 0, KT, tid, rm, cn,
                                                                    acc);
    tile_epilogue<TN>(p, C, tm * kBM, tn * kBN, rm, cn, acc, p.beta, p.beta != 0.f);
  } else {
    __shared__ int abort;
    if (tid == 0) abort = 0;
    const int units = static_cast<int>(gridDim.x);
    WorkItem w;
    for (int n = 0; get_work(static_cast<int>(blockIdx.x), n, units, p.dp_tiles, p.tail_tiles,
                             p.split, KT, 1, w);
         ++n) {
      int tm, tn;
      tile_coords(w.tile, p.tiles_m, p.tiles_n, tm, tn);
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = 0.f;
      tile_mainloop<TN, BK, STAGES, A_T, VEC_A, B_T, VEC_B, kBStride>(
          p, p.A, p.B, sm, tm * kBM, tn * kBN, w.kb0, w.kb1, tid, rm, cn, acc);
      if (w.parts == 1) {
        tile_epilogue<TN>(p, p.C, tm * kBM, tn * kBN, rm, cn, acc, p.beta, p.beta != 0.f);
        continue;
      }
      // k-split tile: part j adds after part j - 1 has stored (in order).
      uint32_t *flag = p.tail_flags + (w.tile - p.dp_tiles);
      if (w.part > 0) {
        if (tid == 0) wait_flag(flag, static_cast<uint32_t>(w.part), &abort, p.err_word);
        __syncthreads();
        tile_epilogue<TN>(p, p.C, tm * kBM, tn * kBN, rm, cn, acc, 1.f, true);
      } else {
        tile_epilogue<TN>(p, p.C, tm * kBM, tn * kBN, rm, cn, acc, p.beta, p.beta != 0.f);
      }
      __threadfence();
      __syncthreads();  // every thread's part of the tile is stored and visible
      if (tid == 0) st_release_gpu(flag, static_cast<uint32_t>(w.part + 1));
    }
  }
}

// CTAs of `kern` (blocks of `threads`) that can be resident at once on the
// device (cached).
int resident_ctas(const DeviceInfo &dev, const void *kern, int threads, size_t smem) {
  static std::mutex mu;
  static std::map<std::tuple<const void *, int>, int> cache;
  std::lock_guard<std::mutex> lock(mu);
  const auto key = std::make_tuple(kern, dev.device);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem) != cudaSuccess)
    per_sm = 0;
  cudaGetLastError();
  const int n = per_sm * dev.sm_count;
  cache[key] = n;
  return n;
}

constexpr int kSimtMaxSplit = 4;  // parts per leftover tile (each adds one pass over its C)
constexpr int kTransposeBMinM = 1024;  // rows from which a transposed B is transposed first
constexpr int kTransposeAMinN = 2048;  // columns from which A is transposed first

// The two kernel shapes: full grids (TN = 16, 8-deep k tiles, 6 stages) and
// under-filled single problems on the k-split grid (TN = 8, 32-deep, 2 stages).
#ifndef DGR_SIMT_WIDE_BK
#define DGR_SIMT_WIDE_BK 8
#endif
#ifndef DGR_SIMT_WIDE_STAGES
#define DGR_SIMT_WIDE_STAGES 6
#endif
struct SimtWide {
  static constexpr int kTN = 16, kBK = DGR_SIMT_WIDE_BK, kStages = DGR_SIMT_WIDE_STAGES;
};
struct SimtNarrow {
  static constexpr int kTN = 8, kBK = 32, kStages = 2;
};

template <class CFG, bool A_T, bool VEC_A, bool B_T, bool VEC_B, int MODE = kModeBatch>
cudaError_t launch_variant(const SimtArgs &a_in, int batch, const DeviceInfo &dev,
                           cudaStream_t stream) {
  constexpr int kTN = CFG::kTN, kBK = CFG::kBK, kStages = CFG::kStages;
  constexpr int kThreads = SimtShape<kTN>::kThreads;
  constexpr size_t smem = sizeof(SimtSmem<kBK, kStages, B_T ? kAStride : kBN>);
  auto kern = sgemm_simt_kernel<kTN, kBK, kStages, A_T, VEC_A, B_T, VEC_B, MODE>;
  cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void *>(kern),
                                       static_cast<int>(smem), dev.device);
  if (e != cudaSuccess) return e;
  SimtArgs a = a_in;
  a.err_word = dev.err_word;
  a.tail_flags = nullptr;
  const int64_t blocks = static_cast<int64_t>(a.tiles_m) * a.tiles_n;
  if constexpr (MODE == kModeSplit) {
    // Persistent grid over the co-resident CTAs, the last wave split along k.
    const int cap = resident_ctas(dev, reinterpret_cast<const void *>(kern), kThreads, smem);
    if (cap <= 0) return cudaErrorLaunchOutOfResources;
    const int KT = (a.K + kBK - 1) / kBK;
    int units = 0;
    plan_work(blocks, KT, 1, cap, kSimtMaxSplit, units, a.dp_tiles, a.tail_tiles, a.split);
    void *flags = nullptr;
    if (a.split > 1) {
      cudaMemPool_t pool;
      e = device_pool(dev, &pool);
      if (e != cudaSuccess) return e;
      const size_t bytes = static_cast<size_t>(a.tail_tiles) * 4;
      e = cudaMallocFromPoolAsync(&flags, bytes, pool, stream);
      if (e != cudaSuccess) return e;
      e = cudaMemsetAsync(flags, 0, bytes, stream);
      a.tail_flags = static_cast<uint32_t *>(flags);
    }
    if (e == cudaSuccess) {
      kern<<<static_cast<unsigned>(units), kThreads, smem, stream>>>(a);
      e = cudaGetLastError();
    }
    if (flags) {
      cudaError_t f = cudaFreeAsync(flags, stream);
      if (e == cudaSuccess) e = f;
    }
    return e;
  }
  // The batch runs on gridDim.y, at most 65535 entries per launch.
  constexpr int kMaxY = 65535;
  for (int b0 = 0; b0 < batch; b0 += kMaxY) {
    SimtArgs c = a;
    c.A += b0 * a.stride_a;
    c.B += b0 * a.stride_b;
    c.C += b0 * a.stride_c;
    const unsigned ny = static_cast<unsigned>(batch - b0 < kMaxY ? batch - b0 : kMaxY);
    kern<<<dim3(static_cast<unsigned>(blocks), ny), kThreads, smem, stream>>>(c);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

template <class CFG, bool A_T, bool VEC_A>
cudaError_t launch_b(const SimtArgs &a, bool b_t, bool vec_b, int batch, const DeviceInfo &dev,
                     cudaStream_t stream) {
  if (b_t) return launch_variant<CFG, A_T, VEC_A, true, false>(a, batch, dev, stream);
  return vec_b ? launch_variant<CFG, A_T, VEC_A, false, true>(a, batch, dev, stream)
               : launch_variant<CFG, A_T, VEC_A, false, false>(a, batch, dev, stream);
}

template <class CFG>
cudaError_t launch_ops(const SimtArgs &a, bool a_t, bool vec_a, bool b_t, bool vec_b, int batch,
                       const DeviceInfo &dev, cudaStream_t stream) {
  if (!a_t) return launch_b<CFG, false, false>(a, b_t, vec_b, batch, dev, stream);
  return vec_a ? launch_b<CFG, true, true>(a, b_t, vec_b, batch, dev, stream)
               : launch_b<CFG, true, false>(a, b_t, vec_b, batch, dev, stream);
}

// 16-byte chunks of a straight copy are safe when the stored matrix (and every
// matrix of a stack) starts 16-byte aligned, its rows are whole 16-byte units
// apart, and its row length `cols` is a multiple of 4 (a chunk never straddles
// the right edge).
bool vec_ok(const float *base, int64_t ld, int64_t cols, int batch, int64_t stride) {
  return (reinterpret_cast<uintptr_t>(base) % 16 == 0) && (ld % 4 == 0) && (cols % 4 == 0) &&
         (batch == 1 || stride % 4 == 0);
}

}  // namespace

namespace {

// The fp32 GEMM; transpose_first enables the one-off transposition of a
// stored-transposed B or a stored A into pool scratch on large problems.
cudaError_t sgemm_simt_run(const DeviceInfo &dev, const BatchOps &ops, int M, int N, int K,
                           float alpha, const float *A, int64_t lda, const float *B, int64_t ldb,
                           float beta, float *C, int64_t ldc, cudaStream_t stream,
                           bool transpose_first) {
  SimtArgs a;
  a.M = M;
  a.N = N;
  a.K = K;
  a.alpha = alpha;
  a.beta = beta;
  a.A = A;
  a.lda = lda;
  a.B = B;
  a.ldb = ldb;
  a.C = C;
  a.ldc = ldc;
  const int batch = ops.batch;
  a.stride_a = batch > 1 ? ops.stride_a : 0;
  a.stride_b = batch > 1 ? ops.stride_b : 0;
  a.stride_c = batch > 1 ? ops.stride_c : 0;
  a.tiles_m = (M + kBM - 1) / kBM;
  a.tiles_n = (N + kBN - 1) / kBN;
  a.c_vec_ok = (reinterpret_cast<uintptr_t>(C) % 16 == 0) && (ldc % 4 == 0) &&
               (batch == 1 || a.stride_c % 4 == 0);
  if (static_cast<int64_t>(a.tiles_m) * a.tiles_n > 0x7fffffffLL) return cudaErrorInvalidValue;
  const bool vec_a = ops.a_t && vec_ok(A, lda, M, batch, a.stride_a);
  const bool vec_b = !ops.b_t && vec_ok(B, ldb, N, batch, a.stride_b);
  // Fewer CTAs than two waves of resident CTAs (2 per SM): a single problem
  // takes the persistent k-split form of the 256-thread shape, a batch or a
  // transposed problem the 256-thread shape one CTA per tile. Otherwise the
  // 128-thread shape, one CTA per tile.
  const int64_t ctas = static_cast<int64_t>(a.tiles_m) * a.tiles_n * batch;
  const bool full = ctas >= 4LL * dev.sm_count;
  // B stored N x K, one problem, a full grid and many rows: B is transposed
  // once into pool scratch (N K values read and written, against the M N K
  // product) and the problem runs with the straight, 16-byte B copy, which
  // measures faster than the transposing one.
  if (transpose_first && ops.b_t && batch == 1 && full && M >= kTransposeBMinM) {
    const int64_t ldn = (static_cast<int64_t>(N) + 3) / 4 * 4;
    cudaMemPool_t pool = nullptr;
    cudaError_t e = device_pool(dev, &pool);
    if (e != cudaSuccess) return e;
    void *scratch = nullptr;
    e = cudaMallocFromPoolAsync(&scratch, static_cast<size_t>(K) * ldn * 4, pool, stream);
    if (e == cudaErrorMemoryAllocation) {  // no room for the copy: the transposing copy path
      cudaGetLastError();
      return sgemm_simt_run(dev, ops, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream, false);
    }
    if (e != cudaSuccess) return e;
    float *bt = static_cast<float *>(scratch);
    e = launch_transpose_f32(dev, B, ldb, N, K, bt, ldn, stream);  // stored N x K -> K x N
    if (e == cudaSuccess) {
      BatchOps straight = ops;
      straight.b_t = false;
      e = sgemm_simt_run(dev, straight, M, N, K, alpha, A, lda, bt, ldn, beta, C, ldc, stream,
                         true);
    }
    cudaError_t f = cudaFreeAsync(scratch, stream);
    return e != cudaSuccess ? e : f;
  }
  // Likewise A stored M x K with many columns: A transposed once (M K values,
  // against the M N K product) lets the k-major A tile be filled by the straight
  // 16-byte copy instead of the 4-byte transposing one.
  if (transpose_first && !ops.a_t && batch == 1 && full && N >= kTransposeAMinN) {
    const int64_t ldm = (static_cast<int64_t>(M) + 3) / 4 * 4;
    cudaMemPool_t pool = nullptr;
    cudaError_t e = device_pool(dev, &pool);
    if (e != cudaSuccess) return e;
    void *scratch = nullptr;
    e = cudaMallocFromPoolAsync(&scratch, static_cast<size_t>(K) * ldm * 4, pool, stream);
    if (e == cudaErrorMemoryAllocation) {  // no room for the copy: the transposing copy path
      cudaGetLastError();
      return sgemm_simt_run(dev, ops, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream, false);
    }
    if (e != cudaSuccess) return e;
    float *at = static_cast<float *>(scratch);
    e = launch_transpose_f32(dev, A, lda, M, K, at, ldm, stream);  // M x K -> K x M
    if (e == cudaSuccess) {
      BatchOps straight = ops;
      straight.a_t = true;
      e = sgemm_simt_run(dev, straight, M, N, K, alpha, at, ldm, B, ldb, beta, C, ldc, stream,
                         true);
    }
    cudaError_t f = cudaFreeAsync(scratch, stream);
    return e != cudaSuccess ? e : f;
  }
  if (ops.plain()) {  // one problem, no transposes
    if (!full)
      return vec_b ? launch_variant<SimtNarrow, false, false, false, true, kModeSplit>(a, 1, dev,
                                                                                      stream)
                   : launch_variant<SimtNarrow, false, false, false, false, kModeSplit>(
                         a, 1, dev, stream);
    return vec_b ? launch_variant<SimtWide, false, false, false, true, kModeTile>(a, 1, dev,
                                                                                 stream)
                 : launch_variant<SimtWide, false, false, false, false, kModeTile>(a, 1, dev,
                                                                                  stream);
  }
  return full ? launch_ops<SimtWide>(a, ops.a_t, vec_a, ops.b_t, vec_b, batch, dev, stream)
              : launch_ops<SimtNarrow>(a, ops.a_t, vec_a, ops.b_t, vec_b, batch, dev, stream);
}

}  // namespace

cudaError_t launch_sgemm_simt_ex(const DeviceInfo &dev, const BatchOps &ops, int M, int N, int K,
                                 float alpha, const float *A, int64_t lda, const float *B,
                                 int64_t ldb, float beta, float *C, int64_t ldc,
                                 cudaStream_t stream) {
  return sgemm_simt_run(dev, ops, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream, true);
}

cudaError_t launch_sgemm_simt(const DeviceInfo &dev, int M, int N, int K, float alpha,
                              const float *A, int64_t lda, const float *B, int64_t ldb,
                              float beta, float *C, int64_t ldc, cudaStream_t stream) {
  return launch_sgemm_simt_ex(dev, BatchOps(), M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
                              stream);
}

}  // namespace dgr
