// sgemm_simt.cu -- exact-fp32 SGEMM on the SIMT FP32 pipe, row-major.
//
//     C = alpha * A * B + beta * C
//
// Design (restated from the pages, rebuilt for sm_103a):
//  * One CTA of 256 threads computes a 128 x 128 tile of C; every thread owns
//    8 x 8 outputs split into four 4 x 4 blocks at row offsets {0, 64} and
//    column offsets {0, 64}, so that neighbouring threads touch neighbouring
//    16-byte chunks of C ("Sgemm [128,128,8]", the kernel's header comment:
//    256 threads, 128x128 tile, 8x8 per thread, cyclic distribution of C for
//    coalescing).
//  * A is staged into shared memory transposed (k-major), so the eight A
//    values a thread needs for one k are two 16-byte shared loads ("Sgemm
//    [128,128,8]", the transposed smema buffer; "CUDA学习之路[11]", section
//    V3 双缓冲, the transposed A tile).
//  * Staging uses cp.async with an S-stage ring (default: two stages of 32
//    values of k) instead of the pages' register prefetch plus two shared
//    buffers: the same overlap of the next tile's load with this tile's FMAs,
//    without holding the prefetch in registers. The transposing copy of A is
//    4 bytes per lane, arranged so a warp's 32 stores hit 32 distinct banks.
//  * The 64 FMAs per k of a thread are issued as 32 packed fma.rn.f32x2
//    (two independent fp32 FMAs, each rounded to nearest like fmaf), which
//    halves the issue slots the FP32 pipe needs on sm_103a.
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
#include <cstdint>

#include <cuda_runtime.h>

#include <map>
#include <mutex>
#include <utility>

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
constexpr int kThreads = 256;
constexpr int kGroupM = 8;  // tiles of M visited together (L2 reuse of B columns)

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
// stores hit 32 distinct banks. rows_valid / k_valid bound the source.
template <int BK>
__device__ __forceinline__ void copy_transposing(const float *src, int64_t ld, float (*dst)[kAStride],
                                                 int r0, int k0, int rows_valid, int k_valid,
                                                 int tid) {
  static_assert(BK % 8 == 0, "transposing copies take k in groups of 8");
  constexpr int kGroupsK = BK / 8;
  const int warp = tid >> 5, lane = tid & 31;
  const int r_lo = lane >> 3, k_lo = lane & 7;
#pragma unroll
  for (int i = 0; i < BK / 2; ++i) {
    const int pair = warp * (BK / 2) + i;        // 0 .. 4*BK-1
    const int r = (pair / kGroupsK) * 4 + r_lo;   // 32 groups of 4 rows
    const int k = (pair % kGroupsK) * 8 + k_lo;   // groups of 8 k
    const int gr = r0 + r, gk = k0 + k;
    const bool ok = gr < rows_valid && gk < k_valid;
    const float *p = ok ? src + static_cast<int64_t>(gr) * ld + gk : src;
    cp_async_4(smem_u32(&dst[k][r]), p, ok ? 4u : 0u);
  }
}

// Copies rows k0 .. k0+BK-1, columns c0 .. c0+127 of a row-major matrix whose
// rows run along k straight into dst[k][col]: 16-byte chunks when VEC (every
// chunk then lies wholly inside or outside the matrix), 4-byte elements
// otherwise.
template <int BK, bool VEC, int Stride>
__device__ __forceinline__ void copy_straight(const float *src, int64_t ld, float (*dst)[Stride],
                                              int k0, int c0, int k_valid, int c_valid, int tid) {
  if constexpr (VEC) {
    constexpr int kChunks = BK * 128 / 4 / kThreads;
#pragma unroll
    for (int i = 0; i < kChunks; ++i) {
      const int c = tid + i * kThreads;
      const int row = c >> 5;
      const int col = (c & 31) * 4;
      const int gk = k0 + row, gc = c0 + col;
      const bool ok = gk < k_valid && gc < c_valid;
      const float *p = ok ? src + static_cast<int64_t>(gk) * ld + gc : src;
      cp_async_16(smem_u32(&dst[row][col]), p, ok ? 16u : 0u);
    }
  } else {
    constexpr int kPer = BK * 128 / kThreads;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int e = tid + i * kThreads;
      const int row = e >> 7;
      const int col = e & 127;
      const int gk = k0 + row, gc = c0 + col;
      const bool ok = gk < k_valid && gc < c_valid;
      const float *p = ok ? src + static_cast<int64_t>(gk) * ld + gc : src;
      cp_async_4(smem_u32(&dst[row][col]), p, ok ? 4u : 0u);
    }
  }
}

// One BK-deep stage: the A tile (k-major, 128 rows of op(A)) and the B tile
// (k rows x 128 columns of op(B)). A_T / B_T: the operand is stored
// transposed; VEC_A / VEC_B: its straight copy may use 16-byte chunks.
template <int BK, bool A_T, bool VEC_A, bool B_T, bool VEC_B, int BStride>
__device__ __forceinline__ void load_tile(const SimtArgs &p, const float *A, const float *B,
                                          float (*sa)[kAStride], float (*sb)[BStride], int m0,
                                          int n0, int k0, int tid) {
  if constexpr (A_T) {
    copy_straight<BK, VEC_A, kAStride>(A, p.lda, sa, k0, m0, p.K, p.M, tid);  // stored K x M
  } else {
    copy_transposing<BK>(A, p.lda, sa, m0, k0, p.M, p.K, tid);  // stored M x K
  }
  if constexpr (B_T) {
    copy_transposing<BK>(B, p.ldb, sb, n0, k0, p.N, p.K, tid);  // stored N x K
  } else {
    copy_straight<BK, VEC_B, BStride>(B, p.ldb, sb, k0, n0, p.K, p.N, tid);  // stored K x N
  }
}

// The k-loop of one 128 x 128 tile at (m0, n0) over k-tiles [kt0, kt1):
// acc += op(A) op(B) over those k. Leaves shared memory free for the next
// tile (every copy waited for, every thread past its last read).
template <int BK, int STAGES, bool A_T, bool VEC_A, bool B_T, bool VEC_B, int BStride>
__device__ __forceinline__ void tile_mainloop(const SimtArgs &p, const float *A, const float *B,
                                              SimtSmem<BK, STAGES, BStride> &sm, int m0, int n0,
                                              int kt0, int kt1, int tid, int rm, int cn,
                                              float (&acc)[8][8]) {
  const int KT = kt1 - kt0;
#pragma unroll
  for (int s = 0; s < STAGES - 1; ++s) {
    if (s < KT)
      load_tile<BK, A_T, VEC_A, B_T, VEC_B, BStride>(p, A, B, sm.a[s], sm.b[s], m0, n0,
                                                      (kt0 + s) * BK, tid);
    cp_async_commit();
  }

  for (int kt = 0; kt < KT; ++kt) {
    cp_async_wait<STAGES - 2>();
    __syncthreads();  // tile kt landed for everyone; tile kt-1 fully consumed
    {
      const int nt = kt + STAGES - 1;
      if (nt < KT) {
        const int s = nt % STAGES;
        load_tile<BK, A_T, VEC_A, B_T, VEC_B, BStride>(p, A, B, sm.a[s], sm.b[s], m0, n0,
                                                        (kt0 + nt) * BK, tid);
      }
      cp_async_commit();
    }
    const int s = kt % STAGES;
#pragma unroll
    for (int k = 0; k < BK; ++k) {
      const float4 a_lo = *reinterpret_cast<const float4 *>(&sm.a[s][k][rm]);
      const float4 a_hi = *reinterpret_cast<const float4 *>(&sm.a[s][k][rm + 64]);
      const float4 b_lo = *reinterpret_cast<const float4 *>(&sm.b[s][k][cn]);
      const float4 b_hi = *reinterpret_cast<const float4 *>(&sm.b[s][k][cn + 64]);
      const float a[8] = {a_lo.x, a_lo.y, a_lo.z, a_lo.w, a_hi.x, a_hi.y, a_hi.z, a_hi.w};
      const float b[8] = {b_lo.x, b_lo.y, b_lo.z, b_lo.w, b_hi.x, b_hi.y, b_hi.z, b_hi.w};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
#if DGR_SIMT_FFMA2
        // Two lanes of one row per instruction: (acc[i][j], acc[i][j+1]) +=
        // a[i] * (b[j], b[j+1]); one IEEE round-to-nearest per lane, as fmaf.
#pragma unroll
        for (int j = 0; j < 8; j += 2) ffma2(acc[i][j], acc[i][j + 1], a[i], b[j], b[j + 1]);
#else
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
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
__device__ __forceinline__ void tile_epilogue(const SimtArgs &p, float *C, int m0, int n0, int rm,
                                              int cn, const float (&acc)[8][8], float beta,
                                              bool use_c) {
  const float alpha = p.alpha;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int row = m0 + rm + (i & 3) + (i >> 2) * 64;
    if (row >= p.M) continue;
    float *crow = C + static_cast<int64_t>(row) * p.ldc;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int col = n0 + cn + h * 64;
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
template <int BK, int STAGES, bool A_T, bool VEC_A, bool B_T, bool VEC_B, int MODE>
__global__ void __launch_bounds__(kThreads, 2) sgemm_simt_kernel(const SimtArgs p) {
  constexpr int kBStride = B_T ? kAStride : kBN;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  auto &sm = *reinterpret_cast<SimtSmem<BK, STAGES, kBStride> *>(smem_raw);

  const int tid = threadIdx.x;
  // Thread -> 8x8 outputs. Warps form a 4 (rows) x 2 (cols) grid, lanes a
  // 4 x 8 grid; rows rm..rm+3 and 64+rm..64+rm+3, cols cn..cn+3 and 64+cn..
  const int warp = tid >> 5, lane = tid & 31;
  const int rm = (warp >> 1) * 16 + (lane >> 3) * 4;
  const int cn = (warp & 1) * 32 + (lane & 7) * 4;
  const int KT = (p.K + BK - 1) / BK;
  float acc[8][8];

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
      for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
    tile_mainloop<BK, STAGES, A_T, VEC_A, B_T, VEC_B, kBStride>(p, A, B, sm, tm * kBM, tn * kBN,
                                                                0, KT, tid, rm, cn, acc);
    tile_epilogue(p, C, tm * kBM, tn * kBN, rm, cn, acc, p.beta, p.beta != 0.f);
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
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
      tile_mainloop<BK, STAGES, A_T, VEC_A, B_T, VEC_B, kBStride>(p, p.A, p.B, sm, tm * kBM,
                                                                  tn * kBN, w.kb0, w.kb1, tid, rm,
                                                                  cn, acc);
      if (w.parts == 1) {
        tile_epilogue(p, p.C, tm * kBM, tn * kBN, rm, cn, acc, p.beta, p.beta != 0.f);
        continue;
      }
      // k-split tile: part j adds after part j - 1 has stored (in order).
      uint32_t *flag = p.tail_flags + (w.tile - p.dp_tiles);
      if (w.part > 0) {
        if (tid == 0) wait_flag(flag, static_cast<uint32_t>(w.part), &abort, p.err_word);
        __syncthreads();
        tile_epilogue(p, p.C, tm * kBM, tn * kBN, rm, cn, acc, 1.f, true);
      } else {
        tile_epilogue(p, p.C, tm * kBM, tn * kBN, rm, cn, acc, p.beta, p.beta != 0.f);
      }
      __threadfence();
      __syncthreads();  // every thread's part of the tile is stored and visible
      if (tid == 0) st_release_gpu(flag, static_cast<uint32_t>(w.part + 1));
    }
  }
}

// CTAs of `kern` that can be resident at once on the device (cached).
int resident_ctas(const DeviceInfo &dev, const void *kern, size_t smem) {
  static std::mutex mu;
  static std::map<std::pair<const void *, int>, int> cache;
  std::lock_guard<std::mutex> lock(mu);
  const auto key = std::make_pair(kern, dev.device);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem) !=
      cudaSuccess)
    per_sm = 0;
  cudaGetLastError();
  const int n = per_sm * dev.sm_count;
  cache[key] = n;
  return n;
}

constexpr int kSimtMaxSplit = 4;  // parts per leftover tile (each adds one pass over its C)

template <int BK, int STAGES, bool A_T, bool VEC_A, bool B_T, bool VEC_B, int MODE = kModeBatch>
cudaError_t launch_variant(const SimtArgs &a_in, int batch, const DeviceInfo &dev,
                           cudaStream_t stream) {
  constexpr size_t smem = sizeof(SimtSmem<BK, STAGES, B_T ? kAStride : kBN>);
  auto kern = sgemm_simt_kernel<BK, STAGES, A_T, VEC_A, B_T, VEC_B, MODE>;
  cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void *>(kern),
                                       static_cast<int>(smem), dev.device);
  if (e != cudaSuccess) return e;
  SimtArgs a = a_in;
  a.err_word = dev.err_word;
  a.tail_flags = nullptr;
  const int64_t blocks = static_cast<int64_t>(a.tiles_m) * a.tiles_n;
  if constexpr (MODE == kModeSplit) {
    // Persistent grid over the co-resident CTAs, the last wave split along k.
    const int cap = resident_ctas(dev, reinterpret_cast<const void *>(kern), smem);
    if (cap <= 0) return cudaErrorLaunchOutOfResources;
    const int KT = (a.K + BK - 1) / BK;
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

#ifndef DGR_SIMT_BK
#define DGR_SIMT_BK 32
#endif
#ifndef DGR_SIMT_STAGES
#define DGR_SIMT_STAGES 2
#endif
constexpr int kSimtBK = DGR_SIMT_BK, kSimtStages = DGR_SIMT_STAGES;

template <bool A_T, bool VEC_A>
cudaError_t launch_b(const SimtArgs &a, bool b_t, bool vec_b, int batch, const DeviceInfo &dev,
                     cudaStream_t stream) {
  if (b_t)
    return launch_variant<kSimtBK, kSimtStages, A_T, VEC_A, true, false>(a, batch, dev, stream);
  return vec_b ? launch_variant<kSimtBK, kSimtStages, A_T, VEC_A, false, true>(a, batch, dev,
                                                                               stream)
               : launch_variant<kSimtBK, kSimtStages, A_T, VEC_A, false, false>(a, batch, dev,
                                                                                stream);
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

cudaError_t launch_sgemm_simt_ex(const DeviceInfo &dev, const BatchOps &ops, int M, int N, int K,
                                 float alpha, const float *A, int64_t lda, const float *B,
                                 int64_t ldb, float beta, float *C, int64_t ldc,
                                 cudaStream_t stream) {
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
  if (ops.plain()) {  // one problem, no transposes
    // Fewer tiles than two waves of resident CTAs (2 per SM): the persistent
    // k-split form keeps every SM busy; otherwise one CTA per tile.
    const int64_t tiles = static_cast<int64_t>(a.tiles_m) * a.tiles_n;
    if (tiles < 4LL * dev.sm_count)
      return vec_b ? launch_variant<kSimtBK, kSimtStages, false, false, false, true, kModeSplit>(
                         a, 1, dev, stream)
                   : launch_variant<kSimtBK, kSimtStages, false, false, false, false, kModeSplit>(
                         a, 1, dev, stream);
    return vec_b ? launch_variant<kSimtBK, kSimtStages, false, false, false, true, kModeTile>(
                       a, 1, dev, stream)
                 : launch_variant<kSimtBK, kSimtStages, false, false, false, false, kModeTile>(
                       a, 1, dev, stream);
  }
  if (!ops.a_t) return launch_b<false, false>(a, ops.b_t, vec_b, batch, dev, stream);
  return vec_a ? launch_b<true, true>(a, ops.b_t, vec_b, batch, dev, stream)
               : launch_b<true, false>(a, ops.b_t, vec_b, batch, dev, stream);
}

cudaError_t launch_sgemm_simt(const DeviceInfo &dev, int M, int N, int K, float alpha,
                              const float *A, int64_t lda, const float *B, int64_t ldb,
                              float beta, float *C, int64_t ldc, cudaStream_t stream) {
  return launch_sgemm_simt_ex(dev, BatchOps(), M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
                              stream);
}

}  // namespace dgr
