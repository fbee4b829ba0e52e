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
#include <cstdint>

#include <cuda_runtime.h>

#include "launch.h"
#include "ptx.cuh"

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
  int tiles_m, tiles_n;
  int c_vec_ok;  // C 16-byte aligned and ldc % 4 == 0
};

// Row stride of the transposed A tile: 132 = 128 + 4 floats. With it, the
// 4-byte copies of one warp (4 rows x 8 consecutive k) land in 32 distinct
// banks, and every 4-float group stays 16-byte aligned for the fragment loads.
constexpr int kAStride = kBM + 4;

template <int BK, int STAGES>
struct SimtSmem {
  float a[STAGES][BK][kAStride];  // A tile, transposed: a[s][k][m]
  float b[STAGES][BK][kBN];       // B tile: b[s][k][n]
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

template <int BK, bool VEC_B>
__device__ __forceinline__ void load_tile(const SimtArgs &p, float (*sa)[kAStride],
                                          float (*sb)[kBN], int m0, int n0, int k0, int tid) {
  // A: one warp instruction copies 4 rows x 8 consecutive k (lane = 8*row + k),
  // i.e. four 32-byte global segments, into the transposed tile. The BK/2
  // instructions of a thread walk (row group, k half) pairs of its warp.
  {
    static_assert(BK % 8 == 0, "A staging copies k in groups of 8");
    constexpr int kGroupsK = BK / 8;
    const int warp = tid >> 5, lane = tid & 31;
    const int r_lo = lane >> 3, k_lo = lane & 7;
#pragma unroll
    for (int i = 0; i < BK / 2; ++i) {
      const int pair = warp * (BK / 2) + i;        // 0 .. 4*BK-1
      const int m = (pair / kGroupsK) * 4 + r_lo;   // 32 groups of 4 rows
      const int k = (pair % kGroupsK) * 8 + k_lo;   // groups of 8 k
      const int gm = m0 + m, gk = k0 + k;
      const bool ok = gm < p.M && gk < p.K;
      const float *src = ok ? p.A + static_cast<int64_t>(gm) * p.lda + gk : p.A;
      cp_async_4(smem_u32(&sa[k][m]), src, ok ? 4u : 0u);
    }
  }
  // B: row-major BK x 128 tile.
  if constexpr (VEC_B) {
    constexpr int kChunks = BK * kBN / 4 / kThreads;
#pragma unroll
    for (int i = 0; i < kChunks; ++i) {
      const int c = tid + i * kThreads;
      const int row = c >> 5;
      const int col = (c & 31) * 4;
      const int gk = k0 + row, gn = n0 + col;
      const bool ok = gk < p.K && gn < p.N;
      const float *src = ok ? p.B + static_cast<int64_t>(gk) * p.ldb + gn : p.B;
      cp_async_16(smem_u32(&sb[row][col]), src, ok ? 16u : 0u);
    }
  } else {
    constexpr int kPer = BK * kBN / kThreads;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int e = tid + i * kThreads;
      const int row = e >> 7;
      const int col = e & (kBN - 1);
      const int gk = k0 + row, gn = n0 + col;
      const bool ok = gk < p.K && gn < p.N;
      const float *src = ok ? p.B + static_cast<int64_t>(gk) * p.ldb + gn : p.B;
      cp_async_4(smem_u32(&sb[row][col]), src, ok ? 4u : 0u);
    }
  }
}

template <int BK, int STAGES, bool VEC_B>
__global__ void __launch_bounds__(kThreads, 2) sgemm_simt_kernel(const SimtArgs p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  auto &sm = *reinterpret_cast<SimtSmem<BK, STAGES> *>(smem_raw);

  const int tid = threadIdx.x;
  int tm, tn;
  tile_coords(blockIdx.x, p.tiles_m, p.tiles_n, tm, tn);
  const int m0 = tm * kBM, n0 = tn * kBN;

  // Thread -> 8x8 outputs. Warps form a 4 (rows) x 2 (cols) grid, lanes a
  // 4 x 8 grid; rows rm..rm+3 and 64+rm..64+rm+3, cols cn..cn+3 and 64+cn..
  const int warp = tid >> 5, lane = tid & 31;
  const int rm = (warp >> 1) * 16 + (lane >> 3) * 4;
  const int cn = (warp & 1) * 32 + (lane & 7) * 4;

  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

  const int KT = (p.K + BK - 1) / BK;
#pragma unroll
  for (int s = 0; s < STAGES - 1; ++s) {
    if (s < KT) load_tile<BK, VEC_B>(p, sm.a[s], sm.b[s], m0, n0, s * BK, tid);
    cp_async_commit();
  }

  for (int kt = 0; kt < KT; ++kt) {
    cp_async_wait<STAGES - 2>();
    __syncthreads();  // tile kt landed for everyone; tile kt-1 fully consumed
    {
      const int nt = kt + STAGES - 1;
      if (nt < KT) {
        const int s = nt % STAGES;
        load_tile<BK, VEC_B>(p, sm.a[s], sm.b[s], m0, n0, nt * BK, tid);
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

  // Epilogue.
  const float alpha = p.alpha, beta = p.beta;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int row = m0 + rm + (i & 3) + (i >> 2) * 64;
    if (row >= p.M) continue;
    float *crow = p.C + static_cast<int64_t>(row) * p.ldc;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int col = n0 + cn + h * 64;
      const float *v = &acc[i][h * 4];
      if (p.c_vec_ok && col + 3 < p.N) {
        float4 out;
        if (beta != 0.f) {
          const float4 c = *reinterpret_cast<const float4 *>(crow + col);
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
            crow[col + j] = (beta != 0.f) ? r + beta * crow[col + j] : r;
          }
        }
      }
    }
  }
}

template <int BK, int STAGES, bool VEC_B>
cudaError_t launch_variant(const SimtArgs &a, int device, cudaStream_t stream) {
  constexpr size_t smem = sizeof(SimtSmem<BK, STAGES>);
  auto kern = sgemm_simt_kernel<BK, STAGES, VEC_B>;
  cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void *>(kern),
                                       static_cast<int>(smem), device);
  if (e != cudaSuccess) return e;
  const int64_t blocks = static_cast<int64_t>(a.tiles_m) * a.tiles_n;
  kern<<<static_cast<unsigned>(blocks), kThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_sgemm_simt(const DeviceInfo &dev, int M, int N, int K, float alpha,
                              const float *A, int64_t lda, const float *B, int64_t ldb,
                              float beta, float *C, int64_t ldc, cudaStream_t stream) {
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
  a.tiles_m = (M + kBM - 1) / kBM;
  a.tiles_n = (N + kBN - 1) / kBN;
  a.c_vec_ok = (reinterpret_cast<uintptr_t>(C) % 16 == 0) && (ldc % 4 == 0);
  if (static_cast<int64_t>(a.tiles_m) * a.tiles_n > 0x7fffffffLL) return cudaErrorInvalidValue;
  const bool vec_b = (reinterpret_cast<uintptr_t>(B) % 16 == 0) && (ldb % 4 == 0) && (N % 4 == 0);
#ifndef DGR_SIMT_BK
#define DGR_SIMT_BK 32
#endif
#ifndef DGR_SIMT_STAGES
#define DGR_SIMT_STAGES 2
#endif
  constexpr int kBK = DGR_SIMT_BK, kStages = DGR_SIMT_STAGES;
  return vec_b ? launch_variant<kBK, kStages, true>(a, dev.device, stream)
               : launch_variant<kBK, kStages, false>(a, dev.device, stream);
}

}  // namespace dgr
