// gemm_small_m.cu -- fp32 and int8 GEMM for short, wide problems (M <= 32).
//
//     C = alpha * A * B + beta * C       A: M x K, B: K x N, C: M x N, row-major
//
// With a handful of rows the GEMM is bound by reading B (K x N) once. Each CTA
// owns 1024 columns of C and one part of the k range:
//   * warp 0 streams the k-slices of B (kc rows x 1024 columns, four TMA boxes)
//     and of A (all M rows x kc) into a 3-stage ring guarded by mbarriers;
//   * 256 threads each compute 4 columns x all M rows in registers:
//       fp32: acc[m][0..3] += A[m][k] * B[k][n..n+3] as packed fp32 FMAs,
//             each lane one IEEE round-to-nearest FMA;
//       int8: four rows of B are transposed in registers (byte permutes) so
//             that one 32-bit word holds B[k..k+3][n], and dp4a adds the
//             4-term dot product with A[m][k..k+3] into an exact int32 sum;
//   * when there are fewer column blocks than SMs, k is split in parts: every
//     part stores its partial sums into a workspace and counts itself done on
//     its column block; once all parts of the block have stored, each part
//     adds one slice of the block's partials in part order and writes
//     alpha * sum + beta * C (deterministic; exact in int32 with
//     wrap-around). The grid is at most one CTA per SM and is launched
//     cooperatively, so all parts are resident at once and this one wait at
//     the end always ends; it is bounded all the same.
// TMA needs 16-byte aligned bases and row strides (fp32: ld % 4 == 0; int8:
// ld % 16 == 0); the entry points use this kernel only then.
//
// Sources: C = alpha*A*B + beta*C, row-major ("Sgemm [128,128,8]", the kernel's
// header comment and host_gemm); signed char inputs with int accumulation (C++
// warp matrix function page, type table). The pages have no small-M kernel.
#include <cstdint>
#include <cstring>
#include <mutex>
#include <type_traits>

#include <cuda.h>
#include <cuda_runtime.h>

#include "launch.h"
#include "ptx.cuh"

namespace dgr {
namespace {

constexpr int kCols = 1024;       // columns of C per CTA
constexpr int kThreads = 32 + 256;
constexpr int kStages = 3;
constexpr int kMaxM = 32;
constexpr int kMaxSplit = 32;

#ifndef DGR_SM_BOX_BYTES
#define DGR_SM_BOX_BYTES 1024
#endif

template <bool kInt>
struct SmCfg {
  using In = typename std::conditional<kInt, int8_t, float>::type;
  using Out = typename std::conditional<kInt, int32_t, float>::type;
  static constexpr int kKC = kInt ? 64 : 16;                       // k rows per stage
  // Width of one TMA box of B in elements (a box row is kBoxBytes long).
  static constexpr int kBoxW = DGR_SM_BOX_BYTES / static_cast<int>(sizeof(In)) > 256
                                   ? 256
                                   : DGR_SM_BOX_BYTES / static_cast<int>(sizeof(In));
  static constexpr int kBoxes = kCols / kBoxW;
  static constexpr uint32_t kBBytes = kKC * kCols * sizeof(In);    // 64 KiB
  static constexpr uint32_t kABytes = kMaxM * kKC * sizeof(In);    // 2 KiB
};

template <bool kInt>
struct __align__(128) SmSmem {
  uint8_t b[kStages][SmCfg<kInt>::kBBytes];  // b[s][k][n]
  uint8_t a[kStages][SmCfg<kInt>::kABytes];  // a[s][m][k] (rows of A)
  // fp32: each consumer warp's k-major copy of the current stage's A tile
  // (row stride kMaxM + 4: rows stay 16-byte aligned, stores spread over banks)
  float at[8][16][kMaxM + 4];
  uint64_t full[kStages];
  uint64_t empty[kStages];
  int abort;
};

template <bool kInt>
struct SmArgs {
  using Out = typename SmCfg<kInt>::Out;
  int M, N, K;
  Out alpha, beta;
  Out *C;
  int64_t ldc;
  int split;
  uint32_t *counters;  // parts done, one per column block (split > 1), zero at launch
  Out *ws;             // partial sums [split][M][blocks * 1024] (split > 1)
  int64_t ws_ld;       // blocks * 1024
  uint32_t *err_word;
  int c_vec_ok;     // C 16-byte aligned and ldc % 4 == 0
};

__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, 256;" ::: "memory");
}

// (c0, c1) = (a0 * b + c0, a1 * b + c1) with one packed fp32 FMA.
__device__ __forceinline__ void ffma2_rows(float &c0, float &c1, float a0, float a1, float b) {
  asm("{\n .reg .b64 ra, rb, rc;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %4};\n"
      " mov.b64 rc, {%0, %1};\n fma.rn.f32x2 rc, ra, rb, rc;\n mov.b64 {%0, %1}, rc;\n}\n"
      : "+f"(c0), "+f"(c1)
      : "f"(a0), "f"(a1), "f"(b));
}

// (c0, c1) = (a * b0 + c0, a * b1 + c1) with one packed fp32 FMA.
__device__ __forceinline__ void ffma2(float &c0, float &c1, float a, float b0, float b1) {
  asm("{\n .reg .b64 ra, rb, rc;\n mov.b64 ra, {%2, %2};\n mov.b64 rb, {%3, %4};\n"
      " mov.b64 rc, {%0, %1};\n fma.rn.f32x2 rc, ra, rb, rc;\n mov.b64 {%0, %1}, rc;\n}\n"
      : "+f"(c0), "+f"(c1)
      : "f"(a), "f"(b0), "f"(b1));
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

// Bounded wait until *count >= target (every part of a column block has
// stored its partial sums). On giving up: sets *abort, records the timeout in
// the error word, returns 0.
__device__ __forceinline__ int wait_count(const uint32_t *count, uint32_t target,
                                          volatile int *abort, uint32_t *err_word) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 0;; ++it) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(count) : "memory");
    if (v >= target) return 1;
    __nanosleep(256);
    if ((it & 63u) == 63u) {
      if (*abort) return 0;
      if (global_timer_ns() - t0 > kWaitLimitNs || it >= kWaitMaxPolls) {
        *abort = 1;
        record_timeout(err_word, kWaitFlag);
        return 0;
      }
    }
  }
}

// Part `part` of column block `blk`: its slice of the block's (row, 4-column
// group) items, each summed over all parts' partial sums in part order (a few
// loads in flight), then alpha * sum + beta * C. Out of line, so that the
// register allocation of the k loop is not shaped by this code.
// The fields it reads are passed by value: a reference to the kernel's
// argument block would make the kernel keep a copy of it in local memory.
template <bool kInt>
struct SliceArgs {
  using Out = typename SmCfg<kInt>::Out;
  const Out *ws;
  int64_t ws_ld, ldc;
  Out *C;
  Out alpha, beta;
  int M, N, split, c_vec_ok;
};
template <bool kInt>
__device__ __noinline__ void reduce_slice(const SliceArgs<kInt> p, int blk, int part, int n0,
                                          int t) {
  using Out = typename SmCfg<kInt>::Out;
  using Vec = typename std::conditional<kInt, int4, float4>::type;
  const bool use_c = p.beta != Out(0);
  constexpr int kGroups = kCols / 4;
  const int items = p.M * kGroups;
  const int i1 = (part + 1) * items / p.split;
#pragma unroll 1
  for (int it = part * items / p.split + t; it < i1; it += 256) {
    const int m = it / kGroups, g = it - (it / kGroups) * kGroups;
    const int64_t wcol = static_cast<int64_t>(blk) * kCols + 4 * g;
    const int nn = n0 + 4 * g;
    Out sum[4] = {Out(0), Out(0), Out(0), Out(0)};
    constexpr int kBatch = 8;  // loads in flight
#pragma unroll 1
    for (int q0 = 0; q0 < p.split; q0 += kBatch) {
      Vec v[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u)
        if (q0 + u < p.split)
          v[u] = __ldcg(reinterpret_cast<const Vec *>(
              p.ws + (static_cast<int64_t>(q0 + u) * p.M + m) * p.ws_ld + wcol));
#pragma unroll
      for (int u = 0; u < kBatch; ++u)
        if (q0 + u < p.split) {
          if constexpr (kInt) {  // int32 wrap-around
            sum[0] = static_cast<int32_t>(static_cast<uint32_t>(sum[0]) + static_cast<uint32_t>(v[u].x));
            sum[1] = static_cast<int32_t>(static_cast<uint32_t>(sum[1]) + static_cast<uint32_t>(v[u].y));
            sum[2] = static_cast<int32_t>(static_cast<uint32_t>(sum[2]) + static_cast<uint32_t>(v[u].z));
            sum[3] = static_cast<int32_t>(static_cast<uint32_t>(sum[3]) + static_cast<uint32_t>(v[u].w));
          } else {
            sum[0] += v[u].x;
            sum[1] += v[u].y;
            sum[2] += v[u].z;
            sum[3] += v[u].w;
          }
        }
    }
    if (nn < p.N) {
      Out *cp = p.C + static_cast<int64_t>(m) * p.ldc + nn;
      if (p.c_vec_ok && nn + 3 < p.N) {
        Vec c = {};
        if (use_c) c = *reinterpret_cast<const Vec *>(cp);
        Vec o;
        o.x = axpby(p.alpha, sum[0], p.beta, c.x, use_c);
        o.y = axpby(p.alpha, sum[1], p.beta, c.y, use_c);
        o.z = axpby(p.alpha, sum[2], p.beta, c.z, use_c);
        o.w = axpby(p.alpha, sum[3], p.beta, c.w, use_c);
        *reinterpret_cast<Vec *>(cp) = o;
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (nn + j < p.N) cp[j] = axpby(p.alpha, sum[j], p.beta, use_c ? cp[j] : Out(0), use_c);
      }
    }
  }
}

// MP: rows of A staged per stage (M rounded up to 1, 2, 4, 8, 16 or 32); every
// per-row loop runs exactly MP times.
template <bool kInt, int MP>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_small_m_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB, const SmArgs<kInt> p) {
  using Cf = SmCfg<kInt>;
  using In = typename Cf::In;
  using Out = typename Cf::Out;
  constexpr int KC = Cf::kKC;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  SmSmem<kInt> &sm = *reinterpret_cast<SmSmem<kInt> *>(smem_raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int *abort = &sm.abort;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&sm.full[s]), 1);
      mbar_init(smem_u32(&sm.empty[s]), 8);  // one arrival per consumer warp
    }
    sm.abort = 0;
    fence_mbar_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  __syncthreads();

  const int blk = static_cast<int>(blockIdx.x) / p.split;
  const int part = static_cast<int>(blockIdx.x) % p.split;
  const int n0 = blk * kCols;
  const int KS = (p.K + KC - 1) / KC;  // k-slices
  const int ks0 = part * KS / p.split;
  const int ks1 = (part + 1) * KS / p.split;
  const uint32_t a_bytes = static_cast<uint32_t>(MP) * KC * sizeof(In);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, issued = 0, issued_parity = 0;
      for (int ks = ks0; ks < ks1; ++ks) {
        if (!mbar_wait_bounded(smem_u32(&sm.empty[stage]), phase ^ 1u, abort, p.err_word,
                               kWaitEmpty))
          break;
        const uint32_t full_bar = smem_u32(&sm.full[stage]);
        mbar_arrive_expect_tx(full_bar, Cf::kBBytes + a_bytes);
#pragma unroll 4
        for (int j = 0; j < Cf::kBoxes; ++j)
          tma_load_2d(smem_u32(sm.b[stage] + j * (Cf::kBBytes / Cf::kBoxes)), &tmB, full_bar,
                      n0 + Cf::kBoxW * j, ks * KC);
        tma_load_2d(smem_u32(sm.a[stage]), &tmA, full_bar, ks * KC, 0);
        issued |= 1u << stage;
        issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      volatile int never = 0;
      for (int s = 0; s < kStages; ++s)
        if (issued & (1u << s))
          mbar_wait_bounded(smem_u32(&sm.full[s]), (issued_parity >> s) & 1u, &never,
                            p.err_word, kWaitDrain);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ consumers
    const int t = threadIdx.x - 32;        // 0..255
    const int col = 4 * t;                 // this thread's first column in the block
    Out acc[MP][4];
#pragma unroll
    for (int m = 0; m < MP; ++m)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[m][j] = Out(0);

    uint32_t stage = 0, phase = 0;
    for (int ks = ks0; ks < ks1; ++ks) {
      int got = 1;
      if (lane == 0)
        got = mbar_wait_bounded(smem_u32(&sm.full[stage]), phase, abort, p.err_word, kWaitFull);
      got = __shfl_sync(0xffffffffu, got, 0);
      if (!got) break;
      const In *bs = reinterpret_cast<const In *>(sm.b[stage]);
      const In *as = reinterpret_cast<const In *>(sm.a[stage]);
      // B box j covers columns kBoxW*j .. of the block: KC rows of kBoxW.
      constexpr int W = Cf::kBoxW;
      const In *bcol = bs + (col / W) * (KC * W) + (col % W);
      if constexpr (!kInt && MP >= 4) {
        // A tile to k-major (at[k][m]) so that rows m, m+1 of one k are a pair
        // in one 16-byte load; then (acc[m][j], acc[m+1][j]) += (a[m], a[m+1])
        // * b[j]: only b[j] is duplicated into a register pair, once per k and
        // column for all rows (with A's rows paired the other way, every row's
        // value needed its own pair).
        // Each warp makes its own copy, so no barrier wider than the warp is
        // needed (the __syncwarp ending the previous stage separates its reads
        // from these writes).
        static_assert(KC == 16, "the k-major copy holds 16 values of k");
        float (*at)[kMaxM + 4] = sm.at[warp - 1];
        for (int e = lane; e < MP * KC; e += 32) at[e % KC][e / KC] = as[e];
        __syncwarp();
#pragma unroll 4
        for (int kq = 0; kq < KC; kq += 4) {
          float4 b4[4];
#pragma unroll
          for (int u = 0; u < 4; ++u)
            b4[u] = *reinterpret_cast<const float4 *>(bcol + (kq + u) * W);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const float b[4] = {b4[u].x, b4[u].y, b4[u].z, b4[u].w};
#pragma unroll
            for (int m = 0; m < MP; m += 4) {
              const float4 a4 = *reinterpret_cast<const float4 *>(&at[kq + u][m]);
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                ffma2_rows(acc[m][j], acc[m + 1][j], a4.x, a4.y, b[j]);
                ffma2_rows(acc[m + 2][j], acc[m + 3][j], a4.z, a4.w, b[j]);
              }
            }
          }
        }
      } else if constexpr (!kInt) {
#pragma unroll 4
        for (int kq = 0; kq < KC; kq += 4) {
          float4 b4[4];
#pragma unroll
          for (int u = 0; u < 4; ++u)
            b4[u] = *reinterpret_cast<const float4 *>(bcol + (kq + u) * W);
#pragma unroll
          for (int m = 0; m < MP; ++m) {
            const float4 a4 = *reinterpret_cast<const float4 *>(as + m * KC + kq);
            const float a[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              ffma2(acc[m][0], acc[m][1], a[u], b4[u].x, b4[u].y);
              ffma2(acc[m][2], acc[m][3], a[u], b4[u].z, b4[u].w);
            }
          }
        }
      } else {
#pragma unroll 4
        for (int kq = 0; kq < KC; kq += 4) {
          // Rows k..k+3 of this thread's 4 columns, one byte per column each.
          const uint32_t w0 = *reinterpret_cast<const uint32_t *>(bcol + (kq + 0) * W);
          const uint32_t w1 = *reinterpret_cast<const uint32_t *>(bcol + (kq + 1) * W);
          const uint32_t w2 = *reinterpret_cast<const uint32_t *>(bcol + (kq + 2) * W);
          const uint32_t w3 = *reinterpret_cast<const uint32_t *>(bcol + (kq + 3) * W);
          // 4 x 4 byte transpose: column j word = (w0.j, w1.j, w2.j, w3.j).
          const uint32_t lo01 = __byte_perm(w0, w1, 0x5140);
          const uint32_t hi01 = __byte_perm(w0, w1, 0x7362);
          const uint32_t lo23 = __byte_perm(w2, w3, 0x5140);
          const uint32_t hi23 = __byte_perm(w2, w3, 0x7362);
          const int c0 = static_cast<int>(__byte_perm(lo01, lo23, 0x5410));
          const int c1 = static_cast<int>(__byte_perm(lo01, lo23, 0x7632));
          const int c2 = static_cast<int>(__byte_perm(hi01, hi23, 0x5410));
          const int c3 = static_cast<int>(__byte_perm(hi01, hi23, 0x7632));
#pragma unroll
          for (int m = 0; m < MP; ++m) {
            const int a4 = *reinterpret_cast<const int *>(as + m * KC + kq);
            acc[m][0] = __dp4a(a4, c0, acc[m][0]);
            acc[m][1] = __dp4a(a4, c1, acc[m][1]);
            acc[m][2] = __dp4a(a4, c2, acc[m][2]);
            acc[m][3] = __dp4a(a4, c3, acc[m][3]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.empty[stage]));
      if (++stage == kStages) {
        stage = 0;
        phase ^= 1u;
      }
    }

    // Epilogue: this thread's 4 columns of every row.
    const int n = n0 + col;
    const bool vec = p.c_vec_ok && n + 3 < p.N;
    using Vec = typename std::conditional<kInt, int4, float4>::type;
    if (p.split == 1) {
      if (!*abort && ks1 > ks0 && n < p.N) {
        const bool use_c = p.beta != Out(0);
#pragma unroll
        for (int m = 0; m < MP; ++m) {
          if (m < p.M) {
            Out *cp = p.C + static_cast<int64_t>(m) * p.ldc + n;
            if (vec) {
              Vec c = {};
              if (use_c) c = *reinterpret_cast<const Vec *>(cp);
              Vec o;
              o.x = axpby(p.alpha, acc[m][0], p.beta, c.x, use_c);
              o.y = axpby(p.alpha, acc[m][1], p.beta, c.y, use_c);
              o.z = axpby(p.alpha, acc[m][2], p.beta, c.z, use_c);
              o.w = axpby(p.alpha, acc[m][3], p.beta, c.w, use_c);
              *reinterpret_cast<Vec *>(cp) = o;
            } else {
#pragma unroll
              for (int j = 0; j < 4; ++j)
                if (n + j < p.N) cp[j] = axpby(p.alpha, acc[m][j], p.beta, use_c ? cp[j] : Out(0), use_c);
            }
          }
        }
      }
    } else {
      // Store this part's partial sums, then count the part done.
      Out *wpart = p.ws + static_cast<int64_t>(part) * p.M * p.ws_ld;
      const int nl = blk * kCols + col;  // column in the workspace
#pragma unroll
      for (int m = 0; m < MP; ++m)
        if (m < p.M) {
          Vec v;
          v.x = acc[m][0];
          v.y = acc[m][1];
          v.z = acc[m][2];
          v.w = acc[m][3];
          *reinterpret_cast<Vec *>(wpart + static_cast<int64_t>(m) * p.ws_ld + nl) = v;
        }
      __threadfence();
      consumer_sync();
      if (t == 0) atomicAdd(p.counters + blk, 1u);
      // Once every part of this column block has stored, each part sums one
      // slice of the block's (row, 4-column group) items over all parts, in
      // part order. All parts are resident at once (a cooperative launch of
      // at most one CTA per SM), so the wait ends; it is bounded all the same.
      __shared__ int ready;
      if (t == 0)
        ready = wait_count(p.counters + blk, static_cast<uint32_t>(p.split), abort, p.err_word);
      consumer_sync();
      if (ready) {
        __threadfence();
        SliceArgs<kInt> sa;
        sa.ws = p.ws;
        sa.ws_ld = p.ws_ld;
        sa.ldc = p.ldc;
        sa.C = p.C;
        sa.alpha = p.alpha;
        sa.beta = p.beta;
        sa.M = p.M;
        sa.N = p.N;
        sa.split = p.split;
        sa.c_vec_ok = p.c_vec_ok;
        reduce_slice<kInt>(sa, blk, part, n0, t);
      }
    }
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

// Row-major rows x cols matrix, element size esize, row stride ld, boxes of
// box_rows x box_cols elements, no swizzle.
bool tmap_plain(CUtensorMap *tm, CUtensorMapDataType dt, int esize, const void *base, int64_t rows,
                int64_t cols, int64_t ld, uint32_t box_rows, uint32_t box_cols) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * esize};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(tm, dt, 2, const_cast<void *>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

template <bool kInt, int MP>
cudaError_t launch(const DeviceInfo &dev, int M, int N, int K, typename SmArgs<kInt>::Out alpha,
                   const void *A, int64_t lda, const void *B, int64_t ldb,
                   typename SmArgs<kInt>::Out beta, typename SmArgs<kInt>::Out *C, int64_t ldc,
                   cudaStream_t stream) {
  using Cf = SmCfg<kInt>;
  const int esize = static_cast<int>(sizeof(typename Cf::In));
  const CUtensorMapDataType dt = kInt ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                      : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  SmArgs<kInt> p;
  p.M = M;
  p.N = N;
  p.K = K;
  p.alpha = alpha;
  p.beta = beta;
  p.C = C;
  p.ldc = ldc;
  p.err_word = dev.err_word;
  p.c_vec_ok = (reinterpret_cast<uintptr_t>(C) % 16 == 0) && (ldc % 4 == 0);
  CUtensorMap tmA, tmB;
  if (!tmap_plain(&tmA, dt, esize, A, M, K, lda, static_cast<uint32_t>(MP), Cf::kKC))
    return cudaErrorInvalidValue;
  if (!tmap_plain(&tmB, dt, esize, B, K, N, ldb, Cf::kKC, Cf::kBoxW)) return cudaErrorInvalidValue;

  const int blocks = (N + kCols - 1) / kCols;
  const int KS = (K + Cf::kKC - 1) / Cf::kKC;
  int split = blocks < dev.sm_count ? dev.sm_count / blocks : 1;
  if (split > kMaxSplit) split = kMaxSplit;
  if (split > KS) split = KS;
  if (split < 1) split = 1;
  p.split = split;

  // split > 1: partial sums [split][M][blocks * 1024] and per-block counters,
  // from the library's stream-ordered pool.
  void *pool_ws = nullptr;
  p.counters = nullptr;
  p.ws = nullptr;
  p.ws_ld = static_cast<int64_t>(blocks) * kCols;
  if (split > 1) {
    cudaMemPool_t pool;
    cudaError_t e = device_pool(dev, &pool);
    if (e != cudaSuccess) return e;
    const size_t ws_bytes = static_cast<size_t>(split) * M * p.ws_ld * sizeof(typename Cf::Out);
    const size_t cnt_off = (ws_bytes + 255) / 256 * 256;
    e = cudaMallocFromPoolAsync(&pool_ws, cnt_off + static_cast<size_t>(blocks) * 4, pool,
                                stream);
    if (e != cudaSuccess) return e;
    p.ws = static_cast<typename Cf::Out *>(pool_ws);
    p.counters = reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(pool_ws) + cnt_off);
    e = cudaMemsetAsync(p.counters, 0, static_cast<size_t>(blocks) * 4, stream);
    if (e != cudaSuccess) {
      cudaFreeAsync(pool_ws, stream);
      return e;
    }
  }
  const size_t smem = sizeof(SmSmem<kInt>);
  static_assert(sizeof(SmSmem<kInt>) <= 232448, "small-M kernel shared memory");
  auto kern = gemm_small_m_kernel<kInt, MP>;
  cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void *>(kern),
                                       static_cast<int>(smem), dev.device);
  if (e == cudaSuccess) {
    // With k split, the parts of a column block wait for one another at the
    // end: a cooperative launch starts the grid only when all of its CTAs can
    // be resident together (another stream's kernels cannot leave it half
    // resident).
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks * split), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = split > 1 ? 1 : 0;
    e = cudaLaunchKernelEx(&cfg, kern, tmA, tmB, p);
    if (e == cudaSuccess) e = cudaGetLastError();
  }
  if (pool_ws) {
    cudaError_t f = cudaFreeAsync(pool_ws, stream);
    if (e == cudaSuccess) e = f;
  }
  return e;
}

}  // namespace

bool small_m_supported(int M, const void *A, int64_t lda, const void *B, int64_t ldb,
                       int esize) {
  if (M < 1 || M > kMaxM) return false;
  const int64_t vec = 16 / esize;  // elements per 16 bytes
  return (reinterpret_cast<uintptr_t>(A) % 16 == 0) && (reinterpret_cast<uintptr_t>(B) % 16 == 0) &&
         (lda % vec == 0) && (ldb % vec == 0);
}

namespace {
template <bool kInt>
cudaError_t launch_mp(const DeviceInfo &dev, int M, int N, int K, typename SmArgs<kInt>::Out alpha,
                      const void *A, int64_t lda, const void *B, int64_t ldb,
                      typename SmArgs<kInt>::Out beta, typename SmArgs<kInt>::Out *C,
                      int64_t ldc, cudaStream_t stream) {
  if (M <= 1) return launch<kInt, 1>(dev, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream);
  if (M <= 2) return launch<kInt, 2>(dev, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream);
  if (M <= 4) return launch<kInt, 4>(dev, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream);
  if (M <= 8) return launch<kInt, 8>(dev, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream);
  if (M <= 16) return launch<kInt, 16>(dev, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream);
  return launch<kInt, 32>(dev, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream);
}
}  // namespace

cudaError_t launch_small_m_f32(const DeviceInfo &dev, int M, int N, int K, float alpha,
                               const float *A, int64_t lda, const float *B, int64_t ldb,
                               float beta, float *C, int64_t ldc, cudaStream_t stream) {
  return launch_mp<false>(dev, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream);
}

cudaError_t launch_small_m_s8(const DeviceInfo &dev, int M, int N, int K, int32_t alpha,
                              const int8_t *A, int64_t lda, const int8_t *B, int64_t ldb,
                              int32_t beta, int32_t *C, int64_t ldc, cudaStream_t stream) {
  return launch_mp<true>(dev, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream);
}

}  // namespace dgr
