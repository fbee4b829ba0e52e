// gemm_tc_skinny.cu -- tensor-core GEMM for short, wide problems (M <= 64).
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
// Cluster form (gemm_tc_skinny_cl_kernel), what every call without caller-
// provided flags takes: the CTAs that split the k range of one column block
// form a thread-block cluster and add their partial sums through distributed
// shared memory, so a call is one launch with no workspace, counters or
// atomics (details at the kernel). Measured on GB300 (bf16, N = K = 8192,
// 50-call loops): M = 1 23.8 us, M = 16 24.7 us, M = 64 26.7 us, against 29.7,
// 35.3 and 37.6 us for the per-block split and the stream-K form it replaces.
// The per-block form remains for callers that supply their own flag memory
// (whole column blocks, no split) and for int8 B as stored with an A whose rows
// are not whole 16-byte units.
//
// int8 as stored (gemm_s8 with 10..64 rows): TMA brings raw byte tiles, and
// converter warps widen each tile exactly to fp16 in shared memory before the
// MMA reads it, so the operands cross HBM once as bytes instead of being
// widened to 16-bit copies first. The cluster form reads A and B this way; the
// per-block form (kRawB) reads B this way and takes a widened A.
//
// Sources: as gemm_tc_kernel.cuh (C = alpha*A*B + beta*C, "Sgemm [128,128,8]"; half /
// bfloat16 x half / bfloat16 -> float and signed char -> int, C++ warp matrix
// function page, type table). The pages have no skinny-shape kernel; this is a
// layout choice for the same computation.
#include <cstdint>
#include <cstring>
#include <mutex>
#include <tuple>
#include <type_traits>
#include <map>

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
  static constexpr int kNumStages = kStages;
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

// int8 B read as stored (the raw-B form of the per-block kernel): TMA brings a
// 64(k) x 128(n) byte tile of B into `raw` (with the A tile into `a`); four
// converter warps write it to `b` as fp16 in the layout TMA gives a 16-bit B
// (two 64-column boxes, 128-byte swizzle) and arrive on `conv`; the MMA waits
// on `conv`. B then crosses HBM once, as bytes, instead of being widened to a
// 16-bit copy first.
constexpr int kI8Stages = 6;
constexpr int kConvWarps = 4;
constexpr int kI8Threads = kThreads + 32 * kConvWarps;
constexpr uint32_t kRawBytes = kBK * kBN;  // 8 KiB: 64 rows of 128 bytes
struct __align__(1024) SkSmemI8 {
  static constexpr int kNumStages = kI8Stages;
  uint8_t b[kI8Stages][kBBytes];
  uint8_t a[kI8Stages][kABytes];
  uint8_t raw[kI8Stages][kRawBytes];
  uint64_t full[kI8Stages];   // TMA: raw B and A landed
  uint64_t conv[kI8Stages];   // converter warps: b written
  uint64_t empty[kI8Stages];  // MMA: stage consumed
  uint64_t tmem_full[2];
  uint64_t tmem_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

// One converter thread's share of a stage (ct in [0, 128)): four 16-byte
// pieces of the raw tile (row k = piece / 8, bytes 16 (piece % 8) ...), each
// widened exactly to 16 fp16 values and stored as two 16-byte chunks of the
// swizzled 16-bit tile: column n = 16 (piece % 8) + t sits in box n / 64, row
// k, chunk (n % 64) / 8, placed at chunk position chunk ^ (k % 8).
// Exact widening of a signed byte x: (x + 128) as the low byte under the fp16
// pattern 0x64 is 1024 + x + 128; subtracting 1152 leaves x (every value
// involved is an integer below 2^11, so fp16 holds it exactly).
__device__ __forceinline__ void widen_s8x16(const uint32_t (&w)[4], uint32_t (&h)[8]) {
  const __half2 bias = __half2half2(__ushort_as_half(0x6480));  // 1152
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint32_t t = w[q] ^ 0x80808080u;
    const uint32_t lo = __byte_perm(t, 0x64646464u, 0x4140);
    const uint32_t hi = __byte_perm(t, 0x64646464u, 0x4342);
    const __half2 l = __hsub2(*reinterpret_cast<const __half2 *>(&lo), bias);
    const __half2 u = __hsub2(*reinterpret_cast<const __half2 *>(&hi), bias);
    h[2 * q] = *reinterpret_cast<const uint32_t *>(&l);
    h[2 * q + 1] = *reinterpret_cast<const uint32_t *>(&u);
  }
}

__device__ __forceinline__ void convert_stage(uint32_t raw, uint32_t b, int ct) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int piece = i * 128 + ct;
    const int k = piece >> 3, c = piece & 7;
    uint32_t w[4];
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];\n"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                 : "r"(raw + static_cast<uint32_t>(k * 128 + c * 16)));
    uint32_t h[8];
    widen_s8x16(w, h);
    const int box = c >> 2;            // 64 columns per box
    const int j0 = (c & 3) * 2;        // first 16-byte chunk of this piece in its row
    const uint32_t row = b + static_cast<uint32_t>(box) * kBBox + static_cast<uint32_t>(k) * 128;
    st_shared_v4(row + static_cast<uint32_t>(((j0) ^ (k & 7)) << 4), h[0], h[1], h[2], h[3]);
    st_shared_v4(row + static_cast<uint32_t>(((j0 + 1) ^ (k & 7)) << 4), h[4], h[5], h[6], h[7]);
  }
}

template <bool kInt>
struct SkArgs {
  using Out = typename std::conditional<kInt, int32_t, float>::type;
  int M, N, K;
  int mp;  // M rounded up to a multiple of 16 (the MMA's N)
  Out alpha, beta;
  Out *C;
  int64_t ldc;
  // Per-block split (gemm_tc_skinny_kernel): every CTA one part of one block.
  int split;           // parts of k per column block
  uint32_t *counters;  // per-block form: parts done, one per column block (split > 1),
                       // zero at launch
  Out *ws;             // per-block form: partial sums [split][M][ws_ld] (split > 1)
  int64_t ws_ld;       // column blocks * 128
  int nunits;          // k-units (k-blocks, or 1024-k chunks in the int mode)
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

__device__ __forceinline__ float add_parts(float a, float b) { return a + b; }
__device__ __forceinline__ int32_t add_parts(int32_t a, int32_t b) {
  return static_cast<int32_t>(static_cast<uint32_t>(a) + static_cast<uint32_t>(b));
}

// C[m][n] = alpha * w[j] + beta * C[m][n] for the rows m = g + j < M of column
// n (a group of 16 rows). Every read of C is issued before the first store: as
// far as the compiler knows a store may alias a later row's read, and
// interleaving them would cost one load latency per row.
template <bool kInt>
__device__ __forceinline__ void write_rows16(const SkArgs<kInt> &p, int n, int g,
                                             typename SkArgs<kInt>::Out (&w)[16]) {
  using Out = typename SkArgs<kInt>::Out;
  const bool use_c = p.beta != Out(0);
#pragma unroll
  for (int j = 0; j < 16; ++j)
    if (g + j < p.M)
      w[j] = axpby(p.alpha, w[j], p.beta,
                   use_c ? p.C[static_cast<int64_t>(g + j) * p.ldc + n] : Out(0), use_c);
#pragma unroll
  for (int j = 0; j < 16; ++j)
    if (g + j < p.M) p.C[static_cast<int64_t>(g + j) * p.ldc + n] = w[j];
}

// kRawB (exact-int mode only): B is int8 as stored, converted to fp16 in
// shared memory by kConvWarps extra warps (SkSmemI8).
template <bool kInt, bool kRawB = false>
__global__ void __launch_bounds__(kRawB ? kI8Threads : kThreads, 1)
    gemm_tc_skinny_kernel(const __grid_constant__ CUtensorMap tmA,
                          const __grid_constant__ CUtensorMap tmB, const SkArgs<kInt> p) {
  static_assert(kInt || !kRawB, "int8 B as stored needs the exact-int mode");
  using Out = typename SkArgs<kInt>::Out;
  using Smem = typename std::conditional<kRawB, SkSmemI8, SkSmem>::type;
  constexpr int kS = Smem::kNumStages;
  extern __shared__ uint8_t smem_raw[];
  Smem &sm = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                       ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int *abort = &sm.abort;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kS; ++s) {
      mbar_init(smem_u32(&sm.full[s]), 1);
      mbar_init(smem_u32(&sm.empty[s]), 1);
      if constexpr (kRawB) mbar_init(smem_u32(&sm.conv[s]), 32 * kConvWarps);
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
    if constexpr (kRawB) {
      // Raw B tiles (converted in shared memory) and their A tiles.
      if (lane == 0) {
        uint32_t stage = 0, phase = 0, issued = 0, issued_parity = 0;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&sm.empty[stage]), phase ^ 1u, abort, p.err_word,
                                 kWaitEmpty))
            break;
          const uint32_t full_bar = smem_u32(&sm.full[stage]);
          mbar_arrive_expect_tx(full_bar, kRawBytes + a_bytes);
          tma_load_2d(smem_u32(sm.raw[stage]), &tmB, full_bar, n0, kb * kBK);
          tma_load_2d(smem_u32(sm.a[stage]), &tmA, full_bar, kb * kBK, 0);
          issued |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == kS) {
            stage = 0;
            phase ^= 1u;
          }
        }
        for (int r = 0; r < kS; ++r)
          if (issued & (1u << r))
            drain_wait(smem_u32(&sm.full[r]), (issued_parity >> r) & 1u, p.err_word);
      }
    } else if (lane == 0) {
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
        if (++stage == kS) {
          stage = 0;
          phase ^= 1u;
        }
      }
      for (int s = 0; s < kS; ++s)
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
          uint32_t ready;
          if constexpr (kRawB)
            ready = smem_u32(&sm.conv[stage]);  // converted by the converter warps
          else
            ready = smem_u32(&sm.full[stage]);
          if (!mbar_wait_bounded(ready, phase, abort, p.err_word, kWaitFull)) {
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
          if (++stage == kS) {
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
  } else if (!kRawB || warp < 2 + kEpiWarps) {
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
    if (p.split == 1) {
      if (n < p.N && !*abort && kb1 > kb0) {
#pragma unroll
        for (int g = 0; g < kMaxM; g += 16) {
          if (g < p.M) {
            Out w[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) w[j] = value(g + j);
            write_rows16<kInt>(p, n, g, w);
          }
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
          // Parts in order (each element's sum in one fixed order); within a
          // part 16 rows at once, so their loads overlap.
#pragma unroll
          for (int g = 0; g < kMaxM; g += 16) {
            if (g < p.M) {
              Out sum[16];
#pragma unroll
              for (int j = 0; j < 16; ++j) sum[j] = Out(0);
#pragma unroll 1
              for (int q = 0; q < p.split; ++q) {
                const Out *src = p.ws + (static_cast<int64_t>(q) * p.M + g) * p.ws_ld + n;
#pragma unroll
                for (int j = 0; j < 16; ++j)
                  if (g + j < p.M)
                    sum[j] = add_parts(sum[j], __ldcg(src + static_cast<int64_t>(j) * p.ws_ld));
              }
              write_rows16<kInt>(p, n, g, sum);
            }
          }
        }
      }
    }
  }

  if constexpr (kRawB) {
    if (warp >= 2 + kEpiWarps) {
      // --------------------------------------------------------- converter
      // Each stage: wait for the raw tile, write its fp16 form, make the
      // writes visible to the tensor core (async proxy), arrive.
      const int ct = static_cast<int>(threadIdx.x) - 32 * (2 + kEpiWarps);
      uint32_t stage = 0, phase = 0;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait_bounded(smem_u32(&sm.full[stage]), phase, abort, p.err_word, kWaitFull))
          break;
        convert_stage(smem_u32(sm.raw[stage]), smem_u32(sm.b[stage]), ct);
        fence_proxy_async_shared();
        mbar_arrive(smem_u32(&sm.conv[stage]));
        if (++stage == kS) {
          stage = 0;
          phase ^= 1u;
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

// ---------------------------------------------------------------- cluster form
//
// Cluster form (gemm_tc_skinny_cl_kernel): the k range of a column block is cut
// into `cl` equal parts (cl = 1, 2, 4 or 8; in the exact-int mode on 1024-k
// chunk boundaries), one per CTA of a thread-block cluster. Each CTA runs the
// pipeline above over its part. Then every CTA puts its 128 x M partial sums in
// its own shared memory, the cluster meets at a barrier, and CTA r adds the cl
// partials of columns [r * 128 / cl, (r + 1) * 128 / cl) in CTA order, reading
// the other CTAs' shared memory directly (distributed shared memory), and
// writes alpha * sum + beta * C. A second barrier keeps every CTA's partials
// in place until the others have read them. There is no workspace, counter or
// atomic in global memory and no second launch: one kernel per call, with a
// result that does not depend on timing (exact in the int mode).
//
// Two CTAs share an SM (shared memory, registers and TMEM are sized for it).
// Measured on GB300, a CTA that streams from DRAM with TMA is capped at about
// 200 box rows per microsecond whatever its ring depth (4 to 24 stages give the
// same rate), while two co-resident CTAs double the SM's rate: the stream, not
// the ring, sets the pace, so the rings here are short and the CTAs many.
//
// kRaw (exact-int mode, int8 A and B as stored): TMA brings byte tiles of A and
// B into a ring of raw stages, and converter warps write their fp16 forms, in
// the layouts TMA gives 16-bit operands, into a ring of 16-bit stages that the
// MMA reads. The converters form kClConvGroups groups of kClGroupWarps warps;
// group g converts k-blocks g, g + kClConvGroups, ..., so one group's fixed
// per-stage costs (waits, the proxy fence, arrivals) overlap another group's
// work. A raw stage is free again once converted, a 16-bit stage once the MMA
// has read it. Neither operand is widened in global memory.
//
// The int8 form is built for a bound kMP on the rows (16, 32 or 64): its A
// tiles and accumulators are sized for kMP rows, so that more stages fit. Both
// rings matter: a raw stage is held from its TMA issue through the
// conversion's loads, a 16-bit stage from its conversion until the MMAs that
// read it complete (measured: with 2 of them the MMA round trip, not the
// stream, set the pace at 0.45 us per k-block; without MMAs 0.22 us).
static_assert(kBK / 16 == 4, "four MMAs of k = 16 per stage");
constexpr int kClMaxCluster = 8;
constexpr int kClCtasPerSm = 2;
constexpr int kClStages = 4;                  // 16-bit form
template <int kMP>
struct ClRaw {
  static constexpr int kStages = kMP <= 16 ? 4 : 3;  // raw (byte) stages
  static constexpr int kWide = kMP <= 32 ? 4 : 3;    // 16-bit stages
  static constexpr uint32_t kABytes = kMP * kBK;          // raw A tile: kMP rows of 64 bytes
  static constexpr uint32_t kWideABytes = kMP * kBK * 2;  // fp16 A tile
};
constexpr int kClConvGroups = 2;
constexpr int kClGroupWarps = 2;
constexpr int kClConvWarps = kClConvGroups * kClGroupWarps;
constexpr int kClRawThreads = 64 + 32 * kEpiWarps + 32 * kClConvWarps;

template <bool kRaw, int kMP>
struct __align__(1024) ClSmem {
  static constexpr int kNumStages = kRaw ? ClRaw<kMP>::kWide : kClStages;  // 16-bit stages
  static constexpr int kNumRaw = kRaw ? ClRaw<kMP>::kStages : 1;      // byte stages
  uint8_t b[kNumStages][kBBytes];  // 16-bit B tile: the MMA's A operand
  uint8_t a[kNumStages][kRaw ? ClRaw<kMP>::kWideABytes : kABytes];  // 16-bit A tile: B operand
  uint8_t rawb[kNumRaw][kRaw ? kRawBytes : 128];
  uint8_t rawa[kNumRaw][kRaw ? ClRaw<kMP>::kABytes : 128];
  uint64_t full[kRaw ? kNumRaw : kNumStages];  // TMA: the stage's tiles landed
  uint64_t raw_free[kNumRaw];                   // kRaw: the converters have read the bytes
  uint64_t conv[kNumStages];                    // kRaw: the converters wrote b and a
  uint64_t empty[kNumStages];                   // MMA: the 16-bit stage consumed
  uint64_t tmem_full[2];
  uint64_t tmem_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};
// The partial sums of a CTA (M x 128 values of 4 bytes, row m at m * 512 bytes)
// reuse the first two B stages once the pipeline is done.
static_assert(2 * kBBytes >= kMaxM * kBN * 4, "partial sums fit in two B stages");

// One raw stage into the 16-bit tiles TMA would give, by converter thread ct of
// a group (kClGroupThreads threads):
//   * B: 64 rows of k x 128 bytes of n, 128-byte swizzled (16-byte chunk c of
//     row k at c ^ (k % 8)). A piece is one chunk: 16 values of n = 16 c ...; it
//     goes to box c / 4 of the 16-bit tile, row k, chunks 2 (c % 4) and the next,
//     each at chunk ^ (k % 8). Eight consecutive pieces cover chunks 0..3 of an
//     even row k and 4..7 of row k + 1, or the other halves: in every group of
//     eight threads the loads and each of the two stores touch eight different
//     16-byte bank groups.
//   * A: mp rows x 64 bytes of k, unswizzled; piece q = row q / 4, bytes 16 (q %
//     4) ...; it goes to row r at r * 128 bytes, chunks 2 (q % 4) and the next
//     at chunk ^ (r % 8).
// All the thread's loads are issued before the first conversion, so their
// latencies overlap.
constexpr int kClGroupThreads = 32 * kClGroupWarps;
// pieces per thread and round (a stage takes kClRounds rounds of loads, then stores)
constexpr int kClRounds = 2;
constexpr int kClBPieces = kRawBytes / 16 / kClGroupThreads / kClRounds;    // 4
// A pieces per thread and round for kMP rows (kMP * 4 pieces of 16 bytes)
template <int kMP>
constexpr int cl_a_pieces() {
  return (kMP * 4 + kClGroupThreads * kClRounds - 1) / (kClGroupThreads * kClRounds);
}
__device__ __forceinline__ void cl_b_piece(int q, int &k, int &c) {
  const int oct = q >> 3, i = q & 7, v = oct & 1;
  k = 2 * (oct >> 1) + (i >> 2);
  c = (i & 3) + 4 * ((i >> 2) ^ v);
}
// Piece numbers of round `rd`: B pieces (rd * kClBPieces + i) * kClGroupThreads +
// ct, A pieces (rd * kClAPieces + i) * kClGroupThreads + ct.
template <int kAP>
__device__ __forceinline__ void cl_load_raw(uint32_t rawb, uint32_t rawa, int mp, int ct, int rd,
                                            uint32_t (&wb)[kClBPieces][4],
                                            uint32_t (&wa)[kAP][4]) {
#pragma unroll
  for (int i = 0; i < kClBPieces; ++i) {
    int k, c;
    cl_b_piece((rd * kClBPieces + i) * kClGroupThreads + ct, k, c);
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];\n"
                 : "=r"(wb[i][0]), "=r"(wb[i][1]), "=r"(wb[i][2]), "=r"(wb[i][3])
                 : "r"(rawb + static_cast<uint32_t>(k * 128 + ((c ^ (k & 7)) << 4))));
  }
#pragma unroll
  for (int i = 0; i < kAP; ++i) {
    const int q = (rd * kAP + i) * kClGroupThreads + ct;
    wa[i][0] = wa[i][1] = wa[i][2] = wa[i][3] = 0;
    if (q < mp * 4)
      asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];\n"
                   : "=r"(wa[i][0]), "=r"(wa[i][1]), "=r"(wa[i][2]), "=r"(wa[i][3])
                   : "r"(rawa + static_cast<uint32_t>(q * 16)));
  }
}
template <int kAP>
__device__ __forceinline__ void cl_store_wide(uint32_t b, uint32_t a, int mp, int ct, int rd,
                                              const uint32_t (&wb)[kClBPieces][4],
                                              const uint32_t (&wa)[kAP][4]) {
#pragma unroll
  for (int i = 0; i < kClBPieces; ++i) {
    int k, c;
    cl_b_piece((rd * kClBPieces + i) * kClGroupThreads + ct, k, c);
    uint32_t h[8];
    widen_s8x16(wb[i], h);
    const uint32_t row = b + static_cast<uint32_t>(c >> 2) * kBBox + static_cast<uint32_t>(k) * 128;
    const int j0 = (c & 3) * 2;
    st_shared_v4(row + static_cast<uint32_t>((j0 ^ (k & 7)) << 4), h[0], h[1], h[2], h[3]);
    st_shared_v4(row + static_cast<uint32_t>(((j0 + 1) ^ (k & 7)) << 4), h[4], h[5], h[6], h[7]);
  }
#pragma unroll
  for (int i = 0; i < kAP; ++i) {
    const int q = (rd * kAP + i) * kClGroupThreads + ct;
    if (q < mp * 4) {
      const int r = q >> 2, c = q & 3;
      uint32_t h[8];
      widen_s8x16(wa[i], h);
      const uint32_t row = a + static_cast<uint32_t>(r) * 128u;
      st_shared_v4(row + static_cast<uint32_t>(((2 * c) ^ (r & 7)) << 4), h[0], h[1], h[2],
                   h[3]);
      st_shared_v4(row + static_cast<uint32_t>(((2 * c + 1) ^ (r & 7)) << 4), h[4], h[5], h[6],
                   h[7]);
    }
  }
}
static_assert(kClRounds * kClBPieces * kClGroupThreads * 16 == kRawBytes,
              "B pieces cover the raw tile");
static_assert(kClRounds * cl_a_pieces<64>() * kClGroupThreads >= 64 * 4 &&
                  kClRounds * cl_a_pieces<16>() * kClGroupThreads >= 16 * 4,
              "A pieces cover the raw tile");

__device__ __forceinline__ void ld_dsmem_v4(uint32_t cluster_addr, uint32_t (&v)[4]) {
  asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];\n"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3])
               : "r"(cluster_addr)
               : "memory");
}

__device__ __forceinline__ float out_from_bits(uint32_t b, float) { return __uint_as_float(b); }
__device__ __forceinline__ int32_t out_from_bits(uint32_t b, int32_t) {
  return static_cast<int32_t>(b);
}
__device__ __forceinline__ uint32_t out_to_bits(float v) { return __float_as_uint(v); }
__device__ __forceinline__ uint32_t out_to_bits(int32_t v) { return static_cast<uint32_t>(v); }

template <bool kInt, bool kRaw, int kMP = kMaxM>
__global__ void __launch_bounds__(kRaw ? kClRawThreads : kThreads, kClCtasPerSm)
    gemm_tc_skinny_cl_kernel(const __grid_constant__ CUtensorMap tmA,
                             const __grid_constant__ CUtensorMap tmB, const SkArgs<kInt> p) {
  static_assert(kInt || !kRaw, "int8 operands as stored need the exact-int mode");
  using Out = typename SkArgs<kInt>::Out;
  using Smem = ClSmem<kRaw, kMP>;
  constexpr int kAccM = kMP;  // rows held per epilogue thread
  constexpr int kS = Smem::kNumStages;
  extern __shared__ uint8_t smem_raw[];
  Smem &sm = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                       ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int *abort = &sm.abort;
  const int cl = p.split;  // CTAs per cluster = parts of k
  const int rank = cl > 1 ? static_cast<int>(cluster_ctarank()) : 0;

  constexpr int kR = Smem::kNumRaw;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kS; ++s) {
      mbar_init(smem_u32(&sm.empty[s]), 1);
      if constexpr (kRaw) {
        mbar_init(smem_u32(&sm.conv[s]), kClGroupWarps);
      } else {
        mbar_init(smem_u32(&sm.full[s]), 1);
      }
    }
    if constexpr (kRaw) {
      for (int s = 0; s < kR; ++s) {
        mbar_init(smem_u32(&sm.full[s]), 1);
        mbar_init(smem_u32(&sm.raw_free[s]), kClGroupWarps);
      }
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
  // Launched as a programmatic dependent of the previous kernel on the stream:
  // the set-up above overlaps that kernel's tail; nothing in global memory is
  // touched before it has completed and its writes are visible.
  grid_dependency_wait();
  grid_launch_dependents();

  // This CTA's part: column block `blk`, k-blocks [kb0, kb1).
  const int blk = static_cast<int>(blockIdx.x) / cl;
  const int n0 = blk * kBN;
  const int KB = (p.K + kBK - 1) / kBK;
  const int kb_unit = kInt ? kChunkKB : 1;
  const int nunits = (KB + kb_unit - 1) / kb_unit;
  const int kb0 = min(KB, (rank * nunits / cl) * kb_unit);
  const int kb1 = min(KB, ((rank + 1) * nunits / cl) * kb_unit);
  const int chunk_kb = kInt ? kChunkKB : KB;
  // bytes per stage of the A tile: mp rows of 64 values
  const uint32_t a_bytes = static_cast<uint32_t>(p.mp) * kBK * (kRaw ? 1 : 2);
  bool have_sums = false;  // epilogue threads: this CTA's partial sums are complete

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      // kRaw: the ring of byte stages (freed by the converters); otherwise the
      // ring of 16-bit stages (freed by the MMA).
      constexpr int kRing = kRaw ? kR : kS;
      uint32_t stage = 0, phase = 0, issued = 0, issued_parity = 0;
      for (int kb = kb0; kb < kb1; ++kb) {
        const uint32_t free_bar =
            kRaw ? smem_u32(&sm.raw_free[stage]) : smem_u32(&sm.empty[stage]);
        if (!mbar_wait_bounded(free_bar, phase ^ 1u, abort, p.err_word, kWaitEmpty)) break;
        const uint32_t full_bar = smem_u32(&sm.full[stage]);
        if constexpr (kRaw) {
          mbar_arrive_expect_tx(full_bar, kRawBytes + a_bytes);
          tma_load_2d(smem_u32(sm.rawb[stage]), &tmB, full_bar, n0, kb * kBK);
          tma_load_2d(smem_u32(sm.rawa[stage]), &tmA, full_bar, kb * kBK, 0);
        } else {
          mbar_arrive_expect_tx(full_bar, kBBytes + a_bytes);
          tma_load_2d(smem_u32(sm.b[stage]), &tmB, full_bar, n0, kb * kBK);
          tma_load_2d(smem_u32(sm.b[stage] + kBBox), &tmB, full_bar, n0 + 64, kb * kBK);
          tma_load_2d(smem_u32(sm.a[stage]), &tmA, full_bar, kb * kBK, 0);
        }
        issued |= 1u << stage;
        issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == kRing) {
          stage = 0;
          phase ^= 1u;
        }
      }
      for (int s = 0; s < kRing; ++s)
        if (issued & (1u << s))
          drain_wait(smem_u32(&sm.full[s]), (issued_parity >> s) & 1u, p.err_word);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, chunk = 0;
      bool ok = true, any = false;
      // Descriptors of stage 0 (as in the per-block form); a stage or a k-step
      // of 16 only moves the start address, the descriptor's low 14 bits
      // (address / 16), so each MMA's descriptors are one add away. A single
      // thread's MMA issue rate is what paces the small-N MMAs here.
      const uint64_t adesc0 = smem_desc(smem_u32(sm.b[0]), kBBox, 1024, 2u);
      const uint64_t bdesc0 = smem_desc(smem_u32(sm.a[0]), 16, 1024, 2u);
      constexpr uint32_t kAStep = sizeof(sm.b[0]) >> 4, kBStep = sizeof(sm.a[0]) >> 4;
      uint32_t a_off = 0, b_off = 0;  // stage offsets in descriptor units
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
          const uint32_t ready = kRaw ? smem_u32(&sm.conv[stage]) : smem_u32(&sm.full[stage]);
          if (!mbar_wait_bounded(ready, phase, abort, p.err_word, kWaitFull)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint64_t ad = adesc0 + a_off, bd = bdesc0 + b_off;
          const uint32_t first = kb == c0 ? 0u : 1u;
          // k-step 16: 16 rows of 128 bytes further in the B tile (N-major),
          // 32 bytes further along the A tile's rows (K-major)
          tc_mma_f16(d_tmem, ad, bd, p.idesc, first);
          tc_mma_f16(d_tmem, ad + 128, bd + 2, p.idesc, 1u);
          tc_mma_f16(d_tmem, ad + 256, bd + 4, p.idesc, 1u);
          tc_mma_f16(d_tmem, ad + 384, bd + 6, p.idesc, 1u);
          any = true;
          tc_commit(smem_u32(&sm.empty[stage]));
          a_off += kAStep;
          b_off += kBStep;
          if (++stage == kS) {
            stage = 0;
            phase ^= 1u;
            a_off = b_off = 0;
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
  } else if (warp < 2 + kEpiWarps) {
    // ------------------------------------------------------------ epilogue
    // Lanes are columns of C: lane -> column n0 + 32 * quarter + lane.
    const int quarter = warp & 3;
    const int col = quarter * 32 + lane;
    const int n = n0 + col;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    uint32_t acc[kInt ? kAccM : 1];
    if constexpr (kInt) {
#pragma unroll
      for (int j = 0; j < kAccM; ++j) acc[j] = 0;
    }
    float facc[kInt ? 1 : kAccM];
    if constexpr (!kInt) {
#pragma unroll
      for (int j = 0; j < kAccM; ++j) facc[j] = 0.f;
    }
    bool done = true;
    uint32_t chunk = 0;
    for (int c0 = kb0; c0 < kb1; c0 += chunk_kb) {
      const uint32_t buf = chunk & 1u, use = (chunk >> 1) & 1u;
      ++chunk;
      int got = 0;
      if (lane == 0)
        got = mbar_wait_bounded(smem_u32(&sm.tmem_full[buf]), use, abort, p.err_word,
                                kWaitTmemFull);
      got = __shfl_sync(0xffffffffu, got, 0);
      if (!got) {
        done = false;
        break;
      }
      tc_fence_after_sync();
      const uint32_t taddr = tmem_base + lane_base + buf * 64;
#pragma unroll
      for (int c = 0; c < kAccM; c += 16) {
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
    have_sums = done && !*abort;
    if (cl == 1) {
      if (n < p.N && have_sums) {
#pragma unroll
        for (int g = 0; g < kAccM; g += 16) {
          if (g < p.M) {
            Out w[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) w[j] = value(g + j);
            write_rows16<kInt>(p, n, g, w);
          }
        }
      }
    } else if (have_sums) {
      // Every MMA has completed (the last accumulator was committed after
      // them) and every TMA copy was consumed by one, so the B stages are free.
      uint32_t *red = reinterpret_cast<uint32_t *>(sm.b[0]);
#pragma unroll
      for (int m = 0; m < kAccM; ++m)
        if (m < p.M) red[m * kBN + col] = out_to_bits(value(m));
    }
  } else {
    if constexpr (kRaw) {
      // --------------------------------------------------------- converter
      // Group g, per k-block kb = kb0 + g, kb0 + g + kClConvGroups, ...: wait
      // for its bytes (raw stage r) and for its 16-bit stage w to be free; load
      // this thread's pieces, release r, write w's fp16 tiles, make them
      // visible to the tensor core (async proxy), arrive on conv[w].
      const int cw = warp - (2 + kEpiWarps);
      const int grp = cw / kClGroupWarps;
      const int ct = (cw % kClGroupWarps) * 32 + lane;
      for (int kb = kb0 + grp; kb < kb1; kb += kClConvGroups) {
        const int i = kb - kb0;
        const int r = i % kR, w = i % kS;
        const uint32_t rphase = static_cast<uint32_t>(i / kR) & 1u;
        const uint32_t wphase = static_cast<uint32_t>(i / kS) & 1u;
        int ok = 1;
        // A ring whose length is not a multiple of the group count (3 raw
        // stages for 17 to 64 rows) alternates each stage between the groups:
        // the previous use of stage r, i - kR, belongs to the other group.
        // Until that use is released, full[r] may still be in its phase, of
        // the other parity, and a parity wait for use i would return at once
        // (TMA copies can complete out of order, so this group can get ahead).
        // Waiting for that release first makes the wait below unambiguous.
        if constexpr (kR % kClConvGroups != 0) {
          if (i >= kR &&
              !mbar_wait_bounded(smem_u32(&sm.raw_free[r]),
                                 static_cast<uint32_t>((i - kR) / kR) & 1u, abort, p.err_word,
                                 kWaitEmpty))
            ok = 0;
        }
        if (!ok ||
            !mbar_wait_bounded(smem_u32(&sm.full[r]), rphase, abort, p.err_word, kWaitFull) ||
            !mbar_wait_bounded(smem_u32(&sm.empty[w]), wphase ^ 1u, abort, p.err_word,
                               kWaitEmpty))
          ok = 0;
        if (!__all_sync(0xffffffffu, ok)) break;
        constexpr int kAP = cl_a_pieces<kMP>();
        uint32_t wb[kClBPieces][4], wa[kAP][4];
#pragma unroll
        for (int rd = 0; rd < kClRounds; ++rd) {
          cl_load_raw(smem_u32(sm.rawb[r]), smem_u32(sm.rawa[r]), p.mp, ct, rd, wb, wa);
          if (rd == kClRounds - 1) {  // every byte of the raw stage is in registers
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&sm.raw_free[r]));
          }
          cl_store_wide(smem_u32(sm.b[w]), smem_u32(sm.a[w]), p.mp, ct, rd, wb, wa);
        }
        fence_proxy_async_shared();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sm.conv[w]));
      }
    }
  }

  __syncwarp();
  if (cl > 1) {
    // ---------------------------------------------------- cluster reduction
    cluster_sync();  // every CTA's partial sums are in its shared memory
    if (warp >= 2 && warp < 2 + kEpiWarps) {
      // All CTAs must have their sums; a CTA whose waits gave up has recorded
      // the error and flags the cluster through its own abort word.
      int bad = 0;
      const uint32_t abort_local = smem_u32(&sm.abort);
      for (int q = 0; q < cl; ++q) {
        uint32_t v;
        asm volatile("ld.shared::cluster.u32 %0, [%1];\n"
                     : "=r"(v)
                     : "r"(mapa_shared(abort_local, static_cast<uint32_t>(q)))
                     : "memory");
        bad |= static_cast<int>(v);
      }
      const int W = kBN / cl;              // columns this CTA finishes
      const int wq = W / 4;                // 4-column groups per row
      const int t = static_cast<int>(threadIdx.x) - 64;
      const uint32_t red_local = smem_u32(sm.b[0]);
      const bool use_c = p.beta != Out(0);
      for (int idx = t; !bad && idx < p.M * wq; idx += 32 * kEpiWarps) {
        const int m = idx / wq;
        const int c = rank * W + (idx - m * wq) * 4;
        const uint32_t off = static_cast<uint32_t>((m * kBN + c) * 4);
        Out s[4] = {Out(0), Out(0), Out(0), Out(0)};
        for (int q = 0; q < cl; ++q) {  // CTA order: one fixed order per element
          uint32_t v[4];
          ld_dsmem_v4(mapa_shared(red_local + off, static_cast<uint32_t>(q)), v);
#pragma unroll
          for (int j = 0; j < 4; ++j) s[j] = add_parts(s[j], out_from_bits(v[j], Out(0)));
        }
        Out *crow = p.C + static_cast<int64_t>(m) * p.ldc + n0 + c;
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (n0 + c + j < p.N)
            crow[j] = axpby(p.alpha, s[j], p.beta, use_c ? crow[j] : Out(0), use_c);
      }
    }
    cluster_sync();  // no CTA leaves while another may still read its sums
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, kTmemCols);
  }
  (void)have_sums;
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

// Whether clusters of cl CTAs of this kernel can be resident on the device
// (queried once per kernel, device and cluster size).
bool clusters_fit(const DeviceInfo &dev, const void *kern, size_t smem, int threads, int cl) {
  static std::mutex mu;
  static std::map<std::tuple<const void *, int, int>, bool> cache;
  std::lock_guard<std::mutex> lock(mu);
  const auto key = std::make_tuple(kern, dev.device, cl);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(cl), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cl);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
  cudaGetLastError();
  cache[key] = n >= 1;
  return n >= 1;
}

// Cluster-form launch: cl = the largest of 1, 2, 4, 8 with blocks * cl CTAs
// at most kClCtasPerSm per SM, at least one k-unit per part, and clusters of
// that size schedulable.
template <bool kInt, bool kRaw, int kMP = kMaxM>
cudaError_t launch_cluster(const DeviceInfo &dev, SkArgs<kInt> p, const CUtensorMap &tmA,
                           const CUtensorMap &tmB, int blocks, int nunits, cudaStream_t stream) {
  // kClCtasPerSm CTAs per SM: 228 KiB of shared memory, 1 KiB of it reserved per CTA
  static_assert(kClCtasPerSm * (sizeof(ClSmem<kRaw, kMP>) + 1024 + 1024) <= 228 * 1024,
                "cluster-form shared memory");
  static_assert(2 * kBBytes >= kMP * kBN * 4, "partial sums fit in two B stages");
  auto kern = gemm_tc_skinny_cl_kernel<kInt, kRaw, kMP>;
  const void *kp = reinterpret_cast<const void *>(kern);
  const size_t smem = sizeof(ClSmem<kRaw, kMP>) + 1024;
  const int threads = kRaw ? kClRawThreads : kThreads;
  cudaError_t e = set_max_dynamic_smem(kp, static_cast<int>(smem), dev.device);
  if (e != cudaSuccess) return e;
  int cl = 1;
  while (cl < kClMaxCluster &&
         static_cast<int64_t>(blocks) * cl * 2 <= static_cast<int64_t>(kClCtasPerSm) * dev.sm_count &&
         cl * 2 <= nunits)
    cl *= 2;
  while (cl > 1 && !clusters_fit(dev, kp, smem, threads, cl)) cl /= 2;
  p.split = cl;
  p.counters = nullptr;
  p.ws = nullptr;
  p.ws_ld = 0;
  p.nunits = nunits;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks * cl), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  // Programmatic dependent launch (the kernel waits for its predecessor before
  // touching global memory), and the cluster shape when k is split.
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = static_cast<unsigned>(cl);
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = cl > 1 ? 2 : 1;
  e = cudaLaunchKernelEx(&cfg, kern, tmA, tmB, p);
  if (e == cudaSuccess) e = cudaGetLastError();
  return e;
}

// One slice per CTA: column blocks times parts of k, at most one CTA per SM
// when k is split (the per-block form of the kernel).
template <bool kInt, bool kRawB>
cudaError_t launch_per_block(const DeviceInfo &dev, SkArgs<kInt> p, const CUtensorMap &tmA,
                             const CUtensorMap &tmB, int blocks, int nunits, cudaStream_t stream,
                             uint32_t *flags_ws) {
  const int M = p.M;
  int split = blocks < dev.sm_count ? dev.sm_count / blocks : 1;
  if (split > kMaxSplit) split = kMaxSplit;
  if (split > nunits) split = nunits;
  if (split < 1) split = 1;

  // split > 1 needs a workspace for the partial sums (from the pool); a caller
  // that provides its own memory gets whole column blocks instead.
  if (flags_ws != nullptr) split = 1;
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

  using Smem = typename std::conditional<kRawB, SkSmemI8, SkSmem>::type;
  const size_t smem = sizeof(Smem) + 1024;
  static_assert(sizeof(SkSmem) + 1024 <= 232448, "skinny kernel shared memory");
  static_assert(sizeof(SkSmemI8) + 1024 <= 232448, "raw-int8 skinny kernel shared memory");
  auto kern = gemm_tc_skinny_kernel<kInt, kRawB>;
  cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void *>(kern),
                                       static_cast<int>(smem), dev.device);
  if (e == cudaSuccess) {
    kern<<<static_cast<unsigned>(blocks * split), kRawB ? kI8Threads : kThreads, smem, stream>>>(
        tmA, tmB, p);
    e = cudaGetLastError();
  }
  if (pool_ws) {
    cudaError_t f = cudaFreeAsync(pool_ws, stream);
    if (e == cudaSuccess) e = f;
  }
  return e;
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

  const int blocks = (N + kBN - 1) / kBN;
  const int KB = (K + kBK - 1) / kBK;
  const int nunits = kInt ? (KB + kChunkKB - 1) / kChunkKB : KB;
  if (flags_ws == nullptr)
    return launch_cluster<kInt, false>(dev, p, tmA, tmB, blocks, nunits, stream);
  (void)flags_words;
  return launch_per_block<kInt, false>(dev, p, tmA, tmB, blocks, nunits, stream, flags_ws);
}

// Row-major rows x cols int8 matrix as bytes, boxes of box_rows rows x
// box_cols columns (by default 64 x 128), unswizzled or with the 128-byte
// swizzle (box_cols = 128): the raw tiles the converter warps read.
bool tmap8(CUtensorMap *tm, const void *base, int64_t rows, int64_t cols, int64_t ld,
           uint32_t box_rows = kBK, uint32_t box_cols = kBN, bool swizzle128 = false) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld)};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}


}  // namespace

bool tc_skinny_route(int M, int N, int sm_count) {
  if (M <= kSkinnyMaxM) return true;
  const int blocks = (N + kBN - 1) / kBN;
  return M <= kMaxM && blocks >= 16 && blocks < sm_count;
}

cudaError_t launch_tc_skinny_float(const DeviceInfo &dev, bool is_bf16, int M, int N, int K,
                                   float alpha, const void *A, int64_t lda, const void *B,
                                   int64_t ldb, float beta, float *C, int64_t ldc,
                                   cudaStream_t stream) {
  return launch<false>(dev,
                       is_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                       is_bf16, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream, nullptr, 0);
}

bool tc_skinny_i8_supported(int M, const void *B, int64_t ldb) {
  return M >= 1 && M <= kMaxM && reinterpret_cast<uintptr_t>(B) % 16 == 0 && ldb % 16 == 0;
}

cudaError_t launch_tc_skinny_i8(const DeviceInfo &dev, int M, int N, int K, int32_t alpha,
                                const void *A16, int64_t lda, const int8_t *B, int64_t ldb,
                                int32_t beta, int32_t *C, int64_t ldc, cudaStream_t stream) {
  if (!tc_skinny_i8_supported(M, B, ldb)) return cudaErrorInvalidValue;
  SkArgs<true> p;
  p.M = M;
  p.N = N;
  p.K = K;
  p.mp = (M + 15) / 16 * 16;
  p.alpha = alpha;
  p.beta = beta;
  p.C = C;
  p.ldc = ldc;
  p.idesc = idesc_f16(false, /*a_mn_major=*/true, /*b_mn_major=*/false, kBN, p.mp);
  p.err_word = dev.err_word;
  CUtensorMap tmA, tmB;
  if (!tmap16(&tmA, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, A16, M, K, lda,
              static_cast<uint32_t>(p.mp)))
    return cudaErrorInvalidValue;
  if (!tmap8(&tmB, B, K, N, ldb)) return cudaErrorInvalidValue;
  const int blocks = (N + kBN - 1) / kBN;
  const int KB = (K + kBK - 1) / kBK;
  const int nunits = (KB + kChunkKB - 1) / kChunkKB;
  return launch_per_block<true, true>(dev, p, tmA, tmB, blocks, nunits, stream, nullptr);
}

cudaError_t launch_tc_skinny_int(const DeviceInfo &dev, int M, int N, int K, int32_t alpha,
                                 const void *A16, int64_t lda, const void *B16, int64_t ldb,
                                 int32_t beta, int32_t *C, int64_t ldc, cudaStream_t stream,
                                 uint32_t *flags, size_t flags_words) {
  return launch<true>(dev, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, false, M, N, K, alpha, A16, lda, B16,
                      ldb, beta, C, ldc, stream, flags, flags_words);
}

bool tc_skinny_s8_supported(int M, const void *A, int64_t lda, const void *B, int64_t ldb) {
  return M >= 1 && M <= kMaxM && reinterpret_cast<uintptr_t>(A) % 16 == 0 && lda % 16 == 0 &&
         reinterpret_cast<uintptr_t>(B) % 16 == 0 && ldb % 16 == 0;
}

cudaError_t launch_tc_skinny_s8(const DeviceInfo &dev, int M, int N, int K, int32_t alpha,
                                const int8_t *A, int64_t lda, const int8_t *B, int64_t ldb,
                                int32_t beta, int32_t *C, int64_t ldc, cudaStream_t stream) {
  if (!tc_skinny_s8_supported(M, A, lda, B, ldb)) return cudaErrorInvalidValue;
  SkArgs<true> p;
  p.M = M;
  p.N = N;
  p.K = K;
  p.mp = (M + 15) / 16 * 16;
  p.alpha = alpha;
  p.beta = beta;
  p.C = C;
  p.ldc = ldc;
  p.idesc = idesc_f16(false, /*a_mn_major=*/true, /*b_mn_major=*/false, kBN, p.mp);
  p.err_word = dev.err_word;
  CUtensorMap tmA, tmB;
  if (!tmap8(&tmA, A, M, K, lda, static_cast<uint32_t>(p.mp), kBK)) return cudaErrorInvalidValue;
  if (!tmap8(&tmB, B, K, N, ldb, kBK, kBN, /*swizzle128=*/true)) return cudaErrorInvalidValue;
  const int blocks = (N + kBN - 1) / kBN;
  const int KB = (K + kBK - 1) / kBK;
  const int nunits = (KB + kChunkKB - 1) / kChunkKB;
  if (p.mp <= 16) return launch_cluster<true, true, 16>(dev, p, tmA, tmB, blocks, nunits, stream);
  if (p.mp <= 32) return launch_cluster<true, true, 32>(dev, p, tmA, tmB, blocks, nunits, stream);
  return launch_cluster<true, true, 64>(dev, p, tmA, tmB, blocks, nunits, stream);
}

}  // namespace dgr
