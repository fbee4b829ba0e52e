// work_split.cuh -- the work list of the persistent GEMM kernels: whole tiles
// round-robin over the resident units, then the leftover tiles of the last
// wave split along k into at most a few parts, one per otherwise idle unit.
// Part j > 0 of a tile adds its partial product into C after part j - 1 has
// stored (a per-tile flag, zero at launch), so every result is computed in
// one fixed order and is reproducible run to run. All units of a launch are
// resident at once (the grid never exceeds the co-resident capacity), so a
// part's wait always ends; the waits are bounded all the same.
#pragma once

#include <cstdint>

#include "launch.h"
#include "ptx.cuh"

namespace dgr {
namespace {

// One item of a unit's work list: a tile and a range of its k-blocks.
struct WorkItem {
  int tile, kb0, kb1, part, parts;
};

// Item n of unit u's work list (false past its end). The first dp_tiles tiles
// (a multiple of the number of units) are whole; each of the remaining
// tail_tiles tiles is split into `split` parts. kb_unit is the k granularity
// of split points in k-blocks.
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

// Splits T tiles of KB k-blocks over at most `cap` units: whole tiles
// round-robin, then the leftover tiles split along k (at most max_split
// parts, in steps of kb_unit k-blocks) so that every unit gets one part.
inline void plan_work(int64_t T, int KB, int kb_unit, int cap, int max_split, int &units,
                      int &dp_tiles, int &tail_tiles, int &split) {
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

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t *p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_gpu(uint32_t *p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Bounded wait until *flag >= value (another unit's part has been stored).
// On giving up: sets *abort, records the timeout in the error word, returns
// false.
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

}  // namespace
}  // namespace dgr
