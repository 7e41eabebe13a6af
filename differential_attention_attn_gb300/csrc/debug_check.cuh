// Bounds checks of the debug build (compiled with -DDIFFATTN_DEBUG; the release
// library compiles every check away).  compute-sanitizer is not available to
// this library's tests, so its kernels check their own accesses instead: every
// tensor-memory column range, shared-memory offset and global index they touch
// is tested against the size of what it addresses.  A failing check records
// DIFFATTN_ERR_BOUNDS | (site << 8) in the call's status word (the first
// failure wins) and the access is skipped, so nothing outside its buffer is
// touched.  Checks that guard a warp-collective instruction (tcgen05.ld/st)
// are agreed over the warp so that the whole warp skips together.
#pragma once

#include <cstdint>

#include "../../include/diffattn.h"

namespace diffattn {

#ifdef DIFFATTN_DEBUG
constexpr bool kDebugChecks = true;
#else
constexpr bool kDebugChecks = false;
#endif

// Per-thread check: records the first failure, returns whether `ok`.
__device__ __forceinline__ bool dbg_ok(bool ok, int32_t *status, int site) {
  if (kDebugChecks && !ok && status != nullptr)
    atomicCAS(status, 0, static_cast<int32_t>(DIFFATTN_ERR_BOUNDS) | (site << 8));
  return !kDebugChecks || ok;
}

// Warp-wide check (every lane of the warp must call it): true only if `ok`
// holds on every lane.
__device__ __forceinline__ bool dbg_ok_warp(bool ok, int32_t *status, int site) {
  if (!kDebugChecks) return true;
  const bool all = __all_sync(0xffffffffu, ok);
  return dbg_ok(all, status, site);
}

// A tensor-memory access spanning `cols` columns from address taddr (lane <<
// 16 | column) by warp `warp`, in an allocation of alloc_cols columns at
// `base`: the columns lie inside the allocation and the lanes (lanes of them
// from the address's lane field) inside the warp's own 32-lane quarter.
__device__ __forceinline__ bool tmem_range_ok(uint32_t taddr, uint32_t cols, uint32_t base,
                                              uint32_t alloc_cols, int warp, uint32_t lanes) {
  const uint32_t col = taddr & 0xFFFFu, lane = taddr >> 16, col0 = base & 0xFFFFu;
  const uint32_t q0 = 32u * static_cast<uint32_t>(warp & 3);
  return col >= col0 && col + cols <= col0 + alloc_cols && lane >= q0 && lane + lanes <= q0 + 32u;
}

// The column range alone, lane 0 (MMA operands and accumulators).
__device__ __forceinline__ bool tmem_cols_ok(uint32_t taddr, uint32_t cols, uint32_t base,
                                             uint32_t alloc_cols) {
  const uint32_t col = taddr & 0xFFFFu, col0 = base & 0xFFFFu;
  return (taddr >> 16) == 0 && col >= col0 && col + cols <= col0 + alloc_cols;
}

}  // namespace diffattn
