// tile_sched.cuh — tile lookup shared by the grouped-GEMM kernels (internal).
#pragma once

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace moe {

struct TileInfo {
  GroupDesc g;
  int m_blk, n_blk;
};

// Tile `tile` of a grouped GEMM: its group (the last group whose first tile
// is <= tile, which skips empty groups) by binary search over the device-built
// prefix of tile counts, then (n block, m block) in the group's order for this
// GEMM: m fastest, or (gate/up only) n fastest.
__device__ __forceinline__ TileInfo decode_tile(int tile, const GemmArgs& a) {
  int lo = 0, hi = a.G - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(a.tile_start + mid) <= tile) lo = mid;
    else hi = mid - 1;
  }
  TileInfo ti;
  ti.g = a.groups[lo];
  const int start = __ldg(a.tile_start + lo);
  const int local = tile - start;
  if (!a.phase_dn && ti.g.order_gu) {
    const int n_tiles = (__ldg(a.tile_start + lo + 1) - start) / ti.g.m_tiles;
    ti.m_blk = local / n_tiles;
    ti.n_blk = local - ti.m_blk * n_tiles;
  } else {
    ti.n_blk = local / ti.g.m_tiles;
    ti.m_blk = local - ti.n_blk * ti.g.m_tiles;
  }
  return ti;
}

// Wait without an abort flag, bounded by `limit_ns`; false on timeout. Used
// only to drain a pipeline that is already shutting down.
__device__ __forceinline__ bool wait_raw(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
  return true;
}

}  // namespace moe
