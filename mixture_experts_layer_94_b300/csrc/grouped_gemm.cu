// grouped_gemm.cu — the expert FFNs as grouped GEMMs on the 5th-generation
// tensor cores (tcgen05.mma, accumulators in TMEM, operands staged by TMA).
//
// What is computed (per group = one routed or shared expert, over its rows):
//   gate/up phase:  g = X W_gate^T, u = X W_up^T, h = bf16(SiLU(g) * u)
//   down phase:     y = h W_down^T, then either
//                   out_acc[token] += w_{t,k} * y   (fused gate-weighted combine)
//                   or y_perm = bf16(y)             (step-wise path)
//   router phase:   partial logits = hidden x (one exact bf16 part of the fp32
//                   router matrix) over a slice of d, written in fp32; the
//                   router's top-K kernel sums the partials in a fixed order
// The expert FFN is the SwiGLU reading of the three-matrix expert ("Mixture of
// Experts Explained: Conditional Computation From Zero", "The slot it replaces,
// and what an expert is"); the weighted sum back to token order is "Chapter 19:
// Mixture-of-Experts Models", §19.3.2 and the §19.2 flowchart ("Sum with gate
// weights"); the shared expert adds with weight 1 ("Mixture of Experts for LLM
// Inference", "Shared experts").
//
// Kernel structure (persistent, 192 threads per CTA, one CTA per SM):
//   warp 0     TMA producer: per K block an activation box and a weight box,
//              128-byte swizzled, into a shared-memory ring.
//   warp 1     allocates 512 TMEM columns; one lane issues tcgen05.mma
//              (bf16 -> fp32, N = 256) into one of two 256-column accumulators
//              and commits stage releases / tile completion to mbarriers.
//   warps 2-5  epilogue: tcgen05.ld the accumulator (warp w reads TMEM lanes
//              32*(w%4)..+31, one output row per thread), apply the fused
//              SwiGLU, weighted scatter-add or logits store, release it.
// PAIR == 1: a CTA computes 128-row tiles alone (M=128; 4-stage x 48 KB ring).
// PAIR == 2: a cluster of two CTAs computes 256-row tiles with the CTA-pair
//   MMA (M=256). Each CTA loads its own 128 activation rows and its own half of
//   the 256 weight rows (the gate tile on the leader, the up tile on the peer;
//   or two halves of the down rows) with ordinary, non-multicast TMA loads into
//   its own 6-stage x 32 KB ring, and each CTA's TMEM receives its own 128
//   rows. The leader's thread issues the MMA; stage releases and tile
//   completion are signalled to both CTAs' barriers. Per CTA this halves the
//   weight bytes pulled from L2 per FLOP and deepens the ring. A group's last
//   tile with at most 128 rows left runs as an M=128 pair MMA, 64 rows per CTA
//   (see is_half_tile), so that it carries at most 127 padding rows, not 255.
// The double-buffered accumulator lets the epilogue of tile i overlap the MMAs
// of tile i+1. Tiles are (group, m block, n block), n-major inside a group so
// CTAs running side by side share weight tiles in L2; a CTA (pair) walks tiles
// unit, unit + units, ... and finds each tile's group by binary search over the
// device-built prefix of tile counts (no host round trip).
// Every mbarrier wait is bounded: on a stall the kernel records a timeout in
// the workspace error word, drains its own copies and MMAs, frees TMEM and exits.
#include <cuda.h>

#include <atomic>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "tile_sched.cuh"

namespace moe {
namespace {

constexpr int kGemmThreads = 192;
constexpr uint32_t kStageA = kBM * kBK * 2;  // 16 KB: 128 activation rows x 64
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCols = 256;
constexpr uint64_t kDrainTimeoutNs = 50000000ull;  // 50 ms per in-flight copy on abort
constexpr size_t kBarrierBytes = 256;

template <int PAIR>
struct Cfg {
  static constexpr int kStages = PAIR == 2 ? 6 : 4;
  static constexpr uint32_t kStageB = PAIR == 2 ? 128 * kBK * 2 : 256 * kBK * 2;  // this CTA's weight rows
  static constexpr uint32_t kStageBytes = kStageA + kStageB;
  static constexpr int kTileRows = kBM * PAIR;
  static constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(128 * PAIR, 256);
  // A pair's tail tile of at most 128 rows: M = 128, 64 rows from each CTA.
  static constexpr uint32_t kIdescHalf = ptx::idesc_bf16_f32(128, 256);
  static constexpr size_t kSmem = 1024 /*alignment slack*/ + (size_t)kStages * kStageBytes + kBarrierBytes;
};

// Whether a pair tile is the half form: the group's last tile with at most
// 128 rows left runs as an M = 128 pair MMA (64 rows from each CTA), which
// halves the padding rows of a group's last tile on average. Its accumulator
// lands folded: TMEM lanes 0-63 of each CTA hold the CTA's 64 rows x the MMA's
// first 128 columns (the leader's B rows), lanes 64-127 the same rows x the
// last 128 (the peer's B rows), both in TMEM columns 0-127. So that SwiGLU
// stays within a thread, a gate/up half tile's B rows are arranged as
// [gate f0..f0+63; up f0..f0+63] on the leader and the next 64 on the peer.
__device__ __forceinline__ bool is_half_tile(const TileInfo& ti) {
  return ti.g.rows - ti.m_blk * 2 * kBM <= kBM;
}

struct RouterTile {
  int m_blk, split, part, kb0, kb1;
};

__device__ __forceinline__ RouterTile decode_router_tile(int tile, const GemmArgs& a) {
  RouterTile r;
  r.m_blk = tile % a.r_m_tiles;
  r.split = tile / a.r_m_tiles;
  r.part = a.r_merged ? 0 : r.split / a.r_dslices;
  const int slice = r.split - r.part * a.r_dslices;
  r.kb0 = slice * a.r_kb_per_slice;
  r.kb1 = min(a.r_nkb_d, r.kb0 + a.r_kb_per_slice);
  return r;
}

template <int PHASE, int EPI, int PAIR>
__global__ void __launch_bounds__(kGemmThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
                        const __grid_constant__ CUtensorMap tmB0, const __grid_constant__ CUtensorMap tmB1,
                        const __grid_constant__ CUtensorMap tmU0, const __grid_constant__ CUtensorMap tmU1,
                        const __grid_constant__ CUtensorMap tmBh0, const __grid_constant__ CUtensorMap tmBh1,
                        const __grid_constant__ CUtensorMap tmUh0, const __grid_constant__ CUtensorMap tmUh1,
                        const GemmArgs a) {
  pdl_trigger();
  using C = Cfg<PAIR>;
  constexpr int kStages = C::kStages;
  constexpr uint32_t kStageB = C::kStageB;
  constexpr uint32_t kStageBytes = C::kStageBytes;
  constexpr int kTileRows = C::kTileRows;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw_base + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw_base);
  const uint32_t sA = base;                              // kStages x 16 KB
  const uint32_t sB = base + kStages * kStageA;          // kStages x kStageB
  const uint32_t sBar = base + kStages * kStageBytes;    // barriers
  uint8_t* gBar = gbase + kStages * kStageBytes;
  auto full_bar = [&](int s) { return sBar + 8u * s; };
  auto empty_bar = [&](int s) { return sBar + 8u * (kStages + s); };
  auto tfull_bar = [&](int i) { return sBar + 8u * (2 * kStages + i); };
  auto tempty_bar = [&](int i) { return sBar + 8u * (2 * kStages + 2 + i); };
  const uint32_t drain_bar = sBar + 8u * (2 * kStages + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gBar + 8 * (2 * kStages + 5));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gBar + 8 * (2 * kStages + 5) + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = PAIR == 2 ? ptx::cluster_ctarank() : 0u;
  const bool leader = rank == 0;
  const int unit = PAIR == 2 ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int units = PAIR == 2 ? (int)(gridDim.x >> 1) : (int)gridDim.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(full_bar(s), 1);
      ptx::mbar_init(empty_bar(s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(tfull_bar(i), 1);
      ptx::mbar_init(tempty_bar(i), 128 * PAIR);
    }
    ptx::mbar_init(drain_bar, 1);
    *abort_flag = 0;
    ptx::fence_mbarrier_init();
    ptx::fence_proxy_async_shared();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tmA0);
    ptx::prefetch_tmap(&tmB0);
    if (PHASE == kPhaseGateUp) ptx::prefetch_tmap(&tmU0);
  }
  if (warp == 1) {
    if (PAIR == 2) {
      ptx::tmem_alloc_pair(ptx::smem_u32(tmem_slot), kTmemCols);
      ptx::tmem_relinquish_pair();
    } else {
      ptx::tmem_alloc(ptx::smem_u32(tmem_slot), kTmemCols);
      ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
  }
  __syncthreads();
  if (PAIR == 2) ptx::cluster_sync();  // the peer's barriers are initialised before any remote use
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // The setup above touches shared memory, TMEM and kernel parameters only;
  // from here on the previous kernel's results are read.
  pdl_wait();
  const int total = (PHASE == kPhaseRouter) ? a.r_tiles : __ldg(a.tile_start + a.G);

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0;
      bool aborted = false;
      for (int tile = unit; tile < total && !aborted && PHASE == kPhaseRouter; tile += units) {
        // Router: A = hidden rows of the m block, B = the router part's columns.
        const RouterTile rt = decode_router_tile(tile, a);
        // merged: the three parts' columns side by side in the B stage
        const uint32_t part_bytes = (uint32_t)a.r_np * kBK * 2u;
        const uint32_t bytes = kStageA + (a.r_merged ? 3u : 1u) * part_bytes;
        for (int kb = rt.kb0; kb < rt.kb1; ++kb) {
          if (!ptx::mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, a.err)) {
            aborted = true;
            break;
          }
          ptx::mbar_arrive_expect_tx(full_bar(stage), bytes);
          ptx::tma_load_2d(sA + stage * kStageA, &tmA0, full_bar(stage), kb * kBK, rt.m_blk * kBM);
          if (a.r_merged) {
            for (int p = 0; p < 3; ++p)
              ptx::tma_load_2d(sB + stage * kStageB + (uint32_t)p * part_bytes, &tmB0, full_bar(stage),
                               p * a.r_d_pad + kb * kBK, 0);
          } else {
            ptx::tma_load_2d(sB + stage * kStageB, &tmB0, full_bar(stage), rt.part * a.r_d_pad + kb * kBK, 0);
          }
          ++issued;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      for (int tile = unit; tile < total && !aborted && PHASE != kPhaseRouter; tile += units) {
        const TileInfo ti = decode_tile(tile, a);
        const int kind = ti.g.kind;
        const CUtensorMap* mA = kind ? &tmA1 : &tmA0;
        const CUtensorMap* mB = kind ? &tmB1 : &tmB0;
        const CUtensorMap* mU = kind ? &tmU1 : &tmU0;
        // a pair's half tile takes 64 rows from each CTA
        const bool half = PAIR == 2 && is_half_tile(ti);
        const int a_row = (PHASE == kPhaseGateUp ? ti.g.a_row0 : ti.g.h_row0) + ti.m_blk * kTileRows +
                          (int)rank * (half ? kBM / 2 : kBM);
        // Weight rows: gate/up -> rows n*128 of the expert in W_gate (and W_up);
        // down -> rows n*256 (+ this CTA's 128-row half in a pair).
        int b_row = ti.g.index * a.w_rows[kind] + ti.n_blk * (PHASE == kPhaseGateUp ? kBNGateUp : kBNDown);
        if (PAIR == 2 && PHASE == kPhaseDown) b_row += (int)rank * (kBNDown / 2);
        const int nkb = a.k_blocks[kind];
        for (int kb = 0; kb < nkb; ++kb) {
          if (!ptx::mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, a.err)) {
            aborted = true;
            break;
          }
          const uint32_t dA = sA + stage * kStageA, dB = sB + stage * kStageB;
          if (PAIR == 2) {
            const uint32_t fb = ptx::mapa_shared(full_bar(stage), 0);  // the leader's barrier
            if (leader) ptx::mbar_arrive_expect_tx(full_bar(stage), 2u * kStageBytes);
            ptx::tma_load_2d_pair(dA, mA, fb, kb * kBK, a_row);
            if (PHASE == kPhaseGateUp && half) {
              // gate and up rows f0..f0+63 on the leader, f0+64..f0+127 on the peer (64-row boxes)
              const int hb = b_row + (int)rank * (kBNGateUp / 2);
              ptx::tma_load_2d_pair(dB, kind ? &tmBh1 : &tmBh0, fb, kb * kBK, hb);
              ptx::tma_load_2d_pair(dB + kStageB / 2, kind ? &tmUh1 : &tmUh0, fb, kb * kBK, hb);
            } else {
              ptx::tma_load_2d_pair(dB, (PHASE == kPhaseGateUp && !leader) ? mU : mB, fb, kb * kBK, b_row);
            }
          } else {
            ptx::mbar_arrive_expect_tx(full_bar(stage), kStageBytes);
            ptx::tma_load_2d(dA, mA, full_bar(stage), kb * kBK, a_row);
            ptx::tma_load_2d(dB, mB, full_bar(stage), kb * kBK, b_row);
            if (PHASE == kPhaseGateUp) ptx::tma_load_2d(dB + kStageB / 2, mU, full_bar(stage), kb * kBK, b_row);
          }
          ++issued;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (aborted && (PAIR == 1 || leader)) {
        // Wait for the copies still in flight into this CTA's ring (the last kStages issues).
        const uint32_t n = issued < (uint32_t)kStages ? issued : (uint32_t)kStages;
        for (uint32_t j = issued - n; j < issued; ++j)
          wait_raw(full_bar(j % kStages), (j / kStages) & 1u, kDrainTimeoutNs);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && (PAIR == 1 || leader)) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool aborted = false;
      for (int tile = unit; tile < total && !aborted; tile += units) {
        int nkb;
        uint32_t idesc = C::kIdesc;
        if (PHASE == kPhaseRouter) {
          const RouterTile rt = decode_router_tile(tile, a);
          nkb = rt.kb1 - rt.kb0;
          idesc = a.r_idesc;
        } else {
          const TileInfo ti = decode_tile(tile, a);
          nkb = a.k_blocks[ti.g.kind];
          if (PAIR == 2 && is_half_tile(ti)) idesc = C::kIdescHalf;
        }
        if (!ptx::mbar_wait(tempty_bar(acc), acc_phase ^ 1u, abort_flag, a.err)) break;
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)acc * kAccCols;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!ptx::mbar_wait(full_bar(stage), phase, abort_flag, a.err)) {
            aborted = true;
            break;
          }
          ptx::tc_fence_after();
          const uint64_t adesc = ptx::smem_desc_sw128(sA + stage * kStageA);
          const uint64_t bdesc = ptx::smem_desc_sw128(sB + stage * kStageB);
          if (PHASE == kPhaseRouter && a.r_merged) {
            // the hi, mid and lo parts of the router matrix into one accumulator
            const uint32_t part_bytes = (uint32_t)a.r_np * kBK * 2u;
            for (int p = 0; p < 3; ++p) {
              const uint64_t pdesc = ptx::smem_desc_sw128(sB + stage * kStageB + (uint32_t)p * part_bytes);
#pragma unroll
              for (int k = 0; k < kBK / 16; ++k)
                ptx::mma_bf16(d_tmem, adesc + 2u * k, pdesc + 2u * k, idesc, (kb | k | p) != 0 ? 1u : 0u);
            }
          } else {
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k) {
              if (PAIR == 2)
                ptx::mma_bf16_pair(d_tmem, adesc + 2u * k, bdesc + 2u * k, idesc, (kb | k) != 0 ? 1u : 0u);
              else
                ptx::mma_bf16(d_tmem, adesc + 2u * k, bdesc + 2u * k, idesc, (kb | k) != 0 ? 1u : 0u);
            }
          }
          if (PAIR == 2) ptx::mma_commit_pair_multicast(empty_bar(stage), 0x3);
          else ptx::mma_commit(empty_bar(stage));
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (aborted) break;
        if (PAIR == 2) ptx::mma_commit_pair_multicast(tfull_bar(acc), 0x3);
        else ptx::mma_commit(tfull_bar(acc));
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // Every MMA this thread issued must finish before TMEM is released.
      if (PAIR == 2) ptx::mma_commit_pair_multicast(drain_bar, 0x1);
      else ptx::mma_commit(drain_bar);
      wait_raw(drain_bar, 0, kWaitTimeoutNs);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;
    const int row_in_tile = (int)rank * kBM + quad * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    int acc = 0;
    uint32_t acc_phase = 0;
    auto release = [&](int i) {
      ptx::tc_fence_before();
      if (PAIR == 2) ptx::mbar_arrive_cluster(ptx::mapa_shared(tempty_bar(i), 0));
      else ptx::mbar_arrive(tempty_bar(i));
    };
    for (int tile = unit; tile < total && PHASE == kPhaseRouter; tile += units) {
      // Router: fp32 partial logits of this (m block, split) for rows < T, experts < N.
      const RouterTile rt = decode_router_tile(tile, a);
      if (!ptx::mbar_wait(tfull_bar(acc), acc_phase, abort_flag, a.err)) break;
      ptx::tc_fence_after();
      const uint32_t tacc = tmem_base + lane_off + (uint32_t)acc * kAccCols;
      const int64_t t = (int64_t)rt.m_blk * kBM + row_in_tile;
      float* prow = a.r_partial + ((int64_t)rt.split * a.r_T + (t < a.r_T ? t : 0)) * a.r_N;
      const bool vec = (a.r_N & 3) == 0;
#pragma unroll 1
      for (int c = 0; c < a.r_np; c += 16) {
        uint32_t v[16];
        ptx::tmem_ld_32x32b_x16(tacc + c, v);
        ptx::tmem_wait_ld();
        if (t < a.r_T) {
          if (vec) {
#pragma unroll
            for (int q = 0; q < 16; q += 4)
              if (c + q < a.r_N)
                *reinterpret_cast<float4*>(prow + c + q) =
                    make_float4(__uint_as_float(v[q]), __uint_as_float(v[q + 1]), __uint_as_float(v[q + 2]),
                                __uint_as_float(v[q + 3]));
          } else {
#pragma unroll
            for (int q = 0; q < 16; ++q)
              if (c + q < a.r_N) prow[c + q] = __uint_as_float(v[q]);
          }
        }
      }
      release(acc);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    for (int tile = unit; tile < total && PHASE != kPhaseRouter; tile += units) {
      const TileInfo ti = decode_tile(tile, a);
      const int kind = ti.g.kind;
      if (!ptx::mbar_wait(tfull_bar(acc), acc_phase, abort_flag, a.err)) break;
      ptx::tc_fence_after();
      const uint32_t tacc = tmem_base + lane_off + (uint32_t)acc * kAccCols;
      // half tile (folded accumulator): lanes 64-127 hold the same 64 rows as
      // lanes 0-63, for the MMA's last 128 columns
      const bool half = PAIR == 2 && is_half_tile(ti);
      const bool upper = half && quad >= 2;
      const int tr = half ? (int)rank * (kBM / 2) + (quad & 1) * 32 + lane : row_in_tile;
      const int r_local = ti.m_blk * kTileRows + tr;
      const bool row_ok = r_local < ti.g.rows;
      if (PHASE == kPhaseGateUp) {
        const int n_ext = a.n_ext[kind];
        const int col0 = ti.n_blk * kBNGateUp;
        __nv_bfloat16* hrow = a.h[kind] + (int64_t)(ti.g.h_row0 + (row_ok ? r_local : 0)) * a.ldh[kind];
        // half tile: gate at TMEM columns 0-63, up at 64-127, for f0 + 64 (upper lanes) + 0..63
        const int nf = half ? kBNGateUp / 2 : kBNGateUp;
        const int fbase = col0 + (upper ? kBNGateUp / 2 : 0);
#pragma unroll 1
        for (int c = 0; c < nf / 32; ++c) {
          uint32_t gv[32], uv[32];
          ptx::tmem_ld_32x32b_x32(tacc + c * 32, gv);
          ptx::tmem_ld_32x32b_x32(tacc + nf + c * 32, uv);
          ptx::tmem_wait_ld();
          if (row_ok) {
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              const int f0 = fbase + c * 32 + v * 8;
              if (f0 < n_ext) {
                uint32_t p[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  const float g0 = __uint_as_float(gv[v * 8 + 2 * j]);
                  const float g1 = __uint_as_float(gv[v * 8 + 2 * j + 1]);
                  const float u0 = __uint_as_float(uv[v * 8 + 2 * j]);
                  const float u1 = __uint_as_float(uv[v * 8 + 2 * j + 1]);
                  p[j] = pack_bf16x2(silu_f(g0) * u0, silu_f(g1) * u1);
                }
                *reinterpret_cast<uint4*>(hrow + f0) = make_uint4(p[0], p[1], p[2], p[3]);
              }
            }
          }
        }
      } else {
        const int col0 = ti.n_blk * kBNDown;
        int64_t t = 0;
        float w = 1.f;
        if (EPI == kEpiScatter && row_ok) {
          if (kind == 0 && a.row_w) {  // expert choice: the row's token and score
            t = __ldg(a.perm_src + ti.g.h_row0 + r_local);
            w = __ldg(a.row_w + ti.g.h_row0 + r_local);
          } else if (kind == 0) {
            const int32_t src = __ldg(a.perm_src + ti.g.h_row0 + r_local);
            t = src / a.top_k;
            w = __ldg(a.topk_w + src);
          } else {
            t = r_local;
          }
        }
        // half tile: TMEM columns 0-127 are output columns col0 + (128 on upper lanes) + 0..127
        const int cbase = col0 + (upper ? kBNDown / 2 : 0);
#pragma unroll 1
        for (int c = 0; c < (half ? kBNDown / 64 : kBNDown / 32); ++c) {
          uint32_t yv[32];
          ptx::tmem_ld_32x32b_x32(tacc + c * 32, yv);
          ptx::tmem_wait_ld();
          if (row_ok) {
            if (EPI == kEpiScatter) {
              float* orow = a.out_acc + t * a.d;
#pragma unroll
              for (int v = 0; v < 8; ++v) {
                const int n0 = cbase + c * 32 + v * 4;
                if (n0 < a.d) {
                  float4 val = make_float4(w * __uint_as_float(yv[v * 4 + 0]), w * __uint_as_float(yv[v * 4 + 1]),
                                           w * __uint_as_float(yv[v * 4 + 2]), w * __uint_as_float(yv[v * 4 + 3]));
                  atomicAdd(reinterpret_cast<float4*>(orow + n0), val);
                }
              }
            } else {
              __nv_bfloat16* yrow = (kind && a.y_sh ? a.y_sh : a.y) + (int64_t)(ti.g.h_row0 + r_local) * a.d;
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                const int n0 = cbase + c * 32 + v * 8;
                if (n0 < a.d) {
                  uint32_t p[4];
#pragma unroll
                  for (int j = 0; j < 4; ++j)
                    p[j] = pack_bf16x2(__uint_as_float(yv[v * 8 + 2 * j]), __uint_as_float(yv[v * 8 + 2 * j + 1]));
                  *reinterpret_cast<uint4*>(yrow + n0) = make_uint4(p[0], p[1], p[2], p[3]);
                }
              }
            }
          }
        }
      }
      release(acc);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  __syncthreads();
  if (PAIR == 2) ptx::cluster_sync();  // no remote arrive or MMA read of this CTA is still pending
  if (warp == 1) {
    ptx::tc_fence_after();
    if (PAIR == 2) ptx::tmem_dealloc_pair(tmem_base, kTmemCols);
    else ptx::tmem_dealloc(tmem_base, kTmemCols);
  }
}

template <int PHASE, int EPI, int PAIR>
cudaError_t launch_t(const GemmMaps& m, const GemmArgs& a, int64_t tile_bound, cudaStream_t s) {
  auto kern = grouped_gemm_kernel<PHASE, EPI, PAIR>;
  constexpr size_t smem = Cfg<PAIR>::kSmem;
  // Per device: the shared-memory opt-in (a function attribute) and, for
  // pairs, how many 2-CTA clusters of this kernel fit on the GPU at once.
  static std::atomic<uint64_t> configured{0};
  static std::atomic<int> max_units[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[1];
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeIgnore;
  if (PAIR == 2) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  if (!(configured.load() & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int units = sms;
    if (PAIR == 2) {
      int clusters = 0;
      cfg.gridDim = dim3((unsigned)(sms & ~1));
      e = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
      if (e != cudaSuccess) return e;
      units = clusters > 0 ? clusters : 1;
    }
    max_units[dev & 63].store(units);
    configured.fetch_or(bit);
  }
  int64_t units = max_units[dev & 63].load();
  if (tile_bound < units) units = tile_bound < 1 ? 1 : tile_bound;
  return launch_attr(kern, dim3((unsigned)(units * PAIR)), dim3(kGemmThreads), smem, s, attr[0], m.a[0], m.a[1],
                     m.b[0], m.b[1], m.bu[0], m.bu[1], m.bh[0], m.bh[1], m.uh[0], m.uh[1], a);
}

}  // namespace

int64_t gemm_tile_bound(int phase, int64_t routed_rows, int32_t N, int32_t S, int64_t T, int32_t F,
                        int32_t Fs, int32_t d, int32_t tile_rows) {
  // sum_e ceil(n_e / BM) <= routed_rows / BM + (experts with rows) <= routed_rows / BM + min(N, routed_rows)
  const int64_t m_routed = routed_rows / tile_rows + (routed_rows < N ? routed_rows : N);
  const int64_t m_shared = (int64_t)S * ((T + tile_rows - 1) / tile_rows);
  if (phase == kPhaseGateUp)
    return m_routed * ((F + kBNGateUp - 1) / kBNGateUp) + m_shared * ((Fs + kBNGateUp - 1) / kBNGateUp);
  return (m_routed + m_shared) * ((d + kBNDown - 1) / kBNDown);
}

cudaError_t launch_grouped_gemm(int phase, int epilogue, int pair, const GemmMaps& maps, const GemmArgs& a,
                                int64_t tile_bound, cudaStream_t s) {
  if (phase == kPhaseRouter) return launch_t<kPhaseRouter, kEpiLogits, 1>(maps, a, tile_bound, s);
  if (pair == 2) {
    if (phase == kPhaseGateUp) return launch_t<kPhaseGateUp, kEpiSwiGLU, 2>(maps, a, tile_bound, s);
    if (epilogue == kEpiScatter) return launch_t<kPhaseDown, kEpiScatter, 2>(maps, a, tile_bound, s);
    return launch_t<kPhaseDown, kEpiStoreY, 2>(maps, a, tile_bound, s);
  }
  if (phase == kPhaseGateUp) return launch_t<kPhaseGateUp, kEpiSwiGLU, 1>(maps, a, tile_bound, s);
  if (epilogue == kEpiScatter) return launch_t<kPhaseDown, kEpiScatter, 1>(maps, a, tile_bound, s);
  return launch_t<kPhaseDown, kEpiStoreY, 1>(maps, a, tile_bound, s);
}

}  // namespace moe
