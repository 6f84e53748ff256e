// grouped_gemm_fp8.cu — the expert FFNs for experts stored as FP8 E4M3 codes
// with one fp32 scale per matrix row.
//
// It computes what grouped_gemm.cu computes (gate/up + SwiGLU, then the down
// projection with the fused gate-weighted scatter-add or a plain store), for
// experts kept in 8 bits. Storing only the experts in low precision is the
// serving recipe of "AI Infrastructure series, Part 12 of 24" ("How do you
// serve an MoE model on your own GPUs?"); it halves the bytes every token
// reads ("Mixture of Experts Explained", "Total versus active parameters"),
// and those bytes are what bound decode.
//
// Data path:
//  * The tensor cores multiply E4M3 by E4M3 (tcgen05.mma kind::f8f6f4, fp32
//    accumulators in TMEM) and read the expert codes exactly as TMA brings
//    them from HBM: no conversion pass, and shared memory carries each code
//    byte twice (TMA write, MMA read). Converting the codes to fp16 in shared
//    memory instead costs three times that, which on this GPU is about the
//    whole shared-memory bandwidth at the HBM rate.
//  * The activations arrive as the two-term E4M3 expansion of act_quant.cu
//    (x ~= s * (hi + lo), bf16-level precision) with the two terms in
//    interleaved rows: a tile of up to 64 tokens is one 128-row MMA operand,
//    token t's hi in row 2t and lo in row 2t+1. TMEM lanes 2t and 2t+1 then
//    hold hi*W and lo*W, which the epilogue adds with one shuffle.
//  * Tokens are the MMA's M, weights its N (256: the gate and up rows of 128
//    FFN units, or 256 rows of W_down); an MMA takes time in proportion to
//    M x K, so the weights go in N. K advances 128 codes (one 128-byte line
//    per row) per pipeline stage, four MMAs of K = 32.
//  * Epilogue: (hi + lo) x the token row's scale x the weight row's scale.
//    Gate/up applies SiLU(g) * u and writes h as fp16 (quantised the same way
//    for the down GEMM). Down either scatter-adds w * y into the token's fp32
//    output row or stores y as bf16.
//
// Warps (192 threads, one CTA per SM, persistent over the tiles):
//   0     TMA producer (token-row box + weight-code boxes per stage)
//   1     TMEM allocation, MMA issue
//   2-5   epilogue (warp w reads TMEM lanes 32*(w%4)..+31)
// Every mbarrier wait is bounded. On a stall the kernel records a timeout in
// the error word, drains its own copies and MMAs, frees TMEM and exits.
#include <cuda.h>

#include <atomic>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "tile_sched.cuh"

namespace moe {
namespace {

constexpr int kThreads = 192;
constexpr int kStages = 4;
constexpr int kKq = 128;            // codes of K per stage (one 128-byte line per row)
constexpr int kARows = 2 * kF8TileRows;  // two operand rows (hi, lo) per token
constexpr int kWRows = 256;         // weight rows per tile (MMA N)
constexpr uint32_t kABytes = (uint32_t)kARows * kKq;   // 16 KB
constexpr uint32_t kBBytes = (uint32_t)kWRows * kKq;   // 32 KB
constexpr uint32_t kStageBytes = kABytes + kBBytes;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCols = 256;
constexpr uint32_t kIdesc = ptx::idesc_f8_f32(kARows, kWRows);
constexpr uint64_t kDrainTimeoutNs = 50000000ull;
constexpr size_t kSmem = 1024 /*alignment slack*/ + (size_t)kStages * kStageBytes + 256;
static_assert(kSmem <= 232448, "shared memory per CTA");

// Operand box for a tile of n tokens: 16 << box_sel(n) rows (>= 2n).
__device__ __forceinline__ int box_sel(int n) { return n <= 8 ? 0 : (n <= 16 ? 1 : (n <= 32 ? 2 : 3)); }

// This lane's sums of 16 accumulator columns of a (hi, lo) lane pair: the
// even lane returns columns 0..15 of `v`, the odd lane columns 16..31, each
// plus its neighbour's same column.
__device__ __forceinline__ void pair_sum16(const uint32_t (&v)[32], int odd, float (&out)[16]) {
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const float mine = __uint_as_float(odd ? v[j + 16] : v[j]);
    const float send = __uint_as_float(odd ? v[j] : v[j + 16]);
    out[j] = mine + __shfl_xor_sync(0xffffffffu, send, 1);
  }
}

template <int PHASE, int EPI>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_fp8_kernel(const __grid_constant__ F8Maps maps, const GemmArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw_base + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw_base);
  const uint32_t sA = base;                           // kStages x 16 KB
  const uint32_t sB = base + kStages * kABytes;       // kStages x 32 KB
  const uint32_t sBar = base + kStages * kStageBytes;
  uint8_t* gBar = gbase + kStages * kStageBytes;
  auto full_bar = [&](int s) { return sBar + 8u * s; };
  auto empty_bar = [&](int s) { return sBar + 8u * (kStages + s); };
  auto tfull_bar = [&](int i) { return sBar + 8u * (2 * kStages + i); };
  auto tempty_bar = [&](int i) { return sBar + 8u * (2 * kStages + 2 + i); };
  const uint32_t drain_bar = sBar + 8u * (2 * kStages + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gBar + 8 * (2 * kStages + 5));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gBar + 8 * (2 * kStages + 5) + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int total = __ldg(a.tile_start + a.G);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(full_bar(s), 1);
      ptx::mbar_init(empty_bar(s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(tfull_bar(i), 1);
      ptx::mbar_init(tempty_bar(i), 128);
    }
    ptx::mbar_init(drain_bar, 1);
    *abort_flag = 0;
    ptx::fence_mbarrier_init();
    ptx::fence_proxy_async_shared();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&maps.w[0]);
    if (PHASE == kPhaseGateUp) ptx::prefetch_tmap(&maps.u[0]);
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), kTmemCols);
    ptx::tmem_relinquish();
    ptx::tc_fence_before();
  }
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, issued = 0;
      bool aborted = false;
      for (int tile = blockIdx.x; tile < total && !aborted; tile += gridDim.x) {
        const TileInfo ti = decode_tile(tile, a);
        const int kind = ti.g.kind;
        const int bsel = box_sel(min(kF8TileRows, ti.g.rows - ti.m_blk * kF8TileRows));
        const uint32_t bytes = (16u << bsel) * kKq + kBBytes;
        const CUtensorMap* mA = &maps.x[kind][bsel];
        const CUtensorMap* mW = &maps.w[kind];
        const CUtensorMap* mU = &maps.u[kind];
        const int a_row = 2 * ((PHASE == kPhaseGateUp ? ti.g.a_row0 : ti.g.h_row0) + ti.m_blk * kF8TileRows);
        // gate/up: rows n*128 of the expert in W_gate and in W_up;
        // down: rows n*256 .. n*256 + 255 of the expert in W_down.
        const int w_row = ti.g.index * a.w_rows[kind] + ti.n_blk * (PHASE == kPhaseGateUp ? kBNGateUp : kBNDown);
        const int nkb = a.k_blocks[kind];
        for (int kb = 0; kb < nkb; ++kb) {
          if (!ptx::mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, a.err)) {
            aborted = true;
            break;
          }
          const uint32_t dA = sA + stage * kABytes, dB = sB + stage * kBBytes;
          ptx::mbar_arrive_expect_tx(full_bar(stage), bytes);
          ptx::tma_load_2d(dA, mA, full_bar(stage), kb * kKq, a_row);
          ptx::tma_load_2d(dB, mW, full_bar(stage), kb * kKq, w_row);
          if (PHASE == kPhaseGateUp) ptx::tma_load_2d(dB + kBBytes / 2, mU, full_bar(stage), kb * kKq, w_row);
          else ptx::tma_load_2d(dB + kBBytes / 2, mW, full_bar(stage), kb * kKq, w_row + kWRows / 2);
          ++issued;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (aborted) {
        // Wait for the copies still in flight into the ring (the last kStages issues).
        const uint32_t n = issued < (uint32_t)kStages ? issued : (uint32_t)kStages;
        for (uint32_t j = issued - n; j < issued; ++j)
          wait_raw(full_bar((int)(j % kStages)), (j / kStages) & 1u, kDrainTimeoutNs);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool aborted = false;
      for (int tile = blockIdx.x; tile < total && !aborted; tile += gridDim.x) {
        const int nkb = a.k_blocks[decode_tile(tile, a).g.kind];
        if (!ptx::mbar_wait(tempty_bar(acc), acc_phase ^ 1u, abort_flag, a.err)) break;
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)acc * kAccCols;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!ptx::mbar_wait(full_bar(stage), phase, abort_flag, a.err)) {
            aborted = true;
            break;
          }
          ptx::tc_fence_after();
          const uint64_t adesc = ptx::smem_desc_sw128(sA + stage * kABytes);
          const uint64_t bdesc = ptx::smem_desc_sw128(sB + stage * kBBytes);
#pragma unroll
          for (int k = 0; k < kKq / 32; ++k)
            ptx::mma_f8(d_tmem, adesc + 2u * k, bdesc + 2u * k, kIdesc, (kb | k) != 0 ? 1u : 0u);
          ptx::mma_commit(empty_bar(stage));
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (aborted) break;
        ptx::mma_commit(tfull_bar(acc));
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // Every MMA this thread issued must finish before TMEM is released.
      ptx::mma_commit(drain_bar);
      wait_raw(drain_bar, 0, kWaitTimeoutNs);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    // Lane pair (2t, 2t+1) of the warp holds token t's hi and lo products;
    // after the pair sum the even lane finishes columns 0..15 of each 32-column
    // chunk and the odd lane columns 16..31.
    const int quad = warp & 3;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const int odd = lane & 1;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool over = false;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      const TileInfo ti = decode_tile(tile, a);
      const int kind = ti.g.kind;
      if (!ptx::mbar_wait(tfull_bar(acc), acc_phase, abort_flag, a.err)) break;
      ptx::tc_fence_after();
      const uint32_t tacc = tmem_base + lane_off + (uint32_t)acc * kAccCols;
      const int r_local = ti.m_blk * kF8TileRows + ((quad * 32 + lane) >> 1);  // token row in the group
      const bool row_ok = r_local < ti.g.rows;
      const int64_t a_idx = (int64_t)(PHASE == kPhaseGateUp ? ti.g.a_row0 : ti.g.h_row0) + (row_ok ? r_local : 0);
      const float sx = row_ok ? __ldg(a.a_scale[kind] + a_idx) : 0.f;
      const int64_t wbase = (int64_t)ti.g.index * a.w_rows[kind];
      if (PHASE == kPhaseGateUp) {
        const int n_ext = a.n_ext[kind];
        __half* hrow = reinterpret_cast<__half*>(a.h[kind]) + (int64_t)(ti.g.h_row0 + (row_ok ? r_local : 0)) * a.ldh[kind];
        const float* sgp = a.w_scale[kind] + wbase;
        const float* sup = a.u_scale[kind] + wbase;
#pragma unroll 1
        for (int c = 0; c < kBNGateUp / 32; ++c) {
          uint32_t gv[32], uv[32];
          ptx::tmem_ld_32x32b_x32(tacc + c * 32, gv);
          ptx::tmem_ld_32x32b_x32(tacc + kBNGateUp + c * 32, uv);
          ptx::tmem_wait_ld();
          float g[16], u[16];
          pair_sum16(gv, odd, g);
          pair_sum16(uv, odd, u);
          const int f0 = ti.n_blk * kBNGateUp + c * 32 + odd * 16;
          if (row_ok && f0 < n_ext) {
            uint32_t p[8];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const float4 sg = __ldg(reinterpret_cast<const float4*>(sgp + f0 + 4 * q));
              const float4 su = __ldg(reinterpret_cast<const float4*>(sup + f0 + 4 * q));
              const float sgv[4] = {sg.x, sg.y, sg.z, sg.w}, suv[4] = {su.x, su.y, su.z, su.w};
              float hv[4];
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const float gg = g[4 * q + j] * sx * sgv[j];
                const float uu = u[4 * q + j] * sx * suv[j];
                hv[j] = silu_f(gg) * uu;
                over |= fabsf(hv[j]) >= 65520.f;
              }
              p[2 * q] = pack_f16x2(hv[0], hv[1]);
              p[2 * q + 1] = pack_f16x2(hv[2], hv[3]);
            }
            *reinterpret_cast<uint4*>(hrow + f0) = make_uint4(p[0], p[1], p[2], p[3]);
            *reinterpret_cast<uint4*>(hrow + f0 + 8) = make_uint4(p[4], p[5], p[6], p[7]);
          }
        }
      } else {
        const float* sdp = a.w_scale[kind] + wbase;
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
        const float ws = w * sx;
#pragma unroll 1
        for (int c = 0; c < kBNDown / 32; ++c) {
          uint32_t yv[32];
          ptx::tmem_ld_32x32b_x32(tacc + c * 32, yv);
          ptx::tmem_wait_ld();
          float y[16];
          pair_sum16(yv, odd, y);
          const int n0 = ti.n_blk * kBNDown + c * 32 + odd * 16;
          if (row_ok && n0 < a.d) {
            if (EPI == kEpiScatter) {
              float* orow = a.out_acc + t * a.d + n0;
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const float4 sd = __ldg(reinterpret_cast<const float4*>(sdp + n0 + 4 * q));
                atomicAdd(reinterpret_cast<float4*>(orow + 4 * q),
                          make_float4(ws * sd.x * y[4 * q], ws * sd.y * y[4 * q + 1], ws * sd.z * y[4 * q + 2],
                                      ws * sd.w * y[4 * q + 3]));
              }
            } else {
              __nv_bfloat16* yrow = a.y + (int64_t)(ti.g.h_row0 + r_local) * a.d + n0;
              uint32_t p[8];
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const float4 sd = __ldg(reinterpret_cast<const float4*>(sdp + n0 + 4 * q));
                p[2 * q] = pack_bf16x2(sx * sd.x * y[4 * q], sx * sd.y * y[4 * q + 1]);
                p[2 * q + 1] = pack_bf16x2(sx * sd.z * y[4 * q + 2], sx * sd.w * y[4 * q + 3]);
              }
              *reinterpret_cast<uint4*>(yrow) = make_uint4(p[0], p[1], p[2], p[3]);
              *reinterpret_cast<uint4*>(yrow + 8) = make_uint4(p[4], p[5], p[6], p[7]);
            }
          }
        }
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(tempty_bar(acc));
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (over) atomicOr(a.err, kErrRange);
  }

  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, kTmemCols);
  }
}

template <int PHASE, int EPI>
cudaError_t launch_t(const F8Maps& m, const GemmArgs& a, int64_t tile_bound, cudaStream_t s) {
  auto kern = grouped_gemm_fp8_kernel<PHASE, EPI>;
  static std::atomic<uint64_t> configured{0};  // per device: the shared-memory opt-in
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(configured.load() & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit);
  }
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  int64_t grid = sms;
  if (tile_bound < grid) grid = tile_bound < 1 ? 1 : tile_bound;
  kern<<<(unsigned)grid, kThreads, kSmem, s>>>(m, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_grouped_gemm_fp8(int phase, int epilogue, const F8Maps& maps, const GemmArgs& a,
                                    int64_t tile_bound, cudaStream_t s) {
  if (phase == kPhaseGateUp) return launch_t<kPhaseGateUp, kEpiSwiGLU>(maps, a, tile_bound, s);
  if (epilogue == kEpiScatter) return launch_t<kPhaseDown, kEpiScatter>(maps, a, tile_bound, s);
  return launch_t<kPhaseDown, kEpiStoreY>(maps, a, tile_bound, s);
}

}  // namespace moe
