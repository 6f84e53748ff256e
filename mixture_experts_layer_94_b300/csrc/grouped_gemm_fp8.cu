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

#include <cuda_fp8.h>

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

// The epilogue warps' loop over this CTA's tiles (warps 2-5, 128 threads):
// tfull_bar(i) / tempty_bar(i) are the accumulator buffers' barriers.
template <int PHASE, int EPI>
__device__ __forceinline__ void epilogue_loop(const GemmArgs& a, int total, uint32_t tmem_base, uint32_t tbar0,
                                              volatile int* abort_flag, int warp, int lane) {
  auto tfull_bar = [&](int i) { return tbar0 + 8u * i; };
  auto tempty_bar = [&](int i) { return tbar0 + 8u * (2 + i); };
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
            __nv_bfloat16* yrow = (kind && a.y_sh ? a.y_sh : a.y) + (int64_t)(ti.g.h_row0 + r_local) * a.d + n0;
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

template <int PHASE, int EPI>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_fp8_kernel(const __grid_constant__ F8Maps maps, const GemmArgs a) {
  pdl_trigger();
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
  // The setup above touches shared memory, TMEM and kernel parameters only;
  // from here on the previous kernel's results are read.
  pdl_wait();
  const int total = __ldg(a.tile_start + a.G);

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
    epilogue_loop<PHASE, EPI>(a, total, tmem_base, tfull_bar(0), abort_flag, warp, lane);
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
  if (const cudaError_t le_ = launch(kern, (unsigned)grid, kThreads, kSmem, s, m, a); le_ != cudaSuccess) return le_;
  return cudaSuccess;
}

// ============================================================================
// MXFP4 experts. The expert matrices are E2M1 codes (two per byte, the even
// element in the low nibble) with one E8M0 power-of-two scale per 32 elements
// of a row (OCP microscaling), the format gpt-oss ships its experts in ("AI
// Infrastructure series, Part 12 of 24", "How do you serve an MoE model on
// your own GPUs?"). They reach the same 8-bit MMAs as FP8 experts:
//  * TMA streams the packed codes (64 bytes = 128 elements of a row per
//    stage, 64-byte swizzle) into a 4-stage ring; half the bytes of FP8.
//  * A preparation pass (mx_prep_kernel) gives every weight row a reference
//    exponent E_row (its largest block exponent - 6) and every block the
//    index of its 8-entry table: E_block - E_row, stored K-block-major so
//    that TMA brings a stage's 256 rows x 4 block indices (1 KB) into the
//    code slot beside the codes.
//  * Converter warps (one thread per weight row) rewrite each 32-element
//    block as E4M3 codes of e2m1 * 2^(E_block - E_row): every block within
//    14 binades of the row's largest converts exactly (E4M3 spans 2^-9 ..
//    448; an E2M1 value has two significant bits); smaller blocks round to
//    nearest. The block's table (its eight magnitudes as E4M3 codes, built
//    once per CTA in shared memory) turns four codes into four bytes with
//    one byte permute; a second permute adds the signs. The E4M3 rows go
//    into a ring in the 128-byte-swizzled K-major layout the MMA reads.
//  * MMA and epilogue as for FP8 experts, with 2^(E_row - 127) as the weight
//    row's scale.
// Warps (480 threads): 0 TMA producer of the codes, 1 MMA, 2-5 epilogue,
// 6-13 converters (two groups of four warps taking alternate stages, so that
// one group converts while the other waits), 14 TMA producer of the token
// rows.

constexpr int kMxConvWarps = 8;
constexpr int kMxGroupWarps = kMxConvWarps / 2;  // converter warps per stage
constexpr int kMxConv0 = 192;
constexpr int kMxXWarp = kMxConv0 / 32 + kMxConvWarps;
constexpr int kMxThreads = (kMxXWarp + 1) * 32;
constexpr int kMxXStages = 3;
constexpr int kMxRStages = 4;  // even: a code slot is always refilled for the same converter group
constexpr int kMxWStages = 3;
constexpr uint32_t kMxRawBytes = (uint32_t)kWRows * (kKq / 2);  // 256 rows x 64 code bytes = 16 KB
constexpr uint32_t kMxIdxBytes = (uint32_t)kWRows * 4;           // 256 rows x 4 block indices
constexpr uint32_t kMxSlotBytes = kMxRawBytes + kMxIdxBytes;      // a multiple of the 512-byte swizzle span
constexpr int kMxTabEntries = 32;                                 // indices 0 .. kMxIdxBias + 6, padded
constexpr int kMxNumBars = 2 * (kMxXStages + kMxRStages + kMxWStages) + 5;
constexpr size_t kMxBarrierBytes = 512;
constexpr size_t kMxSmem = 1024 + (size_t)kMxXStages * kABytes + (size_t)kMxWStages * kBBytes +
                           (size_t)kMxRStages * kMxSlotBytes + 8 * kMxTabEntries + kMxBarrierBytes;
static_assert(8 * kMxNumBars + 8 <= kMxBarrierBytes, "barrier area");
static_assert(kMxSlotBytes % 512 == 0, "code slots keep the 64-byte swizzle's alignment");
static_assert(kMxSmem <= 232448, "shared memory per CTA");
// The code ring's parity waits stay unambiguous because a slot is refilled
// for the group that emptied it (an even ring). The E4M3 ring alternates
// between the groups; a group reaches stage n only after the MMA consumed
// stage n - 3, so its empty-slot wait never skips a phase.
static_assert(kMxRStages % 2 == 0, "code slots stay with one converter group");

// The eight E4M3 codes (as two table words) of the E2M1 magnitudes 0, 0.5,
// 1, 1.5, 2, 3, 4, 6 times 2^k, rounded to nearest (exact for -8 <= k <= 6).
__device__ __forceinline__ uint2 e2m1_table(int k) {
  const float f = exp2f((float)k);
  uint32_t b[8];
  const float mag[8] = {0.f, 0.5f, 1.f, 1.5f, 2.f, 3.f, 4.f, 6.f};
#pragma unroll
  for (int i = 0; i < 8; ++i) b[i] = (uint32_t)__nv_cvt_float_to_fp8(mag[i] * f, __NV_SATFINITE, __NV_E4M3);
  return make_uint2(b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24), b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24));
}

// prmt in its default mode: byte i of the result is source byte (c_i & 7) of
// {b, a}, or, when bit 3 of selector nibble c_i is set, that byte's sign bit
// replicated over all eight bits. Only c's low 16 bits are read.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// Eight E2M1 codes (element i in nibble i of w) -> eight E4M3 codes (elements
// 0-3 in lo, 4-7 in hi, element i in byte i % 4). The magnitude comes from
// the block's table (the code's three low bits select the byte). The sign:
// a permute of 0x80 bytes by the raw codes gives 0x80 for a positive code and
// 0xff (the sign replicated) for a negative one, so bit 6 of each byte is the
// sign; shifted left by one and masked it lands on bit 7.
__device__ __forceinline__ void e2m1x8_to_e4m3x8(uint32_t w, uint2 tab, uint32_t& lo, uint32_t& hi) {
  const uint32_t sel = w & 0x77777777u, wh = w >> 16;
  const uint32_t sl = prmt(0x80808080u, 0x80808080u, w), sh = prmt(0x80808080u, 0x80808080u, wh);
  lo = prmt(tab.x, tab.y, sel) | ((sl << 1) & 0x80808080u);
  hi = prmt(tab.x, tab.y, sel >> 16) | ((sh << 1) & 0x80808080u);
}

template <int PHASE, int EPI>
__global__ void __launch_bounds__(kMxThreads, 1)
    grouped_gemm_mx_kernel(const __grid_constant__ F8Maps maps, const GemmArgs a) {
  pdl_trigger();
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw_base + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw_base);
  const uint32_t sX = base;                          // kMxXStages x 16 KB
  const uint32_t sW = sX + kMxXStages * kABytes;     // kMxWStages x 32 KB
  const uint32_t sRaw = sW + kMxWStages * kBBytes;   // kMxRStages x (16 KB codes + 1 KB block indices)
  const uint32_t sTab = sRaw + kMxRStages * kMxSlotBytes;
  const uint32_t sBar = sTab + 8 * kMxTabEntries;
  uint8_t* gW = gbase + (sW - base);
  const uint8_t* gRaw = gbase + (sRaw - base);
  uint2* gTab = reinterpret_cast<uint2*>(gbase + (sTab - base));
  uint8_t* gBar = gbase + (sBar - base);
  auto xfull_bar = [&](int s) { return sBar + 8u * s; };
  auto xempty_bar = [&](int s) { return sBar + 8u * (kMxXStages + s); };
  auto rfull_bar = [&](int s) { return sBar + 8u * (2 * kMxXStages + s); };
  auto rempty_bar = [&](int s) { return sBar + 8u * (2 * kMxXStages + kMxRStages + s); };
  auto wfull_bar = [&](int s) { return sBar + 8u * (2 * (kMxXStages + kMxRStages) + s); };
  auto wempty_bar = [&](int s) { return sBar + 8u * (2 * (kMxXStages + kMxRStages) + kMxWStages + s); };
  constexpr int kT0 = 2 * (kMxXStages + kMxRStages + kMxWStages);
  auto tfull_bar = [&](int i) { return sBar + 8u * (kT0 + i); };
  auto tempty_bar = [&](int i) { return sBar + 8u * (kT0 + 2 + i); };
  const uint32_t drain_bar = sBar + 8u * (kT0 + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gBar + 8 * kMxNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gBar + 8 * kMxNumBars + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kMxXStages; ++s) {
      ptx::mbar_init(xfull_bar(s), 1);
      ptx::mbar_init(xempty_bar(s), 1);
    }
    for (int s = 0; s < kMxRStages; ++s) {
      ptx::mbar_init(rfull_bar(s), 1);
      ptx::mbar_init(rempty_bar(s), kMxGroupWarps);
    }
    for (int s = 0; s < kMxWStages; ++s) {
      ptx::mbar_init(wfull_bar(s), kMxGroupWarps);
      ptx::mbar_init(wempty_bar(s), 1);
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
    ptx::prefetch_tmap(&maps.kw[0]);
    if (PHASE == kPhaseGateUp) {
      ptx::prefetch_tmap(&maps.u[0]);
      ptx::prefetch_tmap(&maps.ku[0]);
    }
  }
  if (threadIdx.x >= kMxConv0 && threadIdx.x < kMxConv0 + kMxTabEntries) {
    const int i = threadIdx.x - kMxConv0;
    gTab[i] = i <= kMxIdxBias + 6 ? e2m1_table(i - kMxIdxBias) : make_uint2(0u, 0u);
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), kTmemCols);
    ptx::tmem_relinquish();
    ptx::tc_fence_before();
  }
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // The setup above touches shared memory, TMEM and kernel parameters only;
  // from here on the previous kernel's results are read.
  pdl_wait();
  const int total = __ldg(a.tile_start + a.G);

  if (warp == 0 || warp == kMxXWarp) {
    // ------------------------------------------------------------ TMA producers
    // warp 0: the packed codes (two 128-row boxes of 64 bytes per stage);
    // warp kMxXWarp: the token rows.
    if (lane == 0) {
      const bool codes = warp == 0;
      const int stages = codes ? kMxRStages : kMxXStages;
      int stage = 0;
      uint32_t phase = 0, issued = 0;
      bool aborted = false;
      for (int tile = blockIdx.x; tile < total && !aborted; tile += gridDim.x) {
        const TileInfo ti = decode_tile(tile, a);
        const int kind = ti.g.kind;
        const int bsel = box_sel(min(kF8TileRows, ti.g.rows - ti.m_blk * kF8TileRows));
        const uint32_t xbytes = (16u << bsel) * kKq;
        const CUtensorMap* mA = &maps.x[kind][bsel];
        const CUtensorMap* mW = &maps.w[kind];
        const CUtensorMap* mU = &maps.u[kind];
        const CUtensorMap* mKW = &maps.kw[kind];
        const CUtensorMap* mKU = &maps.ku[kind];
        const int a_row = 2 * ((PHASE == kPhaseGateUp ? ti.g.a_row0 : ti.g.h_row0) + ti.m_blk * kF8TileRows);
        const int w_row = ti.g.index * a.w_rows[kind] + ti.n_blk * (PHASE == kPhaseGateUp ? kBNGateUp : kBNDown);
        const int nkb = a.k_blocks[kind];
        for (int kb = 0; kb < nkb; ++kb) {
          const uint32_t full = codes ? rfull_bar(stage) : xfull_bar(stage);
          const uint32_t empty = codes ? rempty_bar(stage) : xempty_bar(stage);
          if (!ptx::mbar_wait(empty, phase ^ 1u, abort_flag, a.err)) {
            aborted = true;
            break;
          }
          if (codes) {
            const uint32_t dR = sRaw + stage * kMxSlotBytes, dI = dR + kMxRawBytes;
            ptx::mbar_arrive_expect_tx(full, kMxSlotBytes);
            ptx::tma_load_2d(dR, mW, full, kb * (kKq / 2), w_row);
            ptx::tma_load_2d(dI, mKW, full, w_row, kb);
            if (PHASE == kPhaseGateUp) {
              ptx::tma_load_2d(dR + kMxRawBytes / 2, mU, full, kb * (kKq / 2), w_row);
              ptx::tma_load_2d(dI + kMxIdxBytes / 2, mKU, full, w_row, kb);
            } else {
              ptx::tma_load_2d(dR + kMxRawBytes / 2, mW, full, kb * (kKq / 2), w_row + kWRows / 2);
              ptx::tma_load_2d(dI + kMxIdxBytes / 2, mKW, full, w_row + kWRows / 2, kb);
            }
          } else {
            ptx::mbar_arrive_expect_tx(full, xbytes);
            ptx::tma_load_2d(sX + stage * kABytes, mA, full, kb * kKq, a_row);
          }
          ++issued;
          if (++stage == stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (aborted) {
        const uint32_t n = issued < (uint32_t)stages ? issued : (uint32_t)stages;
        for (uint32_t j = issued - n; j < issued; ++j) {
          const int s = (int)(j % (uint32_t)stages);
          wait_raw(codes ? rfull_bar(s) : xfull_bar(s), (j / (uint32_t)stages) & 1u, kDrainTimeoutNs);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int xs = 0, ws = 0, acc = 0;
      uint32_t xphase = 0, wphase = 0, acc_phase = 0;
      bool aborted = false;
      for (int tile = blockIdx.x; tile < total && !aborted; tile += gridDim.x) {
        const int nkb = a.k_blocks[decode_tile(tile, a).g.kind];
        if (!ptx::mbar_wait(tempty_bar(acc), acc_phase ^ 1u, abort_flag, a.err)) break;
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)acc * kAccCols;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!ptx::mbar_wait(wfull_bar(ws), wphase, abort_flag, a.err) ||
              !ptx::mbar_wait(xfull_bar(xs), xphase, abort_flag, a.err)) {
            aborted = true;
            break;
          }
          ptx::tc_fence_after();
          const uint64_t adesc = ptx::smem_desc_sw128(sX + xs * kABytes);
          const uint64_t bdesc = ptx::smem_desc_sw128(sW + ws * kBBytes);
#pragma unroll
          for (int k = 0; k < kKq / 32; ++k)
            ptx::mma_f8(d_tmem, adesc + 2u * k, bdesc + 2u * k, kIdesc, (kb | k) != 0 ? 1u : 0u);
          ptx::mma_commit(xempty_bar(xs));
          ptx::mma_commit(wempty_bar(ws));
          if (++xs == kMxXStages) {
            xs = 0;
            xphase ^= 1u;
          }
          if (++ws == kMxWStages) {
            ws = 0;
            wphase ^= 1u;
          }
        }
        if (aborted) break;
        ptx::mma_commit(tfull_bar(acc));
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      ptx::mma_commit(drain_bar);
      wait_raw(drain_bar, 0, kWaitTimeoutNs);
    }
    __syncwarp();
  } else if (threadIdx.x >= kMxConv0) {
    // ------------------------------------------------------------ converters
    // Group grp takes the stages n with n % 2 == grp; its thread t converts
    // weight rows t and t + 128 of the tile (W_gate and W_up row t, or W_down
    // rows t and t + 128). Per row it reads the 64 code bytes (chunk c of the
    // 64-byte-swizzled box row at c ^ ((R >> 1) & 3)) and the four block
    // indices, and writes the row's 128 E4M3 codes: chunk j at j ^ (R & 7) of
    // the 128-byte-swizzled weight tile.
    const int grp = (threadIdx.x - kMxConv0) / (32 * kMxGroupWarps);
    const int t = (threadIdx.x - kMxConv0) % (32 * kMxGroupWarps);
    int rs = 0, ws = 0, n = 0;
    uint32_t rphase = 0, wphase = 0;
    bool aborted = false;
    for (int tile = blockIdx.x; tile < total && !aborted; tile += gridDim.x) {
      const int nkb = a.k_blocks[decode_tile(tile, a).g.kind];
      for (int kb = 0; kb < nkb; ++kb, ++n) {
        if ((n & 1) == grp) {
          if (!ptx::mbar_wait(rfull_bar(rs), rphase, abort_flag, a.err) ||
              !ptx::mbar_wait(wempty_bar(ws), wphase ^ 1u, abort_flag, a.err)) {
            aborted = true;
            break;
          }
          const uint8_t* slot = gRaw + rs * kMxSlotBytes;
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const int R = t + 128 * half;
            const uint4* src = reinterpret_cast<const uint4*>(slot + R * (kKq / 2));
            const int rsw = (R >> 1) & 3;
            uint4 v[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) v[c] = src[c ^ rsw];
            const uint32_t kidx = reinterpret_cast<const uint32_t*>(slot + kMxRawBytes)[R];
            uint4* dst = reinterpret_cast<uint4*>(gW + ws * kBBytes + R * kKq);
            const int wsw = R & 7;
            // Chunk c (16 code bytes = 32 elements) is exactly block 4*kb + c.
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const uint2 tab = gTab[(kidx >> (8 * c)) & (kMxTabEntries - 1)];
              uint32_t r8[8];
              e2m1x8_to_e4m3x8(v[c].x, tab, r8[0], r8[1]);
              e2m1x8_to_e4m3x8(v[c].y, tab, r8[2], r8[3]);
              e2m1x8_to_e4m3x8(v[c].z, tab, r8[4], r8[5]);
              e2m1x8_to_e4m3x8(v[c].w, tab, r8[6], r8[7]);
              dst[(2 * c) ^ wsw] = make_uint4(r8[0], r8[1], r8[2], r8[3]);
              dst[(2 * c + 1) ^ wsw] = make_uint4(r8[4], r8[5], r8[6], r8[7]);
            }
          }
          // Every lane's loads of the code slot have been consumed above.
          __syncwarp();
          if ((threadIdx.x & 31) == 0) ptx::mbar_arrive(rempty_bar(rs));
          ptx::fence_proxy_async_shared();  // generic-proxy writes -> the MMA's async-proxy reads
          __syncwarp();
          if ((threadIdx.x & 31) == 0) ptx::mbar_arrive(wfull_bar(ws));
        }
        if (++rs == kMxRStages) {
          rs = 0;
          rphase ^= 1u;
        }
        if (++ws == kMxWStages) {
          ws = 0;
          wphase ^= 1u;
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    epilogue_loop<PHASE, EPI>(a, total, tmem_base, tfull_bar(0), abort_flag, warp, lane);
  }

  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, kTmemCols);
  }
}

// The preparation of one MXFP4 weight matrix (see launch_mx_prep). A block
// takes kMxPrepRows consecutive rows, whose block scales are one contiguous
// span of global memory: the block copies it with 16-byte loads, all in
// flight at once, into shared memory at a row pitch of an odd number of
// words, so that one thread per row then reads its row without bank
// conflicts; each thread finds its row's reference exponent and writes the
// row's index words K-block-major (consecutive threads store consecutive
// words). Row groups whose experts have no routed rows are skipped.
constexpr int kMxPrepRows = 128;

__device__ __forceinline__ int mx_prep_pitch(int nblk) { return ((nblk + 3) / 4) | 1; }  // words

__global__ void __launch_bounds__(kMxPrepRows) mx_prep_kernel(const uint8_t* __restrict__ bscale, int64_t rows,
                                                              int32_t rows_per_expert, int32_t nblk,
                                                              int32_t kblocks, const int32_t* __restrict__ offsets,
                                                              float* __restrict__ row_scale,
                                                              uint32_t* __restrict__ kidx) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ uint32_t st[];  // [kMxPrepRows][pitch] words
  const int pitch = mx_prep_pitch(nblk);
  const int t = threadIdx.x;
  const bool vec = (reinterpret_cast<uintptr_t>(bscale) & 15u) == 0;
  for (int64_t r0 = (int64_t)blockIdx.x * kMxPrepRows; r0 < rows; r0 += (int64_t)gridDim.x * kMxPrepRows) {
    const int nrows = (int)min((int64_t)kMxPrepRows, rows - r0);
    if (offsets) {  // a group spans the experts of its first and last rows (and any between)
      const int64_t e0 = r0 / rows_per_expert, e1 = (r0 + nrows - 1) / rows_per_expert;
      if (__ldg(offsets + e1 + 1) == __ldg(offsets + e0)) continue;
    }
    const uint8_t* span = bscale + r0 * (int64_t)nblk;
    const int bytes = nrows * nblk;  // a multiple of 16 (rows come in multiples of 32)
    uint8_t* sb = reinterpret_cast<uint8_t*>(st);
    if (vec) {
      constexpr int kUnroll = 4;
      for (int g0 = t; g0 < bytes / 16; g0 += kUnroll * kMxPrepRows) {
        uint4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int g = g0 + u * kMxPrepRows;
          if (g < bytes / 16) v[u] = __ldg(reinterpret_cast<const uint4*>(span) + g);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int g = g0 + u * kMxPrepRows;
          if (g >= bytes / 16) break;
          int row = (16 * g) / nblk, col = 16 * g - row * nblk;
          const uint32_t w4[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
          if ((nblk & 3) == 0) {  // words never straddle two rows
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              st[row * pitch + col / 4] = w4[j];
              col += 4;
              if (col == nblk) {
                col = 0;
                ++row;
              }
            }
          } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              sb[4 * row * pitch + col] = (uint8_t)(w4[j >> 2] >> (8 * (j & 3)));
              if (++col == nblk) {
                col = 0;
                ++row;
              }
            }
          }
        }
      }
    } else {
      for (int o = t; o < bytes; o += kMxPrepRows) {
        const int row = o / nblk;
        sb[4 * row * pitch + (o - row * nblk)] = __ldg(span + o);
      }
    }
    __syncthreads();
    const int64_t r = r0 + t;
    bool live = t < nrows;
    if (live && offsets) {
      const int64_t e = r / rows_per_expert;
      live = __ldg(offsets + e + 1) != __ldg(offsets + e);
    }
    if (live) {
      const uint32_t* row = st + t * pitch;
      int m = 0;
      for (int kb = 0; kb < kblocks; ++kb) {
        const uint32_t w = row[kb];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int v = (int)((w >> (8 * c)) & 255u);
          if (4 * kb + c < nblk && v != 255) m = max(m, v);
        }
      }
      const int e_row = min(max(m - 6, 1), 254);
      row_scale[r] = __uint_as_float((uint32_t)e_row << 23);
      for (int kb = 0; kb < kblocks; ++kb) {
        const uint32_t w = row[kb];
        uint32_t o = 0;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int k = min(max((int)((w >> (8 * c)) & 255u) - e_row, -kMxIdxBias), 6) + kMxIdxBias;
          if (4 * kb + c < nblk) o |= (uint32_t)k << (8 * c);
        }
        kidx[(int64_t)kb * rows + r] = o;
      }
    }
    __syncthreads();
  }
}

template <int PHASE, int EPI>
cudaError_t launch_mx(const F8Maps& m, const GemmArgs& a, int64_t tile_bound, cudaStream_t s) {
  auto kern = grouped_gemm_mx_kernel<PHASE, EPI>;
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(configured.load() & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMxSmem);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit);
  }
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  int64_t grid = sms;
  if (tile_bound < grid) grid = tile_bound < 1 ? 1 : tile_bound;
  if (const cudaError_t le_ = launch(kern, (unsigned)grid, kMxThreads, kMxSmem, s, m, a); le_ != cudaSuccess) return le_;
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_grouped_gemm_fp8(int phase, int epilogue, const F8Maps& maps, const GemmArgs& a,
                                    int64_t tile_bound, cudaStream_t s) {
  if (phase == kPhaseGateUp) return launch_t<kPhaseGateUp, kEpiSwiGLU>(maps, a, tile_bound, s);
  if (epilogue == kEpiScatter) return launch_t<kPhaseDown, kEpiScatter>(maps, a, tile_bound, s);
  return launch_t<kPhaseDown, kEpiStoreY>(maps, a, tile_bound, s);
}

cudaError_t launch_grouped_gemm_mxfp4(int phase, int epilogue, const F8Maps& maps, const GemmArgs& a,
                                      int64_t tile_bound, cudaStream_t s) {
  if (phase == kPhaseGateUp) return launch_mx<kPhaseGateUp, kEpiSwiGLU>(maps, a, tile_bound, s);
  if (epilogue == kEpiScatter) return launch_mx<kPhaseDown, kEpiScatter>(maps, a, tile_bound, s);
  return launch_mx<kPhaseDown, kEpiStoreY>(maps, a, tile_bound, s);
}

cudaError_t launch_mx_prep(const uint8_t* bscale, int64_t rows, int32_t rows_per_expert, int32_t nblk,
                           int32_t kblocks, const int32_t* offsets, float* row_scale, uint32_t* kidx,
                           cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  const size_t smem = (size_t)kMxPrepRows * (size_t)((((nblk + 3) / 4) | 1)) * 4;
  if (smem > kMxPrepMaxSmem) return cudaErrorInvalidValue;
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (smem > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(mx_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  const int64_t want = (rows + kMxPrepRows - 1) / kMxPrepRows;
  const unsigned grid = (unsigned)(want < (int64_t)sms * 16 ? want : (int64_t)sms * 16);
  return launch(mx_prep_kernel, grid, kMxPrepRows, smem, s, bscale, rows, rows_per_expert, nblk, kblocks, offsets,
                row_scale, kidx);
}

}  // namespace moe
