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
//  * The weights are the MMA's A operand (M = 128 weight rows) and the token
//    rows are its B operand (N = 16, 32, 64 or 128). One tile is two 128-row
//    weight sub-tiles against up to 128 token rows of one expert group. The
//    sub-tiles are the gate and up rows of the same 128 FFN units, or 256
//    rows of W_down. With a few tokens per expert (decode) the tensor work
//    per weight byte then scales with the token count rather than with a
//    fixed 128-row tile, so the kernel stays bound by the weight stream.
//  * TMA brings one fp16 activation box (128-byte swizzle; 16, 32, 64 or 128
//    rows, the smallest that holds the tile's rows) and the raw code boxes
//    (no swizzle, 64 codes per row) into a 4-stage ring.
//  * Four converter warps write the codes as fp16 into a 2-stage ring, in the
//    128-byte-swizzled K-major layout the MMA reads. An E4M3 code s.eeee.mmm
//    placed as the fp16 bit pattern s.0eeee.mmm0000000 is exactly 2^-8 times
//    its value. Normal codes map to normal fp16 numbers with the exponent
//    re-biased by 8, and subnormal codes map to fp16 subnormals with the same
//    shift. So the conversion is a byte permute, a shift and two masks per
//    pair of codes, and it never rounds. NaN codes are not supported.
//  * kind::f16 MMA: fp16 x fp16 -> fp32 accumulators in TMEM. Both operands
//    have one type.
//  * Epilogue: accumulator x (2^8 x the weight row's scale). Gate/up applies
//    SiLU(g) * u and writes h as fp16. Down either scatter-adds w * y into
//    the token's fp32 output row or stores y as bf16.
//  The activations are fp16 on this path. A bf16 value is exact in fp16 when
//  2^-14 <= |x| < 65520. Smaller magnitudes keep an absolute error below
//  2^-25. Larger ones overflow and set kErrRange in the error word.
//
// Warps (320 threads, one CTA per SM, persistent over the tiles):
//   0     TMA producer           1    TMEM allocation, MMA issue
//   2-5   epilogue (warp w reads TMEM lanes 32*(w%4)..+31: one weight row per thread)
//   6-9   FP8 -> fp16 converters
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

constexpr int kThreads = 320;
constexpr int kConvThread0 = 192;  // first converter thread (warp 6)
constexpr int kStages = 4;         // TMA ring: activation box + code boxes
constexpr int kWStages = 2;        // converted fp16 weight ring
constexpr int kWRows = 128;        // weight rows per MMA (M)
constexpr uint32_t kXBytes = 128u * kBK * 2u;          // largest activation box: 128 rows x 128 B
constexpr uint32_t kRawBytes = 2u * kWRows * kBK;      // two sub-tiles x 128 rows x 64 codes = 16 KB
constexpr uint32_t kWBytes = 2u * kWRows * kBK * 2u;   // the same rows in fp16 = 32 KB
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCols = 256;  // one accumulator: two sub-tiles x up to 128 token columns
constexpr uint64_t kDrainTimeoutNs = 50000000ull;
constexpr int kNumBars = 2 * kStages + 2 * kWStages + 5;
constexpr size_t kSmem =
    1024 /*alignment slack*/ + (size_t)kStages * (kXBytes + kRawBytes) + (size_t)kWStages * kWBytes + 256;
static_assert(8 * kNumBars + 8 <= 256, "barrier area");

// Two E4M3 codes held in bits 8..15 and 24..31 (zeros elsewhere) -> two fp16
// values 2^-8 times theirs: keep the signs, move the 7 magnitude bits down one.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2_scaled(uint32_t x) {
  return (x & 0x80008000u) | ((x >> 1) & 0x3F803F80u);
}

// 16 codes (in K order) -> 16 fp16 values as two 16-byte chunks.
__device__ __forceinline__ void convert16(const uint4 v, uint4& lo, uint4& hi) {
  lo.x = e4m3x2_to_f16x2_scaled(__byte_perm(v.x, 0u, 0x1404));
  lo.y = e4m3x2_to_f16x2_scaled(__byte_perm(v.x, 0u, 0x3424));
  lo.z = e4m3x2_to_f16x2_scaled(__byte_perm(v.y, 0u, 0x1404));
  lo.w = e4m3x2_to_f16x2_scaled(__byte_perm(v.y, 0u, 0x3424));
  hi.x = e4m3x2_to_f16x2_scaled(__byte_perm(v.z, 0u, 0x1404));
  hi.y = e4m3x2_to_f16x2_scaled(__byte_perm(v.z, 0u, 0x3424));
  hi.z = e4m3x2_to_f16x2_scaled(__byte_perm(v.w, 0u, 0x1404));
  hi.w = e4m3x2_to_f16x2_scaled(__byte_perm(v.w, 0u, 0x3424));
}

// Activation box for a tile with n token rows: 16 << box_sel(n) rows.
__device__ __forceinline__ int box_sel(int n) { return n <= 16 ? 0 : (n <= 32 ? 1 : (n <= 64 ? 2 : 3)); }

__device__ __forceinline__ int tile_rows_valid(const TileInfo& ti) {
  return min(kBM, ti.g.rows - ti.m_blk * kBM);
}

template <int PHASE, int EPI>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_fp8_kernel(const __grid_constant__ F8Maps maps, const GemmArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw_base + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw_base);
  const uint32_t sX = base;                                 // kStages x 16 KB
  const uint32_t sRaw = sX + kStages * kXBytes;             // kStages x 16 KB
  const uint32_t sW = sRaw + kStages * kRawBytes;           // kWStages x 32 KB
  const uint32_t sBar = sW + kWStages * kWBytes;
  const uint8_t* gRaw = gbase + kStages * kXBytes;
  uint8_t* gW = gbase + kStages * (kXBytes + kRawBytes);
  uint8_t* gBar = gW + kWStages * kWBytes;
  auto full_bar = [&](int s) { return sBar + 8u * s; };
  auto empty_bar = [&](int s) { return sBar + 8u * (kStages + s); };
  auto wfull_bar = [&](int s) { return sBar + 8u * (2 * kStages + s); };
  auto wempty_bar = [&](int s) { return sBar + 8u * (2 * kStages + kWStages + s); };
  auto tfull_bar = [&](int i) { return sBar + 8u * (2 * kStages + 2 * kWStages + i); };
  auto tempty_bar = [&](int i) { return sBar + 8u * (2 * kStages + 2 * kWStages + 2 + i); };
  const uint32_t drain_bar = sBar + 8u * (2 * kStages + 2 * kWStages + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gBar + 8 * kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gBar + 8 * kNumBars + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int total = __ldg(a.tile_start + a.G);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(full_bar(s), 1);
      ptx::mbar_init(empty_bar(s), 1);
    }
    for (int s = 0; s < kWStages; ++s) {
      ptx::mbar_init(wfull_bar(s), 4);  // one arrival per converter warp
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
    ptx::prefetch_tmap(&maps.x[0][kF8XBoxes - 1]);
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
        const int bsel = box_sel(tile_rows_valid(ti));
        const uint32_t bytes = ((16u << bsel) * kBK * 2u) + kRawBytes;
        const CUtensorMap* mX = &maps.x[kind][bsel];
        const CUtensorMap* mW = &maps.w[kind];
        const CUtensorMap* mU = &maps.u[kind];
        const int x_row = (PHASE == kPhaseGateUp ? ti.g.a_row0 : ti.g.h_row0) + ti.m_blk * kBM;
        // gate/up: rows n*128 of the expert in W_gate and in W_up;
        // down: rows n*256 and n*256 + 128 of the expert in W_down.
        const int w_row = ti.g.index * a.w_rows[kind] + ti.n_blk * (PHASE == kPhaseGateUp ? kWRows : 2 * kWRows);
        const int nkb = a.k_blocks[kind];
        for (int kb = 0; kb < nkb; ++kb) {
          if (!ptx::mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, a.err)) {
            aborted = true;
            break;
          }
          const uint32_t dRaw = sRaw + stage * kRawBytes;
          ptx::mbar_arrive_expect_tx(full_bar(stage), bytes);
          ptx::tma_load_2d(sX + stage * kXBytes, mX, full_bar(stage), kb * kBK, x_row);
          ptx::tma_load_2d(dRaw, mW, full_bar(stage), kb * kBK, w_row);
          if (PHASE == kPhaseGateUp)
            ptx::tma_load_2d(dRaw + kRawBytes / 2, mU, full_bar(stage), kb * kBK, w_row);
          else
            ptx::tma_load_2d(dRaw + kRawBytes / 2, mW, full_bar(stage), kb * kBK, w_row + kWRows);
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
          wait_raw(full_bar(j % kStages), (j / kStages) & 1u, kDrainTimeoutNs);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0, ws = 0, acc = 0;
      uint32_t phase = 0, wphase = 0, acc_phase = 0;
      bool aborted = false;
      for (int tile = blockIdx.x; tile < total && !aborted; tile += gridDim.x) {
        const TileInfo ti = decode_tile(tile, a);
        const uint32_t idesc = ptx::idesc_f16_f32(kWRows, 16 << box_sel(tile_rows_valid(ti)));
        const int nkb = a.k_blocks[ti.g.kind];
        if (!ptx::mbar_wait(tempty_bar(acc), acc_phase ^ 1u, abort_flag, a.err)) break;
        ptx::tc_fence_after();
        const uint32_t d0 = tmem_base + (uint32_t)acc * kAccCols;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!ptx::mbar_wait(full_bar(stage), phase, abort_flag, a.err) ||
              !ptx::mbar_wait(wfull_bar(ws), wphase, abort_flag, a.err)) {
            aborted = true;
            break;
          }
          ptx::tc_fence_after();
          const uint64_t a0 = ptx::smem_desc_sw128(sW + ws * kWBytes);
          const uint64_t a1 = ptx::smem_desc_sw128(sW + ws * kWBytes + kWBytes / 2);
          const uint64_t b = ptx::smem_desc_sw128(sX + stage * kXBytes);
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            const uint32_t accum = (kb | k) != 0 ? 1u : 0u;
            ptx::mma_f16(d0, a0 + 2u * k, b + 2u * k, idesc, accum);
            ptx::mma_f16(d0 + kWRows, a1 + 2u * k, b + 2u * k, idesc, accum);
          }
          ptx::mma_commit(empty_bar(stage));
          ptx::mma_commit(wempty_bar(ws));
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
          if (++ws == kWStages) {
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
      // Every MMA this thread issued must finish before TMEM is released.
      ptx::mma_commit(drain_bar);
      wait_raw(drain_bar, 0, kWaitTimeoutNs);
    }
    __syncwarp();
  } else if (threadIdx.x >= kConvThread0) {
    // ------------------------------------------------------------ converters
    // Thread ct handles 16-code quarters i = ct, ct + 128, ..., of the 256
    // code rows: row r = i / 4 (64 codes), quarter q = i % 4 -> fp16 chunks
    // 2q and 2q+1 of the 128-byte row, placed at chunk ^ (r % 8) (the
    // 128-byte swizzle the MMA descriptor expects; the ring is 1024-aligned).
    const int ct = threadIdx.x - kConvThread0;
    int stage = 0, ws = 0;
    uint32_t phase = 0, wphase = 0;
    bool aborted = false;
    for (int tile = blockIdx.x; tile < total && !aborted; tile += gridDim.x) {
      const int nkb = a.k_blocks[decode_tile(tile, a).g.kind];
      for (int kb = 0; kb < nkb; ++kb) {
        if (!ptx::mbar_wait(full_bar(stage), phase, abort_flag, a.err) ||
            !ptx::mbar_wait(wempty_bar(ws), wphase ^ 1u, abort_flag, a.err)) {
          aborted = true;
          break;
        }
        const uint8_t* src = gRaw + stage * kRawBytes;
        uint8_t* dst = gW + ws * kWBytes;
#pragma unroll
        for (int it = 0; it < (int)(kRawBytes / 16) / 128; ++it) {
          const int i = it * 128 + ct;
          const int r = i >> 2, q = i & 3, sw = r & 7;
          const uint4 v = *reinterpret_cast<const uint4*>(src + r * kBK + q * 16);
          uint4 lo, hi;
          convert16(v, lo, hi);
          uint8_t* row = dst + r * (kBK * 2);
          *reinterpret_cast<uint4*>(row + (((2 * q) ^ sw) << 4)) = lo;
          *reinterpret_cast<uint4*>(row + (((2 * q + 1) ^ sw) << 4)) = hi;
        }
        ptx::fence_proxy_async_shared();  // generic-proxy writes -> the MMA's async-proxy reads
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(wfull_bar(ws));
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
        if (++ws == kWStages) {
          ws = 0;
          wphase ^= 1u;
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const int wr = quad * 32 + lane;  // weight row inside a 128-row sub-tile
    int acc = 0;
    uint32_t acc_phase = 0;
    bool over = false;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      const TileInfo ti = decode_tile(tile, a);
      const int kind = ti.g.kind;
      const int n_valid = tile_rows_valid(ti);
      if (!ptx::mbar_wait(tfull_bar(acc), acc_phase, abort_flag, a.err)) break;
      ptx::tc_fence_after();
      const uint32_t tacc = tmem_base + lane_off + (uint32_t)acc * kAccCols;
      const int64_t wbase = (int64_t)ti.g.index * a.w_rows[kind];
      if (PHASE == kPhaseGateUp) {
        const int f = ti.n_blk * kWRows + wr;
        const bool f_ok = f < a.n_ext[kind];
        const float sg = f_ok ? __ldg(a.w_scale[kind] + wbase + f) * 256.f : 0.f;
        const float su = f_ok ? __ldg(a.u_scale[kind] + wbase + f) * 256.f : 0.f;
        const int64_t ldh = a.ldh[kind];
        __half* hcol = reinterpret_cast<__half*>(a.h[kind]) + (int64_t)(ti.g.h_row0 + ti.m_blk * kBM) * ldh + f;
#pragma unroll 1
        for (int c = 0; c < n_valid; c += 16) {
          uint32_t gv[16], uv[16];
          ptx::tmem_ld_32x32b_x16(tacc + c, gv);
          ptx::tmem_ld_32x32b_x16(tacc + kWRows + c, uv);
          ptx::tmem_wait_ld();
          if (f_ok) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              if (c + j < n_valid) {
                const float g = __uint_as_float(gv[j]) * sg;
                const float u = __uint_as_float(uv[j]) * su;
                const float hv = silu_f(g) * u;
                over |= fabsf(hv) >= 65520.f;
                hcol[(int64_t)(c + j) * ldh] = __float2half_rn(hv);
              }
            }
          }
        }
      } else {
#pragma unroll 1
        for (int sub = 0; sub < 2; ++sub) {
          const int i = ti.n_blk * 2 * kWRows + sub * kWRows + wr;  // output feature
          const bool i_ok = i < a.d;
          const float sd = i_ok ? __ldg(a.w_scale[kind] + wbase + i) * 256.f : 0.f;
#pragma unroll 1
          for (int c = 0; c < n_valid; c += 16) {
            uint32_t yv[16];
            ptx::tmem_ld_32x32b_x16(tacc + sub * kWRows + c, yv);
            ptx::tmem_wait_ld();
            if (!i_ok) continue;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              if (c + j >= n_valid) continue;
              const int r_local = ti.m_blk * kBM + c + j;
              const float y = __uint_as_float(yv[j]) * sd;
              if (EPI == kEpiScatter) {
                int64_t t;
                float w;
                if (kind == 0 && a.row_w) {  // expert choice: the row's token and score
                  t = __ldg(a.perm_src + ti.g.h_row0 + r_local);
                  w = __ldg(a.row_w + ti.g.h_row0 + r_local);
                } else if (kind == 0) {
                  const int32_t src = __ldg(a.perm_src + ti.g.h_row0 + r_local);
                  t = src / a.top_k;
                  w = __ldg(a.topk_w + src);
                } else {
                  t = r_local;
                  w = 1.f;
                }
                atomicAdd(a.out_acc + t * a.d + i, w * y);
              } else {
                a.y[(int64_t)(ti.g.h_row0 + r_local) * a.d + i] = __float2bfloat16_rn(y);
              }
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
