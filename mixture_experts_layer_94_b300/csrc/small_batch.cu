// small_batch.cu — the expert FFNs of a decode-sized batch on the CUDA cores
// (internal).
//
// With T <= 4 tokens every expert holds at most T packed rows, so a grouped
// GEMM tile (128 activation rows) is almost all padding and its 256 weight
// rows per tile leave most SMs idle (8 touched experts x 12 tiles at T = 1).
// The work is a stream of weight rows, each used by at most T activation rows:
// HBM-bound, with nothing for the tensor cores to gain. An item is four weight
// rows of one expert (gate rows f, f+1 and up rows f, f+1; or W_down rows
// j..j+3). One 512-thread CTA per SM walks its share of the items: warp 0
// streams each item's rows from HBM into a ring of shared-memory stages with
// 1-D bulk copies (the bytes in flight then hold no registers), and the other
// 15 warps take one item each, dot its rows with the expert's activation rows
// and write the results.
//
// Two launches do the whole FFN part of the layer. The gate/up kernel stages
// the batch's T token rows of hidden in shared memory as fp32, rounded once as
// the activation format holds them (no permuted copy in global memory), and
// clears the fp32 accumulator; the down kernel adds the gate-weighted rows
// into it, and its last CTA to finish rounds it to the bf16 output (no
// separate finalise launch).
//
// Formats: bf16 weights with bf16 activations, or FP8 E4M3 codes with fp32 row
// scales and fp16 activations. Products and sums are fp32; h is rounded once,
// to bf16 (fp16 for FP8 experts), as the grouped GEMMs store it.
//
// Every mbarrier wait is bounded (kWaitTimeoutNs); a wait that gives up
// records kErrTimeout, raises the CTA's abort flag so the other waits return,
// and the copy warp waits (bounded) for its copies in flight before the CTA
// exits.

#include <cuda_fp8.h>

#include <atomic>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "tile_sched.cuh"

namespace moe {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kConsumers = kWarps - 1;  // warp 0 issues the copies
constexpr int kRowsPerItem = 4;         // weight rows of one item
constexpr int kMaxStages = 32;

// Elements in one 16-byte unit of weight codes.
__host__ __device__ constexpr int unit_elems(int fmt) { return fmt == kSmallBf16 ? 8 : 16; }
// Bytes per weight element.
__host__ __device__ constexpr int elem_bytes(int fmt) { return fmt == kSmallBf16 ? 2 : 1; }

__host__ __device__ constexpr size_t align128(size_t x) { return (x + 127) & ~(size_t)127; }

__device__ __forceinline__ float2 half2_bits_to_f32(uint32_t bits) {
  __half2 h;
  *reinterpret_cast<uint32_t*>(&h) = bits;
  return __half22float2(h);
}

// 8 activations (16 bytes: bf16, or fp16 when F16) to fp32.
template <bool F16>
__device__ __forceinline__ void act8(const uint4 v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (F16) {
      const float2 p = half2_bits_to_f32(w[i]);
      f[2 * i] = p.x;
      f[2 * i + 1] = p.y;
    } else {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
}

// Two E4M3 codes (low 16 bits of c; the lower byte is the earlier element).
// Measured: placing each code's bits into an fp32 word on the integer pipe
// instead made the one-token FP8 gate/up stage slower (42 against 31-39 us).
__device__ __forceinline__ float2 e4m3x2_f32(uint32_t c) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(c & 0xFFFFu), __NV_E4M3);
  return half2_bits_to_f32((uint32_t)h.x | ((uint32_t)h.y << 16));
}

// Elements 8s .. 8s+7 of a 16-byte unit of weight codes as fp32 (FP8 row
// scales are applied by the caller).
template <int FMT>
__device__ __forceinline__ void w8(const uint4 u, int s, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
  if (FMT == kSmallBf16) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  } else {  // 16 E4M3 codes per unit: words 2s, 2s+1
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const uint32_t c = w[2 * s + i];
      const float2 lo = e4m3x2_f32(c), hi = e4m3x2_f32(c >> 16);
      f[4 * i] = lo.x;
      f[4 * i + 1] = lo.y;
      f[4 * i + 2] = hi.x;
      f[4 * i + 3] = hi.y;
    }
  }
}

__device__ __forceinline__ float round_bf16(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }

// x rounded to fp16 (nearest even); `over` is set when a finite x lies beyond
// fp16's range, as the row gather reports it.
__device__ __forceinline__ float round_f16(float x, bool& over) {
  const float m = fabsf(x);
  over |= (m >= 65520.f) && (m <= 3.402823466e38f);
  return __half2float(__float2half_rn(x));
}

// Where the dot products' activation rows come from.
enum XSource {
  kXShared = 0,  // fp32 token rows staged in shared memory (gate/up)
  kXAct16 = 1,   // rows in the activation format in global memory (h: bf16, or fp16 for FP8 experts)
};

// Elements 8v .. 8v+7 of activation row `row` as fp32.
template <int XS, int FMT>
__device__ __forceinline__ void x8(const void* row, int64_t v, float (&f)[8]) {
  if (XS == kXShared) {
    const float4* p = static_cast<const float4*>(row) + 2 * v;
    const float4 a = p[0], b = p[1];
    f[0] = a.x;
    f[1] = a.y;
    f[2] = a.z;
    f[3] = a.w;
    f[4] = b.x;
    f[5] = b.y;
    f[6] = b.z;
    f[7] = b.w;
  } else {
    act8<FMT != kSmallBf16>(__ldg(static_cast<const uint4*>(row) + v), f);
  }
}

// acc[q][r] = (weight row q of the stage) . (activation row r), summed over
// the warp. Row q of the stage starts at stage + q * srow; `units` 16-byte
// units of codes per row (unit j covers elements j*E .. j*E+E-1); activation
// row r starts at xr[r]; rows >= `rows` are skipped.
template <int FMT, int R, int XS>
__device__ __forceinline__ void dot_stage(const uint8_t* stage, int srow, const void* const (&xr)[R], int rows,
                                          int units, int lane, float (&acc)[kRowsPerItem][R]) {
  constexpr int SUB = unit_elems(FMT) / 8;
#pragma unroll
  for (int q = 0; q < kRowsPerItem; ++q)
#pragma unroll
    for (int r = 0; r < R; ++r) acc[q][r] = 0.f;
#pragma unroll 2
  for (int j = lane; j < units; j += 32) {
    uint4 wv[kRowsPerItem];
#pragma unroll
    for (int q = 0; q < kRowsPerItem; ++q)
      wv[q] = *reinterpret_cast<const uint4*>(stage + (size_t)q * srow + (size_t)j * 16);
#pragma unroll
    for (int s = 0; s < SUB; ++s) {
      float xf[R][8];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        if (r < rows) x8<XS, FMT>(xr[r], (int64_t)j * SUB + s, xf[r]);
      }
#pragma unroll
      for (int q = 0; q < kRowsPerItem; ++q) {
        float wf[8];
        w8<FMT>(wv[q], s, wf);
#pragma unroll
        for (int r = 0; r < R; ++r) {
          if (r < rows) {
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[q][r] = fmaf(wf[i], xf[r][i], acc[q][r]);
          }
        }
      }
    }
  }
#pragma unroll
  for (int q = 0; q < kRowsPerItem; ++q)
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc[q][r] += __shfl_xor_sync(0xFFFFFFFFu, acc[q][r], off);
}

// Item `item` of a phase: its group (a routed expert from the list of those
// holding rows, then the shared experts) and its row block within the group.
struct ItemRef {
  int g, blk;
};
__device__ __forceinline__ ItemRef item_ref(int64_t item, int64_t n_r, int per_r, int per_s, int N,
                                            const int32_t* s_list) {
  ItemRef ir;
  if (item < n_r) {
    ir.g = s_list[item / per_r];
    ir.blk = (int)(item % per_r);
  } else {
    const int64_t i2 = item - n_r;
    ir.g = N + (int)(i2 / per_s);
    ir.blk = (int)(i2 % per_s);
  }
  return ir;
}

// First weight row of an item in its stacked matrix (gate / up rows f0, f0+1
// for phase 0, W_down rows j0..j0+3 for phase 1), and the row length.
template <int PHASE>
__device__ __forceinline__ int64_t item_row0(const SmallBatchArgs& a, int g, int blk, int* klen) {
  const int kind = g < a.N ? 0 : 1, e = kind ? g - a.N : g;
  const int Fk = kind ? a.Fs : a.F;
  if (PHASE == 0) {
    *klen = a.d;
    return (int64_t)e * Fk + 2 * blk;
  }
  *klen = Fk;
  return (int64_t)e * a.d + kRowsPerItem * blk;
}

// PHASE 0: stage the T token rows of hidden (bf16 when HB, else fp32) in
// shared memory, rounded to the activation format (bf16, or fp16 for FP8
// experts); clear out_acc and the down kernel's completion count; then
// h[row r][f, f+1] = SiLU(g) * u for the item's gate rows f, f+1 and up rows
// f, f+1. PHASE 1: out_acc[token of r][j..j+3] += w_r * y for W_down rows
// j..j+3; the last CTA to finish writes out = bf16(out_acc). Items: every
// routed expert holding rows (F/2 or d/4 items each), then every shared expert
// (Fs/2 or d/4 items each); CTA b takes items b, b + grid, b + 2 grid, ... in
// order, its k-th in stage k % stages, handled by consumer warp 1 + k % 15.
template <int FMT, int R, int PHASE, bool HB>
__global__ void __launch_bounds__(kThreads, 1) small_batch_ffn_kernel(const SmallBatchArgs a) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ __align__(128) uint8_t s_dyn[];  // [x rows (phase 0)][stages]
  __shared__ int32_t s_list[kMaxExperts];
  __shared__ int32_t s_count[kWarps];
  __shared__ __align__(8) uint64_t s_full[kMaxStages], s_empty[kMaxStages];
  __shared__ int s_abort;
  __shared__ bool s_last;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = a.N, S = a.stages;
  constexpr bool kF16 = FMT != kSmallBf16;
  bool over = false;
  const size_t x_bytes = PHASE == 0 ? align128((size_t)a.T * a.d * 4) : 0;
  float4* s_rows4 = reinterpret_cast<float4*>(s_dyn);
  const float* s_rows = reinterpret_cast<const float*>(s_dyn);
  uint8_t* s_stage = s_dyn + x_bytes;
  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int s = 0; s < S; ++s) {
      ptx::mbar_init(ptx::smem_u32(&s_full[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&s_empty[s]), 1);
    }
    ptx::fence_mbarrier_init();
  }
  if (PHASE == 0) {
    const int64_t nacc = a.T * a.d / 4;
    const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x; i < nacc; i += (int64_t)gridDim.x * kThreads)
      reinterpret_cast<float4*>(a.out_acc)[i] = zero;
    if (blockIdx.x == 0 && threadIdx.x == 0) *a.done = 0u;
    // the token rows, 8 elements per step, as the row gather would store them
    const int nvec = (int)(a.T * (a.d / 8));
    for (int i = threadIdx.x; i < nvec; i += kThreads) {
      float f[8];
      if (HB) {
        act8<false>(__ldg(static_cast<const uint4*>(a.hidden) + i), f);
        if (kF16) {
#pragma unroll
          for (int k = 0; k < 8; ++k) f[k] = round_f16(f[k], over);
        }
      } else {
        const float4* p = static_cast<const float4*>(a.hidden) + 2 * (int64_t)i;
        const float4 u = __ldg(p), v = __ldg(p + 1);
        const float t[8] = {u.x, u.y, u.z, u.w, v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 8; ++k) f[k] = kF16 ? round_f16(t[k], over) : round_bf16(t[k]);
      }
      s_rows4[2 * i] = make_float4(f[0], f[1], f[2], f[3]);
      s_rows4[2 * i + 1] = make_float4(f[4], f[5], f[6], f[7]);
    }
  }
  // the routed experts that hold rows, in expert order (N <= 256 < kThreads)
  const bool has = (int)threadIdx.x < N && a.groups[threadIdx.x].rows > 0;
  const uint32_t ball = __ballot_sync(0xFFFFFFFFu, has);
  if (lane == 0) s_count[warp] = __popc(ball);
  __syncthreads();
  int base = 0, nr = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const int c = s_count[w];
    base += w < warp ? c : 0;
    nr += c;
  }
  if (has) s_list[base + __popc(ball & ((1u << lane) - 1u))] = (int32_t)threadIdx.x;
  __syncthreads();

  const int per_r = PHASE == 0 ? a.F / 2 : a.d / kRowsPerItem;
  const int per_s = PHASE == 0 ? a.Fs / 2 : a.d / kRowsPerItem;
  const int64_t n_r = (int64_t)nr * per_r;
  const int64_t total = n_r + (a.S > 0 ? (int64_t)a.S * per_s : 0);
  const int srow = a.stage_row_bytes;
  constexpr int EB = elem_bytes(FMT);

  if (warp == 0) {
    // copies: item k of this CTA into stage k % S once its previous use is released
    if (lane == 0) {
      int issued = 0;
      for (int k = 0;; ++k) {
        const int64_t item = blockIdx.x + (int64_t)k * gridDim.x;
        if (item >= total) break;
        const int s = k % S;
        const uint32_t n = (uint32_t)(k / S);
        if (k >= S && !ptx::mbar_wait(ptx::smem_u32(&s_empty[s]), (n - 1) & 1u, &s_abort, a.err)) break;
        const ItemRef ir = item_ref(item, n_r, per_r, per_s, N, s_list);
        int klen = 0;
        const int64_t row0 = item_row0<PHASE>(a, ir.g, ir.blk, &klen);
        const uint32_t bytes = (uint32_t)klen * EB;
        const int kind = ir.g < N ? 0 : 1;
        const uint8_t* src[kRowsPerItem];
        if (PHASE == 0) {
          const uint8_t* wg = static_cast<const uint8_t*>(kind ? a.s_gate : a.w_gate);
          const uint8_t* wu = static_cast<const uint8_t*>(kind ? a.s_up : a.w_up);
          src[0] = wg + row0 * bytes;
          src[1] = wg + (row0 + 1) * bytes;
          src[2] = wu + row0 * bytes;
          src[3] = wu + (row0 + 1) * bytes;
        } else {
          const uint8_t* wd = static_cast<const uint8_t*>(kind ? a.s_down : a.w_down);
#pragma unroll
          for (int q = 0; q < kRowsPerItem; ++q) src[q] = wd + (row0 + q) * bytes;
        }
        const uint32_t bar = ptx::smem_u32(&s_full[s]);
        ptx::mbar_arrive_expect_tx(bar, kRowsPerItem * bytes);
        const uint32_t dst = ptx::smem_u32(s_stage + (size_t)s * kRowsPerItem * srow);
#pragma unroll
        for (int q = 0; q < kRowsPerItem; ++q) ptx::bulk_load(dst + (uint32_t)q * srow, src[q], bytes, bar);
        issued = k + 1;
      }
      // the copies still in flight land before the CTA may exit (the normal
      // path has consumed them all; after an abort, wait a bounded time)
      for (int k = issued > S ? issued - S : 0; k < issued; ++k)
        wait_raw(ptx::smem_u32(&s_full[k % S]), (uint32_t)(k / S) & 1u, kWaitTimeoutNs);
    }
  } else {
    for (int k = warp - 1;; k += kConsumers) {
      const int64_t item = blockIdx.x + (int64_t)k * gridDim.x;
      if (item >= total) break;
      const int s = k % S;
      const uint32_t n = (uint32_t)(k / S);
      const bool ok = ptx::mbar_wait(ptx::smem_u32(&s_full[s]), n & 1u, &s_abort, a.err);
      if (!__all_sync(0xFFFFFFFFu, ok)) break;
      const ItemRef ir = item_ref(item, n_r, per_r, per_s, N, s_list);
      const GroupDesc gd = a.groups[ir.g];
      const int kind = ir.g < N ? 0 : 1;
      int rows = gd.rows;
      if (rows > R) {  // cannot happen for token choice with T <= R
        if (lane == 0) atomicOr(a.err, kErrBounds);
        rows = R;
      }
      int klen = 0;
      const int64_t row0 = item_row0<PHASE>(a, ir.g, ir.blk, &klen);
      const int Fk = kind ? a.Fs : a.F;
      const uint8_t* stage = s_stage + (size_t)s * kRowsPerItem * srow;
      const int units = klen / unit_elems(FMT);
      float acc[kRowsPerItem][R];
      if (PHASE == 0) {
        // row r's token: its packed copy's source slot / K (routed), or r (shared)
        int tok = 0;
        if (lane < rows) {
          if (kind) {
            tok = lane;
          } else {
            const int32_t src = __ldg(a.perm_src + gd.a_row0 + lane);
            if (src >= 0 && (int64_t)src < a.T * a.K) tok = src / a.K;
            else atomicOr(a.err, kErrBounds);
          }
        }
        const void* xr[R];
#pragma unroll
        for (int r = 0; r < R; ++r) xr[r] = s_rows + (int64_t)__shfl_sync(0xFFFFFFFFu, tok, r) * a.d;
        dot_stage<FMT, R, kXShared>(stage, srow, xr, rows, units, lane, acc);
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&s_empty[s]));
        const int f0 = 2 * ir.blk;
        float gs0 = 1.f, gs1 = 1.f, us0 = 1.f, us1 = 1.f;
        if (FMT == kSmallE4M3) {
          const float* sg = static_cast<const float*>(kind ? a.s_gate_scale : a.w_gate_scale);
          const float* su = static_cast<const float*>(kind ? a.s_up_scale : a.w_up_scale);
          gs0 = __ldg(sg + row0);
          gs1 = __ldg(sg + row0 + 1);
          us0 = __ldg(su + row0);
          us1 = __ldg(su + row0 + 1);
        }
        uint32_t* h = static_cast<uint32_t*>(kind ? a.h_sh : a.h);
#pragma unroll
        for (int r = 0; r < R; ++r) {
          if (lane == r && r < rows) {
            const float h0 = silu_f(gs0 * acc[0][r]) * (us0 * acc[2][r]);
            const float h1 = silu_f(gs1 * acc[1][r]) * (us1 * acc[3][r]);
            if (kF16) over |= fmaxf(fabsf(h0), fabsf(h1)) >= 65520.f;
            h[((int64_t)(gd.h_row0 + r) * Fk + f0) / 2] = kF16 ? pack_f16x2(h0, h1) : pack_bf16x2(h0, h1);
          }
        }
      } else {
        const uint16_t* hb = static_cast<const uint16_t*>(kind ? a.h_sh : a.h);
        const void* xr[R];
#pragma unroll
        for (int r = 0; r < R; ++r) xr[r] = hb + (int64_t)(gd.h_row0 + r) * Fk;
        dot_stage<FMT, R, kXAct16>(stage, srow, xr, rows, units, lane, acc);
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&s_empty[s]));
        const int j0 = kRowsPerItem * ir.blk;
        const int q = lane & (kRowsPerItem - 1), rl = lane / kRowsPerItem;
        if (rl < rows) {
          float y = 0.f;
#pragma unroll
          for (int r = 0; r < R; ++r)
#pragma unroll
            for (int qq = 0; qq < kRowsPerItem; ++qq)
              if (r == rl && qq == q) y = acc[qq][r];
          if (FMT == kSmallE4M3)
            y *= __ldg(static_cast<const float*>(kind ? a.s_down_scale : a.w_down_scale) + row0 + q);
          int64_t t = rl;
          float wt = 1.f;
          bool valid = true;
          if (kind == 0) {
            const int32_t src = __ldg(a.perm_src + gd.h_row0 + rl);
            valid = src >= 0 && (int64_t)src < a.T * a.K;
            t = valid ? src / a.K : 0;
            wt = valid ? __ldg(a.topk_w + src) : 0.f;
            if (!valid) atomicOr(a.err, kErrBounds);
          }
          if (valid) atomicAdd(a.out_acc + t * a.d + j0 + q, wt * y);
        }
      }
    }
  }
  if (over) atomicOr(a.err, kErrRange);
  __syncthreads();
  if (PHASE == 1) {
    // the last CTA to finish rounds the accumulator to the bf16 output
    if (threadIdx.x == 0) {
      __threadfence();
      s_last = atomicAdd(a.done, 1u) == gridDim.x - 1;
    }
    __syncthreads();
    if (s_last) {
      __threadfence();
      const int64_t nvec = a.T * a.d / 8;
      const float4* acc4 = reinterpret_cast<const float4*>(a.out_acc);
      for (int64_t v = threadIdx.x; v < nvec; v += kThreads) {
        const float4 p = __ldcg(acc4 + 2 * v), q = __ldcg(acc4 + 2 * v + 1);
        reinterpret_cast<uint4*>(a.out)[v] =
            make_uint4(pack_bf16x2(p.x, p.y), pack_bf16x2(p.z, p.w), pack_bf16x2(q.x, q.y), pack_bf16x2(q.z, q.w));
      }
    }
  }
}

// Shared memory of a phase: the staged token rows (phase 0) and the stages
// (four rows of the longest weight row each); 0 stages if fewer than 2 fit.
struct SmemPlan {
  int stages;
  int stage_row_bytes;
  size_t bytes;
};
SmemPlan smem_plan(int fmt, int phase, int64_t T, int32_t d, int32_t F, int32_t Fs, int32_t S) {
  SmemPlan p{};
  const size_t x_bytes = phase == 0 ? align128((size_t)T * d * 4) : 0;
  const int klen = phase == 0 ? d : (S > 0 && Fs > F ? Fs : F);
  p.stage_row_bytes = (int)align128((size_t)klen * elem_bytes(fmt));
  const size_t stage = (size_t)kRowsPerItem * p.stage_row_bytes;
  if (x_bytes + 2 * stage > kSmallBatchMaxSmem) return SmemPlan{};
  const size_t fit = (kSmallBatchMaxSmem - x_bytes) / stage;
  p.stages = (int)(fit < (size_t)kMaxStages ? fit : (size_t)kMaxStages);
  p.bytes = x_bytes + (size_t)p.stages * stage;
  return p;
}

// These grids are launched without programmatic stream serialisation (their
// griddepcontrol.wait is then a no-op): measured, letting them start early
// behind the previous kernel made a 2-token layer 13 % and a 4-token layer
// 14 % slower, with every stage's own time unchanged. Their dynamic shared
// memory exceeds the default 48 KB; the limit is raised once per kernel and
// device.
template <int FMT, int R, int PHASE, bool HB>
cudaError_t launch_k(const SmallBatchArgs& a, unsigned grid, size_t smem, cudaStream_t s) {
  void (*kern)(const SmallBatchArgs) = small_batch_ffn_kernel<FMT, R, PHASE, HB>;
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(configured.load() & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmallBatchMaxSmem);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit);
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = nullptr;
  cfg.numAttrs = 0;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

template <int FMT, int R>
cudaError_t launch_fr(const SmallBatchArgs& a, int phase, unsigned grid, size_t smem, cudaStream_t s) {
  if (phase == 1) return launch_k<FMT, R, 1, true>(a, grid, smem, s);
  return a.hidden_bf16 ? launch_k<FMT, R, 0, true>(a, grid, smem, s) : launch_k<FMT, R, 0, false>(a, grid, smem, s);
}

}  // namespace

bool small_batch_fits(int fmt, int64_t T, int32_t d, int32_t F, int32_t Fs, int32_t S) {
  return smem_plan(fmt, 0, T, d, F, Fs, S).stages >= 2 && smem_plan(fmt, 1, T, d, F, Fs, S).stages >= 2;
}

cudaError_t launch_small_batch_ffn(const SmallBatchArgs& args, int phase, cudaStream_t s) {
  SmallBatchArgs a = args;
  if (a.max_rows < 1 || a.max_rows > kSmallBatchMaxRows || a.N > kMaxExperts) return cudaErrorInvalidValue;
  if (a.fmt == kSmallE4M3 ? a.max_rows != 1 : a.fmt != kSmallBf16) return cudaErrorInvalidValue;
  if (a.T < 1 || a.T > a.max_rows) return cudaErrorInvalidValue;
  const SmemPlan sp = smem_plan(a.fmt, phase, a.T, a.d, a.F, a.Fs, a.S);
  if (sp.stages < 2) return cudaErrorInvalidValue;
  a.stages = sp.stages;
  a.stage_row_bytes = sp.stage_row_bytes;
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // items: at most min(N, rows) routed experts hold rows
  const int64_t touched = a.N < a.routed_rows ? a.N : a.routed_rows;
  const int64_t per_r = phase == 0 ? a.F / 2 : a.d / kRowsPerItem;
  const int64_t per_s = phase == 0 ? a.Fs / 2 : a.d / kRowsPerItem;
  const int64_t items = touched * per_r + (a.S > 0 ? a.S * per_s : 0);
  int64_t want = (items + kConsumers - 1) / kConsumers;
  if (want < 1) want = 1;
  const unsigned grid = (unsigned)(want < sms ? want : sms);
  if (a.fmt == kSmallE4M3) return launch_fr<kSmallE4M3, 1>(a, phase, grid, sp.bytes, s);
  if (a.max_rows <= 1) return launch_fr<kSmallBf16, 1>(a, phase, grid, sp.bytes, s);
  if (a.max_rows <= 2) return launch_fr<kSmallBf16, 2>(a, phase, grid, sp.bytes, s);
  return launch_fr<kSmallBf16, 4>(a, phase, grid, sp.bytes, s);
}

}  // namespace moe
