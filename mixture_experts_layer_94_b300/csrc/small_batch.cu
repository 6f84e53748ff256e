// small_batch.cu — the expert FFNs of a decode-sized batch on the CUDA cores
// (internal).
//
// With T <= 4 tokens every expert holds at most T packed rows, so a grouped
// GEMM tile (128 activation rows) is almost all padding and its 256 weight
// rows per tile leave most SMs idle (8 touched experts x 12 tiles at T = 1).
// The work is a stream of weight rows, each used by at most T activation rows:
// HBM-bound, with nothing for the tensor cores to gain. Here a warp takes four
// weight rows of one expert (gate rows f, f+1 and up rows f, f+1; or W_down
// rows j..j+3), streams them from HBM once in 16-byte units, and dots them with
// the expert's activation rows. One 512-thread CTA per SM walks all (expert,
// row block) items, so every SM streams weights.
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

#include <cuda_fp8.h>

#include <atomic>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kRowsPerItem = 4;  // weight rows a warp streams together

// Elements in one 16-byte unit of weight codes.
__host__ __device__ constexpr int unit_elems(int fmt) { return fmt == kSmallBf16 ? 8 : 16; }

// 16 bytes of weight codes, read once: no L1 allocation.
__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}

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

// acc[q][r] += (weight row q) . (activation row r) over `units` 16-byte units
// of codes (unit j covers elements j*E .. j*E+E-1), then summed over the warp.
// Activation row r starts at xr[r]; rows >= `rows` are skipped.
template <int FMT, int R, int XS>
__device__ __forceinline__ void dot_rows(const uint4* const (&w)[kRowsPerItem], const void* const (&xr)[R],
                                         int rows, int units, int lane, float (&acc)[kRowsPerItem][R]) {
  constexpr int E = unit_elems(FMT), SUB = E / 8;
  constexpr int U = R == 1 ? 4 : 2;  // units per row in flight per lane
  for (int j0 = lane; j0 < units; j0 += 32 * U) {
    uint4 wv[kRowsPerItem][U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int j = j0 + 32 * u;
#pragma unroll
      for (int q = 0; q < kRowsPerItem; ++q) wv[q][u] = j < units ? ld_stream(w[q] + j) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int j = j0 + 32 * u;
      if (j < units) {
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
            w8<FMT>(wv[q][u], s, wf);
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
    }
  }
#pragma unroll
  for (int q = 0; q < kRowsPerItem; ++q)
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc[q][r] += __shfl_xor_sync(0xFFFFFFFFu, acc[q][r], off);
}

// 16-byte units of codes in one weight row of `k` elements.
__device__ __forceinline__ int64_t row_units(int k, int fmt) { return k / unit_elems(fmt); }

// PHASE 0: stage the T token rows of hidden (bf16 when HB, else fp32) in
// shared memory, rounded to the activation format (bf16, or fp16 for FP8
// experts); clear out_acc and the down kernel's completion count; then
// h[row r][f, f+1] = SiLU(g) * u for the item's gate rows f, f+1 and up rows
// f, f+1. PHASE 1: out_acc[token of r][j..j+3] += w_r * y for W_down rows
// j..j+3; the last CTA to finish writes out = bf16(out_acc). Items: every
// routed expert holding rows (F/2 or d/4 items each), then every shared expert
// (Fs/2 or d/4 items each); item i goes to warp i / gridDim.x of CTA
// i % gridDim.x, so a partial last round still spreads over every SM.
template <int FMT, int R, int PHASE, bool HB>
__global__ void __launch_bounds__(kThreads, 1) small_batch_ffn_kernel(const SmallBatchArgs a) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ float4 s_rows4[];  // PHASE 0: [T][d] fp32
  __shared__ int32_t s_list[kMaxExperts];
  __shared__ int32_t s_count[kWarps];
  __shared__ bool s_last;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = a.N;
  constexpr bool kF16 = FMT != kSmallBf16;
  bool over = false;
  const float* s_rows = reinterpret_cast<const float*>(s_rows4);
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
  for (int64_t item = (int64_t)warp * gridDim.x + blockIdx.x; item < total; item += (int64_t)gridDim.x * kWarps) {
    int g, blk;
    if (item < n_r) {
      g = s_list[item / per_r];
      blk = (int)(item % per_r);
    } else {
      const int64_t i2 = item - n_r;
      g = N + (int)(i2 / per_s);
      blk = (int)(i2 % per_s);
    }
    const GroupDesc gd = a.groups[g];
    const int kind = g < N ? 0 : 1;
    const int e = kind ? g - N : g;
    int rows = gd.rows;
    if (rows > R) {  // cannot happen for token choice with T <= R
      if (lane == 0) atomicOr(a.err, kErrBounds);
      rows = R;
    }
    const int Fk = kind ? a.Fs : a.F;
    float acc[kRowsPerItem][R];
#pragma unroll
    for (int q = 0; q < kRowsPerItem; ++q)
#pragma unroll
      for (int r = 0; r < R; ++r) acc[q][r] = 0.f;

    if (PHASE == 0) {
      const int f0 = 2 * blk;
      const int64_t units = row_units(a.d, FMT);
      const int64_t row0 = (int64_t)e * Fk + f0;  // gate / up row f0 of this expert
      const uint4* wg = static_cast<const uint4*>(kind ? a.s_gate : a.w_gate);
      const uint4* wu = static_cast<const uint4*>(kind ? a.s_up : a.w_up);
      const uint4* const w[kRowsPerItem] = {wg + row0 * units, wg + (row0 + 1) * units, wu + row0 * units,
                                            wu + (row0 + 1) * units};
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
      dot_rows<FMT, R, kXShared>(w, xr, rows, (int)units, lane, acc);
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
      const int j0 = kRowsPerItem * blk;
      const int64_t units = row_units(Fk, FMT);
      const int64_t row0 = (int64_t)e * a.d + j0;  // W_down row j0 of this expert
      const uint4* wd = static_cast<const uint4*>(kind ? a.s_down : a.w_down);
      const uint4* const w[kRowsPerItem] = {wd + row0 * units, wd + (row0 + 1) * units, wd + (row0 + 2) * units,
                                            wd + (row0 + 3) * units};
      const uint16_t* hb = static_cast<const uint16_t*>(kind ? a.h_sh : a.h);
      const void* xr[R];
#pragma unroll
      for (int r = 0; r < R; ++r) xr[r] = hb + (int64_t)(gd.h_row0 + r) * Fk;
      dot_rows<FMT, R, kXAct16>(w, xr, rows, (int)units, lane, acc);
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
        bool ok = true;
        if (kind == 0) {
          const int32_t src = __ldg(a.perm_src + gd.h_row0 + rl);
          ok = src >= 0 && (int64_t)src < a.T * a.K;
          t = ok ? src / a.K : 0;
          wt = ok ? __ldg(a.topk_w + src) : 0.f;
          if (!ok) atomicOr(a.err, kErrBounds);
        }
        if (ok) atomicAdd(a.out_acc + t * a.d + j0 + q, wt * y);
      }
    }
  }
  if (over) atomicOr(a.err, kErrRange);
  if (PHASE == 1) {
    // the last CTA to finish rounds the accumulator to the bf16 output
    __syncthreads();
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

// These grids are launched without programmatic stream serialisation (their
// griddepcontrol.wait is then a no-op): measured, letting them start early
// behind the previous kernel made a 2-token layer 13 % and a 4-token layer
// 14 % slower, with every stage's own time unchanged. The gate/up grid's
// dynamic shared memory (the token rows) may exceed the default 48 KB; its
// limit is raised once per kernel and device.
template <int FMT, int R, int PHASE, bool HB>
cudaError_t launch_k(const SmallBatchArgs& a, unsigned grid, size_t smem, cudaStream_t s) {
  void (*kern)(const SmallBatchArgs) = small_batch_ffn_kernel<FMT, R, PHASE, HB>;
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (PHASE == 0 && !(configured.load() & bit)) {
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
cudaError_t launch_fr(const SmallBatchArgs& a, int phase, unsigned grid, cudaStream_t s) {
  if (phase == 1) return launch_k<FMT, R, 1, true>(a, grid, 0, s);
  const size_t smem = (size_t)a.T * a.d * 4;
  return a.hidden_bf16 ? launch_k<FMT, R, 0, true>(a, grid, smem, s) : launch_k<FMT, R, 0, false>(a, grid, smem, s);
}

}  // namespace

cudaError_t launch_small_batch_ffn(const SmallBatchArgs& a, int phase, cudaStream_t s) {
  if (a.max_rows < 1 || a.max_rows > kSmallBatchMaxRows || a.N > kMaxExperts) return cudaErrorInvalidValue;
  if (a.fmt == kSmallE4M3 ? a.max_rows != 1 : a.fmt != kSmallBf16) return cudaErrorInvalidValue;
  if (a.T < 1 || a.T > a.max_rows || (size_t)a.T * a.d * 4 > kSmallBatchMaxSmem) return cudaErrorInvalidValue;
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // items: at most min(N, rows) routed experts hold rows
  const int64_t touched = a.N < a.routed_rows ? a.N : a.routed_rows;
  const int64_t per_r = phase == 0 ? a.F / 2 : a.d / kRowsPerItem;
  const int64_t per_s = phase == 0 ? a.Fs / 2 : a.d / kRowsPerItem;
  const int64_t items = touched * per_r + (a.S > 0 ? a.S * per_s : 0);
  int64_t want = (items + kWarps - 1) / kWarps;
  if (want < 1) want = 1;
  const unsigned grid = (unsigned)(want < sms ? want : sms);
  if (a.fmt == kSmallE4M3) return launch_fr<kSmallE4M3, 1>(a, phase, grid, s);
  if (a.max_rows <= 1) return launch_fr<kSmallBf16, 1>(a, phase, grid, s);
  if (a.max_rows <= 2) return launch_fr<kSmallBf16, 2>(a, phase, grid, s);
  return launch_fr<kSmallBf16, 4>(a, phase, grid, s);
}

}  // namespace moe
