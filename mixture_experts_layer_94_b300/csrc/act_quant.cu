// act_quant.cu — the activations of the FP8-weight expert GEMMs as a two-term
// E4M3 expansion.
//
// The tensor cores multiply E4M3 by E4M3 (kind::f8f6f4) at twice the fp16
// rate and read the expert codes straight from shared memory, but both
// operands must be 8-bit. The experts' weights are E4M3 already; an
// activation row x (K fp16 values) is carried as a row scale and two E4M3
// rows:
//   s  = max_k |x_k| / 448                  (1 for an all-zero row)
//   hi = e4m3(x / s),  lo = e4m3(x / s - hi)    (round to nearest even, saturating)
//   x ~= s * (hi + lo)
// hi keeps |x/s - hi| <= 2^-4 |x/s|, so lo's own rounding leaves
// |x/s - hi - lo| <= 2^-8 |x/s| wherever lo is a normal number (|x/s| >= 2^-2),
// and an absolute 2^-10 below: the precision of a bf16 activation, which is
// what the bf16-weight path multiplies with. The GEMM sums hi*W and lo*W in
// fp32.
// Output rows interleave the terms: row 2r holds hi of row r, row 2r+1 its lo,
// so the GEMM loads one box of 2n rows for n tokens and adds neighbouring
// accumulator lanes.
// The same split fused with the row gather of the layer (launch_gather_quant)
// reads each routed row straight from hidden, rounded to fp16 exactly as the
// gather would store it, so the permuted fp16 copy is never written.
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "act_convert.cuh"
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

// 8 fp16 values (one 16-byte vector) as floats.
__device__ __forceinline__ void unpack8(const uint4 v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float2 p = __half22float2(*reinterpret_cast<const __half2*>(&w[j]));
    f[2 * j] = p.x;
    f[2 * j + 1] = p.y;
  }
}

// Two floats -> two E4M3 codes (the first in the low byte), saturating.
__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
  return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}

// Two E4M3 codes (low byte first) -> their exact values.
__device__ __forceinline__ float2 e4m3x2_value(uint32_t c) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)c, __NV_E4M3);
  return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

// Two floats of a quantised row: their E4M3 hi and lo codes.
__device__ __forceinline__ void split2(float f0, float f1, float s, uint32_t& hi, uint32_t& lo) {
  const float q0 = __fdiv_rn(f0, s), q1 = __fdiv_rn(f1, s);
  hi = e4m3x2(q0, q1);
  const float2 h = e4m3x2_value(hi);
  lo = e4m3x2(q0 - h.x, q1 - h.y);
}

// Eight values (one 16-byte source vector) -> 8 hi codes and 8 lo codes.
__device__ __forceinline__ void quant8(const uint4 v, float s, uint2& hi, uint2& lo) {
  float f[8];
  unpack8(v, f);
  uint32_t h[4], l[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) split2(f[2 * j], f[2 * j + 1], s, h[j], l[j]);
  hi = make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
  lo = make_uint2(l[0] | (l[1] << 16), l[2] | (l[3] << 16));
}

__device__ __forceinline__ float amax8(const uint4 v, float m) {
  float f[8];
  unpack8(v, f);
#pragma unroll
  for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(f[j]));
  return m;
}

// Row sources. open(r, &src) gives output row r's source row (false: the row
// is skipped, left as it is); vec(src, i, over) its 16-byte vector i as 8
// fp16 values.
// An fp16 matrix [rows][K].
struct F16Rows {
  const __half* src;
  int K;
  __device__ void init() {}
  __device__ bool open(int64_t r, int64_t& row) const {
    row = r;
    return true;
  }
  __device__ uint4 vec(int64_t row, int i, bool&) const {
    return __ldg(reinterpret_cast<const uint4*>(src + row * K) + i);
  }
};

// Rows of hidden ([T][d], bf16 or fp32) rounded to fp16: output row r <
// routed is the token of packed row r (perm_src / K, or row_token), rows
// routed .. routed + T - 1 are the tokens in order (the shared experts'
// rows). Packed rows at or beyond offsets[N] are not placed.
struct HiddenRows {
  const void* hidden;
  bool hidden_bf16;
  int d, K;
  int64_t T, routed;
  const int32_t* perm_src;
  const int32_t* row_token;
  const int32_t* placed_at;  // &offsets[N]
  int64_t placed;
  __device__ void init() { placed = min(routed, (int64_t)__ldg(placed_at)); }
  __device__ bool open(int64_t r, int64_t& t) const {
    if (r >= routed) {
      t = r - routed;
      return true;
    }
    if (r >= placed) return false;
    if (row_token) {
      t = row_token[r];
      return t >= 0 && t < T;
    }
    const int32_t src = perm_src[r];
    t = src / K;
    return src >= 0 && src < routed;
  }
  __device__ uint4 vec(int64_t t, int i, bool& over) const {
    return hidden_vec(hidden, hidden_bf16, d, t, i, true, over);
  }
};

// Where a quantised row goes: rows below `split` to (dst0, scale0) at r, the
// rest to (dst1, scale1) at r - split. Optionally the kernel also clears
// zero [zero_n4 float4s] and reports an fp16 overflow in err.
struct QuantOut {
  uint8_t* dst0;
  float* scale0;
  uint8_t* dst1;
  float* scale1;
  int64_t split;
  float* zero;
  int64_t zero_n4;
  uint32_t* err;
};

__device__ __forceinline__ void quant_dest(const QuantOut& o, int64_t r, int K, uint2*& hi, uint2*& lo,
                                           float*& scale) {
  const bool second = r >= o.split;
  const int64_t q = second ? r - o.split : r;
  uint8_t* dst = second ? o.dst1 : o.dst0;
  hi = reinterpret_cast<uint2*>(dst + (2 * q) * (int64_t)K);
  lo = reinterpret_cast<uint2*>(dst + (2 * q + 1) * (int64_t)K);
  scale = (second ? o.scale1 : o.scale0) + q;
}

__device__ __forceinline__ void quant_tail(const QuantOut& o, bool over) {
  if (o.zero) {
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    float4* zp = reinterpret_cast<float4*>(o.zero);
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (int64_t i = tid; i < o.zero_n4; i += (int64_t)gridDim.x * blockDim.x) zp[i] = z;
  }
  if (over && o.err) atomicOr(o.err, kErrRange);
}

// Large batches: one warp per row, grid-stride over rows (many rows in
// flight per SM).
template <class Src>
__global__ void __launch_bounds__(256) quant_warp_kernel(Src src, int64_t rows, int K, QuantOut o) {
  pdl_trigger();
  pdl_wait();
  src.init();
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int nvec = K / 8;
  bool over = false;
  for (int64_t r = warp0; r < rows; r += nwarps) {
    int64_t sr;
    if (!src.open(r, sr)) continue;
    float amax = 0.f;
    for (int v = lane; v < nvec; v += 32) amax = amax8(src.vec(sr, v, over), amax);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    const float s = amax > 0.f ? amax / 448.f : 1.f;
    uint2 *hi_row, *lo_row;
    float* scale;
    quant_dest(o, r, K, hi_row, lo_row, scale);
    for (int v = lane; v < nvec; v += 32) {
      bool unused = false;
      quant8(src.vec(sr, v, unused), s, hi_row[v], lo_row[v]);
    }
    if (lane == 0) *scale = s;
  }
  quant_tail(o, over);
}

// Small batches: one 256-thread block per row, grid-stride over rows. A row's
// first kQV * 256 vectors are loaded once, all in flight together, and kept in
// registers for both passes (the block-wide max, then the split), so a short
// batch pays one load latency per row; the rest of a longer row is read again
// in the second pass.
constexpr int kQThreads = 256;
constexpr int kQV = 8;

template <class Src>
__global__ void __launch_bounds__(kQThreads, 2) quant_block_kernel(Src src, int64_t rows, int K, QuantOut o) {
  pdl_trigger();
  pdl_wait();
  src.init();
  __shared__ float s_max[kQThreads / 32];
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int nvec = K / 8;
  bool over = false;
  for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
    int64_t sr;
    if (!src.open(r, sr)) continue;  // uniform across the block
    uint4 v[kQV];
    float amax = 0.f;
#pragma unroll
    for (int q = 0; q < kQV; ++q) {
      const int i = t + q * kQThreads;
      if (i < nvec) v[q] = src.vec(sr, i, over);
    }
#pragma unroll
    for (int q = 0; q < kQV; ++q)
      if (t + q * kQThreads < nvec) amax = amax8(v[q], amax);
    for (int i = t + kQV * kQThreads; i < nvec; i += kQThreads) amax = amax8(src.vec(sr, i, over), amax);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    if (lane == 0) s_max[warp] = amax;
    __syncthreads();
    amax = s_max[0];
#pragma unroll
    for (int w = 1; w < kQThreads / 32; ++w) amax = fmaxf(amax, s_max[w]);
    const float s = amax > 0.f ? amax / 448.f : 1.f;
    uint2 *hi_row, *lo_row;
    float* scale;
    quant_dest(o, r, K, hi_row, lo_row, scale);
#pragma unroll
    for (int q = 0; q < kQV; ++q) {
      const int i = t + q * kQThreads;
      if (i < nvec) quant8(v[q], s, hi_row[i], lo_row[i]);
    }
    for (int i = t + kQV * kQThreads; i < nvec; i += kQThreads) {
      bool unused = false;
      quant8(src.vec(sr, i, unused), s, hi_row[i], lo_row[i]);
    }
    if (t == 0) *scale = s;
    __syncthreads();  // s_max is rewritten for the next row
  }
  quant_tail(o, over);
}

// Token-major form of the fused gather for large token-choice batches: one
// warp per token splits its hidden row once and stores the two E4M3 rows and
// the scale to each of the token's K packed rows (inv_row; -1 = dropped) and,
// with shared experts, to the token's shared row. The split is a function of
// the token's row alone, so every copy is the one the row-major form writes.
__global__ void __launch_bounds__(256) quant_token_kernel(HiddenRows src, const int32_t* __restrict__ inv_row,
                                                          int64_t shared_rows, QuantOut o) {
  pdl_trigger();
  pdl_wait();
  const int64_t placed = min(src.routed, (int64_t)__ldg(src.placed_at));
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int K = src.d, nvec = K / 8, topk = src.K;
  bool over = false;
  for (int64_t t = warp0; t < src.T; t += nwarps) {
    // lane k < topk holds copy k's packed row, or -1
    int32_t r_own = lane < topk ? __ldg(inv_row + t * topk + lane) : -1;
    if (r_own >= placed) r_own = -1;
    float amax = 0.f;
    for (int v = lane; v < nvec; v += 32) amax = amax8(src.vec(t, v, over), amax);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    const float sc = amax > 0.f ? amax / 448.f : 1.f;
    for (int v0 = 0; v0 < nvec; v0 += 32) {  // warp-uniform trips: every lane takes part in the shuffles
      const int v = v0 + lane;
      const bool on = v < nvec;
      bool unused = false;
      uint2 hi = make_uint2(0u, 0u), lo = hi;
      if (on) quant8(src.vec(t, v, unused), sc, hi, lo);
      for (int k = 0; k < topk; ++k) {
        const int32_t r = __shfl_sync(0xffffffffu, r_own, k);
        if (r < 0 || !on) continue;
        reinterpret_cast<uint2*>(o.dst0 + (2 * (int64_t)r) * K)[v] = hi;
        reinterpret_cast<uint2*>(o.dst0 + (2 * (int64_t)r + 1) * K)[v] = lo;
      }
      if (shared_rows && on) {
        reinterpret_cast<uint2*>(o.dst1 + (2 * t) * K)[v] = hi;
        reinterpret_cast<uint2*>(o.dst1 + (2 * t + 1) * K)[v] = lo;
      }
    }
    if (r_own >= 0) o.scale0[r_own] = sc;
    if (shared_rows && lane == 0) o.scale1[t] = sc;
  }
  quant_tail(o, over);
}

template <class Src>
cudaError_t launch_quant(const Src& src, int64_t rows, int32_t K, const QuantOut& o, cudaStream_t s) {
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (rows <= 2 * (int64_t)sms)
    return launch(quant_block_kernel<Src>, (unsigned)(rows < 1 ? 1 : rows), kQThreads, 0, s, src, rows, K, o);
  const int64_t want = (rows + 7) / 8;  // 8 rows (warps) per 256-thread CTA
  const unsigned grid = (unsigned)(want < (int64_t)sms * 8 ? want : (int64_t)sms * 8);
  return launch(quant_warp_kernel<Src>, grid, 256, 0, s, src, rows, K, o);
}

}  // namespace

cudaError_t launch_act_quant(const void* src, int64_t rows, int32_t K, uint8_t* dst, float* scale, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  QuantOut o{dst, scale, nullptr, nullptr, rows, nullptr, 0, nullptr};
  return launch_quant(F16Rows{static_cast<const __half*>(src), K}, rows, K, o, s);
}

cudaError_t launch_gather_quant(const PermuteArgs& a, int64_t rows, int64_t shared_rows, cudaStream_t s) {
  HiddenRows src{a.hidden, a.hidden_bf16, a.d, a.K, a.T, rows, a.perm_src, a.row_token, a.offsets + a.N, 0};
  QuantOut o{a.xq, a.sx, a.xq_sh, a.sx_sh, rows, a.zero_rows, a.zero_rows ? a.T * a.d / 4 : 0, a.err};
  if (!a.row_token && rows == a.T * a.K && rows >= kTokenMajorMinRows) {
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t want = (a.T + 7) / 8;  // 8 tokens (warps) per 256-thread CTA
    const unsigned grid = (unsigned)(want < (int64_t)sms * 8 ? want : (int64_t)sms * 8);
    return launch(quant_token_kernel, grid, 256, 0, s, src, (const int32_t*)a.inv_row, shared_rows, o);
  }
  return launch_quant(src, rows + shared_rows, a.d, o, s);
}

}  // namespace moe
