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
#include <cuda_fp16.h>
#include <cuda_fp8.h>

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

// Large batches: one warp per row, grid-stride over rows (many rows in
// flight per SM); 16-byte vectors (K % 8 == 0).
__global__ void __launch_bounds__(256) act_quant_warp_kernel(const __half* __restrict__ src, int64_t rows, int K,
                                                             uint8_t* __restrict__ dst, float* __restrict__ scale) {
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int nvec = K / 8;
  for (int64_t r = warp0; r < rows; r += nwarps) {
    const uint4* row = reinterpret_cast<const uint4*>(src + r * K);
    float amax = 0.f;
    for (int v = lane; v < nvec; v += 32) {
      float f[8];
      unpack8(__ldg(row + v), f);
#pragma unroll
      for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(f[j]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float s = amax > 0.f ? amax / 448.f : 1.f;
    uint2* hi_row = reinterpret_cast<uint2*>(dst + (2 * r) * (int64_t)K);
    uint2* lo_row = reinterpret_cast<uint2*>(dst + (2 * r + 1) * (int64_t)K);
    for (int v = lane; v < nvec; v += 32) {
      float f[8];
      unpack8(__ldg(row + v), f);
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float q0 = __fdiv_rn(f[2 * j], s), q1 = __fdiv_rn(f[2 * j + 1], s);
        hi[j] = e4m3x2(q0, q1);
        const float2 h = e4m3x2_value(hi[j]);
        lo[j] = e4m3x2(q0 - h.x, q1 - h.y);
      }
      hi_row[v] = make_uint2(hi[0] | (hi[1] << 16), hi[2] | (hi[3] << 16));
      lo_row[v] = make_uint2(lo[0] | (lo[1] << 16), lo[2] | (lo[3] << 16));
    }
    if (lane == 0) scale[r] = s;
  }
}


// Small batches: one 256-thread block per row, grid-stride over rows; 16-byte vectors (K %
// 8 == 0). A row's first kQV * 256 vectors are loaded once, all in flight
// together, and kept in registers for both passes (the block-wide max, then
// the split), so a short batch pays one load latency per row; the rest of a
// longer row is read again from L2 in the second pass.
constexpr int kQThreads = 256;
constexpr int kQV = 8;

__global__ void __launch_bounds__(kQThreads, 2) act_quant_block_kernel(const __half* __restrict__ src, int64_t rows, int K,
                                                                    uint8_t* __restrict__ dst, float* __restrict__ scale) {
  pdl_trigger();
  pdl_wait();
  __shared__ float s_max[kQThreads / 32];
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int nvec = K / 8;
  for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
    const uint4* row = reinterpret_cast<const uint4*>(src + r * K);
    uint4 v[kQV];
    float amax = 0.f;
#pragma unroll
    for (int q = 0; q < kQV; ++q) {
      const int i = t + q * kQThreads;
      if (i < nvec) v[q] = __ldg(row + i);
    }
#pragma unroll
    for (int q = 0; q < kQV; ++q)
      if (t + q * kQThreads < nvec) amax = amax8(v[q], amax);
    for (int i = t + kQV * kQThreads; i < nvec; i += kQThreads) amax = amax8(__ldg(row + i), amax);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if (lane == 0) s_max[warp] = amax;
    __syncthreads();
    amax = s_max[0];
#pragma unroll
    for (int w = 1; w < kQThreads / 32; ++w) amax = fmaxf(amax, s_max[w]);
    const float s = amax > 0.f ? amax / 448.f : 1.f;
    uint2* hi_row = reinterpret_cast<uint2*>(dst + (2 * r) * (int64_t)K);
    uint2* lo_row = reinterpret_cast<uint2*>(dst + (2 * r + 1) * (int64_t)K);
#pragma unroll
    for (int q = 0; q < kQV; ++q) {
      const int i = t + q * kQThreads;
      if (i < nvec) quant8(v[q], s, hi_row[i], lo_row[i]);
    }
    for (int i = t + kQV * kQThreads; i < nvec; i += kQThreads) quant8(__ldg(row + i), s, hi_row[i], lo_row[i]);
    if (t == 0) scale[r] = s;
    __syncthreads();  // s_max is rewritten for the next row
  }
}

}  // namespace

cudaError_t launch_act_quant(const void* src, int64_t rows, int32_t K, uint8_t* dst, float* scale, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const __half* x = static_cast<const __half*>(src);
  if (rows <= 2 * (int64_t)sms) return launch(act_quant_block_kernel, (unsigned)rows, kQThreads, 0, s, x, rows, K, dst, scale);
  const int64_t want = (rows + 7) / 8;  // 8 rows (warps) per 256-thread CTA
  const unsigned grid = (unsigned)(want < (int64_t)sms * 8 ? want : (int64_t)sms * 8);
  return launch(act_quant_warp_kernel, grid, 256, 0, s, x, rows, K, dst, scale);
}

}  // namespace moe
