// act_convert.cuh — hidden rows in the activation format (internal).
#pragma once

#include "common.cuh"

namespace moe {

__device__ __forceinline__ uint4 cvt8_bf16(const float4 p, const float4 q) {
  return make_uint4(pack_bf16x2(p.x, p.y), pack_bf16x2(p.z, p.w), pack_bf16x2(q.x, q.y), pack_bf16x2(q.z, q.w));
}

__device__ __forceinline__ float4 bf16x4_to_f32(uint32_t lo, uint32_t hi) {
  return make_float4(__uint_as_float(lo << 16), __uint_as_float(lo & 0xFFFF0000u), __uint_as_float(hi << 16),
                     __uint_as_float(hi & 0xFFFF0000u));
}

// 8 values to fp16 (round to nearest even). `over` is set when a finite value
// lies beyond fp16's range (|v| >= 65520 rounds to infinity).
__device__ __forceinline__ uint4 cvt8_f16(const float4 p, const float4 q, bool& over) {
  const float m = fmaxf(fmaxf(fmaxf(fabsf(p.x), fabsf(p.y)), fmaxf(fabsf(p.z), fabsf(p.w))),
                        fmaxf(fmaxf(fabsf(q.x), fabsf(q.y)), fmaxf(fabsf(q.z), fabsf(q.w))));
  over |= (m >= 65520.f) && (m <= 3.402823466e38f);
  return make_uint4(pack_f16x2(p.x, p.y), pack_f16x2(p.z, p.w), pack_f16x2(q.x, q.y), pack_f16x2(q.z, q.w));
}

// One 16-byte vector (8 elements, vector v) of row t of hidden ([T][d], bf16
// or fp32) in the activation format: bf16, or fp16 when act_f16.
__device__ __forceinline__ uint4 hidden_vec(const void* hidden, bool hidden_bf16, int d, int64_t t, int v,
                                            bool act_f16, bool& over) {
  if (hidden_bf16) {
    const uint4 x = __ldg(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(hidden) + t * d) + v);
    if (!act_f16) return x;
    return cvt8_f16(bf16x4_to_f32(x.x, x.y), bf16x4_to_f32(x.z, x.w), over);
  }
  const float4* sp = reinterpret_cast<const float4*>(static_cast<const float*>(hidden) + t * d);
  const float4 p = __ldg(sp + 2 * v), q = __ldg(sp + 2 * v + 1);
  return act_f16 ? cvt8_f16(p, q, over) : cvt8_bf16(p, q);
}

}  // namespace moe
