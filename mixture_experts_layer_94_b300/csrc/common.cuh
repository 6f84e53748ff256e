// common.cuh — shared device helpers of libmoe (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

// Bits of the device error word (first 4 bytes of every workspace).
constexpr uint32_t kErrTimeout = 1u;  // a bounded pipeline wait gave up
constexpr uint32_t kErrBounds = 2u;   // an input index was out of range
constexpr uint32_t kErrRange = 4u;    // an fp16 activation (FP8-weight experts) overflowed

// Bound on any single pipeline wait. The longest legitimate wait in this
// library is one output tile of MMA work (well under a millisecond), so two
// seconds only ever trips on a genuine stall.
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;

constexpr int kTokensPerChunk = 32;  // route-and-pack chunk: one warp, one token per lane
constexpr int kMaxExperts = 256;
constexpr int kMaxTopK = 32;
constexpr int kMaxShared = 8;

// GEMM tiling shared by host and device.
constexpr int kBM = 128;        // rows of the activation tile (MMA M)
constexpr int kBK = 64;         // K elements per pipeline stage (128 B of bf16 = one swizzle atom)
constexpr int kBNGateUp = 128;  // gate columns per tile (the up tile adds another 128 -> MMA N = 256)
constexpr int kBNDown = 256;    // output columns per down-projection tile (MMA N = 256)

// One GEMM group: a routed expert (kind 0) or a shared expert (kind 1).
struct GroupDesc {
  int32_t kind;       // 0 routed, 1 shared
  int32_t index;      // expert index within its kind
  int32_t a_row0;     // first row of the group in its activation matrix
  int32_t rows;       // rows of the group
  int32_t m_tiles;    // ceil(rows / kBM)
  int32_t h_row0;     // first row in the group's h / y matrix
  int32_t pad0, pad1;
};

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + __expf(-z)); }

}  // namespace moe
