// router.cu — router logits, scoring, top-K and gate weights.
//
// "Mixture of Experts for LLM Inference", section "Opening the router": one raw
// score per expert from a small linear layer, a softmax (or, for DeepSeek-V3, a
// sigmoid affinity), top-K, renormalisation of the survivors.
// "Chapter 19: Mixture-of-Experts Models", §19.3.2: softmax over the chosen
// logits equals full softmax + renormalisation; §19.3.4: the balancing bias
// shifts the scores used for selection only.
//
// Design: a CTA takes 32 tokens; d is walked in 32-wide chunks staged in shared
// memory (the router matrix chunk is shared by all 32 tokens). Each warp owns 4
// tokens and keeps their logits in registers, fp32 FMA. Lanes split the experts
// (lane owns experts lane, lane+32, ... when N > 32) or, for N <= 32, split d
// into 32/Npad lane groups that are reduced by shuffles at the end. Top-K is a
// K-round shuffle argmax over (key desc, expert asc); slot k ends in lane k.
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kRouterWarps = 8;
constexpr int kTokPerWarp = 4;
constexpr int kTokPerCta = kRouterWarps * kTokPerWarp;  // 32
constexpr int kDChunk = 32;

template <typename T>
__device__ __forceinline__ float load_as_float(const T* p);
template <>
__device__ __forceinline__ float load_as_float<float>(const float* p) {
  return *p;
}
template <>
__device__ __forceinline__ float load_as_float<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}

// EPL: experts per lane (N > 32), LPE: lanes per expert (N <= 32; d split).
template <int EPL, int LPE, typename XT>
__global__ void __launch_bounds__(kRouterWarps * 32) router_topk_kernel(const RouterArgs a) {
  constexpr int NCOL = (LPE == 1) ? 32 * EPL : 32 / LPE;  // staged router columns
  __shared__ float ws[kDChunk][NCOL];
  __shared__ float xs[kTokPerCta][kDChunk];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t t0 = (int64_t)blockIdx.x * kTokPerCta;
  const XT* __restrict__ x = static_cast<const XT*>(a.hidden);
  const int N = a.N, d = a.d;

  const int ecol = (LPE == 1) ? lane : (lane % NCOL);  // lane's first expert column
  const int jgrp = (LPE == 1) ? 0 : (lane / NCOL);     // lane's d sub-lattice

  float acc[kTokPerWarp][EPL];
#pragma unroll
  for (int t = 0; t < kTokPerWarp; ++t)
#pragma unroll
    for (int i = 0; i < EPL; ++i) acc[t][i] = 0.f;

  for (int j0 = 0; j0 < d; j0 += kDChunk) {
    for (int i = tid; i < kDChunk * NCOL; i += kRouterWarps * 32) {
      const int j = i / NCOL, e = i % NCOL;
      ws[j][e] = (e < N && j0 + j < d) ? a.w_router[(int64_t)(j0 + j) * N + e] : 0.f;
    }
    for (int i = tid; i < kTokPerCta * kDChunk; i += kRouterWarps * 32) {
      const int tk = i / kDChunk, j = i % kDChunk;
      const int64_t t = t0 + tk;
      xs[tk][j] = (t < a.T && j0 + j < d) ? load_as_float<XT>(x + t * d + j0 + j) : 0.f;
    }
    __syncthreads();
#pragma unroll 4
    for (int jj = 0; jj < kDChunk / LPE; ++jj) {
      const int j = jj * LPE + jgrp;
      float w[EPL];
#pragma unroll
      for (int i = 0; i < EPL; ++i) w[i] = ws[j][ecol + 32 * i];
#pragma unroll
      for (int t = 0; t < kTokPerWarp; ++t) {
        const float xv = xs[warp * kTokPerWarp + t][j];
#pragma unroll
        for (int i = 0; i < EPL; ++i) acc[t][i] = fmaf(xv, w[i], acc[t][i]);
      }
    }
    __syncthreads();
  }
  if (LPE > 1) {
#pragma unroll
    for (int off = NCOL; off < 32; off <<= 1)
#pragma unroll
      for (int t = 0; t < kTokPerWarp; ++t) acc[t][0] += __shfl_xor_sync(0xffffffffu, acc[t][0], off);
  }

  const int K = a.K;
#pragma unroll
  for (int tk = 0; tk < kTokPerWarp; ++tk) {
    const int64_t t = t0 + warp * kTokPerWarp + tk;
    if (t >= a.T) continue;  // uniform across the warp
    float key[EPL], sc[EPL];
    bool valid[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = ecol + 32 * i;
      valid[i] = (e < N) && (jgrp == 0);
      float l = acc[tk][i];
      if (valid[i] && a.router_bias) l += a.router_bias[e];
      if (valid[i] && a.logits) a.logits[t * N + e] = l;
      if (a.score_fn == 0) {
        sc[i] = l;
        key[i] = l;
      } else {
        const float s = 1.0f / (1.0f + expf(-l));
        sc[i] = s;
        key[i] = s + ((valid[i] && a.sel_bias) ? a.sel_bias[e] : 0.f);
      }
    }
    uint32_t taken = 0;
    int my_e = -1;
    float my_sc = 0.f;
    for (int k = 0; k < K; ++k) {
      float bv = -INFINITY;
      int be = 0x7fffffff;
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        const int e = ecol + 32 * i;
        if (valid[i] && !((taken >> i) & 1u) && (key[i] > bv || (key[i] == bv && e < be))) {
          bv = key[i];
          be = e;
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
        const int oe = __shfl_xor_sync(0xffffffffu, be, off);
        if (ov > bv || (ov == bv && oe < be)) {
          bv = ov;
          be = oe;
        }
      }
      // Owner of expert be: lane (be % 32) slot be/32 (N > 32) or lane be (N <= 32).
      const int owner = (LPE == 1) ? (be & 31) : be;
      const int slot = (LPE == 1) ? (be >> 5) : 0;
      float v = 0.f;
#pragma unroll
      for (int i = 0; i < EPL; ++i)
        if (i == slot) v = sc[i];
      if (lane == owner) taken |= 1u << slot;
      v = __shfl_sync(0xffffffffu, v, owner & 31);
      if (lane == k) {
        my_e = be;
        my_sc = v;
      }
    }
    float w;
    if (a.score_fn == 0) {
      const float lmax = __shfl_sync(0xffffffffu, my_sc, 0);  // slot 0 holds the largest logit
      const float ex = (lane < K) ? expf(my_sc - lmax) : 0.f;
      float z = 0.f;
      if (a.renormalize) {
        z = ex;
      } else {
#pragma unroll
        for (int i = 0; i < EPL; ++i)
          if (valid[i]) z += expf(sc[i] - lmax);
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
      w = ex / z;
    } else {
      float z = (lane < K) ? my_sc : 0.f;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
      w = a.renormalize ? my_sc / z : my_sc;
    }
    if (lane < K) {
      a.topk_idx[t * K + lane] = my_e;
      a.topk_w[t * K + lane] = w;
    }
  }
}

template <typename XT>
cudaError_t launch_router_t(const RouterArgs& a, cudaStream_t s) {
  const dim3 grid((unsigned)((a.T + kTokPerCta - 1) / kTokPerCta));
  const dim3 block(kRouterWarps * 32);
  const int N = a.N;
  if (N <= 1) router_topk_kernel<1, 32, XT><<<grid, block, 0, s>>>(a);
  else if (N <= 2) router_topk_kernel<1, 16, XT><<<grid, block, 0, s>>>(a);
  else if (N <= 4) router_topk_kernel<1, 8, XT><<<grid, block, 0, s>>>(a);
  else if (N <= 8) router_topk_kernel<1, 4, XT><<<grid, block, 0, s>>>(a);
  else if (N <= 16) router_topk_kernel<1, 2, XT><<<grid, block, 0, s>>>(a);
  else if (N <= 32) router_topk_kernel<1, 1, XT><<<grid, block, 0, s>>>(a);
  else if (N <= 64) router_topk_kernel<2, 1, XT><<<grid, block, 0, s>>>(a);
  else if (N <= 128) router_topk_kernel<4, 1, XT><<<grid, block, 0, s>>>(a);
  else router_topk_kernel<8, 1, XT><<<grid, block, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_router(const RouterArgs& a, bool hidden_bf16, cudaStream_t s) {
  if (a.T == 0) return cudaSuccess;
  return hidden_bf16 ? launch_router_t<__nv_bfloat16>(a, s) : launch_router_t<float>(a, s);
}

}  // namespace moe
