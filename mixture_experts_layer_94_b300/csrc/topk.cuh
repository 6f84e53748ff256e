// topk.cuh — one token's scoring, group limit and top-K on one warp (internal).
//
// "Mixture of Experts for LLM Inference", "Opening the router": softmax scores
// (or, for DeepSeek-V3, a sigmoid affinity), the K largest kept, their weights
// renormalised. "Chapter 19", §19.3.2: the softmax over the chosen logits equals
// the full softmax renormalised over them; §19.3.4: a per-expert bias moves the
// selection only, never the weights. Group-limited routing ("Mixture of Experts
// for LLM Inference", "Three tricks that tame the all-to-alls"): a token picks
// only from its topk_groups best groups of consecutive experts.
//
// Lane l holds experts l, l + 32, ... (EPL of them). Every decision is taken in
// fp32 with ties going to the lower index, so any warp that runs these steps
// on the same logits reaches the same experts and weights.
#pragma once

#include <math.h>

#include "common.cuh"

namespace moe {

// The lane's experts' scores and selection keys from their logits `lg`
// (router bias already added): softmax keeps the logit as both; sigmoid gives
// s = sigmoid(l) and key = s + sel_bias.
template <int EPL>
__device__ __forceinline__ void router_scores(const float (&lg)[EPL], const bool (&valid)[EPL], int lane,
                                              int score_fn, const float* sel_bias, float (&sc)[EPL],
                                              float (&key)[EPL]) {
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    const float l = lg[i];
    if (score_fn == 0) {
      sc[i] = l;
      key[i] = l;
    } else {
      const float sg = 1.0f / (1.0f + expf(-l));
      sc[i] = sg;
      key[i] = sg + ((valid[i] && sel_bias) ? sel_bias[e] : 0.f);
    }
  }
}

// Group-limited routing: a group's score is the sum of its two largest keys
// (its one key for groups of one); the topk_groups best groups (score desc,
// group asc) stay valid, every other expert is dropped from `valid`.
// s_key / s_kept: this warp's scratch in shared memory (N floats, n_groups bytes).
template <int EPL>
__device__ __forceinline__ void router_group_limit(const float (&key)[EPL], bool (&valid)[EPL], int lane, int N,
                                                   int n_groups, int topk_groups, float* s_key,
                                                   unsigned char* s_kept) {
  const int G = n_groups, gs = N / G;
#pragma unroll
  for (int i = 0; i < EPL; ++i)
    if (valid[i]) s_key[lane + 32 * i] = key[i];
  __syncwarp();
  float gsc[kMaxExperts / 32];
#pragma unroll
  for (int j = 0; j < kMaxExperts / 32; ++j) {
    const int g = lane + 32 * j;
    float b1 = -INFINITY, b2 = -INFINITY;
    if (g < G) {
      for (int e = g * gs; e < (g + 1) * gs; ++e) {
        const float v = s_key[e];
        if (v > b1) {
          b2 = b1;
          b1 = v;
        } else if (v > b2) {
          b2 = v;
        }
      }
      gsc[j] = gs > 1 ? b1 + b2 : b1;
      s_kept[g] = 0;
    } else {
      gsc[j] = -INFINITY;
    }
  }
  uint32_t gtaken = 0;
  for (int r = 0; r < topk_groups; ++r) {
    float bv = -INFINITY;
    int bg = 0x7fffffff;
#pragma unroll
    for (int j = 0; j < kMaxExperts / 32; ++j) {
      const int g = lane + 32 * j;
      if (g < G && !((gtaken >> j) & 1u) && (gsc[j] > bv || (gsc[j] == bv && g < bg))) {
        bv = gsc[j];
        bg = g;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int og = __shfl_xor_sync(0xffffffffu, bg, off);
      if (ov > bv || (ov == bv && og < bg)) {
        bv = ov;
        bg = og;
      }
    }
    if (lane == (bg & 31)) {
      gtaken |= 1u << (bg >> 5);
      s_kept[bg] = 1;
    }
  }
  __syncwarp();
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    if (valid[i] && !s_kept[e / gs]) valid[i] = false;
  }
  __syncwarp();
}

// K rounds of a shuffle argmax over (key desc, expert asc) among the valid
// experts; slot k ends in lane k: its expert (`my_e`) and gate weight
// (`my_w`): softmax over the chosen logits or the chosen sigmoid scores over
// their sum; without renormalisation the full-softmax probability over the
// valid experts, or the raw sigmoid score. Lanes >= K get my_e = -1.
template <int EPL>
__device__ __forceinline__ void router_select(const float (&sc)[EPL], const float (&key)[EPL],
                                              const bool (&valid)[EPL], int lane, int K, int score_fn,
                                              int renormalize, int& my_e, float& my_w) {
  uint32_t taken = 0;
  my_e = -1;
  float my_sc = 0.f;
  for (int k = 0; k < K; ++k) {
    float bv = -INFINITY;
    int be = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
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
    const int owner = be & 31, slot = be >> 5;
    float v = 0.f;
#pragma unroll
    for (int i = 0; i < EPL; ++i)
      if (i == slot) v = sc[i];
    if (lane == owner) taken |= 1u << slot;
    v = __shfl_sync(0xffffffffu, v, owner);
    if (lane == k) {
      my_e = be;
      my_sc = v;
    }
  }
  if (score_fn == 0) {
    const float lmax = __shfl_sync(0xffffffffu, my_sc, 0);  // slot 0 holds the largest logit
    const float ex = (lane < K) ? expf(my_sc - lmax) : 0.f;
    float z = 0.f;
    if (renormalize) {
      z = ex;
    } else {
#pragma unroll
      for (int i = 0; i < EPL; ++i)
        if (valid[i]) z += expf(sc[i] - lmax);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
    my_w = ex / z;
  } else {
    float z = (lane < K) ? my_sc : 0.f;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
    my_w = renormalize ? my_sc / z : my_sc;
  }
}

}  // namespace moe
