// router.cu — router logits, scoring, top-K and gate weights.
//
// "Mixture of Experts for LLM Inference", section "Opening the router": one raw
// score per expert from a small linear layer, a softmax (or, for DeepSeek-V3, a
// sigmoid affinity), top-K, renormalisation of the survivors.
// "Chapter 19: Mixture-of-Experts Models", §19.3.2: softmax over the chosen
// logits equals full softmax + renormalisation; §19.3.4: the balancing bias
// shifts the scores used for selection only.
//
// fp32 throughout (the router is kept in higher precision than the experts,
// "Chapter 19", §19.6.2 table). For a bf16 hidden of more than 64 tokens the
// logits run on the tensor cores (the grouped GEMM's router phase, see
// split_router_kernel below); for an fp32 hidden or a small batch, on CUDA
// cores:
//   R1 router_logits: partial logits over a slice of d, for a tile of tokens.
//      The d axis is split into S slices when there are too few token tiles to
//      fill the GPU (decode batches), so every SM streams part of W_router.
//      N <= 32: lanes split d (8 consecutive inputs per lane, 16-byte loads),
//      each lane keeps TPW tokens x N logits in registers, and a butterfly
//      reduction ends the tile. N > 32: lanes split the experts (lane owns
//      experts lane, lane+32, ...), each warp owns 4 tokens, and 32-wide chunks
//      of hidden and W_router are staged in shared memory with the next chunk
//      prefetched into registers while the current one is consumed.
//   R2 router_topk: one warp per token sums the S partials in a fixed order
//      (deterministic), adds the router bias, scores, and selects K by a
//      K-round shuffle argmax over (key desc, expert asc); slot k ends in lane k.
#include <math.h>

#include <atomic>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "topk.cuh"

namespace moe {
namespace {

constexpr int kWarps = 8;

template <typename XT>
__device__ __forceinline__ void load8(const XT* p, float (&v)[8]);
template <>
__device__ __forceinline__ void load8<float>(const float* p, float (&v)[8]) {
  const float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

template <>
__device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16* p, float (&v)[8]) {
  const uint4 a = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    v[2 * q] = __uint_as_float(w[q] << 16);
    v[2 * q + 1] = __uint_as_float(w[q] & 0xFFFF0000u);
  }
}

template <typename T>
__device__ __forceinline__ float to_f(T v);
template <>
__device__ __forceinline__ float to_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

// ---------------------------------------------------------------- R1, N <= 32
// NP: N rounded up to a power of two; TPW tokens per warp.
template <int NP, int TPW, typename XT>
__global__ void __launch_bounds__(kWarps * 32) logits_small_n_kernel(const RouterArgs a) {
  pdl_trigger();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = a.N, d = a.d;
  const int64_t t0 = ((int64_t)blockIdx.x * kWarps + warp) * TPW;
  if (t0 >= a.T) return;
  const int s = blockIdx.y;
  const int j_begin = s * a.d_slice, j_end = min(d, j_begin + a.d_slice);
  const XT* x = static_cast<const XT*>(a.hidden);
  float acc[TPW][NP];
#pragma unroll
  for (int t = 0; t < TPW; ++t)
#pragma unroll
    for (int e = 0; e < NP; ++e) acc[t][e] = 0.f;
  const bool vec_w = (N == NP) && (NP % 4 == 0);
  for (int j0 = j_begin + lane * 8; j0 < j_end; j0 += 256) {
    float xv[TPW][8];
#pragma unroll
    for (int t = 0; t < TPW; ++t) {
      if (t0 + t < a.T) load8<XT>(x + (t0 + t) * d + j0, xv[t]);
      else {
#pragma unroll
        for (int q = 0; q < 8; ++q) xv[t][q] = 0.f;
      }
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float* wrow = a.w_router + (int64_t)(j0 + q) * N;
      float w[NP];
      if (vec_w) {
#pragma unroll
        for (int e = 0; e < NP; e += 4) {
          const float4 v = __ldg(reinterpret_cast<const float4*>(wrow + e));
          w[e] = v.x; w[e + 1] = v.y; w[e + 2] = v.z; w[e + 3] = v.w;
        }
      } else {
#pragma unroll
        for (int e = 0; e < NP; ++e) w[e] = (e < N) ? __ldg(wrow + e) : 0.f;
      }
#pragma unroll
      for (int t = 0; t < TPW; ++t)
#pragma unroll
        for (int e = 0; e < NP; ++e) acc[t][e] = fmaf(xv[t][q], w[e], acc[t][e]);
    }
  }
#pragma unroll
  for (int t = 0; t < TPW; ++t)
#pragma unroll
    for (int e = 0; e < NP; ++e)
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc[t][e] += __shfl_xor_sync(0xffffffffu, acc[t][e], off);
  float* part = a.partial + (int64_t)s * a.T * N;
#pragma unroll
  for (int t = 0; t < TPW; ++t) {
    if (t0 + t >= a.T) break;
    float v = 0.f;
#pragma unroll
    for (int e = 0; e < NP; ++e)
      if (e == lane) v = acc[t][e];
    if (lane < N) part[(t0 + t) * N + lane] = v;
  }
}

// ---------------------------------------------------------------- R1, N > 32
constexpr int kTokPerWarpL = 4;
constexpr int kTokPerCtaL = kWarps * kTokPerWarpL;  // 32
constexpr int kDChunk = 32;

template <int EPL, typename XT>
__global__ void __launch_bounds__(kWarps * 32) logits_large_n_kernel(const RouterArgs a) {
  pdl_trigger();
  pdl_wait();
  constexpr int NCOL = 32 * EPL;
  constexpr int W_PER_THR = kDChunk * NCOL / (kWarps * 32);       // EPL * 4
  constexpr int X_PER_THR = kTokPerCtaL * kDChunk / (kWarps * 32);  // 4
  __shared__ float ws[kDChunk][NCOL];
  __shared__ float xs[kTokPerCtaL][kDChunk];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t t0 = (int64_t)blockIdx.x * kTokPerCtaL;
  const int N = a.N, d = a.d;
  const int s = blockIdx.y;
  const int j_begin = s * a.d_slice, j_end = min(d, j_begin + a.d_slice);
  const XT* x = static_cast<const XT*>(a.hidden);

  float acc[kTokPerWarpL][EPL];
#pragma unroll
  for (int t = 0; t < kTokPerWarpL; ++t)
#pragma unroll
    for (int i = 0; i < EPL; ++i) acc[t][i] = 0.f;

  float wr[W_PER_THR], xr[X_PER_THR];
  auto fetch = [&](int j0) {
#pragma unroll
    for (int q = 0; q < W_PER_THR; ++q) {
      const int i = tid + q * kWarps * 32;
      const int j = i / NCOL, e = i % NCOL;
      wr[q] = (e < N && j0 + j < j_end) ? __ldg(a.w_router + (int64_t)(j0 + j) * N + e) : 0.f;
    }
#pragma unroll
    for (int q = 0; q < X_PER_THR; ++q) {
      const int i = tid + q * kWarps * 32;
      const int tk = i / kDChunk, j = i % kDChunk;
      const int64_t t = t0 + tk;
      xr[q] = (t < a.T && j0 + j < j_end) ? to_f<XT>(x[t * d + j0 + j]) : 0.f;
    }
  };
  auto stash = [&]() {
#pragma unroll
    for (int q = 0; q < W_PER_THR; ++q) {
      const int i = tid + q * kWarps * 32;
      ws[i / NCOL][i % NCOL] = wr[q];
    }
#pragma unroll
    for (int q = 0; q < X_PER_THR; ++q) {
      const int i = tid + q * kWarps * 32;
      xs[i / kDChunk][i % kDChunk] = xr[q];
    }
  };
  fetch(j_begin);
  for (int j0 = j_begin; j0 < j_end; j0 += kDChunk) {
    __syncthreads();  // previous chunk fully consumed
    stash();
    __syncthreads();
    if (j0 + kDChunk < j_end) fetch(j0 + kDChunk);  // in flight during the FMAs below
#pragma unroll 8
    for (int j = 0; j < kDChunk; ++j) {
      float w[EPL];
#pragma unroll
      for (int i = 0; i < EPL; ++i) w[i] = ws[j][lane + 32 * i];
#pragma unroll
      for (int t = 0; t < kTokPerWarpL; ++t) {
        const float xv = xs[warp * kTokPerWarpL + t][j];
#pragma unroll
        for (int i = 0; i < EPL; ++i) acc[t][i] = fmaf(xv, w[i], acc[t][i]);
      }
    }
  }
  float* part = a.partial + (int64_t)s * a.T * N;
#pragma unroll
  for (int t = 0; t < kTokPerWarpL; ++t) {
    const int64_t tt = t0 + warp * kTokPerWarpL + t;
    if (tt >= a.T) break;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      if (e < N) part[tt * N + e] = acc[t][i];
    }
  }
}

// ---------------------------------------------------------------- R1, N > 32, staged
// The same partial logits when a CTA's d slice fits in shared memory (decode
// batches): the slice of W_router (rows j_begin.., N floats each, contiguous)
// and of the tile's 32 token rows are copied in with cp.async, every 16-byte
// piece in flight at once, so the CTA pays one load latency instead of one per
// 32-row chunk; then the FMAs read shared memory only. N % 4 == 0 and d % 8 ==
// 0 (16-byte pieces of both rows).
constexpr size_t kStagedMaxSmem = 100 * 1024;

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, bool valid) {
  const uint32_t sa = (uint32_t)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(sa), "l"(gmem), "r"(valid ? 16 : 0)
               : "memory");
}

template <int EPL, typename XT>
size_t staged_smem(int d_slice) {
  return (size_t)d_slice * 32 * EPL * sizeof(float) + (size_t)kTokPerCtaL * d_slice * sizeof(XT);
}

template <int EPL, typename XT>
__global__ void __launch_bounds__(kWarps * 32) logits_staged_kernel(const RouterArgs a) {
  pdl_trigger();
  pdl_wait();
  constexpr int NCOL = 32 * EPL;
  constexpr int XV = 16 / sizeof(XT);  // elements of hidden per 16-byte piece
  extern __shared__ __align__(16) float st[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t t0 = (int64_t)blockIdx.x * kTokPerCtaL;
  const int N = a.N, d = a.d, ds = a.d_slice;
  const int j_begin = blockIdx.y * ds, jn = min(d - j_begin, ds);
  float* ws = st;                                         // [ds][NCOL]
  XT* xs = reinterpret_cast<XT*>(st + (size_t)ds * NCOL);  // [kTokPerCtaL][ds]
  const XT* x = static_cast<const XT*>(a.hidden);
  for (int i = tid; i < ds * (NCOL / 4); i += kWarps * 32) {
    const int j = i / (NCOL / 4), c = 4 * (i % (NCOL / 4));
    const bool ok = j < jn && c < N;
    cp_async16(ws + j * NCOL + c, ok ? a.w_router + (int64_t)(j_begin + j) * N + c : a.w_router, ok);
  }
  for (int i = tid; i < kTokPerCtaL * (ds / XV); i += kWarps * 32) {
    const int tk = i / (ds / XV), c = XV * (i % (ds / XV));
    const bool ok = t0 + tk < a.T && c < jn;
    cp_async16(xs + tk * ds + c, ok ? x + (t0 + tk) * d + j_begin + c : x, ok);
  }
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
  __syncthreads();
  float acc[kTokPerWarpL][EPL];
#pragma unroll
  for (int t = 0; t < kTokPerWarpL; ++t)
#pragma unroll
    for (int i = 0; i < EPL; ++i) acc[t][i] = 0.f;
  const XT* xw = xs + warp * kTokPerWarpL * ds;
#pragma unroll 4
  for (int j = 0; j < jn; ++j) {
    float w[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) w[i] = ws[j * NCOL + lane + 32 * i];
#pragma unroll
    for (int t = 0; t < kTokPerWarpL; ++t) {
      const float xv = to_f<XT>(xw[t * ds + j]);
#pragma unroll
      for (int i = 0; i < EPL; ++i) acc[t][i] = fmaf(xv, w[i], acc[t][i]);
    }
  }
  float* part = a.partial + (int64_t)blockIdx.y * a.T * N;
#pragma unroll
  for (int t = 0; t < kTokPerWarpL; ++t) {
    const int64_t tt = t0 + warp * kTokPerWarpL + t;
    if (tt >= a.T) break;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      if (e < N) part[tt * N + e] = acc[t][i];
    }
  }
}

// ---------------------------------------------------------------- R2
template <int EPL>
__global__ void __launch_bounds__(kWarps * 32) topk_kernel(const RouterArgs a) {
  pdl_trigger();
  pdl_wait();
  __shared__ float s_key[kWarps][kMaxExperts];
  __shared__ unsigned char s_kept[kWarps][kMaxExperts];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t t = (int64_t)blockIdx.x * kWarps + warp;
  if (t >= a.T) return;
  const int N = a.N, K = a.K;
  float key[EPL], sc[EPL], lg[EPL];
  bool valid[EPL];
  // Partials summed in split order (deterministic). All of a lane's experts
  // load kSplitBatch splits at a time, so EPL x kSplitBatch loads are in
  // flight together (two round trips for the 32 splits of a decode batch).
  {
    constexpr int kSplitBatch = EPL <= 4 ? 16 : 8;
    const int64_t stride = a.T * N;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      valid[i] = lane + 32 * i < N;
      lg[i] = 0.f;
    }
    for (int s0 = 0; s0 < a.splits; s0 += kSplitBatch) {
      float v[EPL][kSplitBatch];
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        const float* pp = a.partial + t * N + lane + 32 * i;
#pragma unroll
        for (int q = 0; q < kSplitBatch; ++q)
          v[i][q] = (valid[i] && s0 + q < a.splits) ? __ldg(pp + (int64_t)(s0 + q) * stride) : 0.f;
      }
#pragma unroll
      for (int i = 0; i < EPL; ++i)
#pragma unroll
        for (int q = 0; q < kSplitBatch; ++q) lg[i] += v[i][q];
    }
  }
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    if (valid[i]) {
      if (a.router_bias) lg[i] += a.router_bias[e];
      if (a.logits) a.logits[t * N + e] = lg[i];
    }
  }
  router_scores<EPL>(lg, valid, lane, a.score_fn, a.sel_bias, sc, key);
  if (a.n_groups > 1 && a.topk_groups < a.n_groups)
    router_group_limit<EPL>(key, valid, lane, N, a.n_groups, a.topk_groups, s_key[warp], s_kept[warp]);
  if (a.scores_t) {
    // Expert choice: the token's score for every expert, stored transposed
    // (S[e][t]) for the per-expert selection.
    float sv[EPL];
    if (a.score_fn == 0) {
      float mx = -INFINITY;
#pragma unroll
      for (int i = 0; i < EPL; ++i)
        if (valid[i]) mx = fmaxf(mx, sc[i]);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      float z = 0.f;
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        sv[i] = valid[i] ? expf(sc[i] - mx) : 0.f;
        z += sv[i];
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
#pragma unroll
      for (int i = 0; i < EPL; ++i) sv[i] /= z;
    } else {
#pragma unroll
      for (int i = 0; i < EPL; ++i) sv[i] = sc[i];
    }
#pragma unroll
    for (int i = 0; i < EPL; ++i)
      if (valid[i]) a.scores_t[(int64_t)(lane + 32 * i) * a.T + t] = sv[i];
    return;
  }
  int my_e;
  float w;
  router_select<EPL>(sc, key, valid, lane, K, a.score_fn, a.renormalize, my_e, w);
  if (lane < K) {
    a.topk_idx[t * K + lane] = my_e;
    a.topk_w[t * K + lane] = w;
  }
}

// ---------------------------------------------------------------- tensor-core path
// W3[e][part * d_pad + j] for part 0, 1, 2 = hi, mid, lo with
//   hi = bf16(w), mid = bf16(w - hi), lo = bf16(w - hi - mid),  w = W_router[j][e].
// hi + mid + lo == w exactly for every normal fp32 w (8 + 8 + 8 significand
// bits), and each bf16 x bf16 product is exact in fp32, so hidden x W3 over the
// three parts is an fp32 dot product. Rows e >= N and columns j >= d are zero.
// 32 x 32 tiles through shared memory: coalesced reads along e, writes along j.
__global__ void __launch_bounds__(256) split_router_kernel(const float* __restrict__ w, int d, int N, int np,
                                                           int d_pad, __nv_bfloat16* __restrict__ w3) {
  pdl_trigger();
  pdl_wait();
  __shared__ float tile[32][33];
  const int j0 = blockIdx.x * 32, e0 = blockIdx.y * 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8
  for (int r = ty; r < 32; r += 8) {
    const int j = j0 + r, e = e0 + tx;
    tile[r][tx] = (j < d && e < N) ? w[(int64_t)j * N + e] : 0.f;
  }
  __syncthreads();
  for (int r = ty; r < 32; r += 8) {
    const int e = e0 + r, j = j0 + tx;
    if (e < np && j < d_pad) {
      const float v = tile[tx][r];
      const __nv_bfloat16 hi = __float2bfloat16_rn(v);
      const float r1 = v - __bfloat162float(hi);
      const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
      const __nv_bfloat16 lo = __float2bfloat16_rn(r1 - __bfloat162float(mid));
      __nv_bfloat16* row = w3 + (int64_t)e * 3 * d_pad;
      row[j] = hi;
      row[d_pad + j] = mid;
      row[2 * d_pad + j] = lo;
    }
  }
}

cudaError_t launch_tensor_logits(const RouterArgs& a, const RouterPlan& pl, cudaStream_t s) {
  const dim3 sgrid((unsigned)((pl.d_pad + 31) / 32), (unsigned)((pl.np + 31) / 32));
  if (const cudaError_t le_ = launch(split_router_kernel, sgrid, 256, 0, s, a.w_router, a.d, a.N, pl.np, pl.d_pad, a.w3); le_ != cudaSuccess) return le_;
  GemmMaps m{};
  if (!make_tmap_bf16(&m.a[0], a.hidden, (uint64_t)a.d, (uint64_t)a.T, kBM) ||
      !make_tmap_bf16(&m.b[0], a.w3, (uint64_t)3 * pl.d_pad, (uint64_t)pl.np, (uint32_t)pl.np))
    return cudaErrorInvalidValue;
  m.a[1] = m.a[0];
  m.b[1] = m.bu[0] = m.bu[1] = m.b[0];
  m.bh[0] = m.bh[1] = m.uh[0] = m.uh[1] = m.b[0];
  GemmArgs g{};
  g.err = nullptr;
  g.r_m_tiles = (int32_t)pl.token_tiles;
  g.r_dslices = pl.dslices;
  g.r_kb_per_slice = pl.kb_per_slice;
  g.r_nkb_d = pl.nkb_d;
  g.r_d_pad = pl.d_pad;
  g.r_np = pl.np;
  g.r_merged = pl.merged ? 1 : 0;
  g.r_N = a.N;
  g.r_T = a.T;
  g.r_tiles = (int32_t)(pl.token_tiles * pl.splits);
  g.r_idesc = ptx::idesc_bf16_f32(128, pl.np);
  g.r_partial = a.partial;
  return launch_grouped_gemm(kPhaseRouter, kEpiLogits, 1, m, g, g.r_tiles, s);
}

// ---------------------------------------------------------------- expert choice
// One CTA per expert: the C-th largest score key is found by a 4-pass radix
// select over the 32-bit keys (scores are >= 0, so their bit patterns order
// like the values), then the tokens with a larger key, and the lowest-indexed
// tokens equal to it, are written in ascending token order. Two block-wide
// scans (ties, then picks) keep the result deterministic.
constexpr int kSelThreads = 1024;

__device__ __forceinline__ int block_exclusive_scan(int v, int* s_warp, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int w = lane < (kSelThreads / 32) ? s_warp[lane] : 0;
    int wi = w;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, wi, off);
      if (lane >= off) wi += o;
    }
    s_warp[lane] = wi - w;  // exclusive prefix of warp sums
    if (lane == 31) s_warp[32] = wi;
  }
  __syncthreads();
  const int res = s_warp[warp] + incl - v;
  total = s_warp[32];
  __syncthreads();
  return res;
}

__global__ void __launch_bounds__(kSelThreads) expert_choice_select_kernel(const float* __restrict__ scores_t,
                                                                            int64_t T, int32_t N, int32_t C,
                                                                            int32_t* row_token, float* row_w,
                                                                            int32_t* offsets, int32_t* counts) {
  pdl_trigger();
  pdl_wait();
  __shared__ int hist[256];
  __shared__ int s_warp[33];
  __shared__ uint32_t s_prefix;
  __shared__ int s_need;
  const int e = blockIdx.x;
  const uint32_t* keys = reinterpret_cast<const uint32_t*>(scores_t) + (int64_t)e * T;
  uint32_t prefix = 0, pmask = 0;
  int need = C;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    for (int64_t t = threadIdx.x; t < T; t += blockDim.x) {
      const uint32_t k = __ldg(keys + t);
      if ((k & pmask) == prefix) atomicAdd(&hist[(k >> shift) & 255u], 1);
    }
    __syncthreads();
    if (threadIdx.x == 0) {  // the bin holding the need-th largest key
      int above = 0, b = 255;
      for (; b > 0; --b) {
        if (above + hist[b] >= need) break;
        above += hist[b];
      }
      s_prefix = prefix | ((uint32_t)b << shift);
      s_need = need - above;
    }
    __syncthreads();
    prefix = s_prefix;
    need = s_need;
    pmask |= 255u << shift;
    __syncthreads();
  }
  // prefix: the C-th largest key; `need` tokens equal to it are taken (lowest
  // indices first). Each thread owns a contiguous run of tokens.
  const int64_t per = (T + blockDim.x - 1) / blockDim.x;
  const int64_t t0 = min((int64_t)threadIdx.x * per, T), t1 = min(t0 + per, T);
  int n_eq = 0;
  for (int64_t t = t0; t < t1; ++t) n_eq += __ldg(keys + t) == prefix;
  int tot;
  const int eq_before = block_exclusive_scan(n_eq, s_warp, tot);
  int n_pick = 0, eq_seen = eq_before;
  for (int64_t t = t0; t < t1; ++t) {
    const uint32_t k = __ldg(keys + t);
    if (k > prefix) ++n_pick;
    else if (k == prefix) n_pick += (eq_seen++ < need);
  }
  int pos = block_exclusive_scan(n_pick, s_warp, tot);
  eq_seen = eq_before;
  for (int64_t t = t0; t < t1; ++t) {
    const uint32_t k = __ldg(keys + t);
    const bool take = k > prefix || (k == prefix && eq_seen++ < need);
    if (take) {
      row_token[(int64_t)e * C + pos] = (int32_t)t;
      row_w[(int64_t)e * C + pos] = __uint_as_float(k);
      ++pos;
    }
  }
  if (threadIdx.x == 0) {
    offsets[e] = e * C;
    if (e == N - 1) offsets[N] = N * C;
    if (counts) counts[e] = C;
  }
}

// N > 32: the staged kernel when the slice fits in shared memory and the rows
// split into 16-byte pieces, else the chunked one.
template <int EPL, typename XT>
cudaError_t launch_large_n(const RouterArgs& a, const RouterPlan& pl, dim3 grid, dim3 block, cudaStream_t s) {
  const size_t smem = staged_smem<EPL, XT>(pl.d_slice);
  if (a.N % 4 == 0 && a.d % 8 == 0 && smem <= kStagedMaxSmem) {
    static std::atomic<uint64_t> configured{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(configured.load() & bit)) {
      e = cudaFuncSetAttribute(logits_staged_kernel<EPL, XT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)kStagedMaxSmem);
      if (e != cudaSuccess) return e;
      configured.fetch_or(bit);
    }
    return launch(logits_staged_kernel<EPL, XT>, grid, block, smem, s, a);
  }
  return launch(logits_large_n_kernel<EPL, XT>, grid, block, 0, s, a);
}

template <typename XT>
cudaError_t launch_logits(const RouterArgs& a, const RouterPlan& pl, cudaStream_t s) {
  const dim3 grid((unsigned)pl.token_tiles, (unsigned)pl.splits), block(kWarps * 32);
  const int N = a.N;
  if (N <= 32) {
    if (pl.np == 1) { if (const cudaError_t le_ = launch(logits_small_n_kernel<1, 4, XT>, grid, block, 0, s, a); le_ != cudaSuccess) return le_; }
    else if (pl.np == 2) { if (const cudaError_t le_ = launch(logits_small_n_kernel<2, 4, XT>, grid, block, 0, s, a); le_ != cudaSuccess) return le_; }
    else if (pl.np == 4) { if (const cudaError_t le_ = launch(logits_small_n_kernel<4, 4, XT>, grid, block, 0, s, a); le_ != cudaSuccess) return le_; }
    else if (pl.np == 8) { if (const cudaError_t le_ = launch(logits_small_n_kernel<8, 4, XT>, grid, block, 0, s, a); le_ != cudaSuccess) return le_; }
    else if (pl.np == 16) { if (const cudaError_t le_ = launch(logits_small_n_kernel<16, 2, XT>, grid, block, 0, s, a); le_ != cudaSuccess) return le_; }
    else { if (const cudaError_t le_ = launch(logits_small_n_kernel<32, 1, XT>, grid, block, 0, s, a); le_ != cudaSuccess) return le_; }
  } else if (N <= 64) {
    return launch_large_n<2, XT>(a, pl, grid, block, s);
  } else if (N <= 128) {
    return launch_large_n<4, XT>(a, pl, grid, block, s);
  } else {
    return launch_large_n<8, XT>(a, pl, grid, block, s);
  }
  return cudaSuccess;
}

}  // namespace

// Batches of at most this many tokens take the CUDA-core logits kernels even
// with a bf16 hidden: they read the fp32 router matrix once, split over d
// across CTAs, instead of splitting it into three bf16 parts for a tensor-core
// GEMM with a single token tile.
constexpr int64_t kCudaCoreMaxT = 64;
// Most d slices the CUDA-core path splits a token tile into (the top-K kernel
// sums this many partials per logit).
constexpr int64_t kMaxSplits = 32;

RouterPlan router_plan(int64_t T, int32_t d, int32_t N, bool hidden_bf16) {
  // Aim at ~2 CTAs per SM of a 148-SM part; the plan depends on sizes only so
  // that workspace sizes are a host-side function of the problem.
  constexpr int64_t kTargetCtas = 296;
  RouterPlan pl{};
  if (hidden_bf16 && T > kCudaCoreMaxT) {
    // Tensor cores: one CTA per SM; tiles = 128-token blocks x 3 parts x
    // slices. With few experts (np <= kRouterMergedMaxNp) the three parts'
    // columns fit one B stage side by side, and a tile adds all three into
    // one accumulator: each hidden tile is then read once, and the tile's
    // k-block loop (its TMA round trips) is a third as long for the same
    // number of tiles.
    constexpr int64_t kTargetTiles = 148;
    pl.tensor = true;
    pl.np = (N + 15) / 16 * 16;
    pl.token_tiles = (T + kBM - 1) / kBM;
    pl.nkb_d = (d + kBK - 1) / kBK;
    pl.d_pad = pl.nkb_d * kBK;
    pl.merged = pl.np <= kRouterMergedMaxNp;
    const int64_t per_slice = pl.merged ? pl.token_tiles : pl.token_tiles * 3;
    // d slices: the fewest that minimise what one CTA runs, waves of tiles x
    // (k-blocks per tile + about two k-blocks of per-tile overhead); a last,
    // partly filled wave costs a whole one. At most 16 partials per logit
    // merged, 24 (8 x 3) otherwise, and at most 32 MB of partials (a quarter
    // of the L2; beyond that they evict what the next stages read).
    const int64_t max_slices = pl.merged ? 16 : 8;
    const int64_t part_bytes = (pl.merged ? 1 : 3) * T * (int64_t)N * 4;
    int64_t slices = 1, best = -1;
    for (int64_t sl = 1; sl <= max_slices && sl <= pl.nkb_d && (sl == 1 || sl * part_bytes <= (32ll << 20)); ++sl) {
      const int64_t kbs = (pl.nkb_d + sl - 1) / sl;
      const int64_t used = (pl.nkb_d + kbs - 1) / kbs;  // slices that hold k-blocks
      const int64_t cost = (per_slice * used + kTargetTiles - 1) / kTargetTiles * (kbs + 2);
      if (best < 0 || cost < best) {
        best = cost;
        slices = sl;
      }
    }
    pl.kb_per_slice = (int32_t)((pl.nkb_d + slices - 1) / slices);
    pl.dslices = (pl.nkb_d + pl.kb_per_slice - 1) / pl.kb_per_slice;
    pl.splits = (pl.merged ? 1 : 3) * pl.dslices;
    pl.d_slice = pl.kb_per_slice * kBK;
    return pl;
  }
  int chunk;
  if (N <= 32) {
    pl.np = 1;
    while (pl.np < N) pl.np <<= 1;
    const int tpw = pl.np <= 8 ? 4 : (pl.np == 16 ? 2 : 1);
    pl.token_tiles = (T + (int64_t)kWarps * tpw - 1) / ((int64_t)kWarps * tpw);
    chunk = 256;  // 32 lanes x 8 inputs
  } else {
    pl.np = 0;
    pl.token_tiles = (T + kTokPerCtaL - 1) / kTokPerCtaL;
    chunk = kDChunk;
  }
  const int64_t max_splits = (d + chunk - 1) / chunk;
  int64_t splits = 1;
  if (pl.token_tiles > 0 && pl.token_tiles < kTargetCtas) splits = (kTargetCtas + pl.token_tiles - 1) / pl.token_tiles;
  if (splits > kMaxSplits) splits = kMaxSplits;
  if (splits > max_splits) splits = max_splits;
  if (splits < 1) splits = 1;
  int64_t slice = (d + splits - 1) / splits;
  slice = (slice + chunk - 1) / chunk * chunk;
  pl.d_slice = (int32_t)slice;
  pl.splits = (int32_t)((d + slice - 1) / slice);
  return pl;
}

cudaError_t launch_expert_choice_select(const float* scores_t, int64_t T, int32_t N, int32_t C,
                                        int32_t* row_token, float* row_w, int32_t* offsets, int32_t* counts,
                                        cudaStream_t s) {
  if (const cudaError_t le_ = launch(expert_choice_select_kernel, N, kSelThreads, 0, s, scores_t, T, N, C, row_token, row_w, offsets, counts); le_ != cudaSuccess) return le_;
  return cudaSuccess;
}

cudaError_t launch_router(const RouterArgs& a0, bool hidden_bf16, cudaStream_t s) {
  if (a0.T == 0) return cudaSuccess;
  const RouterPlan pl = router_plan(a0.T, a0.d, a0.N, hidden_bf16);
  RouterArgs a = a0;
  a.splits = pl.splits;
  a.d_slice = pl.d_slice;
  cudaError_t e = pl.tensor ? launch_tensor_logits(a, pl, s)
                  : (hidden_bf16 ? launch_logits<__nv_bfloat16>(a, pl, s) : launch_logits<float>(a, pl, s));
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)((a.T + kWarps - 1) / kWarps);
  if (a.N <= 32) { if (const cudaError_t le_ = launch(topk_kernel<1>, grid, kWarps * 32, 0, s, a); le_ != cudaSuccess) return le_; }
  else if (a.N <= 64) { if (const cudaError_t le_ = launch(topk_kernel<2>, grid, kWarps * 32, 0, s, a); le_ != cudaSuccess) return le_; }
  else if (a.N <= 128) { if (const cudaError_t le_ = launch(topk_kernel<4>, grid, kWarps * 32, 0, s, a); le_ != cudaSuccess) return le_; }
  else { if (const cudaError_t le_ = launch(topk_kernel<8>, grid, kWarps * 32, 0, s, a); le_ != cudaSuccess) return le_; }
  return cudaSuccess;
}

}  // namespace moe
