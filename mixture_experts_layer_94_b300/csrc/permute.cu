// permute.cu — route and pack: per-expert histogram, prefix sum and a stable
// expert-major permutation of the T*K token copies, plus the row gather.
//
// "Chapter 19: Mixture-of-Experts Models", §19.6.3 "How expert parallelism
// dispatches tokens": token hidden states are routed and packed so that each
// expert receives its tokens as one contiguous batch ("Route and pack"), and
// results are later returned to the original tokens.
//
// Design (deterministic, no ordering races): tokens are cut into 32-token
// chunks, one warp per chunk, one token per lane. For every expert a warp
// builds a 32-bit lane mask in shared memory (atomicOr: order-independent);
// popc(mask) is the chunk's count, popc(mask & lanes_below) a copy's rank
// inside the chunk. One CTA scans counts over chunks and experts, giving each
// (expert, chunk) its first output row. A copy's row is then
//   offsets[e] + rows of e in earlier chunks + rank in its chunk,
// i.e. expert ascending, token ascending: the same order as a stable sort.
// The gather moves each hidden row to its permuted rows with 16-byte vectors.
// With an expert capacity C ("Chapter 19", §19.6.1) a copy whose rank inside
// its expert is C or more is dropped (inv_row = -1) and offsets count kept
// copies: min(count, C) per expert.
#include "act_convert.cuh"
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kHistWarps = 8;

__device__ void schedule_block(int N, int S, int F, int Fs, int d, int tile_rows, int64_t T,
                               const int32_t* offs, GroupDesc* groups, int32_t* ts_gu, int32_t* ts_dn);

__device__ __forceinline__ void build_chunk_masks(uint32_t* masks, const int32_t* __restrict__ idx,
                                                  int64_t T, int K, int N, int64_t chunk, int lane,
                                                  uint32_t* err) {
  for (int e = lane; e < N; e += 32) masks[e] = 0u;
  __syncwarp();
  const int64_t t = chunk * kTokensPerChunk + lane;
  if (t < T) {
    for (int k = 0; k < K; ++k) {
      const int e = idx[t * K + k];
      if (e < 0 || e >= N) {
        atomicOr(err, kErrBounds);
      } else {
        atomicOr(&masks[e], 1u << lane);
      }
    }
  }
  __syncwarp();
}

__global__ void __launch_bounds__(kHistWarps * 32) route_hist_kernel(const PermuteArgs a) {
  pdl_trigger();
  pdl_wait();
  __shared__ uint32_t masks[kHistWarps][kMaxExperts];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t c = (int64_t)blockIdx.x * kHistWarps + warp;
  if (c >= a.C) return;  // whole warp
  build_chunk_masks(masks[warp], a.topk_idx, a.T, a.K, a.N, c, lane, a.err);
  for (int e = lane; e < a.N; e += 32) a.chunk_counts[(int64_t)e * a.C + c] = __popc(masks[warp][e]);
}

// One CTA: counts[e] = sum over chunks, offsets = exclusive scan over experts
// of the kept counts min(counts[e], capacity), and
// chunk_counts[e][c] <- sum_{c' < c} chunk_counts[e][c'] (the rank base).
__global__ void __launch_bounds__(1024) route_scan_kernel(const PermuteArgs a) {
  pdl_trigger();
  pdl_wait();
  __shared__ int32_t s_counts[kMaxExperts];
  __shared__ int32_t s_offsets[kMaxExperts + 1];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  const int N = a.N;
  const int64_t C = a.C;
  for (int e = warp; e < N; e += nwarps) {
    const int32_t* row = a.chunk_counts + (int64_t)e * C;
    int32_t s = 0;
    for (int64_t c = lane; c < C; c += 32) s += row[c];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (lane == 0) s_counts[e] = s;
  }
  __syncthreads();
  if (warp == 0) {  // exclusive scan of N <= 256 counts, 8 per lane
    int32_t v[kMaxExperts / 32];
    int32_t local = 0;
#pragma unroll
    for (int i = 0; i < kMaxExperts / 32; ++i) {
      const int e = lane * (kMaxExperts / 32) + i;
      v[i] = (e < N) ? min(s_counts[e], a.capacity) : 0;
      local += v[i];
    }
    int32_t incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int32_t o = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += o;
    }
    int32_t run = incl - local;
#pragma unroll
    for (int i = 0; i < kMaxExperts / 32; ++i) {
      const int e = lane * (kMaxExperts / 32) + i;
      if (e < N) s_offsets[e] = run;
      run += v[i];
    }
    if (lane == 31) s_offsets[N] = incl;
  }
  __syncthreads();
  for (int e = threadIdx.x; e <= N; e += blockDim.x) {
    a.offsets[e] = s_offsets[e];
    if (e < N && a.counts) a.counts[e] = s_counts[e];
  }
  for (int e = warp; e < N; e += nwarps) {  // per chunk: the expert rank of its first copy
    int32_t* row = a.chunk_counts + (int64_t)e * C;
    int32_t run = 0;
    for (int64_t c0 = 0; c0 < C; c0 += 32) {
      const int64_t c = c0 + lane;
      const int32_t v = (c < C) ? row[c] : 0;
      int32_t incl = v;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int32_t o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
      }
      if (c < C) row[c] = run + incl - v;
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  if (a.groups) {
    __syncthreads();
    schedule_block(N, a.S, a.F, a.Fs, a.d, a.tile_rows, a.T, s_offsets, a.groups, a.ts_gu, a.ts_dn);
  }
}

constexpr int kScatterWarps = 8;

// One warp per chunk: each copy's row = its chunk's base for the expert plus
// its rank among the chunk's earlier tokens that chose the same expert.
__global__ void __launch_bounds__(kScatterWarps * 32) route_scatter_kernel(const PermuteArgs a) {
  pdl_trigger();
  pdl_wait();
  __shared__ uint32_t masks[kScatterWarps][kMaxExperts];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t c = (int64_t)blockIdx.x * kScatterWarps + warp;
  if (c >= a.C) return;
  const int K = a.K, N = a.N;
  uint32_t* m = masks[warp];
  build_chunk_masks(m, a.topk_idx, a.T, K, N, c, lane, a.err);
  const int64_t t = c * kTokensPerChunk + lane;
  if (t < a.T) {
    const uint32_t below = (1u << lane) - 1u;
    for (int k = 0; k < K; ++k) {
      const int e = a.topk_idx[t * K + k];
      if (e >= 0 && e < N) {
        const int32_t rank = a.chunk_counts[(int64_t)e * a.C + c] + __popc(m[e] & below);
        if (rank < a.capacity) {
          const int32_t r = __ldg(a.offsets + e) + rank;
          a.perm_src[r] = (int32_t)(t * K + k);
          a.inv_row[t * K + k] = r;
        } else {
          a.inv_row[t * K + k] = -1;
        }
      } else {
        a.inv_row[t * K + k] = -1;  // out-of-range expert (reported by the histogram)
      }
    }
  }
}

// One 16-byte output vector (8 elements) of hidden row t, vector v, in the
// activation format.
__device__ __forceinline__ uint4 act_vec(const PermuteArgs& a, int64_t t, int v, bool& over) {
  return hidden_vec(a.hidden, a.hidden_bf16, a.d, t, v, a.act_f16, over);
}

// Row gather into expert order: one thread per 16-byte output vector (8
// elements), grid-stride, each thread with kGatherBatch vectors' loads in
// flight at once, so that a small batch (a few rows) costs one index load and
// one data load of latency rather than a chain of them. The fused layer also
// clears the fp32 accumulator and writes a copy of hidden in the activation
// format (shared experts) when hidden is not already in it. Activations are
// bf16 for bf16 experts and fp16 for FP8 experts; a value beyond fp16's range
// is reported through the error word.
constexpr int kGatherBatch = 4;

__global__ void __launch_bounds__(256) gather_rows_kernel(const PermuteArgs a, int64_t rows) {
  pdl_trigger();
  pdl_wait();
  const int d = a.d, nvec = d / 8;
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t nthr = (int64_t)gridDim.x * blockDim.x;
  // Only rows [0, offsets[N]) are placed; fewer than T*K when an input index
  // was out of range (reported through the error word).
  const int64_t placed = min(rows, (int64_t)__ldg(a.offsets + a.N));
  const int64_t total = placed * nvec;
  bool over = false;
  uint4* xp = reinterpret_cast<uint4*>(a.x_perm);
  // Item i = (row i / nvec, vector i % nvec). A thread's items are tid + k *
  // nthr; their (row, vector) pairs advance by a fixed step, so no division
  // is done per vector.
  const int64_t adv = (int64_t)kGatherBatch * nthr;
  const int64_t adv_r = adv / nvec;
  const int adv_v = (int)(adv - adv_r * nvec);
  int64_t rr[kGatherBatch];
  int vv[kGatherBatch];
#pragma unroll
  for (int u = 0; u < kGatherBatch; ++u) {
    const int64_t i = tid + u * nthr;
    rr[u] = i / nvec;
    vv[u] = (int)(i - rr[u] * nvec);
  }
  for (int64_t i0 = tid; i0 < total; i0 += adv) {
    uint4 val[kGatherBatch];
    int64_t at[kGatherBatch];
#pragma unroll
    for (int u = 0; u < kGatherBatch; ++u) {
      const int64_t i = i0 + u * nthr;
      const int64_t r = rr[u];
      const int v = vv[u];
      vv[u] += adv_v;
      rr[u] += adv_r;
      if (vv[u] >= nvec) {
        vv[u] -= nvec;
        ++rr[u];
      }
      at[u] = -1;
      if (i >= total) continue;
      int64_t t;
      if (a.row_token) {
        t = a.row_token[r];
        if (t < 0 || t >= a.T) continue;
      } else {
        const int32_t src = a.perm_src[r];
        if (src < 0 || src >= rows) continue;
        t = src / a.K;
      }
      val[u] = act_vec(a, t, v, over);
      at[u] = i;
    }
#pragma unroll
    for (int u = 0; u < kGatherBatch; ++u)
      if (at[u] >= 0) xp[at[u]] = val[u];
  }
  if (a.zero_rows) {
    const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
    float4* z = reinterpret_cast<float4*>(a.zero_rows);
    for (int64_t i = tid; i < a.T * d / 4; i += nthr) z[i] = zero;
  }
  if (a.x_act) {
    uint4* dp = reinterpret_cast<uint4*>(a.x_act);
    for (int64_t i = tid; i < a.T * nvec; i += nthr) dp[i] = act_vec(a, i / nvec, (int)(i % nvec), over);
  }
  if (over && a.err) atomicOr(a.err, kErrRange);
}

// The GEMM groups (routed experts from offsets, then shared experts over all
// T tokens) and the exclusive prefix of their tile counts per phase. Called by
// every thread of one CTA; `offs` may be shared or global memory.
__device__ void schedule_block(int N, int S, int F, int Fs, int d, int tile_rows, int64_t T,
                               const int32_t* offs, GroupDesc* groups, int32_t* ts_gu, int32_t* ts_dn) {
  __shared__ int32_t s_gu[kMaxExperts + kMaxShared + 1];
  __shared__ int32_t s_dn[kMaxExperts + kMaxShared + 1];
  const int G = N + S;
  const int nt_dn = (d + kBNDown - 1) / kBNDown;
  for (int g = threadIdx.x; g < G; g += blockDim.x) {
    GroupDesc gd;
    int Fg;
    if (g < N) {
      gd.kind = 0;
      gd.index = g;
      gd.a_row0 = offs[g];
      gd.rows = offs[g + 1] - offs[g];
      gd.h_row0 = gd.a_row0;
      Fg = F;
    } else {
      gd.kind = 1;
      gd.index = g - N;
      gd.a_row0 = 0;
      gd.rows = (int32_t)T;
      gd.h_row0 = (int32_t)((int64_t)gd.index * T);
      Fg = Fs;
    }
    gd.m_tiles = (gd.rows + tile_rows - 1) / tile_rows;
    // n fastest where the group's activation rows outweigh its 2 Fg gate/up
    // weight rows (the same K, d)
    gd.order_gu = gd.rows > 2 * Fg ? 1 : 0;
    gd.pad = 0;
    groups[g] = gd;
    s_gu[g] = gd.m_tiles * ((Fg + kBNGateUp - 1) / kBNGateUp);
    s_dn[g] = gd.m_tiles * nt_dn;
  }
  __syncthreads();
  if (threadIdx.x < 32) {  // exclusive scans of G <= 264 counts, one warp
    const int lane = threadIdx.x;
    int32_t run_gu = 0, run_dn = 0;
    for (int g0 = 0; g0 < G; g0 += 32) {
      const int g = g0 + lane;
      const int32_t vg = g < G ? s_gu[g] : 0, vd = g < G ? s_dn[g] : 0;
      int32_t ig = vg, id = vd;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int32_t og = __shfl_up_sync(0xffffffffu, ig, off), od = __shfl_up_sync(0xffffffffu, id, off);
        if (lane >= off) {
          ig += og;
          id += od;
        }
      }
      if (g < G) {
        ts_gu[g] = run_gu + ig - vg;
        ts_dn[g] = run_dn + id - vd;
      }
      run_gu += __shfl_sync(0xffffffffu, ig, 31);
      run_dn += __shfl_sync(0xffffffffu, id, 31);
    }
    if (lane == 0) {
      ts_gu[G] = run_gu;
      ts_dn[G] = run_dn;
    }
  }
}

__global__ void __launch_bounds__(512) schedule_kernel(const ScheduleArgs a) {
  pdl_trigger();
  pdl_wait();
  schedule_block(a.N, a.S, a.F, a.Fs, a.d, a.tile_rows, a.T, a.offsets, a.groups, a.tile_start_gu,
                 a.tile_start_dn);
}

// Small batches (at most 32 chunks = 1024 tokens): one CTA does the histogram,
// both scans, the scatter and the schedule; one warp per chunk.
constexpr int kSmallChunks = 32;

__global__ void __launch_bounds__(1024) route_small_kernel(const PermuteArgs a) {
  pdl_trigger();
  pdl_wait();
  __shared__ uint32_t masks[kSmallChunks][kMaxExperts];
  __shared__ int32_t s_offsets[kMaxExperts + 1];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = a.N, K = a.K, C = a.C;
  if (warp < C) build_chunk_masks(masks[warp], a.topk_idx, a.T, K, N, warp, lane, a.err);
  __syncthreads();
  if (warp == 0) {  // counts and exclusive scan over experts, 8 experts per lane
    int32_t v[kMaxExperts / 32];
    int32_t local = 0;
#pragma unroll
    for (int i = 0; i < kMaxExperts / 32; ++i) {
      const int e = lane * (kMaxExperts / 32) + i;
      int32_t c = 0;
      if (e < N)
        for (int ch = 0; ch < C; ++ch) c += __popc(masks[ch][e]);
      v[i] = c;
      local += min(c, a.capacity);
    }
    int32_t incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int32_t o = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += o;
    }
    int32_t run = incl - local;
#pragma unroll
    for (int i = 0; i < kMaxExperts / 32; ++i) {
      const int e = lane * (kMaxExperts / 32) + i;
      if (e < N) {
        s_offsets[e] = run;
        a.offsets[e] = run;
        if (a.counts) a.counts[e] = v[i];
      }
      run += min(v[i], a.capacity);
    }
    if (lane == 31) {
      s_offsets[N] = incl;
      a.offsets[N] = incl;
    }
  }
  __syncthreads();
  if (warp < C) {
    const int64_t t = (int64_t)warp * kTokensPerChunk + lane;
    if (t < a.T) {
      const uint32_t below = (1u << lane) - 1u;
      for (int k = 0; k < K; ++k) {
        const int e = a.topk_idx[t * K + k];
        if (e >= 0 && e < N) {
          int32_t rank = __popc(masks[warp][e] & below);
          for (int ch = 0; ch < warp; ++ch) rank += __popc(masks[ch][e]);
          if (rank < a.capacity) {
            const int32_t r = s_offsets[e] + rank;
            a.perm_src[r] = (int32_t)(t * K + k);
            a.inv_row[t * K + k] = r;
          } else {
            a.inv_row[t * K + k] = -1;
          }
        } else {
          a.inv_row[t * K + k] = -1;
        }
      }
    }
  }
  if (a.groups) {
    __syncthreads();
    schedule_block(N, a.S, a.F, a.Fs, a.d, a.tile_rows, a.T, s_offsets, a.groups, a.ts_gu, a.ts_dn);
  }
}

// Token-major form of the same copy, for large token-choice batches: a thread
// reads a 16-byte vector of hidden row t once and stores it to each of the
// token's K packed rows (inv_row; -1 = dropped). Hidden is then streamed from
// HBM once, where the row-major gather above re-reads a row for each of its K
// copies (in expert order, long after the first read once hidden and the
// packed rows outgrow L2). Clears the accumulator and writes the
// activation-format copy of hidden like the gather.
constexpr int kScatterBatch = 2;

__global__ void __launch_bounds__(256) scatter_rows_kernel(const PermuteArgs a) {
  pdl_trigger();
  pdl_wait();
  const int d = a.d, nvec = d / 8, K = a.K;
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t nthr = (int64_t)gridDim.x * blockDim.x;
  const int64_t placed = min(a.T * K, (int64_t)__ldg(a.offsets + a.N));
  const int64_t total = a.T * nvec;
  bool over = false;
  uint4* xp = reinterpret_cast<uint4*>(a.x_perm);
  uint4* dp = reinterpret_cast<uint4*>(a.x_act);
  const int64_t adv = (int64_t)kScatterBatch * nthr;
  const int64_t adv_t = adv / nvec;
  const int adv_v = (int)(adv - adv_t * nvec);
  int64_t tt[kScatterBatch];
  int vv[kScatterBatch];
#pragma unroll
  for (int u = 0; u < kScatterBatch; ++u) {
    const int64_t i = tid + u * nthr;
    tt[u] = i / nvec;
    vv[u] = (int)(i - tt[u] * nvec);
  }
  for (int64_t i0 = tid; i0 < total; i0 += adv) {
    uint4 val[kScatterBatch];
    int64_t t_of[kScatterBatch];
    int v_of[kScatterBatch];
#pragma unroll
    for (int u = 0; u < kScatterBatch; ++u) {
      const int64_t i = i0 + u * nthr;
      t_of[u] = i < total ? tt[u] : -1;
      v_of[u] = vv[u];
      vv[u] += adv_v;
      tt[u] += adv_t;
      if (vv[u] >= nvec) {
        vv[u] -= nvec;
        ++tt[u];
      }
      if (t_of[u] >= 0) val[u] = act_vec(a, t_of[u], v_of[u], over);
    }
#pragma unroll
    for (int u = 0; u < kScatterBatch; ++u) {
      if (t_of[u] < 0) continue;
      const int32_t* ir = a.inv_row + t_of[u] * K;
      for (int k = 0; k < K; ++k) {
        const int32_t r = __ldg(ir + k);
        if (r >= 0 && r < placed) xp[(int64_t)r * nvec + v_of[u]] = val[u];
      }
      if (dp) dp[t_of[u] * nvec + v_of[u]] = val[u];
    }
  }
  if (a.zero_rows) {
    const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
    float4* z = reinterpret_cast<float4*>(a.zero_rows);
    for (int64_t i = tid; i < a.T * d / 4; i += nthr) z[i] = zero;
  }
  if (over && a.err) atomicOr(a.err, kErrRange);
}

}  // namespace

cudaError_t launch_permute(const PermuteArgs& a, cudaStream_t s) {
  if (a.C == 0) {  // T == 0: empty histogram, offsets all zero
    if (const cudaError_t le_ = launch(route_scan_kernel, 1, 1024, 0, s, a); le_ != cudaSuccess) return le_;
    return cudaSuccess;
  }
  if (a.C <= kSmallChunks) {
    if (const cudaError_t le_ = launch(route_small_kernel, 1, 1024, 0, s, a); le_ != cudaSuccess) return le_;
  } else {
    if (const cudaError_t le_ = launch(route_hist_kernel, (unsigned)((a.C + kHistWarps - 1) / kHistWarps), kHistWarps * 32, 0, s, a); le_ != cudaSuccess) return le_;
    if (const cudaError_t le_ = launch(route_scan_kernel, 1, 1024, 0, s, a); le_ != cudaSuccess) return le_;
    if (const cudaError_t le_ = launch(route_scatter_kernel, (unsigned)((a.C + kScatterWarps - 1) / kScatterWarps), kScatterWarps * 32, 0, s, a); le_ != cudaSuccess) return le_;
  }
  if (a.xq) return launch_gather_quant(a, a.T * a.K, a.xq_sh ? a.T : 0, s);
  return launch_gather(a, a.T * a.K, s);
}

cudaError_t launch_gather(const PermuteArgs& a, int64_t rows, cudaStream_t s) {
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (!a.row_token && rows >= kTokenMajorMinRows) {
    const int64_t want = (a.T * (a.d / 8) + 255) / 256;
    const unsigned grid = (unsigned)(want < (int64_t)sms * 8 ? (want < 1 ? 1 : want) : (int64_t)sms * 8);
    return launch(scatter_rows_kernel, grid, 256, 0, s, a);
  }
  const int64_t want = (rows * (a.d / 8) + 255) / 256;  // one 16-byte vector per thread
  const unsigned grid = (unsigned)(want < (int64_t)sms * 8 ? (want < 1 ? 1 : want) : (int64_t)sms * 8);
  return launch(gather_rows_kernel, grid, 256, 0, s, a, rows);
}

cudaError_t launch_schedule(const ScheduleArgs& a, cudaStream_t s) {
  if (const cudaError_t le_ = launch(schedule_kernel, 1, 512, 0, s, a); le_ != cudaSuccess) return le_;
  return cudaSuccess;
}

}  // namespace moe
