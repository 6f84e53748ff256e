// decode_layer.cu — the whole layer for a decode-sized token-choice batch in
// one kernel (internal).
//
// With T <= 4 tokens (bf16 or FP8 E4M3 experts) the layer is a stream of the touched experts' weight
// rows, each used by at most T activation rows ("Mixture of Experts
// Explained", "2. Why batching erodes the advantage": at small batch every
// token pays for reading its own experts' weights; "AI Infrastructure series,
// Part 12", "What happens when many users share the GPU?"). Launch and
// synchronisation latency would then cost as much as the router itself, so
// every step runs in one cooperative grid, one CTA per SM, with two grid-wide
// barriers:
//
//   phase 0  router logits ("Mixture of Experts for LLM Inference", "Opening
//            the router"; "Chapter 19", §19.3.2): CTA c < rsplits sums its
//            slice of d for all T tokens and N experts (fp32) into a partial;
//            every CTA stages the T token rows, rounded to the activation
//            format (bf16, or fp16 for FP8 experts), in shared memory.
//   barrier
//   phase 1  every CTA sums the partials in split order (the same fp32
//            result everywhere), scores, applies the group limit, takes the
//            top-K (topk.cuh), the capacity drops ("Chapter 19", §19.6.1: the
//            first C copies of an expert in token order stay), and lists the
//            touched experts; the last CTA stores the per-expert counts.
//   phase 2  gate/up: groups of 8 weight rows, gate rows f..f+3 and up rows
//            f..f+3 of one touched (or shared) expert. The groups' steps are
//            split into equal contiguous ranges over the grid's warps; a warp
//            streams its steps once from HBM and stores h = SiLU(g) * u
//            (16-bit) for each token that chose the expert.
//   barrier  (each warp first issues its first down-row loads, so HBM stays
//            busy across the barrier; while it completes, every CTA computes
//            the gate weights, which nothing needs before the down phase, and
//            CTA 0 stores topk_idx and topk_w)
//   phase 3  down: groups of 8 consecutive rows W_down[e][8b..8b+7] of every
//            touched (and shared) expert, split the same way. When the last
//            group of output block b is done, the warp that finished it sums
//            out[t][8b..8b+7] = sum_k w[t][k] y_{e(t,k)} in slot order, plus the
//            shared experts with weight 1 ("Chapter 19", §19.3.2 and the §19.2
//            flowchart; "Mixture of Experts for LLM Inference", "Shared
//            experts"), and stores the bf16 output.
//
// A warp reads one group's 8 rows 64 bytes per row per step: lane (g, t4)
// loads 16 bytes of row g, and the step's dot products with the token rows
// are one (bf16) or four (FP8, codes widened to fp16) mma.sync m16n8k16 with
// the weights as the 8-column operand and the token rows as the 16-row one
// (rows beyond the group's tokens are zero). The contraction's element order
// inside a step is permuted identically on both operands, so each lane's 16
// loaded bytes feed the MMA as they are. fp32 accumulation throughout.
// kDepth steps per lane are in flight in a register ring, across group
// boundaries.
//
// Every weight row is read from HBM once per call. A warp's range is at least
// one group long, so a group is split between at most two warps; the two
// halves meet in a slot, and the one arriving second adds them (fp32 addition
// of two terms does not depend on their order). Every result is therefore
// the same from run to run.
//
// The grid barriers are counters in the workspace's first 256 bytes (zeroed
// once by the caller, as the error word is). Waits are bounded: a wait that
// runs out sets kErrTimeout and the CTA skips the rest of its work; the last
// CTA to leave returns the counters to zero.

#include <cuda_fp8.h>

#include <atomic>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "topk.cuh"

namespace moe {
namespace {

constexpr int kThreads = kDecodeThreads;
constexpr int kWarps = kThreads / 32;
constexpr int kDepth = 8;  // 16-byte weight loads in flight per lane
constexpr int kMaxU = kMaxTopK * kDecodeMaxTokens + kMaxShared;  // touched routed + shared entries
constexpr uint64_t kBarrierTimeoutNs = 1000000000ull;
constexpr int kRouterRowsPerThread = 16;

// 16 bytes of weights, read once: no L1 allocation; the L2 fetches the
// whole 256-byte span, which holds this row's next three steps.
__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ float round_f16(float x, bool& over) {
  const float m = fabsf(x);
  over |= (m >= 65520.f) && (m <= 3.402823466e38f);
  return __half2float(__float2half_rn(x));
}

// D += A B for one m16n8k16 tile, fp32 accumulation. A's rows 8..15 are zero
// (a1 = a3 = 0): only token slots 0..7 exist.
template <bool F16>
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a2, uint32_t b0, uint32_t b1) {
  if (F16)
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
  else
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}

// Two E4M3 codes (the low 16 bits of c; the lower byte is the earlier element)
// as an fp16 pair, exactly.
__device__ __forceinline__ uint32_t e4m3x2_f16x2(uint32_t c) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(c & 0xFFFFu), __NV_E4M3);
  return (uint32_t)h.x | ((uint32_t)h.y << 16);
}

// One step of a group: this lane's 16 bytes of weights `w` (8 bf16, or 16
// E4M3 codes) against the token row's same elements at `x` in shared memory
// (16-bit; a zero row for a token slot the group does not have).
template <int FMT>
__device__ __forceinline__ void mma_step(float (&c)[4], const uint4 w, const uint16_t* x) {
  if (FMT == kDecodeBf16) {
    const uint4 xv = *reinterpret_cast<const uint4*>(x);
    mma16816<false>(c, xv.x, xv.y, w.x, w.y);
    mma16816<false>(c, xv.z, xv.w, w.z, w.w);
  } else {
    const uint4 x0 = reinterpret_cast<const uint4*>(x)[0], x1 = reinterpret_cast<const uint4*>(x)[1];
    mma16816<true>(c, x0.x, x0.y, e4m3x2_f16x2(w.x), e4m3x2_f16x2(w.x >> 16));
    mma16816<true>(c, x0.z, x0.w, e4m3x2_f16x2(w.y), e4m3x2_f16x2(w.y >> 16));
    mma16816<true>(c, x1.x, x1.y, e4m3x2_f16x2(w.z), e4m3x2_f16x2(w.z >> 16));
    mma16816<true>(c, x1.z, x1.w, e4m3x2_f16x2(w.w), e4m3x2_f16x2(w.w >> 16));
  }
}

// The layer's routing as every CTA computes it (shared memory).
struct Routing {
  int32_t idx[kDecodeMaxTokens][kMaxTopK];
  float w[kDecodeMaxTokens][kMaxTopK];
  uint8_t keep[kDecodeMaxTokens][kMaxTopK];
  int16_t tk_u[kDecodeMaxTokens][kMaxTopK];  // entry of copy (t, k), or -1 when dropped
  int8_t tk_r[kDecodeMaxTokens][kMaxTopK];   // its token slot in that entry
  // touched entries: routed experts holding kept copies (expert order), then
  // the shared experts. Entry u: expert index (routed) or N + s (shared), and
  // its token slots: token t and h row (t*K + k routed; T*K + s*T + t shared).
  int32_t n_entries, n_routed;
  int32_t ent_e[kMaxU];
  int32_t ent_n[kMaxU];
  int8_t ent_tok[kMaxU][kDecodeMaxTokens];
  int16_t ent_col[kMaxU][kDecodeMaxTokens];
};

// Waits until *ctr >= target (one thread), bounded; false on timeout.
__device__ bool wait_count(const uint32_t* ctr, uint32_t target) {
  const uint64_t t0 = globaltimer_ns();
  uint32_t spins = 0;
  while (ld_acquire(ctr) < target) {
    if ((++spins & 63u) == 0 && globaltimer_ns() - t0 > kBarrierTimeoutNs) return false;
  }
  return true;
}

// Grid barrier number `gen` (1, 2): every CTA adds one (grid_arrive), then
// waits for gen*G (grid_wait); a CTA may work in between.
__device__ void grid_arrive(uint32_t* ctr) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(ctr, 1u);
  }
}

__device__ bool grid_wait(uint32_t* ctr, uint32_t gen, uint32_t* err, bool* s_ok) {
  if (threadIdx.x == 0) {
    const bool ok = wait_count(ctr, gen * gridDim.x);
    if (!ok) atomicOr(err, kErrTimeout);
    __threadfence();
    *s_ok = ok;
  }
  __syncthreads();
  return *s_ok;
}

__device__ bool grid_barrier(uint32_t* ctr, uint32_t gen, uint32_t* err, bool* s_ok) {
  grid_arrive(ctr);
  return grid_wait(ctr, gen, err, s_ok);
}

// Adds the other half of a group split between two warps. `slot` holds two
// halves of 64 floats (each lane's fragment c0, c1); `mine` is 0 for the half
// that starts the group, 1 for the one that ends it. Returns true in the warp
// that arrives second, whose `c` then holds the sum.
__device__ __forceinline__ bool join_halves(float (&c)[4], float* slot, uint32_t* cnt, int mine, int lane) {
  reinterpret_cast<float2*>(slot + 64 * mine)[lane] = make_float2(c[0], c[1]);
  __threadfence();
  __syncwarp();
  uint32_t prev = 0;
  if (lane == 0) prev = atomicAdd(cnt, 1u);
  prev = __shfl_sync(0xFFFFFFFFu, prev, 0);
  if (prev != 1u) return false;
  __threadfence();
  const float2 o = __ldcg(reinterpret_cast<const float2*>(slot + 64 * (1 - mine)) + lane);
  c[0] += o.x;
  c[1] += o.y;
  return true;
}

// Token t's scores, group limit, top-K and gate weights from its summed
// logits lg_s[t][.] (router bias added here); slot k's expert and weight
// land in idx[k], w[k]. Group-limited routing only: kept out of line, so
// that the rank-based path the other problems take stays compact (the
// kernel's code is fetched cold from DRAM once per launch).
template <int EPL>
__device__ __noinline__ void topk_token(const DecodeArgs& a, const float* lg_s, int t, int lane, int N, int K,
                                           float* s_key, unsigned char* s_kept, int32_t* idx, float* w) {
  float lg[EPL], sc[EPL], key[EPL];
  bool valid[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    valid[i] = e < N;
    lg[i] = valid[i] ? lg_s[t * N + e] + (a.router_bias ? a.router_bias[e] : 0.f) : 0.f;
  }
  router_scores<EPL>(lg, valid, lane, a.score_fn, a.sel_bias, sc, key);
  if (a.n_groups > 1 && a.topk_groups < a.n_groups)
    router_group_limit<EPL>(key, valid, lane, N, a.n_groups, a.topk_groups, s_key, s_kept);
  int my_e;
  float my_w;
  router_select<EPL>(sc, key, valid, lane, K, a.score_fn, a.renormalize, my_e, my_w);
  if (lane < K) {
    idx[lane] = my_e;
    w[lane] = my_w;
  }
}

template <int FMT, bool HB>
__global__ void __launch_bounds__(kThreads, 1) decode_layer_kernel(const DecodeArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ Routing rt;
  __shared__ float s_key[kDecodeMaxTokens][kMaxExperts];
  __shared__ unsigned char s_kept[kDecodeMaxTokens][kMaxExperts];
  __shared__ bool s_ok;
  __shared__ int32_t s_wcount[kWarps];
  __shared__ uint8_t s_slot[kDecodeMaxTokens][kMaxExperts];
  __shared__ __align__(8) uint64_t s_hbar;  // the h rows' bulk copies (phase 3)
  __shared__ int s_abort;
  constexpr bool kF16 = FMT != kDecodeBf16;
  constexpr int EPS = FMT == kDecodeBf16 ? 32 : 64;  // elements of a row per step
  constexpr int EPL = EPS / 4;                       // elements per lane per step
  constexpr int BPS = 64;                            // bytes of a row per step
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int T = (int)a.T, N = a.N, K = a.K, d = a.d;
  const int G = gridDim.x, c = blockIdx.x;
  const int64_t GW = (int64_t)G * kWarps, gw = (int64_t)c * kWarps + warp;
  bool over = false;
  bool ok = true;
  if (tid == 0) {
    ptx::mbar_init(ptx::smem_u32(&s_hbar), 1);
    ptx::fence_mbarrier_init();
    s_abort = 0;
  }

  // ------------------------------------------------------------ phase 0
  // shared memory: the zero row [z_len], then the token rows [T][x_stride]
  // (phases 0-2) or the h rows [T*K + S*T][hsm_stride] (phase 3), and the
  // router scratch after the token rows
  uint16_t* zrow = reinterpret_cast<uint16_t*>(smem);
  uint16_t* xs = zrow + a.z_len;
  const int xstride = a.x_stride;
  float* red = reinterpret_cast<float*>(smem + (size_t)a.smem_x_bytes);
  // the counters of this launch's split groups and output blocks start at zero
  for (int64_t i = (int64_t)c * kThreads + tid; i < GW + 1; i += (int64_t)G * kThreads) a.bnd_cnt[i] = 0u;
  for (int i = c * kThreads + tid; i < d / 8; i += G * kThreads) a.blk_cnt[i] = 0u;
  // h rows are padded to whole blocks of steps; the down phase reads the
  // padding (against zero weights), so it must hold zeros
  {
    const int pr = a.h_stride - a.F, ps = a.hs_stride - a.Fs;
    const int nr = T * K * pr, ns = a.S * T * ps;
    for (int i = c * kThreads + tid; i < nr + ns; i += G * kThreads) {
      if (i < nr) static_cast<uint16_t*>(a.h)[(int64_t)(i / pr) * a.h_stride + a.F + i % pr] = 0;
      else static_cast<uint16_t*>(a.h_sh)[(int64_t)((i - nr) / ps) * a.hs_stride + a.Fs + (i - nr) % ps] = 0;
    }
  }
  // Router CTAs issue their first batch of router weights before anything
  // else, so that its DRAM round trip overlaps the token rows' below.
  const bool router_cta = c < a.rsplits;
  const int j0 = c * a.r_slice, nj = router_cta ? min(a.r_slice, d - j0) : 0;
  const int Q = kThreads / N;  // threads per expert, splitting the slice's rows
  const int q = tid / N, e = tid - q * N;
  float wv[kRouterRowsPerThread];
#pragma unroll
  for (int u = 0; u < kRouterRowsPerThread; ++u) {
    const int j = q + u * Q;
    wv[u] = router_cta && q < Q && j < nj ? __ldg(a.w_router + (int64_t)(j0 + j) * N + e) : 0.f;
  }
  // the zero row, then the token rows rounded to the activation format and
  // zero-padded to x_stride
  for (int i = tid; i < (a.z_len + T * xstride) / 8; i += kThreads) {
    const int j = i - a.z_len / 8;
    const int t = j < 0 ? -1 : j / (xstride / 8), v = j - t * (xstride / 8);
    uint4 o = make_uint4(0u, 0u, 0u, 0u);
    if (t >= 0 && 8 * v < d) {
      float f[8];
      if (HB) {
        const uint4 hv = __ldg(static_cast<const uint4*>(a.hidden) + ((int64_t)t * d) / 8 + v);
        const uint32_t hw[4] = {hv.x, hv.y, hv.z, hv.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          f[2 * k] = __uint_as_float(hw[k] << 16);
          f[2 * k + 1] = __uint_as_float(hw[k] & 0xFFFF0000u);
        }
      } else {
        const float4* p = static_cast<const float4*>(a.hidden) + ((int64_t)t * d) / 4 + 2 * v;
        const float4 u0 = __ldg(p), u1 = __ldg(p + 1);
        f[0] = u0.x; f[1] = u0.y; f[2] = u0.z; f[3] = u0.w;
        f[4] = u1.x; f[5] = u1.y; f[6] = u1.z; f[7] = u1.w;
      }
      if (kF16) {
#pragma unroll
        for (int k = 0; k < 8; ++k) f[k] = round_f16(f[k], over);
        o = make_uint4(pack_f16x2(f[0], f[1]), pack_f16x2(f[2], f[3]), pack_f16x2(f[4], f[5]),
                       pack_f16x2(f[6], f[7]));
      } else {
        o = make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                       pack_bf16x2(f[6], f[7]));
      }
    }
    reinterpret_cast<uint4*>(zrow)[i] = o;
  }
  // bf16 hidden with bf16 experts: the staged rows hold the hidden values
  // exactly, and the router reads its slice from them
  constexpr bool kXsExact = HB && !kF16;
  if (router_cta) {
    float* xsl = red;                   // [T][r_slice] fp32 slice of the token rows (otherwise)
    float* part = red + T * a.r_slice;  // [Q][T][N]
    if (!kXsExact) {
      for (int i = tid; i < T * nj; i += kThreads) {
        const int t = i / nj, j = i - t * nj;
        const int64_t xi = (int64_t)t * d + j0 + j;
        xsl[t * a.r_slice + j] = HB ? __bfloat162float(static_cast<const __nv_bfloat16*>(a.hidden)[xi])
                                    : static_cast<const float*>(a.hidden)[xi];
      }
    }
    __syncthreads();
    auto xval = [&](int t, int j) {
      return kXsExact ? __uint_as_float((uint32_t)xs[(int64_t)t * xstride + j0 + j] << 16) : xsl[t * a.r_slice + j];
    };
    if (q < Q) {
      float acc[kDecodeMaxTokens] = {0.f, 0.f, 0.f, 0.f};
      for (int jb = q;; jb += kRouterRowsPerThread * Q) {
#pragma unroll
        for (int u = 0; u < kRouterRowsPerThread; ++u) {
          const int j = jb + u * Q;
          if (j < nj) {
#pragma unroll
            for (int t = 0; t < kDecodeMaxTokens; ++t)
              if (t < T) acc[t] = fmaf(xval(t, j), wv[u], acc[t]);
          }
        }
        const int jn = jb + kRouterRowsPerThread * Q;
        if (jn >= nj) break;
#pragma unroll
        for (int u = 0; u < kRouterRowsPerThread; ++u) {
          const int j = jn + u * Q;
          wv[u] = j < nj ? __ldg(a.w_router + (int64_t)(j0 + j) * N + e) : 0.f;
        }
      }
#pragma unroll
      for (int t = 0; t < kDecodeMaxTokens; ++t)
        if (t < T) part[((int64_t)q * T + t) * N + e] = acc[t];
    }
    __syncthreads();
    // the Q partial sums of each (token, expert), in order
    for (int i = tid; i < T * N; i += kThreads) {
      float s = 0.f;
      for (int qq = 0; qq < Q; ++qq) s += part[(int64_t)qq * T * N + i];
      a.router_part[(int64_t)c * T * N + i] = s;
    }
  }
  ok = grid_barrier(a.sync, 1u, a.err, &s_ok);

  // ------------------------------------------------------------ phase 1
  if (ok) {
    // logits: the rsplits partials of every (token, expert) summed in split
    // order by P threads each (P a power of two), then the P sums in order
    const int pairs = T * N;
    float* lg_s = red;          // [T][N]
    float* psum = red + pairs;  // [P][pairs]
    int P = 1;
    while (P * 2 * pairs <= kThreads && P * 2 <= a.rsplits) P *= 2;
    // (up to 64 loads per thread in one batch: one L2 round trip for the
    // partials of up to 4 tokens of 128 experts)
    for (int i = tid; i < P * pairs; i += kThreads) {
      const int p = i / pairs, pr = i - p * pairs;
      float s = 0.f;
      for (int sp0 = p; sp0 < a.rsplits; sp0 += 64 * P) {
        float v[64];
#pragma unroll
        for (int u = 0; u < 64; ++u) {
          const int sp = sp0 + u * P;
          v[u] = sp < a.rsplits ? __ldcg(a.router_part + (int64_t)sp * pairs + pr) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < 64; ++u) s += v[u];
      }
      psum[i] = s;
    }
    __syncthreads();
    const bool grouped = a.n_groups > 1 && a.topk_groups < a.n_groups;
    // The P sums in order, and for the rank-based top-K every (token, expert)
    // pair's selection key and score (the same fp32 arithmetic as
    // router_scores). key_s and sc_s overlay psum's first two rows, whose
    // column i only this thread reads, before it writes.
    float* key_s = red + pairs;     // [T][N]
    float* sc_s = red + 2 * pairs;  // [T][N]
    for (int i = tid; i < pairs; i += kThreads) {
      float s = 0.f;
      for (int p = 0; p < P; ++p) s += psum[p * pairs + i];
      lg_s[i] = s;
      if (!grouped) {
        const int e = i - (i / N) * N;
        const float l = s + (a.router_bias ? a.router_bias[e] : 0.f);
        if (a.score_fn == 0) {
          key_s[i] = l;
          sc_s[i] = l;
        } else {
          const float sg = 1.0f / (1.0f + expf(-l));
          sc_s[i] = sg;
          key_s[i] = sg + (a.sel_bias ? a.sel_bias[e] : 0.f);
        }
      }
    }
    __syncthreads();
    if (grouped) {
      // group-limited routing: one warp per token (topk.cuh)
      if (warp < T) {
        if (N <= 128) topk_token<4>(a, lg_s, warp, lane, N, K, s_key[warp], s_kept[warp], rt.idx[warp], rt.w[warp]);
        else topk_token<8>(a, lg_s, warp, lane, N, K, s_key[warp], s_kept[warp], rt.idx[warp], rt.w[warp]);
      }
      // slot of expert e in token t's choice (0xFF: not chosen)
      for (int i = tid; i < T * N; i += kThreads) s_slot[i / N][i % N] = 0xFF;
      __syncthreads();
      for (int i = tid; i < T * K; i += kThreads) s_slot[i / K][rt.idx[i / K][i % K]] = (uint8_t)(i % K);
    } else {
      // Each pair's rank: the number of experts whose key is larger, or
      // equal at a lower index. The experts of rank below K are the top-K,
      // and the rank is the slot (key descending, ties to the lower index);
      // it also gives the slot map (0xFF: not chosen). P threads share a
      // pair's comparisons.
      int lp = 0;  // P = 2^lp
      while (lp < 5 && (2 << lp) * pairs <= kThreads) ++lp;
      const int P = 1 << lp;
      for (int i0 = 0; i0 < pairs * P; i0 += kThreads) {
        const int i = i0 + tid;
        const int pr = i >> lp, p = i & (P - 1);
        // token t = pr / N for T <= 4, without a division
        const int t = (pr >= N) + (pr >= 2 * N) + (pr >= 3 * N), e = pr - t * N;
        int cnt = 0;
        if (pr < pairs) {
          // this thread's contiguous share [j0, j1) of the token's keys, four at a time where aligned
          const float ke = key_s[pr];
          const float* kt = key_s + t * N;
          const int j0 = (N * p) >> lp, j1 = (N * (p + 1)) >> lp;
          int j = j0;
          if (((reinterpret_cast<uintptr_t>(kt + j0)) & 15u) == 0) {
#pragma unroll 4
            for (; j + 4 <= j1; j += 4) {
              const float4 k4 = *reinterpret_cast<const float4*>(kt + j);
              cnt += (k4.x > ke) || (k4.x == ke && j < e);
              cnt += (k4.y > ke) || (k4.y == ke && j + 1 < e);
              cnt += (k4.z > ke) || (k4.z == ke && j + 2 < e);
              cnt += (k4.w > ke) || (k4.w == ke && j + 3 < e);
            }
          }
          for (; j < j1; ++j) {
            const float kj = kt[j];
            cnt += (kj > ke) || (kj == ke && j < e);
          }
        }
        for (int off = 1; off < P; off <<= 1) cnt += __shfl_xor_sync(0xFFFFFFFFu, cnt, off);
        if (pr < pairs && p == 0) {
          s_slot[t][e] = cnt < K ? (uint8_t)cnt : (uint8_t)0xFF;
          if (cnt < K) rt.idx[t][cnt] = e;
        }
      }
      // (the gate weights follow during the second grid barrier: nothing
      // needs them before the down phase)
    }
    __syncthreads();
    {
      // capacity: the first `capacity` copies of each expert in token order
      // stay. One thread per expert counts its kept copies; a block-wide count
      // of the experts holding any gives each its entry (expert order).
      const int e = tid;
      int kept = 0;
      if (e < N) {
        int seen = 0;
        for (int t = 0; t < T; ++t) {
          const int k = s_slot[t][e];
          if (k != 0xFF) {
            const bool keep = seen < a.capacity;
            ++seen;
            rt.keep[t][k] = keep;
            rt.tk_u[t][k] = -1;
            kept += keep;
          }
        }
      }
      const uint32_t ball = __ballot_sync(0xFFFFFFFFu, kept > 0);
      if (lane == 0) s_wcount[warp] = __popc(ball);
      __syncthreads();
      int base = 0, nr = 0;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const int cw = s_wcount[w];
        base += w < warp ? cw : 0;
        nr += cw;
      }
      if (kept > 0) {
        const int n = base + __popc(ball & ((1u << lane) - 1u));
        rt.ent_e[n] = e;
        rt.ent_n[n] = kept;
        int r = 0;
        for (int t = 0; t < T; ++t) {
          const int k = s_slot[t][e];
          if (k != 0xFF && rt.keep[t][k]) {
            rt.ent_tok[n][r] = (int8_t)t;
            rt.ent_col[n][r] = (int16_t)(t * K + k);
            rt.tk_u[t][k] = (int16_t)n;
            rt.tk_r[t][k] = (int8_t)r;
            ++r;
          }
        }
      }
      if (tid < a.S) {
        const int n = nr + tid;
        rt.ent_e[n] = N + tid;
        rt.ent_n[n] = T;
        for (int t = 0; t < T; ++t) {
          rt.ent_tok[n][t] = (int8_t)t;
          rt.ent_col[n][t] = (int16_t)(T * K + tid * T + t);
        }
      }
      if (tid == 0) {
        rt.n_routed = nr;
        rt.n_entries = nr + a.S;
      }
    }
    __syncthreads();
    // the per-expert counts from the last CTA (the same tables in every CTA)
    if (c == G - 1 && a.counts) {
      for (int e = tid; e < N; e += kThreads) {
        int cnt = 0;
        for (int t = 0; t < T; ++t) cnt += s_slot[t][e] != 0xFF;
        a.counts[e] = cnt;
      }
    }
  }

  // ------------------------------------------------------------ phase 3 setup
  // groups: output block ob (8 elements) x entry u, entry fastest; a routed
  // entry's group is BF blocks of kDepth steps, a shared one BFs
  const int BF = ((a.F + EPS - 1) / EPS + kDepth - 1) / kDepth;
  const int BFs = a.S > 0 ? ((a.Fs + EPS - 1) / EPS + kDepth - 1) / kDepth : 0;
  const int nR = ok ? rt.n_routed : 0;
  const int per_ob = nR * BF + a.S * BFs;  // blocks per output block
  const int tb3 = (d / 8) * per_ob;
  const int bmax = BF > BFs ? BF : BFs;
  int nw3 = tb3 / bmax;  // every range at least one group long
  if (nw3 > GW) nw3 = (int)GW;
  if (nw3 < 1 && tb3 > 0) nw3 = 1;
  const bool active3 = ok && gw < nw3;
  const int b0 = active3 ? (int)((int64_t)tb3 * gw / nw3) : 0;
  const int b1 = active3 ? (int)((int64_t)tb3 * (gw + 1) / nw3) : 0;
  const int rows_h = T * K + a.S * T;                // h rows; row rows_h is zero
  const int ycols = rows_h;                          // y columns: (token, slot) pairs, then shared
  // the group of flat block x: output block, entry, its first block, its length
  auto locate3 = [&](int x, int& ob, int& u, int& start, int& len) {
    ob = x / per_ob;
    const int r = x - ob * per_ob;
    if (r < nR * BF) {
      u = r / BF;
      start = ob * per_ob + u * BF;
      len = BF;
    } else {
      const int s = (r - nR * BF) / BFs;
      u = nR + s;
      start = ob * per_ob + nR * BF + s * BFs;
      len = BFs;
    }
  };
  // this lane's weight row of the group at flat block x, and that row's length
  auto row3 = [&](int x, int& rowlen) {
    int ob, u, start, len;
    locate3(x, ob, u, start, len);
    const int e = rt.ent_e[u];
    const int64_t eb = FMT == kDecodeBf16 ? 2 : 1;
    rowlen = e < N ? a.F : a.Fs;
    return (e < N ? static_cast<const uint8_t*>(a.w_down) + ((int64_t)e * d + 8 * ob + g) * a.F * eb
                  : static_cast<const uint8_t*>(a.s_down) + ((int64_t)(e - N) * d + 8 * ob + g) * a.Fs * eb) +
           16 * t4;
  };
  // ------------------------------------------------------------ phase 2
  // group j: entry u's gate rows f0..f0+3 (lane rows g < 4) and up rows
  // f0..f0+3 (g >= 4); the routed entries have F/4 groups each, then the
  // shared entries Fs/4. A group is B2 blocks of kDepth steps (steps past the
  // row's end load zeros); warp ranges are whole blocks, each at least one
  // group long, so the unrolled loop below never meets a group's end inside
  // a block.
  if (ok) {
    const int B2 = ((d + EPS - 1) / EPS + kDepth - 1) / kDepth;
    const int gr_routed = rt.n_routed * (a.F / 4);
    const int groups = gr_routed + a.S * (a.Fs / 4);
    const int nw = GW < groups ? (int)GW : groups;
    const int tb = groups * B2;
    const int64_t row_bytes = (int64_t)d * (FMT == kDecodeBf16 ? 2 : 1);
    auto locate2 = [&](int j, int& u, int& f0) {
      if (j < gr_routed) {
        u = j / (a.F / 4);
        f0 = 4 * (j - u * (a.F / 4));
      } else {
        const int s = (j - gr_routed) / (a.Fs / 4);
        u = rt.n_routed + s;
        f0 = 4 * (j - gr_routed - s * (a.Fs / 4));
      }
    };
    // this lane's weight row of group j (at its first step)
    auto row2 = [&](int j) {
      int u, f0;
      locate2(j, u, f0);
      const int e = rt.ent_e[u];
      const int f = f0 + (g & 3);
      const bool up = g >= 4;
      const uint8_t* base =
          e < N ? static_cast<const uint8_t*>(up ? a.w_up : a.w_gate) + ((int64_t)e * a.F + f) * row_bytes
                : static_cast<const uint8_t*>(up ? a.s_up : a.s_gate) + ((int64_t)(e - N) * a.Fs + f) * row_bytes;
      return base + 16 * t4;
    };
    // this lane's token row of entry u (the zero row past the entry's tokens)
    auto xrow2 = [&](int u) {
      return (g < rt.ent_n[u] ? xs + (int64_t)rt.ent_tok[u][g] * xstride : zrow) + EPL * t4;
    };
    if (gw < nw) {
      const int b0 = (int)((int64_t)tb * gw / nw), b1 = (int)((int64_t)tb * (gw + 1) / nw);
      int lj = b0 / B2, lbg = b0 - lj * B2;  // the block being loaded: group, block in the group
      const uint8_t* lp = row2(lj);
      uint4 ring[kDepth];
#pragma unroll
      for (int i = 0; i < kDepth; ++i) {
        const int st = lbg * kDepth + i;
        ring[i] = st * EPS + EPL * t4 < d ? ld_stream(lp + (int64_t)st * BPS) : make_uint4(0u, 0u, 0u, 0u);
      }
      int cj = lj, cbg = lbg, cfirst = lbg;  // the block being consumed, and where this piece began
      int cu, cf0;
      locate2(cj, cu, cf0);
      const uint16_t* cx = xrow2(cu);
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      for (int b = b0; b < b1; ++b) {
        const bool more = b + 1 < b1;
        if (more && ++lbg == B2) {
          lbg = 0;
          lp = row2(++lj);
        }
        const int ls0 = lbg * kDepth, cs0 = cbg * kDepth;
#pragma unroll
        for (int i = 0; i < kDepth; ++i) {
          const uint4 v = ring[i];
          if (more)
            ring[i] = (ls0 + i) * EPS + EPL * t4 < d ? ld_stream(lp + (int64_t)(ls0 + i) * BPS)
                                                     : make_uint4(0u, 0u, 0u, 0u);
          mma_step<FMT>(acc, v, cx + (cs0 + i) * EPS);
        }
        const bool end_group = ++cbg == B2;
        if (end_group || !more) {
          // this warp's piece of group cj is done: the whole group, or one
          // of its two halves
          bool have = true;
          if (cfirst != 0 || !end_group) {
            const int mine = cfirst != 0 ? 1 : 0;
            const int bslot = mine ? (int)gw : (int)gw + 1;
            have = join_halves(acc, a.bnd_val + (int64_t)bslot * 128, a.bnd_cnt + bslot, mine, lane);
          }
          if (have) {
            // lane (slot g, t4 < 2) holds gate rows f0+2t4, f0+2t4+1; lane t4+2 the up rows
            const float up0 = __shfl_down_sync(0xFFFFFFFFu, acc[0], 2);
            const float up1 = __shfl_down_sync(0xFFFFFFFFu, acc[1], 2);
            const int e = rt.ent_e[cu];
            if (t4 < 2 && g < rt.ent_n[cu]) {
              const int f = cf0 + 2 * t4;
              float g0 = acc[0], g1 = acc[1], u0 = up0, u1 = up1;
              if (FMT == kDecodeE4M3) {
                const float* sg = e < N ? static_cast<const float*>(a.w_gate_scale) + (int64_t)e * a.F
                                        : static_cast<const float*>(a.s_gate_scale) + (int64_t)(e - N) * a.Fs;
                const float* su = e < N ? static_cast<const float*>(a.w_up_scale) + (int64_t)e * a.F
                                        : static_cast<const float*>(a.s_up_scale) + (int64_t)(e - N) * a.Fs;
                g0 *= __ldg(sg + f);
                g1 *= __ldg(sg + f + 1);
                u0 *= __ldg(su + f);
                u1 *= __ldg(su + f + 1);
              }
              const float h0 = silu_f(g0) * u0, h1 = silu_f(g1) * u1;
              if (kF16) over |= fmaxf(fabsf(h0), fabsf(h1)) >= 65520.f;
              const uint32_t hv = kF16 ? pack_f16x2(h0, h1) : pack_bf16x2(h0, h1);
              const int col = rt.ent_col[cu][g];
              uint16_t* hp = e < N ? static_cast<uint16_t*>(a.h) + (int64_t)col * a.h_stride + f
                                   : static_cast<uint16_t*>(a.h_sh) + (int64_t)(col - T * K) * a.hs_stride + f;
              *reinterpret_cast<uint32_t*>(hp) = hv;
            }
          }
          acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
          if (end_group && more) {
            cbg = 0;
            cfirst = 0;
            ++cj;
            locate2(cj, cu, cf0);
            cx = xrow2(cu);
          }
        }
      }
    }
  }

  uint4 ring3[kDepth];
  int lx = b0, lbg = 0, llen = 1, lK = 0;  // the block being loaded, its place in the group
  const uint8_t* lp3 = nullptr;
  if (active3) {
    int ob, u, start;
    locate3(lx, ob, u, start, llen);
    lbg = lx - start;
    lp3 = row3(lx, lK);
  }
#pragma unroll
  for (int i = 0; i < kDepth; ++i) {
    const int st = lbg * kDepth + i;
    ring3[i] = active3 && st * EPS + EPL * t4 < lK ? ld_stream(lp3 + (int64_t)st * BPS) : make_uint4(0u, 0u, 0u, 0u);
  }
  if (ok) {
    grid_arrive(a.sync);
    // while the barrier completes: the gate weights of the rank-based top-K,
    // warp t for token t, as router_select computes them (the group-limited
    // path set them with its selection), then topk_idx / topk_w from CTA 0
    const bool grouped = a.n_groups > 1 && a.topk_groups < a.n_groups;
    if (!grouped && warp < T) {
      const float* sc_s = red + 2 * T * N;
      const float* sct = sc_s + warp * N;
      const int my_e = lane < K ? rt.idx[warp][lane] : 0;
      const float my_sc = lane < K ? sct[my_e] : 0.f;
      float w;
      if (a.score_fn == 0) {
        const float lmax = __shfl_sync(0xffffffffu, my_sc, 0);  // slot 0 holds the largest logit
        const float ex = lane < K ? expf(my_sc - lmax) : 0.f;
        float z = 0.f;
        if (a.renormalize) {
          z = ex;
        } else {
          for (int e = lane; e < N; e += 32) z += expf(sct[e] - lmax);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
        w = ex / z;
      } else {
        float z = lane < K ? my_sc : 0.f;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
        w = a.renormalize ? my_sc / z : my_sc;
      }
      if (lane < K) rt.w[warp][lane] = w;
    }
    __syncthreads();
    if (c == 0) {
      for (int i = tid; i < T * K; i += kThreads) {
        a.topk_idx[i] = rt.idx[i / K][i % K];
        a.topk_w[i] = rt.w[i / K][i % K];
      }
    }
    ok = grid_wait(a.sync, 2u, a.err, &s_ok);
  }

  uint16_t* hs = xs;  // phase 3: the h rows reuse the token rows' space
  const int hsm = a.hsm_stride;
  if (ok) {
    // h rows into shared memory (routed rows t*K + k, then the shared rows):
    // one bulk copy per row, issued by warp 0 and counted on one mbarrier.
    // Unlike loads from every thread, the copies do not queue behind the
    // down-row loads already in flight.
    const uint32_t bar = ptx::smem_u32(&s_hbar);
    if (warp == 0) {
      if (lane == 0)
        ptx::mbar_arrive_expect_tx(bar, (uint32_t)(T * K * a.h_stride + a.S * T * a.hs_stride) * 2u);
      __syncwarp();
      // the copies write shared memory the token rows held (read through the
      // generic proxy) and read h rows other CTAs wrote before the barrier
      ptx::fence_proxy_async_shared();
      ptx::fence_proxy_async_global();
      for (int r = lane; r < rows_h; r += 32) {
        const bool sh = r >= T * K;
        const int len = sh ? a.hs_stride : a.h_stride;
        const uint16_t* src = static_cast<const uint16_t*>(sh ? a.h_sh : a.h) + (int64_t)(sh ? r - T * K : r) * len;
        ptx::bulk_load(ptx::smem_u32(hs + (int64_t)r * hsm), src, (uint32_t)len * 2u, bar);
      }
    }
    ptx::mbar_wait(bar, 0, &s_abort, a.err);
    __syncthreads();
    if (s_abort) {
      // timed out: the copies may still be landing; wait for them (bounded)
      // before this CTA leaves
      ok = false;
      if (tid == 0) {
        const uint64_t t0 = globaltimer_ns();
        while (!ptx::mbar_try_wait(bar, 0) && globaltimer_ns() - t0 < kWaitTimeoutNs) {
        }
      }
      __syncthreads();
    }
  }
  if (ok && active3) {
    int cob, cu, cstart, clen;
    locate3(b0, cob, cu, cstart, clen);
    int cbg = b0 - cstart, cfirst = cbg;
    // this lane's h row of entry u (the zero row past the entry's tokens)
    auto hrow3 = [&](int u) {
      return (g < rt.ent_n[u] ? hs + (int64_t)rt.ent_col[u][g] * hsm : zrow) + EPL * t4;
    };
    const uint16_t* ch = hrow3(cu);
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int b = b0; b < b1; ++b) {
      const bool more = b + 1 < b1;
      if (more) {
        ++lx;
        if (++lbg == llen) {
          int ob, u, start;
          locate3(lx, ob, u, start, llen);
          lbg = 0;
          lp3 = row3(lx, lK);
        }
      }
      const int ls0 = lbg * kDepth, cs0 = cbg * kDepth;
#pragma unroll
      for (int i = 0; i < kDepth; ++i) {
        const uint4 v = ring3[i];
        if (more)
          ring3[i] = (ls0 + i) * EPS + EPL * t4 < lK ? ld_stream(lp3 + (int64_t)(ls0 + i) * BPS)
                                                     : make_uint4(0u, 0u, 0u, 0u);
        mma_step<FMT>(acc, v, ch + (cs0 + i) * EPS);
      }
      const bool end_group = ++cbg == clen;
      if (end_group || !more) {
        // store this piece of y (0: it starts the group, 1: it ends it; a
        // whole group also zeroes its second half) per (token, slot) column,
        // then count its blocks towards the output block
        const int piece = cfirst != 0 ? 1 : 0;
        const bool whole = cfirst == 0 && end_group;
        if (g < rt.ent_n[cu]) {
          float y0 = acc[0], y1 = acc[1];
          if (FMT == kDecodeE4M3) {
            const int e = rt.ent_e[cu];
            const float* sd = e < N ? static_cast<const float*>(a.w_down_scale) + (int64_t)e * d
                                    : static_cast<const float*>(a.s_down_scale) + (int64_t)(e - N) * d;
            y0 *= __ldg(sd + 8 * cob + 2 * t4);
            y1 *= __ldg(sd + 8 * cob + 2 * t4 + 1);
          }
          float* yb = a.ybuf + ((int64_t)cob * 2 * ycols + rt.ent_col[cu][g]) * 8 + 2 * t4;
          *reinterpret_cast<float2*>(yb + (int64_t)piece * ycols * 8) = make_float2(y0, y1);
          if (whole) *reinterpret_cast<float2*>(yb + (int64_t)ycols * 8) = make_float2(0.f, 0.f);
        }
        __threadfence();
        __syncwarp();
        const uint32_t done = (uint32_t)(cbg - cfirst);
        uint32_t prev = 0;
        if (lane == 0) prev = atomicAdd(a.blk_cnt + cob, done);
        prev = __shfl_sync(0xFFFFFFFFu, prev, 0);
        if (prev + done == (uint32_t)per_ob) {
          // the output block's last piece: out[t][8 ob + n] for lane (t, n) =
          // sum_k w[t][k] y[t,k][n] (slot order; dropped copies add nothing)
          // + the shared experts' y[T*K + s*T + t][n]
          __threadfence();
          const int t = lane >> 3, n = lane & 7;
          if (t < T) {
            const float* yb = a.ybuf + (int64_t)cob * 2 * ycols * 8 + n;
            const int64_t half = (int64_t)ycols * 8;
            float o = 0.f;
            for (int k0 = 0; k0 < K; k0 += 8) {
              float yv[8], wv[8];
#pragma unroll
              for (int q = 0; q < 8; ++q) {
                const int k = k0 + q;
                const bool use = k < K && rt.keep[t][k];
                const float* p = yb + (int64_t)(t * K + (use ? k : 0)) * 8;
                yv[q] = use ? __ldcg(p) + __ldcg(p + half) : 0.f;
                wv[q] = use ? rt.w[t][k] : 0.f;
              }
#pragma unroll
              for (int q = 0; q < 8; ++q) o = fmaf(wv[q], yv[q], o);
            }
            for (int s0 = 0; s0 < a.S; ++s0) {
              const float* p = yb + (int64_t)(T * K + s0 * T + t) * 8;
              o += __ldcg(p) + __ldcg(p + half);
            }
            a.out[(int64_t)t * d + 8 * cob + n] = __float2bfloat16_rn(o);
          }
        }
        acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
        if (end_group && more) {
          locate3(b + 1, cob, cu, cstart, clen);
          cbg = 0;
          cfirst = 0;
          ch = hrow3(cu);
        }
      }
    }
  }
  if (over) atomicOr(a.err, kErrRange);

  // the last CTA to leave returns the barrier counters to zero
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(a.sync + 1, 1u) == (uint32_t)G - 1) {
      atomicExch(a.sync, 0u);
      atomicExch(a.sync + 1, 0u);
    }
  }
}

template <int FMT, bool HB>
cudaError_t launch_fh(const DecodeArgs& a, cudaStream_t s) {
  void (*kern)(const DecodeArgs) = decode_layer_kernel<FMT, HB>;
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(configured.load() & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDecodeMaxSmem);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit);
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)a.grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = a.smem_bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace

DecodePlan decode_plan(const moe_problem_t& p, int sms) {
  DecodePlan pl{};
  const int64_t T = p.T;
  const bool fp8 = p.expert_dtype == MOE_EXPERT_FP8_E4M3;
  const int E = fp8 ? 16 : 8;     // weights per 16-byte unit
  const int EPS = fp8 ? 64 : 32;  // elements of a row per step
  pl.grid = sms;
  // router slices: at most kRouterRowsPerThread rows per thread, one batch
  // of loads, over at most min(grid, kDecodeMaxSplits) CTAs
  const int Q = p.n_experts > 0 ? kDecodeThreads / p.n_experts : 1;
  const int max_splits = sms < kDecodeMaxSplits ? sms : kDecodeMaxSplits;
  int slice = kRouterRowsPerThread * (Q > 0 ? Q : 1);
  if ((p.d_model + slice - 1) / slice > max_splits) slice = (p.d_model + max_splits - 1) / max_splits;
  pl.r_slice = slice;
  pl.rsplits = (p.d_model + slice - 1) / slice;
  // 16-bit rows in shared memory, zero-padded to whole blocks of kDepth
  // steps; a row stride of 64 bytes past a multiple of 128 puts two token
  // rows in one wavefront
  auto stride = [&](int k) {
    const int64_t blocks = ((int64_t)(k + EPS - 1) / EPS + kDepth - 1) / kDepth;
    const int64_t padded = blocks * kDepth * EPS;
    return (int)(((padded * 2 + 127) / 128 * 128 + 64) / 2);
  };
  pl.x_stride = stride(p.d_model);
  auto padded = [&](int k) { return (int)(((int64_t)(k + EPS - 1) / EPS + kDepth - 1) / kDepth * kDepth * EPS); };
  pl.h_stride = padded(p.ffn);
  pl.hs_stride = p.n_shared > 0 ? padded(p.shared_ffn) : 0;
  const int hmax = pl.h_stride > pl.hs_stride ? pl.h_stride : pl.hs_stride;
  pl.hsm_stride = (int)(((int64_t)hmax * 2 + 127) / 128 * 128 + 64) / 2;
  const int Fmax = p.n_shared > 0 && p.shared_ffn > p.ffn ? p.shared_ffn : p.ffn;
  const int hs = stride(Fmax);
  pl.z_len = pl.x_stride > hs ? pl.x_stride : hs;
  const int64_t hrows = T * p.top_k + (int64_t)p.n_shared * T;
  const size_t x_bytes = ((size_t)T * pl.x_stride + pl.z_len) * 2;
  const size_t ph3 = ((size_t)hrows * pl.hsm_stride + pl.z_len) * 2;
  const size_t red0 = ((size_t)T * slice + (size_t)(Q > 0 ? Q : 1) * T * p.n_experts) * 4;
  const size_t red1 = ((size_t)T * p.n_experts + (3 * (size_t)T * p.n_experts > kDecodeThreads
                                                      ? 2 * (size_t)T * p.n_experts : kDecodeThreads)) * 4;
  const size_t red_bytes = red0 > red1 ? red0 : red1;
  pl.smem_x_bytes = (x_bytes + 127) / 128 * 128;
  pl.smem_bytes = pl.smem_x_bytes + red_bytes > ph3 ? pl.smem_x_bytes + red_bytes : ph3;
  pl.ok = p.routing == MOE_ROUTING_TOKEN_CHOICE && T >= 1 && T <= kDecodeMaxTokens && p.top_k <= kMaxTopK &&
          p.n_experts >= 1 && p.n_experts <= kMaxExperts && p.n_shared <= kMaxShared && (p.d_model % E) == 0 &&
          (p.ffn % E) == 0 && (p.n_shared == 0 || (p.shared_ffn % E) == 0) && pl.smem_bytes <= kDecodeMaxSmem &&
          hrows <= 32767 && pl.rsplits <= max_splits;
  return pl;
}

size_t decode_h_elems(const moe_problem_t& p, bool shared) {
  const bool fp8 = p.expert_dtype == MOE_EXPERT_FP8_E4M3;
  const int EPS = fp8 ? 64 : 32;
  const int k = shared ? p.shared_ffn : p.ffn;
  const int64_t stride = ((int64_t)(k + EPS - 1) / EPS + kDepth - 1) / kDepth * kDepth * EPS;
  const int64_t rows = shared ? (int64_t)p.n_shared * p.T : p.T * (int64_t)p.top_k;
  return (size_t)(rows * stride);
}

size_t decode_ybuf_floats(const moe_problem_t& p) {
  // the down phase's results: per output block of 8 elements, two pieces of
  // every (token, slot) column and every shared (expert, token) column
  const int64_t cols = p.T * (int64_t)p.top_k + (int64_t)p.n_shared * p.T;
  return (size_t)(p.d_model / 8) * 2 * (size_t)cols * 8;
}

cudaError_t launch_decode_layer(const DecodeArgs& a, cudaStream_t s) {
  if (a.T < 1 || a.T > kDecodeMaxTokens || a.grid < 1) return cudaErrorInvalidValue;
  if (a.fmt == kDecodeE4M3)
    return a.hidden_bf16 ? launch_fh<kDecodeE4M3, true>(a, s) : launch_fh<kDecodeE4M3, false>(a, s);
  if (a.fmt != kDecodeBf16) return cudaErrorInvalidValue;
  return a.hidden_bf16 ? launch_fh<kDecodeBf16, true>(a, s) : launch_fh<kDecodeBf16, false>(a, s);
}

}  // namespace moe
