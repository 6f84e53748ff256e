/*
 * moe_oracle.c — the ORACLE for the token-choice MoE FFN layer forward pass.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the plain, slow, obviously correct CPU
 * statement of what the layer computes. Only the test suite, the smoke check
 * and the benchmark's CPU-baseline leg may load it. It shares no code, header,
 * table or helper with the CUDA library, and the CUDA library never calls it.
 *
 * Arithmetic: fp64 throughout, plain loops in the order the definition states,
 * with one deliberate exception. The router is an fp32 layer ("Chapter 19:
 * Mixture-of-Experts Models", §19.6.2 table, "Higher-precision router": the
 * router is kept in higher precision than the bf16 experts). So each logit is
 * the fp64 dot product rounded once to fp32, and the top-K decision compares
 * fp32 keys: the same precision the device kernel decides in. Everything after
 * the decision (weights, expert FFNs, combine) is fp64.
 *
 * Expert weights arrive as bf16 bit patterns (uint16), as FP8 E4M3 codes
 * (uint8) with one fp32 scale per matrix row, or as MXFP4 (E2M1 codes two
 * per byte with one E8M0 scale per 32 elements of a row) ("AI Infrastructure series, Part
 * 12 of 24", "How do you serve an MoE model on your own GPUs?": quantise the
 * experts' weights, keep the router in 16 bits or more; "Mixture of Experts
 * Explained", "Total versus active parameters": the bytes a token reads fall
 * by the same factor as the storage); either way each weight is widened
 * exactly to fp64 element by element. Hidden rows arrive as fp32 (a bf16
 * hidden is widened exactly by the caller).
 *
 * Parity status of every function: pinned (see the tests of the oracle).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_ERR_ARG -1
#define ORACLE_ERR_MISSING_EXPERT -2

static double bf16_bits_to_double(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* OCP FP8 E4M3 ("fn": no infinities): sign, 4 exponent bits with bias 7,
 * 3 mantissa bits; exponent 0 encodes subnormals m/8 * 2^-6; S.1111.111 is
 * NaN. */
double moe_oracle_e4m3_to_double(uint8_t b) {
  const int s = b >> 7, e = (b >> 3) & 15, m = b & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) v = ldexp((double)m / 8.0, -6);
  else v = ldexp(1.0 + (double)m / 8.0, e - 7);
  return s ? -v : v;
}

/* OCP FP4 E2M1: sign, 2 exponent bits with bias 1, 1 mantissa bit; exponent
 * 0 encodes the subnormal m * 0.5. Values 0, 0.5, 1, 1.5, 2, 3, 4, 6 and
 * their negatives. */
double moe_oracle_e2m1_to_double(uint8_t c) {
  const int s = (c >> 3) & 1, e = (c >> 1) & 3, m = c & 1;
  const double v = e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
  return s ? -v : v;
}

/* OCP E8M0 shared scale: 2^(E - 127); E = 255 is NaN. */
double moe_oracle_e8m0_to_double(uint8_t e) { return e == 255 ? NAN : ldexp(1.0, (int)e - 127); }

/* Expert weights in one of three storage formats:
 *   0  bf16 values;
 *   1  FP8 E4M3 codes with one fp32 scale per matrix row: w = e4m3(q) * scale[row];
 *   2  MXFP4 (OCP microscaling): E2M1 codes packed two per byte (element 2i
 *      in the low nibble, 2i+1 in the high nibble) and one E8M0 scale per 32
 *      consecutive elements of a row: w = e2m1(q) * 2^(bscale[row][col/32] - 127). */
typedef struct {
  int fmt;
  const void* q;
  const float* scale;     /* fmt 1: [rows] */
  const uint8_t* bscale;  /* fmt 2: [rows][ld / 32] */
} wmat_t;

static double wload(wmat_t w, int64_t row, int64_t ld, int64_t col) {
  if (w.fmt == 0) return bf16_bits_to_double(((const uint16_t*)w.q)[row * ld + col]);
  if (w.fmt == 1) return moe_oracle_e4m3_to_double(((const uint8_t*)w.q)[row * ld + col]) * (double)w.scale[row];
  const uint8_t byte = ((const uint8_t*)w.q)[row * (ld / 2) + col / 2];
  const uint8_t code = (col & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 15);
  return moe_oracle_e2m1_to_double(code) * moe_oracle_e8m0_to_double(w.bscale[row * (ld / 32) + col / 32]);
}

/* A set of experts' matrices, one pointer per expert (NULL: not provided),
 * all in one format; the scale arrays (fp32 row scales for fmt 1, E8M0 block
 * scales for fmt 2) are unused for bf16. */
typedef struct {
  int fmt;
  const void* const* gate;
  const void* const* up;
  const void* const* down;
  const void* const* s_gate;
  const void* const* s_up;
  const void* const* s_down;
} wset_t;

/* Expert e of a set; returns 0 if any of its matrices (or scales) is missing. */
static int wset_expert(const wset_t* ws, int32_t e, wmat_t* g, wmat_t* u, wmat_t* dn) {
  if (!ws->gate[e] || !ws->up[e] || !ws->down[e]) return 0;
  if (ws->fmt != 0 && (!ws->s_gate || !ws->s_up || !ws->s_down || !ws->s_gate[e] || !ws->s_up[e] ||
                       !ws->s_down[e]))
    return 0;
  g->fmt = u->fmt = dn->fmt = ws->fmt;
  g->q = ws->gate[e];
  u->q = ws->up[e];
  dn->q = ws->down[e];
  g->scale = ws->fmt == 1 ? (const float*)ws->s_gate[e] : NULL;
  u->scale = ws->fmt == 1 ? (const float*)ws->s_up[e] : NULL;
  dn->scale = ws->fmt == 1 ? (const float*)ws->s_down[e] : NULL;
  g->bscale = ws->fmt == 2 ? (const uint8_t*)ws->s_gate[e] : NULL;
  u->bscale = ws->fmt == 2 ? (const uint8_t*)ws->s_up[e] : NULL;
  dn->bscale = ws->fmt == 2 ? (const uint8_t*)ws->s_down[e] : NULL;
  return 1;
}

int moe_oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* SiLU(z) = z * sigmoid(z) = z / (1 + e^-z): the gate nonlinearity of the
 * SwiGLU reading of "an ordinary MLP" with "3 matrices" ("AI Infrastructure
 * series Part 12", "What is a Mixture of Experts model?"; "Mixture of Experts
 * Explained", "The slot it replaces"). */
double moe_oracle_silu(double z) { return z / (1.0 + exp(-z)); }

/* Logistic sigmoid, the DeepSeek-V3 affinity ("Mixture of Experts for LLM
 * Inference", "Opening the router": sigmoid + normalisation instead of a
 * softmax). */
static double sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }

/*
 * Router for one token ("Mixture of Experts for LLM Inference", "Opening the
 * router"; "Chapter 19", §19.3.2 and §19.3.4; "AI Infrastructure series Part
 * 12", "How does the router decide? A worked example").
 *
 * 1. logit_e = sum_j x_j * W_router[j][e]  (+ router_bias_e), fp64, j ascending;
 *    then rounded once to fp32.
 * 2. softmax scoring: key_e = logit_e; probs_e = full softmax over all N.
 *    sigmoid scoring: s_e = sigmoid(logit_e); key_e = fp32(s_e + sel_bias_e);
 *    probs_e = s_e.
 * 3. top-K: repeatedly take the largest remaining key; equal keys go to the
 *    lower expert index. Slot k holds the k-th pick.
 * 4. margin = the smallest gap between consecutive keys among the first
 *    min(K+1, N) picks: how far the token is from a different choice or a
 *    different slot order.
 *    Group-limited routing (n_groups > 1, topk_groups < n_groups): the N
 *    experts form n_groups equal groups of consecutive indices; a group's
 *    score is the sum of its two largest keys (its one key for groups of one);
 *    the topk_groups best groups (score desc, group index asc) are kept and
 *    the top-K picks above range over their experts only. The margin then
 *    also covers the gaps between consecutive group scores among the first
 *    topk_groups + 1 groups ("Mixture of Experts for LLM Inference", "Three
 *    tricks that tame the all-to-alls": node-limited routing caps how many
 *    nodes a token may visit; "AI Infrastructure series Part 12": at most 4
 *    servers per token).
 * 5. weights: softmax + renormalise -> exp(l_j - l_max) / sum over the chosen;
 *    softmax, no renormalise -> probs of the chosen;
 *    sigmoid + renormalise -> s_j / sum of chosen s (unbiased: the selection
 *    bias never reaches the weights); sigmoid, no renormalise -> s_j.
 */
static void router_one_token(int32_t d, int32_t N, int32_t K, int32_t score_fn,
                             int32_t renormalize, int32_t n_groups, int32_t topk_groups,
                             const float* x,
                             const float* w_router, const float* router_bias,
                             const float* sel_bias, double* logits_out,
                             double* probs_out, float* keys_out,
                             int32_t* idx_out, double* w_out, double* margin_out,
                             float* l32, double* prob, float* key,
                             unsigned char* taken, int32_t* order) {
  for (int32_t e = 0; e < N; ++e) {
    double acc = 0.0;
    for (int32_t j = 0; j < d; ++j) acc += (double)x[j] * (double)w_router[(int64_t)j * N + e];
    if (router_bias) acc += (double)router_bias[e];
    l32[e] = (float)acc;
    if (logits_out) logits_out[e] = (double)l32[e];
  }
  if (score_fn == 0) {
    double mx = -INFINITY;
    for (int32_t e = 0; e < N; ++e) if ((double)l32[e] > mx) mx = (double)l32[e];
    double z = 0.0;
    for (int32_t e = 0; e < N; ++e) z += exp((double)l32[e] - mx);
    for (int32_t e = 0; e < N; ++e) {
      prob[e] = exp((double)l32[e] - mx) / z;
      key[e] = l32[e];
    }
  } else {
    for (int32_t e = 0; e < N; ++e) {
      prob[e] = sigmoid((double)l32[e]);
      double b = sel_bias ? (double)sel_bias[e] : 0.0;
      key[e] = (float)(prob[e] + b);
    }
  }
  if (probs_out) for (int32_t e = 0; e < N; ++e) probs_out[e] = prob[e];
  if (keys_out) for (int32_t e = 0; e < N; ++e) keys_out[e] = key[e];

  /* Experts a token may pick: all, or those of the kept groups. taken[e] = 1
   * marks an expert already picked or not allowed. */
  int32_t allowed = N;
  double margin = INFINITY;
  for (int32_t e = 0; e < N; ++e) taken[e] = 0;
  if (n_groups > 1 && topk_groups < n_groups) {
    const int32_t gs = N / n_groups;
    double gscore[256];
    unsigned char gkept[256];
    for (int32_t g = 0; g < n_groups; ++g) {
      int32_t b1 = -1, b2 = -1; /* the group's two largest keys */
      for (int32_t e = g * gs; e < (g + 1) * gs; ++e) {
        if (b1 < 0 || key[e] > key[b1]) {
          b2 = b1;
          b1 = e;
        } else if (b2 < 0 || key[e] > key[b2]) {
          b2 = e;
        }
      }
      gscore[g] = (double)key[b1] + (b2 >= 0 ? (double)key[b2] : 0.0);
      gkept[g] = 0;
    }
    int32_t gpicks = (topk_groups + 1 < n_groups) ? topk_groups + 1 : n_groups;
    int32_t gorder[257];
    for (int32_t k = 0; k < gpicks; ++k) {
      int32_t best = -1;
      for (int32_t g = 0; g < n_groups; ++g) {
        if (gkept[g]) continue;
        if (best < 0 || gscore[g] > gscore[best]) best = g;
      }
      gkept[best] = 1;
      gorder[k] = best;
    }
    for (int32_t k = 0; k + 1 < gpicks; ++k) {
      double gap = gscore[gorder[k]] - gscore[gorder[k + 1]];
      if (gap < margin) margin = gap;
    }
    for (int32_t g = 0; g < n_groups; ++g) gkept[g] = 0;
    for (int32_t k = 0; k < topk_groups; ++k) gkept[gorder[k]] = 1;
    allowed = topk_groups * gs;
    for (int32_t e = 0; e < N; ++e)
      if (!gkept[e / gs]) taken[e] = 1;
  }
  int32_t picks = (K + 1 < allowed) ? K + 1 : allowed;
  for (int32_t k = 0; k < picks; ++k) {
    int32_t best = -1;
    for (int32_t e = 0; e < N; ++e) {
      if (taken[e]) continue;
      if (best < 0 || key[e] > key[best]) best = e; /* strict: ties keep the lower index */
    }
    taken[best] = 1;
    order[k] = best;
  }
  for (int32_t k = 0; k + 1 < picks; ++k) {
    double gap = (double)key[order[k]] - (double)key[order[k + 1]];
    if (gap < margin) margin = gap;
  }
  *margin_out = margin;

  for (int32_t k = 0; k < K; ++k) idx_out[k] = order[k];
  if (score_fn == 0) {
    if (renormalize) {
      double lmax = (double)l32[order[0]];
      double z = 0.0;
      for (int32_t k = 0; k < K; ++k) z += exp((double)l32[order[k]] - lmax);
      for (int32_t k = 0; k < K; ++k) w_out[k] = exp((double)l32[order[k]] - lmax) / z;
    } else {
      for (int32_t k = 0; k < K; ++k) w_out[k] = prob[order[k]];
    }
  } else {
    if (renormalize) {
      double z = 0.0;
      for (int32_t k = 0; k < K; ++k) z += prob[order[k]];
      for (int32_t k = 0; k < K; ++k) w_out[k] = prob[order[k]] / z;
    } else {
      for (int32_t k = 0; k < K; ++k) w_out[k] = prob[order[k]];
    }
  }
}

static int router_args_ok(int64_t T, int32_t d, int32_t N, int32_t K, int32_t score_fn,
                          int32_t n_groups, int32_t topk_groups,
                          const float* hidden, const float* w_router) {
  if (T < 0 || d <= 0 || N <= 0 || K <= 0 || K > N) return 0;
  if (n_groups > 1) {
    if (N % n_groups != 0 || n_groups > 256 || topk_groups < 1 || topk_groups > n_groups) return 0;
    if (K > topk_groups * (N / n_groups)) return 0;
  }
  if (score_fn != 0 && score_fn != 1) return 0;
  if ((T > 0 && !hidden) || !w_router) return 0;
  return 1;
}

/*
 * Router over T tokens (rows of `hidden`, fp32 [T][d]). Outputs per token:
 * logits/probs (fp64 [T][N], nullable), keys (fp32 [T][N], nullable),
 * topk_idx [T][K], topk_w (fp64 [T][K]), margin (fp64 [T]).
 */
int moe_oracle_router(int64_t T, int32_t d, int32_t N, int32_t K, int32_t score_fn,
                      int32_t renormalize, int32_t n_groups, int32_t topk_groups,
                      const float* hidden, const float* w_router,
                      const float* router_bias, const float* sel_bias,
                      double* logits_out, double* probs_out, float* keys_out,
                      int32_t* topk_idx, double* topk_w, double* margin) {
  if (!router_args_ok(T, d, N, K, score_fn, n_groups, topk_groups, hidden, w_router)) return ORACLE_ERR_ARG;
  if (!topk_idx || !topk_w || !margin) return ORACLE_ERR_ARG;
  int failed = 0;
#pragma omp parallel
  {
    float* l32 = (float*)malloc(sizeof(float) * (size_t)N);
    double* prob = (double*)malloc(sizeof(double) * (size_t)N);
    float* key = (float*)malloc(sizeof(float) * (size_t)N);
    unsigned char* taken = (unsigned char*)malloc((size_t)N);
    int32_t* order = (int32_t*)malloc(sizeof(int32_t) * (size_t)N);
    if (!l32 || !prob || !key || !taken || !order) {
#pragma omp atomic write
      failed = 1;
    } else {
#pragma omp for schedule(dynamic, 4)
      for (int64_t t = 0; t < T; ++t) {
        router_one_token(d, N, K, score_fn, renormalize, n_groups, topk_groups, hidden + t * d, w_router,
                         router_bias, sel_bias, logits_out ? logits_out + t * N : NULL,
                         probs_out ? probs_out + t * N : NULL,
                         keys_out ? keys_out + t * N : NULL, topk_idx + t * K,
                         topk_w + t * K, margin + t, l32, prob, key, taken, order);
      }
    }
    free(l32); free(prob); free(key); free(taken); free(order);
  }
  return failed ? ORACLE_ERR_ARG : ORACLE_OK;
}

/*
 * Expert capacity ("Chapter 19", §19.6.1): C = ceil(c * T * K / N) for
 * capacity factor c > 0. Returns -1 (no cap) for c <= 0.
 */
int64_t moe_oracle_capacity(double c, int64_t T, int32_t K, int32_t N) {
  if (!(c > 0.0)) return -1;
  return (int64_t)ceil(c * (double)T * (double)K / (double)N);
}

/*
 * Route and pack ("Chapter 19", §19.6.3): a counting sort of the T*K token
 * copies by expert.
 *   counts[e]    = number of copies whose expert is e (histogram)
 *   offsets[0]   = 0, offsets[e+1] = offsets[e] + counts[e] (exclusive scan)
 *   perm_src[r]  = t*K + k for the copies in expert-major order; inside one
 *                  expert the copies keep their (t, k) order, i.e. token
 *                  ascending (a token picks an expert at most once)
 *   inv_row[t*K+k] = r, the inverse permutation.
 * Returns ORACLE_ERR_ARG if an index lies outside [0, N).
 */
/*
 * With a capacity cap >= 0 ("Chapter 19", §19.6.1 "capacity-limited";
 * "Mixture of Experts Explained", "Routing collapses unless you stop it":
 * copies beyond the cap skip the FFN and pass on the residual alone), only the
 * first `cap` copies of each expert in (t, k) order are placed: offsets count
 * kept copies, inv_row of a dropped copy is -1, counts still count every copy
 * routed to the expert. cap < 0: no cap.
 */
int moe_oracle_permute_cap(int64_t T, int32_t K, int32_t N, int64_t cap, const int32_t* topk_idx,
                           int32_t* counts, int32_t* offsets, int32_t* perm_src, int32_t* inv_row) {
  if (T < 0 || K <= 0 || N <= 0 || !counts || !offsets) return ORACLE_ERR_ARG;
  if (T > 0 && (!topk_idx || !perm_src || !inv_row)) return ORACLE_ERR_ARG;
  const int64_t n = T * K;
  for (int32_t e = 0; e < N; ++e) counts[e] = 0;
  for (int64_t i = 0; i < n; ++i) {
    int32_t e = topk_idx[i];
    if (e < 0 || e >= N) return ORACLE_ERR_ARG;
    counts[e] += 1;
  }
  offsets[0] = 0;
  for (int32_t e = 0; e < N; ++e) {
    int64_t kept = counts[e];
    if (cap >= 0 && kept > cap) kept = cap;
    offsets[e + 1] = offsets[e] + (int32_t)kept;
  }
  int32_t* seen = (int32_t*)malloc(sizeof(int32_t) * (size_t)N);
  if (!seen) return ORACLE_ERR_ARG;
  for (int32_t e = 0; e < N; ++e) seen[e] = 0;
  for (int64_t i = 0; i < n; ++i) {
    int32_t e = topk_idx[i];
    int32_t rank = seen[e]++;
    if (cap >= 0 && rank >= cap) {
      inv_row[i] = -1;
      continue;
    }
    int32_t r = offsets[e] + rank;
    perm_src[r] = (int32_t)i;
    inv_row[i] = r;
  }
  free(seen);
  return ORACLE_OK;
}

int moe_oracle_permute(int64_t T, int32_t K, int32_t N, const int32_t* topk_idx,
                       int32_t* counts, int32_t* offsets, int32_t* perm_src,
                       int32_t* inv_row) {
  if (T < 0 || K <= 0 || N <= 0 || !counts || !offsets) return ORACLE_ERR_ARG;
  if (T > 0 && (!topk_idx || !perm_src || !inv_row)) return ORACLE_ERR_ARG;
  const int64_t n = T * K;
  for (int32_t e = 0; e < N; ++e) counts[e] = 0;
  for (int64_t i = 0; i < n; ++i) {
    int32_t e = topk_idx[i];
    if (e < 0 || e >= N) return ORACLE_ERR_ARG;
    counts[e] += 1;
  }
  offsets[0] = 0;
  for (int32_t e = 0; e < N; ++e) offsets[e + 1] = offsets[e] + counts[e];
  int32_t* cursor = (int32_t*)malloc(sizeof(int32_t) * (size_t)N);
  if (!cursor) return ORACLE_ERR_ARG;
  for (int32_t e = 0; e < N; ++e) cursor[e] = offsets[e];
  for (int64_t i = 0; i < n; ++i) {
    int32_t r = cursor[topk_idx[i]]++;
    perm_src[r] = (int32_t)i;
    inv_row[i] = r;
  }
  free(cursor);
  return ORACLE_OK;
}

/*
 * One expert FFN on one token, SwiGLU reading:
 *   g = W_gate x,  u = W_up x         (W_gate, W_up: [F][d])
 *   h_f = SiLU(g_f) * u_f
 *   y = W_down h                      (W_down: [d][F])
 * Each weight is decoded from its stored format (bf16, or FP8 E4M3 code times
 * its row's scale) to an exact double. `h` is caller scratch of F doubles; y
 * is fp64 [d].
 */
static void expert_ffn_w(int32_t d, int32_t F, const double* x, wmat_t wg, wmat_t wu, wmat_t wd,
                         double* h, double* y) {
  for (int32_t f = 0; f < F; ++f) {
    double g = 0.0, u = 0.0;
    for (int32_t j = 0; j < d; ++j) {
      g += wload(wg, f, d, j) * x[j];
      u += wload(wu, f, d, j) * x[j];
    }
    h[f] = moe_oracle_silu(g) * u;
  }
  for (int32_t i = 0; i < d; ++i) {
    double acc = 0.0;
    for (int32_t f = 0; f < F; ++f) acc += wload(wd, i, F, f) * h[f];
    y[i] = acc;
  }
}

void moe_oracle_expert_ffn(int32_t d, int32_t F, const double* x, const uint16_t* w_gate,
                           const uint16_t* w_up, const uint16_t* w_down, double* h,
                           double* y) {
  const wmat_t wg = {0, w_gate, NULL, NULL}, wu = {0, w_up, NULL, NULL}, wd = {0, w_down, NULL, NULL};
  expert_ffn_w(d, F, x, wg, wu, wd, h, y);
}

/* The same expert with FP8 E4M3 weights and per-row scales: W_gate, W_up
 * codes [F][d] with scales [F]; W_down codes [d][F] with scales [d]. */
void moe_oracle_expert_ffn_fp8(int32_t d, int32_t F, const double* x, const uint8_t* q_gate,
                               const float* s_gate, const uint8_t* q_up, const float* s_up,
                               const uint8_t* q_down, const float* s_down, double* h, double* y) {
  const wmat_t wg = {1, q_gate, s_gate, NULL}, wu = {1, q_up, s_up, NULL}, wd = {1, q_down, s_down, NULL};
  expert_ffn_w(d, F, x, wg, wu, wd, h, y);
}

/* The same expert with MXFP4 weights: W_gate, W_up codes [F][d/2] with E8M0
 * block scales [F][d/32]; W_down codes [d][F/2] with block scales [d][F/32]
 * (d and F multiples of 32). */
void moe_oracle_expert_ffn_mxfp4(int32_t d, int32_t F, const double* x, const uint8_t* q_gate,
                                 const uint8_t* b_gate, const uint8_t* q_up, const uint8_t* b_up,
                                 const uint8_t* q_down, const uint8_t* b_down, double* h, double* y) {
  const wmat_t wg = {2, q_gate, NULL, b_gate}, wu = {2, q_up, NULL, b_up}, wd = {2, q_down, NULL, b_down};
  expert_ffn_w(d, F, x, wg, wu, wd, h, y);
}

/*
 * Gate-weighted combine for one token ("Chapter 19", §19.3.2 and the §19.2
 * flowchart "Sum with gate weights"; "AI Infrastructure series Part 12",
 * worked example): out = sum_k w_k * y_k  (+ shared, weight 1, if given).
 *   w [K], y [K][d], shared [d] or NULL, out [d].
 */
void moe_oracle_combine(int32_t K, int32_t d, const double* w, const double* y,
                        const double* shared, double* out) {
  for (int32_t i = 0; i < d; ++i) {
    double acc = 0.0;
    for (int32_t k = 0; k < K; ++k) acc += w[k] * y[(int64_t)k * d + i];
    if (shared) acc += shared[i];
    out[i] = acc;
  }
}

/*
 * Expert-choice routing ("Mixture of Experts for LLM Inference", "Token choice
 * vs expert choice": each expert picks its own top tokens up to a fixed
 * capacity; "Chapter 19", §19.6.1 "Expert Choice"; "Mixture of Experts
 * Explained", "Expert-choice versus token-choice routing").
 *   1. logits as in the router (fp64 sum, rounded to fp32), + router_bias;
 *   2. score S[t][e]: softmax over the N experts of token t, or sigmoid;
 *      rounded to fp32 (the precision the selection is decided in);
 *   3. expert e takes the C tokens with the largest S[.][e] (equal scores:
 *      lower token first); its rows list them in ascending token order;
 *      row weight = S[t][e] in fp64 (no renormalisation);
 *   4. margin[e] = S of e's C-th pick minus S of its (C+1)-th (fp32 values),
 *      +inf when C >= T.
 * Outputs: row_token [N][C], row_w fp64 [N][C], margin fp64 [N].
 */
int moe_oracle_expert_choice(int64_t T, int32_t d, int32_t N, int32_t score_fn, int64_t C,
                             const float* hidden, const float* w_router, const float* router_bias,
                             int32_t* row_token, double* row_w, double* margin) {
  if (T <= 0 || d <= 0 || N <= 0 || C <= 0 || C > T || !hidden || !w_router) return ORACLE_ERR_ARG;
  if (!row_token || !row_w || !margin || (score_fn != 0 && score_fn != 1)) return ORACLE_ERR_ARG;
  double* s64 = (double*)malloc(sizeof(double) * (size_t)T * (size_t)N);
  float* s32 = (float*)malloc(sizeof(float) * (size_t)T * (size_t)N);
  if (!s64 || !s32) {
    free(s64);
    free(s32);
    return ORACLE_ERR_ARG;
  }
#pragma omp parallel for schedule(dynamic, 8)
  for (int64_t t = 0; t < T; ++t) {
    float l[256];
    for (int32_t e = 0; e < N; ++e) {
      double acc = 0.0;
      for (int32_t j = 0; j < d; ++j) acc += (double)hidden[t * d + j] * (double)w_router[(int64_t)j * N + e];
      if (router_bias) acc += (double)router_bias[e];
      l[e] = (float)acc;
    }
    if (score_fn == 0) {
      double mx = -INFINITY, z = 0.0;
      for (int32_t e = 0; e < N; ++e) if ((double)l[e] > mx) mx = (double)l[e];
      for (int32_t e = 0; e < N; ++e) z += exp((double)l[e] - mx);
      for (int32_t e = 0; e < N; ++e) s64[t * N + e] = exp((double)l[e] - mx) / z;
    } else {
      for (int32_t e = 0; e < N; ++e) s64[t * N + e] = sigmoid((double)l[e]);
    }
    for (int32_t e = 0; e < N; ++e) s32[t * N + e] = (float)s64[t * N + e];
  }
  int status = ORACLE_OK;
#pragma omp parallel
  {
    unsigned char* picked = (unsigned char*)malloc((size_t)T);
    if (!picked) {
#pragma omp atomic write
      status = ORACLE_ERR_ARG;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (int32_t e = 0; e < N; ++e) {
        for (int64_t t = 0; t < T; ++t) picked[t] = 0;
        float last = 0.f;
        for (int64_t c = 0; c < C; ++c) { /* selection: largest score, lower token on ties */
          int64_t best = -1;
          for (int64_t t = 0; t < T; ++t) {
            if (picked[t]) continue;
            if (best < 0 || s32[t * N + e] > s32[best * N + e]) best = t;
          }
          picked[best] = 1;
          last = s32[best * N + e];
        }
        double gap = INFINITY;
        if (C < T) {
          int64_t next = -1;
          for (int64_t t = 0; t < T; ++t) {
            if (picked[t]) continue;
            if (next < 0 || s32[t * N + e] > s32[next * N + e]) next = t;
          }
          gap = (double)last - (double)s32[next * N + e];
        }
        margin[e] = gap;
        int64_t r = 0;
        for (int64_t t = 0; t < T; ++t) {
          if (!picked[t]) continue;
          row_token[(int64_t)e * C + r] = (int32_t)t;
          row_w[(int64_t)e * C + r] = s64[t * N + e];
          ++r;
        }
      }
    }
    free(picked);
  }
  free(s64);
  free(s32);
  return status;
}

/*
 * The layer under a given routing: out[t] = sum_k w[t][k] * E_{idx[t][k]}(x_t)
 * (+ the shared experts), skipping slots with idx < 0. Used for expert-choice
 * routing, where the number of experts per token varies (0..N).
 *   idx int32 [n][M], w fp64 [n][M]; other arguments as moe_oracle_layer.
 */
static int layer_routed_impl(int64_t n_rows, int32_t d, int32_t N, int32_t M, int32_t F, int32_t S,
                             int32_t Fs, const float* hidden, const int32_t* idx, const double* w,
                             const wset_t* routed, const wset_t* shared, double* out) {
  if (n_rows < 0 || d <= 0 || N <= 0 || M <= 0 || F <= 0 || S < 0 || (S > 0 && Fs <= 0)) return ORACLE_ERR_ARG;
  if (!hidden || !idx || !w || !routed->gate || !routed->up || !routed->down || !out) return ORACLE_ERR_ARG;
  if (S > 0 && (!shared->gate || !shared->up || !shared->down)) return ORACLE_ERR_ARG;
  const int32_t Fmax = (S > 0 && Fs > F) ? Fs : F;
  int status = ORACLE_OK;
#pragma omp parallel
  {
    double* x = (double*)malloc(sizeof(double) * (size_t)d);
    double* h = (double*)malloc(sizeof(double) * (size_t)Fmax);
    double* y = (double*)malloc(sizeof(double) * (size_t)M * (size_t)d);
    double* wk = (double*)malloc(sizeof(double) * (size_t)M);
    double* sh = (double*)malloc(sizeof(double) * (size_t)d);
    double* ys = (double*)malloc(sizeof(double) * (size_t)d);
    if (!x || !h || !y || !wk || !sh || !ys) {
#pragma omp atomic write
      status = ORACLE_ERR_ARG;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (int64_t t = 0; t < n_rows; ++t) {
        for (int32_t j = 0; j < d; ++j) x[j] = (double)hidden[t * d + j];
        int bad = 0;
        for (int32_t k = 0; k < M; ++k) {
          const int32_t e = idx[t * M + k];
          wk[k] = 0.0;
          for (int32_t i = 0; i < d; ++i) y[(int64_t)k * d + i] = 0.0;
          if (e < 0) continue;
          wmat_t wg, wu, wd;
          if (e >= N || !wset_expert(routed, e, &wg, &wu, &wd)) {
            bad = 1;
            break;
          }
          expert_ffn_w(d, F, x, wg, wu, wd, h, y + (int64_t)k * d);
          wk[k] = w[t * M + k];
        }
        for (int32_t i = 0; i < d; ++i) sh[i] = 0.0;
        for (int32_t s = 0; s < S && !bad; ++s) {
          wmat_t wg, wu, wd;
          if (!wset_expert(shared, s, &wg, &wu, &wd)) {
            bad = 1;
            break;
          }
          expert_ffn_w(d, Fs, x, wg, wu, wd, h, ys);
          for (int32_t i = 0; i < d; ++i) sh[i] += ys[i];
        }
        if (bad) {
#pragma omp atomic write
          status = ORACLE_ERR_MISSING_EXPERT;
          continue;
        }
        moe_oracle_combine(M, d, wk, y, S > 0 ? sh : NULL, out + t * d);
      }
    }
    free(x); free(h); free(y); free(wk); free(sh); free(ys);
  }
  return status;
}

int moe_oracle_layer_routed(int64_t n_rows, int32_t d, int32_t N, int32_t M, int32_t F, int32_t S,
                            int32_t Fs, const float* hidden, const int32_t* idx, const double* w,
                            const uint16_t* const* w_gate, const uint16_t* const* w_up,
                            const uint16_t* const* w_down, const uint16_t* const* ws_gate,
                            const uint16_t* const* ws_up, const uint16_t* const* ws_down, double* out) {
  const wset_t routed = {0, (const void* const*)w_gate, (const void* const*)w_up,
                         (const void* const*)w_down, NULL, NULL, NULL};
  const wset_t shared = {0, (const void* const*)ws_gate, (const void* const*)ws_up,
                         (const void* const*)ws_down, NULL, NULL, NULL};
  return layer_routed_impl(n_rows, d, N, M, F, S, Fs, hidden, idx, w, &routed, &shared, out);
}

/* moe_oracle_layer_routed with FP8 E4M3 experts: codes and per-row scales as
 * moe_oracle_layer_fp8. */
int moe_oracle_layer_routed_fp8(int64_t n_rows, int32_t d, int32_t N, int32_t M, int32_t F, int32_t S,
                                int32_t Fs, const float* hidden, const int32_t* idx, const double* w,
                                const uint8_t* const* q_gate, const uint8_t* const* q_up,
                                const uint8_t* const* q_down, const float* const* s_gate,
                                const float* const* s_up, const float* const* s_down,
                                const uint8_t* const* qs_gate, const uint8_t* const* qs_up,
                                const uint8_t* const* qs_down, const float* const* ss_gate,
                                const float* const* ss_up, const float* const* ss_down, double* out) {
  if (!s_gate || !s_up || !s_down) return ORACLE_ERR_ARG;
  if (S > 0 && (!ss_gate || !ss_up || !ss_down)) return ORACLE_ERR_ARG;
  const wset_t routed = {1, (const void* const*)q_gate, (const void* const*)q_up,
                         (const void* const*)q_down, (const void* const*)s_gate, (const void* const*)s_up,
                         (const void* const*)s_down};
  const wset_t shared = {1, (const void* const*)qs_gate, (const void* const*)qs_up,
                         (const void* const*)qs_down, (const void* const*)ss_gate, (const void* const*)ss_up,
                         (const void* const*)ss_down};
  return layer_routed_impl(n_rows, d, N, M, F, S, Fs, hidden, idx, w, &routed, &shared, out);
}

/* moe_oracle_layer_routed with MXFP4 experts: packed E2M1 codes and E8M0
 * block scales as moe_oracle_layer_mxfp4. */
int moe_oracle_layer_routed_mxfp4(int64_t n_rows, int32_t d, int32_t N, int32_t M, int32_t F, int32_t S,
                                  int32_t Fs, const float* hidden, const int32_t* idx, const double* w,
                                  const uint8_t* const* q_gate, const uint8_t* const* q_up,
                                  const uint8_t* const* q_down, const uint8_t* const* b_gate,
                                  const uint8_t* const* b_up, const uint8_t* const* b_down,
                                  const uint8_t* const* qs_gate, const uint8_t* const* qs_up,
                                  const uint8_t* const* qs_down, const uint8_t* const* bs_gate,
                                  const uint8_t* const* bs_up, const uint8_t* const* bs_down, double* out) {
  if (!b_gate || !b_up || !b_down) return ORACLE_ERR_ARG;
  if (S > 0 && (!bs_gate || !bs_up || !bs_down)) return ORACLE_ERR_ARG;
  if ((d % 32) != 0 || (F % 32) != 0 || (S > 0 && (Fs % 32) != 0)) return ORACLE_ERR_ARG;
  const wset_t routed = {2, (const void* const*)q_gate, (const void* const*)q_up,
                         (const void* const*)q_down, (const void* const*)b_gate, (const void* const*)b_up,
                         (const void* const*)b_down};
  const wset_t shared = {2, (const void* const*)qs_gate, (const void* const*)qs_up,
                         (const void* const*)qs_down, (const void* const*)bs_gate, (const void* const*)bs_up,
                         (const void* const*)bs_down};
  return layer_routed_impl(n_rows, d, N, M, F, S, Fs, hidden, idx, w, &routed, &shared, out);
}

/*
 * The whole layer for `n_rows` tokens whose hidden rows are given (fp32
 * [n_rows][d]): router, top-K, every chosen expert's FFN, the always-on shared
 * experts ("Mixture of Experts for LLM Inference", "Shared experts": they run
 * for every token and never go through the router; added with weight 1), and
 * the weighted combine.
 *
 * Expert weights are passed as one pointer per expert (each expert is its own
 * allocation, as "Mixture of Experts Explained", "Three honest caveats" notes);
 * a NULL pointer means "not provided" and is an error only if a token picks it.
 *   w_gate[e], w_up[e]: bf16 [F][d];  w_down[e]: bf16 [d][F]
 *   ws_gate[s], ws_up[s]: bf16 [Fs][d]; ws_down[s]: bf16 [d][Fs]
 * keep: uint8 [n][K] or NULL; keep[t][k] == 0 marks a copy dropped by its
 * expert's capacity: it contributes nothing (topk_w still reports the router's
 * weight; the kept weights are not renormalised).
 * Outputs: topk_idx [n][K], topk_w fp64 [n][K], margin fp64 [n], out fp64 [n][d].
 */
static int layer_impl(int64_t n_rows, int32_t d, int32_t N, int32_t K, int32_t F,
                      int32_t S, int32_t Fs, int32_t score_fn, int32_t renormalize,
                      int32_t n_groups, int32_t topk_groups,
                      const float* hidden, const float* w_router, const float* router_bias,
                      const float* sel_bias, const wset_t* routed, const wset_t* shared,
                      const unsigned char* keep,
                      int32_t* topk_idx, double* topk_w, double* margin, double* out) {
  if (!router_args_ok(n_rows, d, N, K, score_fn, n_groups, topk_groups, hidden, w_router))
    return ORACLE_ERR_ARG;
  if (F <= 0 || S < 0 || (S > 0 && Fs <= 0)) return ORACLE_ERR_ARG;
  if (!routed->gate || !routed->up || !routed->down || !topk_idx || !topk_w || !margin || !out)
    return ORACLE_ERR_ARG;
  if (S > 0 && (!shared->gate || !shared->up || !shared->down)) return ORACLE_ERR_ARG;
  int status = ORACLE_OK;
  const int32_t Fmax = (S > 0 && Fs > F) ? Fs : F;
#pragma omp parallel
  {
    float* l32 = (float*)malloc(sizeof(float) * (size_t)N);
    double* prob = (double*)malloc(sizeof(double) * (size_t)N);
    float* key = (float*)malloc(sizeof(float) * (size_t)N);
    unsigned char* taken = (unsigned char*)malloc((size_t)N);
    int32_t* order = (int32_t*)malloc(sizeof(int32_t) * (size_t)N);
    double* x = (double*)malloc(sizeof(double) * (size_t)d);
    double* h = (double*)malloc(sizeof(double) * (size_t)Fmax);
    double* y = (double*)malloc(sizeof(double) * (size_t)K * (size_t)d);
    double* sh = (double*)malloc(sizeof(double) * (size_t)d);
    double* ys = (double*)malloc(sizeof(double) * (size_t)d);
    double* wk = (double*)malloc(sizeof(double) * (size_t)K);
    if (!l32 || !prob || !key || !taken || !order || !x || !h || !y || !sh || !ys || !wk) {
#pragma omp atomic write
      status = ORACLE_ERR_ARG;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (int64_t t = 0; t < n_rows; ++t) {
        const float* xr = hidden + t * d;
        int32_t* idx = topk_idx + t * K;
        double* w = topk_w + t * K;
        router_one_token(d, N, K, score_fn, renormalize, n_groups, topk_groups, xr, w_router, router_bias,
                         sel_bias, NULL, NULL, NULL, idx, w, margin + t, l32, prob, key,
                         taken, order);
        for (int32_t j = 0; j < d; ++j) x[j] = (double)xr[j];
        int missing = 0;
        for (int32_t k = 0; k < K; ++k) {
          wmat_t wg, wu, wd;
          if (!wset_expert(routed, idx[k], &wg, &wu, &wd)) { missing = 1; break; }
          expert_ffn_w(d, F, x, wg, wu, wd, h, y + (int64_t)k * d);
        }
        if (missing) {
#pragma omp atomic write
          status = ORACLE_ERR_MISSING_EXPERT;
          continue;
        }
        for (int32_t i = 0; i < d; ++i) sh[i] = 0.0;
        for (int32_t s = 0; s < S && !missing; ++s) {
          wmat_t wg, wu, wd;
          if (!wset_expert(shared, s, &wg, &wu, &wd)) { missing = 1; break; }
          expert_ffn_w(d, Fs, x, wg, wu, wd, h, ys);
          for (int32_t i = 0; i < d; ++i) sh[i] += ys[i];
        }
        if (missing) {
#pragma omp atomic write
          status = ORACLE_ERR_MISSING_EXPERT;
          continue;
        }
        /* a copy dropped by its expert's capacity contributes nothing */
        for (int32_t k = 0; k < K; ++k) wk[k] = (keep && !keep[t * K + k]) ? 0.0 : w[k];
        moe_oracle_combine(K, d, wk, y, S > 0 ? sh : NULL, out + t * d);
      }
    }
    free(l32); free(prob); free(key); free(taken); free(order);
    free(x); free(h); free(y); free(sh); free(ys); free(wk);
  }
  return status;
}

int moe_oracle_layer(int64_t n_rows, int32_t d, int32_t N, int32_t K, int32_t F,
                     int32_t S, int32_t Fs, int32_t score_fn, int32_t renormalize,
                     int32_t n_groups, int32_t topk_groups,
                     const float* hidden, const float* w_router, const float* router_bias,
                     const float* sel_bias, const uint16_t* const* w_gate,
                     const uint16_t* const* w_up, const uint16_t* const* w_down,
                     const uint16_t* const* ws_gate, const uint16_t* const* ws_up,
                     const uint16_t* const* ws_down, const unsigned char* keep,
                     int32_t* topk_idx, double* topk_w, double* margin, double* out) {
  const wset_t routed = {0, (const void* const*)w_gate, (const void* const*)w_up,
                         (const void* const*)w_down, NULL, NULL, NULL};
  const wset_t shared = {0, (const void* const*)ws_gate, (const void* const*)ws_up,
                         (const void* const*)ws_down, NULL, NULL, NULL};
  return layer_impl(n_rows, d, N, K, F, S, Fs, score_fn, renormalize, n_groups, topk_groups, hidden,
                    w_router, router_bias, sel_bias, &routed, &shared, keep, topk_idx, topk_w, margin,
                    out);
}

/*
 * The same layer with every expert matrix (routed and shared) stored as FP8
 * E4M3 codes with one fp32 scale per matrix row, as moe_oracle_expert_ffn_fp8:
 *   q_gate[e], q_up[e]: uint8 [F][d] with s_gate[e], s_up[e]: fp32 [F]
 *   q_down[e]: uint8 [d][F] with s_down[e]: fp32 [d]
 *   qs_* / ss_*: the same for the S shared experts (Fs in place of F).
 * The router stays in full precision ("AI Infrastructure series, Part 12 of
 * 24", "How do you serve an MoE model on your own GPUs?": only the experts'
 * weights go to low precision).
 */
int moe_oracle_layer_fp8(int64_t n_rows, int32_t d, int32_t N, int32_t K, int32_t F,
                         int32_t S, int32_t Fs, int32_t score_fn, int32_t renormalize,
                         int32_t n_groups, int32_t topk_groups,
                         const float* hidden, const float* w_router, const float* router_bias,
                         const float* sel_bias, const uint8_t* const* q_gate,
                         const uint8_t* const* q_up, const uint8_t* const* q_down,
                         const float* const* s_gate, const float* const* s_up,
                         const float* const* s_down, const uint8_t* const* qs_gate,
                         const uint8_t* const* qs_up, const uint8_t* const* qs_down,
                         const float* const* ss_gate, const float* const* ss_up,
                         const float* const* ss_down, const unsigned char* keep,
                         int32_t* topk_idx, double* topk_w, double* margin, double* out) {
  if (!s_gate || !s_up || !s_down) return ORACLE_ERR_ARG;
  if (S > 0 && (!ss_gate || !ss_up || !ss_down)) return ORACLE_ERR_ARG;
  const wset_t routed = {1, (const void* const*)q_gate, (const void* const*)q_up,
                         (const void* const*)q_down, (const void* const*)s_gate, (const void* const*)s_up,
                         (const void* const*)s_down};
  const wset_t shared = {1, (const void* const*)qs_gate, (const void* const*)qs_up,
                         (const void* const*)qs_down, (const void* const*)ss_gate, (const void* const*)ss_up,
                         (const void* const*)ss_down};
  return layer_impl(n_rows, d, N, K, F, S, Fs, score_fn, renormalize, n_groups, topk_groups, hidden,
                    w_router, router_bias, sel_bias, &routed, &shared, keep, topk_idx, topk_w, margin,
                    out);
}

/*
 * The layer with every expert matrix (routed and shared) in MXFP4, as
 * moe_oracle_expert_ffn_mxfp4: codes q_* [rows][K/2] and E8M0 block scales
 * b_* [rows][K/32] per expert (shared: qs_*, bs_*). The router stays fp32.
 */
int moe_oracle_layer_mxfp4(int64_t n_rows, int32_t d, int32_t N, int32_t K, int32_t F,
                           int32_t S, int32_t Fs, int32_t score_fn, int32_t renormalize,
                           int32_t n_groups, int32_t topk_groups,
                           const float* hidden, const float* w_router, const float* router_bias,
                           const float* sel_bias, const uint8_t* const* q_gate,
                           const uint8_t* const* q_up, const uint8_t* const* q_down,
                           const uint8_t* const* b_gate, const uint8_t* const* b_up,
                           const uint8_t* const* b_down, const uint8_t* const* qs_gate,
                           const uint8_t* const* qs_up, const uint8_t* const* qs_down,
                           const uint8_t* const* bs_gate, const uint8_t* const* bs_up,
                           const uint8_t* const* bs_down, const unsigned char* keep,
                           int32_t* topk_idx, double* topk_w, double* margin, double* out) {
  if (!b_gate || !b_up || !b_down) return ORACLE_ERR_ARG;
  if (S > 0 && (!bs_gate || !bs_up || !bs_down)) return ORACLE_ERR_ARG;
  if ((d % 32) != 0 || (F % 32) != 0 || (S > 0 && (Fs % 32) != 0)) return ORACLE_ERR_ARG;
  const wset_t routed = {2, (const void* const*)q_gate, (const void* const*)q_up,
                         (const void* const*)q_down, (const void* const*)b_gate, (const void* const*)b_up,
                         (const void* const*)b_down};
  const wset_t shared = {2, (const void* const*)qs_gate, (const void* const*)qs_up,
                         (const void* const*)qs_down, (const void* const*)bs_gate, (const void* const*)bs_up,
                         (const void* const*)bs_down};
  return layer_impl(n_rows, d, N, K, F, S, Fs, score_fn, renormalize, n_groups, topk_groups, hidden,
                    w_router, router_bias, sel_bias, &routed, &shared, keep, topk_idx, topk_w, margin,
                    out);
}
