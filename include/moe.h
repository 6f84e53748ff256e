/*
 * moe.h — C ABI of a B300-native (sm_103a) forward pass of one token-choice
 * Mixture-of-Experts FFN layer.
 *
 * The layer, as the source pages state it:
 *   - "Mixture of Experts for LLM Inference", section "Opening the router":
 *     a small linear layer gives one raw score per expert, a softmax turns the
 *     scores into shares, top-K keeps the K largest and renormalises them, and
 *     those K weights blend the chosen experts' outputs. Some models (DeepSeek-V3)
 *     use a sigmoid affinity plus normalisation over the chosen K instead.
 *   - "Chapter 19: Mixture-of-Experts Models", §19.3.2 "A concrete router
 *     computation": logits = hidden_state @ W_router; softmax over the top-K
 *     logits equals full softmax + renormalisation over the chosen K.
 *   - same chapter, §19.3.4: a per-expert bias shifts the scores used for
 *     top-K selection only; the mixing weights come from the unbiased scores.
 *   - "Mixture of Experts for LLM Inference", "Shared experts: stop relearning
 *     the basics": a shared expert runs on every token, outside the router.
 *   - "Chapter 19", §19.6.3 "How expert parallelism dispatches tokens" ("Route
 *     and pack"): token copies are grouped by expert before the expert FFNs run
 *     and returned to token order for the weighted aggregation.
 *   - Each expert is an FFN with three matrices ("Mixture of Experts Explained:
 *     Conditional Computation From Zero", "The slot it replaces, and what an
 *     expert is"); this library reads it as SwiGLU:
 *       E(x) = W_down (SiLU(W_gate x) * (W_up x)),  SiLU(z) = z * sigmoid(z).
 *
 * Conventions for every entry point:
 *   - Every pointer argument is a DEVICE pointer owned by the caller, unless
 *     stated otherwise. The library allocates no device memory and keeps no
 *     per-call global state; scratch lives in a caller-provided workspace.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     All work is enqueued asynchronously on it; no entry point synchronises
 *     except moe_get_device_status.
 *   - Arguments are validated on the host before anything is enqueued; an
 *     invalid call returns an error status and enqueues nothing.
 *   - A workspace's first 256 bytes hold the device error word: zero them
 *     once before the workspace's first use (moe_get_device_status clears the
 *     word after reading it).
 *   - Launch failures return MOE_ERR_CUDA. Faults the kernels detect on the
 *     device (an expert index out of range, a pipeline wait that ran out of
 *     time) are recorded in an error word inside the workspace and reported by
 *     moe_get_device_status; kernels never trap.
 *   - Row-major layouts throughout. bf16 is IEEE bfloat16 stored as uint16;
 *     fp16 is IEEE binary16; FP8 E4M3 is the OCP 8-bit float with 4 exponent
 *     bits (bias 7), 3 mantissa bits and no infinities, stored as uint8.
 *   - Layer outputs exclude the residual stream (the residual path lies
 *     outside the FFN slot the layer replaces).
 */
#ifndef MOE_B300_H
#define MOE_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = -1,   /* a null required pointer, a bad size or flag */
  MOE_ERR_UNSUPPORTED = -2,   /* a valid problem this build does not handle */
  MOE_ERR_WORKSPACE = -3,     /* ws is NULL, misaligned or smaller than needed */
  MOE_ERR_CUDA = -4,          /* a CUDA runtime call or a launch failed */
  MOE_ERR_TIMEOUT = -5,       /* device: a bounded pipeline wait gave up */
  MOE_ERR_DEVICE_BOUNDS = -6, /* device: an input index was out of range */
  MOE_ERR_RANGE = -7          /* device: an fp16 activation of the FP8-weight
                                 path overflowed (|value| >= 65520) */
} moe_status_t;

typedef enum { MOE_SCORE_SOFTMAX = 0, MOE_SCORE_SIGMOID = 1 } moe_score_fn_t;
typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype_t;
typedef enum { MOE_ROUTING_TOKEN_CHOICE = 0, MOE_ROUTING_EXPERT_CHOICE = 1 } moe_routing_t;

/*
 * Storage format of the expert matrices (routed and shared alike; the router
 * is always fp32). Storing only the experts in low precision is the serving
 * recipe of "AI Infrastructure series, Part 12 of 24", "How do you serve an
 * MoE model on your own GPUs?"; it cuts the bytes a token reads by the same
 * factor ("Mixture of Experts Explained", "Total versus active parameters").
 *   MOE_EXPERT_BF16      bf16 matrices
 *   MOE_EXPERT_FP8_E4M3  FP8 E4M3 codes with one fp32 scale per matrix row:
 *                        weight = e4m3(code) * scale[row]. NaN codes
 *                        (0x7F, 0xFF) are not supported. The activations
 *                        between the calls (x_perm, h_perm) are then fp16
 *                        rows instead of bf16 (exact for bf16 values of
 *                        magnitude 2^-14 .. 65504, within 2^-25 below that;
 *                        an overflow beyond it is reported as MOE_ERR_RANGE).
 *                        Inside the expert GEMMs the tensor cores multiply
 *                        the E4M3 codes by a two-term E4M3 expansion of each
 *                        activation row, x ~= s_row * (hi + lo), whose
 *                        relative error is at most 2^-8 (that of a bf16
 *                        activation), with fp32 accumulation.
 *   MOE_EXPERT_MXFP4     OCP microscaling FP4 (the format gpt-oss ships its
 *                        experts in): E2M1 codes packed two per byte (the
 *                        even element of a row in the low nibble) and one
 *                        E8M0 scale per 32 consecutive elements of a row:
 *                        weight = e2m1(code) * 2^(scale - 127). Activations
 *                        as for FP8. Inside the GEMMs each 32-element block
 *                        becomes E4M3 codes relative to its row's reference
 *                        exponent (the row's largest block exponent - 6):
 *                        exact for blocks within 14 binades of the row's
 *                        largest, rounded to nearest below that.
 */
typedef enum { MOE_EXPERT_BF16 = 0, MOE_EXPERT_FP8_E4M3 = 1, MOE_EXPERT_MXFP4 = 2 } moe_expert_dtype_t;

/* Which call a workspace is sized for (moe_workspace_bytes). */
typedef enum {
  MOE_CALL_PERMUTE = 0,
  MOE_CALL_GROUPED_SWIGLU = 1,
  MOE_CALL_LAYER_FORWARD = 2,
  MOE_CALL_ROUTER = 3
} moe_call_t;

/*
 * The problem statement, in the pages' terms: T tokens, d_model, N routed
 * experts, K chosen per token, the FFN width of a routed expert, the number of
 * always-on shared experts and their width, and the score function.
 */
typedef struct moe_problem {
  int64_t T;             /* tokens in this call, >= 0 (T == 0 is a no-op)      */
  int32_t d_model;       /* hidden size d, > 0, multiple of 8                  */
  int32_t n_experts;     /* N routed experts, 1..256                           */
  int32_t top_k;         /* K experts per token, 1..min(N, 32)                 */
  int32_t ffn;           /* F, routed expert FFN width, > 0, multiple of 8     */
  int32_t n_shared;      /* S always-on shared experts, >= 0                   */
  int32_t shared_ffn;    /* Fs, shared expert width (multiple of 8 if S > 0)   */
  int32_t score_fn;      /* moe_score_fn_t                                     */
  int32_t renormalize;   /* 1: chosen weights renormalised to sum to 1;
                            0: softmax -> the full-softmax probability of each
                               chosen expert, sigmoid -> its raw sigmoid score */
  int32_t hidden_dtype;  /* moe_dtype_t of `hidden`                           */
  int32_t n_groups;      /* group-limited routing: experts form n_groups equal
                            groups of consecutive indices (0 or 1: off)      */
  int32_t topk_groups;   /* groups a token may pick from (1..n_groups); a
                            group's score is the sum of its two largest
                            selection keys ("Mixture of Experts for LLM
                            Inference", "Three tricks that tame the
                            all-to-alls": node-limited routing)              */
  double capacity_factor; /* expert capacity C = ceil(c * T * K / N) for c > 0
                            ("Chapter 19", §19.6.1); copies beyond the first
                            C of an expert (token order) are dropped: they
                            skip the FFN and contribute nothing, the kept
                            weights are not renormalised; C is computed in
                            double precision. 0: dropless                  */
  int32_t routing;       /* moe_routing_t: token choice (every token picks K
                            experts) or expert choice (every expert picks
                            C = min(ceil(c T K / N), T) tokens, c =
                            capacity_factor or 1 when 0; K is then the mean
                            number of experts per token)                    */
  int32_t expert_dtype;  /* moe_expert_dtype_t of every expert matrix. FP8
                            requires d_model, ffn and shared_ffn to be
                            multiples of 16, MXFP4 multiples of 32 (and at
                            most 32768, else MOE_ERR_UNSUPPORTED)          */
} moe_problem_t;

/*
 * Weights of one layer. Routed experts are stacked: w_gate/w_up are
 * bf16 [N][F][d] (row f of expert e holds the d inputs of unit f, i.e. the
 * operand is K-major), w_down is bf16 [N][d][F]. Shared experts likewise:
 * ws_gate/ws_up bf16 [S][Fs][d], ws_down bf16 [S][d][Fs]; NULL when S == 0.
 * The router is fp32 (kept in higher precision than the experts, per
 * "Chapter 19", §19.6.2 table, "Higher-precision router"):
 *   w_router     fp32 [d][N]   logits = hidden @ w_router (+ router_bias)
 *   router_bias  fp32 [N] or NULL: the bias term of the router's linear layer,
 *                added to every logit
 *   sel_bias     fp32 [N] or NULL: selection-only bias, added to the sigmoid
 *                score before top-K, never to the mixing weights (sigmoid
 *                scoring only)
 * With expert_dtype == MOE_EXPERT_FP8_E4M3 the expert matrices hold uint8
 * codes in the same layouts, and the *_scale arrays hold one fp32 scale per
 * matrix row (16-byte aligned):
 *   w_gate_scale, w_up_scale [N][F]; w_down_scale [N][d];
 *   ws_gate_scale, ws_up_scale [S][Fs]; ws_down_scale [S][d] (NULL when S == 0).
 * With expert_dtype == MOE_EXPERT_MXFP4 the expert matrices hold packed E2M1
 * codes, half the bytes of each row (w_gate, w_up [N][F][d/2], w_down
 * [N][d][F/2]; shared likewise), and the *_scale arrays hold the E8M0 block
 * scales as uint8: w_gate_scale, w_up_scale [N][F][d/32], w_down_scale
 * [N][d][F/32]; ws_* [S][Fs][d/32], [S][Fs][d/32], [S][d][Fs/32].
 * The scale arrays are ignored for bf16 experts.
 * mx_prep (MXFP4 only, else ignored): NULL, or a buffer moe_mxfp4_prepare
 * filled from these same block scales for a problem with the same n_experts,
 * n_shared, d_model, ffn and shared_ffn. With it a call skips the per-call
 * preparation of the experts it uses (three launches, six with shared
 * experts); the results are bit-identical. The caller prepares again after
 * changing the block scales.
 */
typedef struct moe_weights {
  const float* w_router;
  const float* router_bias;
  const float* sel_bias;
  const void* w_gate;
  const void* w_up;
  const void* w_down;
  const void* ws_gate;
  const void* ws_up;
  const void* ws_down;
  const void* w_gate_scale;   /* fp32 row scales (FP8) or uint8 E8M0 block scales (MXFP4) */
  const void* w_up_scale;
  const void* w_down_scale;
  const void* ws_gate_scale;
  const void* ws_up_scale;
  const void* ws_down_scale;
  const void* mx_prep;
} moe_weights_t;

/* Human-readable name of a moe_status_t. Never NULL. Host only. */
const char* moe_status_string(int32_t status);

/*
 * Host-only validation of a problem statement (no CUDA call). Returns MOE_OK,
 * MOE_ERR_INVALID_ARG (p NULL, a size out of range, a bad enum) or
 * MOE_ERR_UNSUPPORTED (a valid statement this build does not handle).
 */
moe_status_t moe_problem_check(const moe_problem_t* p);

/*
 * Bytes of workspace the given call needs for problem p (host only, no CUDA
 * call). Returns 0 if p is invalid. The workspace must be 256-byte aligned.
 */
size_t moe_workspace_bytes(const moe_problem_t* p, int32_t call);

/*
 * Router, scoring, top-K and gate weights, per token ("Mixture of Experts for
 * LLM Inference", "Opening the router"; "Chapter 19", §19.3.2 and §19.3.4;
 * "AI Infrastructure series Part 12", "How does the router decide? A worked
 * example").
 *   hidden      [T][d], p->hidden_dtype
 *   w_router    fp32 [d][N];  router_bias, sel_bias: fp32 [N] or NULL
 *   topk_idx    out int32 [T][K]: chosen experts in descending key order;
 *               equal keys are broken toward the lower expert index
 *   topk_w      out fp32 [T][K]: gate weight of each chosen expert
 *   logits_opt  out fp32 [T][N] or NULL: the router logits (debug)
 *   ws          workspace of moe_workspace_bytes(p, MOE_CALL_ROUTER) bytes
 *               (partial logits when the d axis is split across CTAs)
 * Key used for selection: softmax -> the logit (monotone in the softmax);
 * sigmoid -> sigmoid(logit) + sel_bias. Weights: softmax -> softmax over the
 * chosen logits; sigmoid -> chosen sigmoid scores / their sum.
 * sel_bias with softmax scoring returns MOE_ERR_UNSUPPORTED. Deterministic.
 */
moe_status_t moe_router_topk(const moe_problem_t* p, const void* hidden,
                             const float* w_router, const float* router_bias,
                             const float* sel_bias, int32_t* topk_idx,
                             float* topk_w, float* logits_opt, void* ws,
                             size_t ws_bytes, void* stream);

/*
 * Route and pack ("Chapter 19", §19.6.3): per-expert histogram, exclusive
 * prefix sum and a stable expert-major permutation of the T*K token copies
 * (expert ascending, then token ascending), plus the gather of the hidden rows
 * into that order.
 *   topk_idx   int32 [T][K], every entry in [0, N), the K entries of a token
 *              distinct (as top-K selection gives them)
 *   hidden     [T][d], p->hidden_dtype
 *   counts     out int32 [N]:   counts[e] = #{(t,k) : topk_idx[t][k] == e}
 *   offsets    out int32 [N+1]: offsets[0] = 0, offsets[e+1] = offsets[e] + counts[e]
 *   perm_src   out int32 [T*K]: permuted row r holds token copy perm_src[r] = t*K + k
 *   inv_row    out int32 [T*K]: inv_row[t*K + k] = r (the inverse of perm_src);
 *              -1 for a copy dropped by its expert's capacity (p->capacity_factor
 *              > 0), in which case offsets count kept copies only, perm_src lists
 *              offsets[N] rows and counts still count every copy routed to e
 *   x_perm     out [T*K][d]: x_perm[r] = hidden[perm_src[r] / K] rounded to
 *              bf16, or to fp16 when p->expert_dtype is FP8 (an fp16 overflow
 *              sets MOE_ERR_RANGE in the workspace error word)
 *   ws         workspace of moe_workspace_bytes(p, MOE_CALL_PERMUTE) bytes
 * Token-choice problems only (MOE_ERR_INVALID_ARG otherwise).
 * The result is deterministic. An index outside [0, N) sets
 * MOE_ERR_DEVICE_BOUNDS in the workspace error word; outputs are then undefined.
 */
moe_status_t moe_permute(const moe_problem_t* p, const int32_t* topk_idx,
                         const void* hidden, int32_t* counts, int32_t* offsets,
                         int32_t* perm_src, int32_t* inv_row, void* x_perm,
                         void* ws, size_t ws_bytes, void* stream);

/*
 * Expert-choice routing ("Mixture of Experts for LLM Inference", "Token choice
 * vs expert choice": each expert picks its own top tokens up to a fixed
 * capacity; "Chapter 19", §19.6.1 "Expert Choice"), for problems with
 * p->routing == MOE_ROUTING_EXPERT_CHOICE:
 *   score S[t][e] = softmax over the experts of token t's fp32 logits, or
 *   sigmoid(logit); expert e takes the C tokens with the largest S[.][e]
 *   (equal scores: lower token first), C = min(ceil(c T K / N), T).
 *   row_token out int32 [N][C]: expert e's tokens in ascending order
 *   row_w     out fp32 [N][C]: their scores S[t][e] (not renormalised)
 *   offsets   out int32 [N+1]: e * C (every expert is full by construction)
 *   ws        workspace of moe_workspace_bytes(p, MOE_CALL_ROUTER) bytes
 * A token no expert picks gets no routed contribution. Deterministic.
 * Requires p->score_fn's router inputs as in moe_router_topk; no selection
 * bias, no group limit (MOE_ERR_UNSUPPORTED otherwise).
 */
/*
 * The number of tokens C every expert takes under expert-choice routing:
 * C = min(ceil(c * T * K / N), T), c = p->capacity_factor, or 1 when it is 0
 * ("Chapter 19", §19.6.1, the capacity equation; here applied per expert to
 * tokens instead of to token copies). Sizes row_token / row_w below and the
 * layer's packed rows (N * C). Host only, no CUDA call; p->routing is not
 * read. Returns -1 for an invalid problem.
 */
int64_t moe_expert_choice_capacity(const moe_problem_t* p);

moe_status_t moe_expert_choice_select(const moe_problem_t* p, const void* hidden,
                                      const float* w_router, const float* router_bias,
                                      int32_t* row_token, float* row_w, int32_t* offsets,
                                      void* ws, size_t ws_bytes, void* stream);

/*
 * moe_permute_static: the same route and pack as moe_permute, for callers that
 * cannot allocate device memory. The source pages have no counterpart to this
 * entry point; it exists only for how the library is deployed.
 *
 * Who needs it: a caller that must not call cudaMalloc (or any allocator) on
 * the routing path, e.g. a server that reserves all GPU memory up front and
 * accounts for every byte, a plug-in inside a framework that owns the device
 * allocator, or a latency-critical loop that cannot afford cudaMalloc's cost
 * and implicit device synchronisation. moe_permute needs a workspace for its
 * per-chunk expert counts; here that scratch is a fixed array compiled into
 * the library, so the caller passes only the inputs and outputs below, with
 * the same meaning, layout and results as in moe_permute.
 *
 * Limit: n_experts * ceil(T / 32) <= MOE_PERMUTE_STATIC_MAX_CHUNK_COUNTS
 * (e.g. 256 experts with up to 8192 tokens, 8 experts with up to 262144);
 * larger problems return MOE_ERR_UNSUPPORTED and enqueue nothing. The array
 * (256 KB + 256 bytes) is reserved on every GPU that loads the library, until
 * the process exits. The entry point allocates nothing.
 *
 * The first call on a device looks up the array's device address on that
 * device (cudaGetSymbolAddress); make that first call before any stream
 * capture. The address is cached per device together with the CUDA context
 * it was looked up in, and looked up again when a call comes from another
 * context. After cudaDeviceReset the primary context (and the array) is
 * created anew and may reuse the old context handle: make a first call again
 * before any capture, and do not reuse the array's contents across a reset.
 * For FP8 and MXFP4 experts x_perm holds fp16 rows, as in moe_permute.
 * Every call on a device shares the one array and leaves its contents
 * behind: calls whose work overlaps on the GPU (different streams or host
 * threads without ordering between them) race and give wrong results, so
 * order them. The call clears the array's error word itself. There is no
 * error word to read afterwards: an expert index outside [0, N) is skipped,
 * and shows as offsets[N] < T*K.
 */
#define MOE_PERMUTE_STATIC_MAX_CHUNK_COUNTS 65536
moe_status_t moe_permute_static(const moe_problem_t* p, const int32_t* topk_idx,
                                const void* hidden, int32_t* counts,
                                int32_t* offsets, int32_t* perm_src,
                                int32_t* inv_row, void* x_perm, void* stream);

/*
 * The routed experts' SwiGLU FFNs over the packed rows, as grouped GEMMs on
 * the tensor cores (bf16 operands, fp32 accumulation):
 *   for every expert e and row r in [offsets[e], offsets[e+1]):
 *     h_perm[r] = bf16( SiLU(W_gate[e] x_perm[r]) * (W_up[e] x_perm[r]) )
 *     y_perm[r] = bf16( W_down[e] h_perm[r] )          (not yet weighted)
 *   x_perm  bf16 [T*K][d];  offsets int32 [N+1] as written by moe_permute
 *   w_gate, w_up bf16 [N][F][d];  w_down bf16 [N][d][F]
 *   h_perm  out bf16 [T*K][F];  y_perm out bf16 [T*K][d]
 *   ws      workspace of moe_workspace_bytes(p, MOE_CALL_GROUPED_SWIGLU) bytes
 * p->n_shared is ignored here. A shared expert runs through this same call as
 * one group over every token: n_experts = 1, top_k = 1, offsets = {0, T},
 * x_perm = the hidden rows in bf16, weights = that shared expert's.
 * For an expert-choice problem the packed rows are the N*C picks
 * (moe_expert_choice_select) and offsets are e*C.
 * bf16 experts only (p->expert_dtype == MOE_EXPERT_BF16, else
 * MOE_ERR_INVALID_ARG); FP8 experts use moe_grouped_swiglu_fp8.
 */
moe_status_t moe_grouped_swiglu(const moe_problem_t* p, const void* x_perm,
                                const int32_t* offsets, const void* w_gate,
                                const void* w_up, const void* w_down,
                                void* h_perm, void* y_perm, void* ws,
                                size_t ws_bytes, void* stream);

/*
 * moe_grouped_swiglu for FP8 E4M3 experts (p->expert_dtype ==
 * MOE_EXPERT_FP8_E4M3, else MOE_ERR_INVALID_ARG):
 *   h_perm[r] = fp16( SiLU(g) * u ),  g_f = sg[e][f] * (Q_gate[e] x_perm[r])_f,
 *                                     u_f = su[e][f] * (Q_up[e] x_perm[r])_f
 *   y_perm[r] = bf16( sd[e][i] * (Q_down[e] h_perm[r])_i )
 * with Q the decoded E4M3 codes (exact), fp32 accumulation.
 *   x_perm  fp16 [rows][d] (moe_permute writes fp16 for FP8 problems)
 *   w_gate, w_up uint8 [N][F][d], w_gate_scale, w_up_scale fp32 [N][F]
 *   w_down uint8 [N][d][F], w_down_scale fp32 [N][d]
 *   h_perm  out fp16 [rows][F];  y_perm out bf16 [rows][d]
 *   ws      workspace of moe_workspace_bytes(p, MOE_CALL_GROUPED_SWIGLU) bytes
 * rows, offsets and shared experts as moe_grouped_swiglu (a shared expert is
 * one group over every token with its own codes and scales). An h value
 * beyond fp16's range sets MOE_ERR_RANGE in the workspace error word.
 */
moe_status_t moe_grouped_swiglu_fp8(const moe_problem_t* p, const void* x_perm,
                                    const int32_t* offsets, const void* w_gate,
                                    const float* w_gate_scale, const void* w_up,
                                    const float* w_up_scale, const void* w_down,
                                    const float* w_down_scale, void* h_perm,
                                    void* y_perm, void* ws, size_t ws_bytes,
                                    void* stream);

/*
 * moe_grouped_swiglu_fp8 for MXFP4 experts (p->expert_dtype ==
 * MOE_EXPERT_MXFP4, else MOE_ERR_INVALID_ARG): w_gate, w_up uint8 [N][F][d/2]
 * packed E2M1 codes with E8M0 block scales w_gate_bscale, w_up_bscale uint8
 * [N][F][d/32]; w_down [N][d][F/2] with w_down_bscale [N][d][F/32]. Other
 * arguments, layouts and results as moe_grouped_swiglu_fp8.
 */
moe_status_t moe_grouped_swiglu_mxfp4(const moe_problem_t* p, const void* x_perm,
                                      const int32_t* offsets, const void* w_gate,
                                      const void* w_gate_bscale, const void* w_up,
                                      const void* w_up_bscale, const void* w_down,
                                      const void* w_down_bscale, void* h_perm,
                                      void* y_perm, void* ws, size_t ws_bytes,
                                      void* stream);

/*
 * Gate-weighted combine back to token order ("Chapter 19", §19.2 flowchart,
 * "Sum with gate weights"; "Mixture of Experts for LLM Inference", "The MoE
 * change is surprisingly local"):
 *   out[t] = bf16( sum_k topk_w[t][k] * y_perm[inv_row[t*K + k]]
 *                  + shared_out[t] )
 * with fp32 accumulation in slot order k = 0..K-1 (deterministic); slots with
 * inv_row == -1 (dropped by capacity) are skipped.
 *   y_perm bf16 [T*K][d]; inv_row int32 [T*K]; topk_w fp32 [T][K]
 *   shared_out bf16 [T][d] or NULL;  out bf16 [T][d]
 */
moe_status_t moe_combine(const moe_problem_t* p, const void* y_perm,
                         const int32_t* inv_row, const float* topk_w,
                         const void* shared_out, void* out, void* stream);

/*
 * The whole layer: router + top-K, route and pack, grouped SwiGLU with the
 * SiLU*up product fused into the up-projection epilogue and the gate-weighted
 * scatter-add fused into the down-projection epilogue, the shared experts
 * (weight 1) and the final fp32 -> bf16 rounding.
 *   w            the layer's weights (device pointers inside)
 *   hidden       [T][d], p->hidden_dtype
 *   out          out bf16 [T][d]
 *   topk_idx_opt, topk_w_opt  out int32/fp32 [T][K] or NULL
 *   counts_opt   out int32 [N] or NULL (per-expert token counts)
 *   ws           workspace of moe_workspace_bytes(p, MOE_CALL_LAYER_FORWARD)
 * The fp32 scatter-add makes `out` reproducible only up to the order of
 * floating-point additions (last-bit differences between runs are possible);
 * the step-wise calls above are bit-reproducible.
 * With p->routing == MOE_ROUTING_EXPERT_CHOICE the experts pick their tokens
 * (moe_expert_choice_select) and each picked (token, expert) pair adds
 * S[t][e] * E_e(x_t); topk_idx_opt and topk_w_opt must then be NULL and
 * counts_opt receives C for every expert.
 * With p->expert_dtype == MOE_EXPERT_FP8_E4M3 (or MOE_EXPERT_MXFP4) every
 * expert (routed and shared) reads its codes and scales from `w` and the
 * expert GEMMs run on fp16 activations (see moe_expert_dtype_t).
 * Decode-sized token-choice batches (moe_layer_small_batch) run the whole
 * layer as one kernel instead; its result is reproducible bit for bit.
 */
moe_status_t moe_layer_forward(const moe_problem_t* p, const moe_weights_t* w,
                               const void* hidden, void* out,
                               int32_t* topk_idx_opt, float* topk_w_opt,
                               int32_t* counts_opt, void* ws, size_t ws_bytes,
                               void* stream);

/*
 * moe_layer_forward with stage timing: identical work and kernels, plus a
 * cudaEventRecord on `stream` before the first kernel and after each stage.
 *   stage_events  array of MOE_LAYER_STAGES cudaEvent_t (passed as void*),
 *                 created by the caller; event i+1 minus event i is stage i:
 *                 0 router+top-K, 1 route and pack, 2 GEMM schedule (built
 *                 inside route and pack: an empty stage),
 *                 3 gate/up GEMM + SwiGLU, 4 down GEMM + weighted scatter-add,
 *                 5 fp32 -> bf16 finalise. A decode-sized batch
 *                 (moe_layer_small_batch) is one kernel: stage 0 holds it
 *                 and stages 1 to 5 are empty.
 * Used by the benchmark to time each kernel inside the timed region.
 */
#define MOE_LAYER_STAGES 6
moe_status_t moe_layer_forward_profiled(const moe_problem_t* p, const moe_weights_t* w,
                                        const void* hidden, void* out, void* ws,
                                        size_t ws_bytes, void* const* stage_events,
                                        void* stream);

/*
 * Number of kernels one moe_layer_forward call launches for problem p and
 * weights w (host only, no CUDA call; only w->mx_prep is read, and w may be
 * NULL: no prepared buffer); 0 if p is invalid.
 */
int32_t moe_layer_forward_kernel_count(const moe_problem_t* p, const moe_weights_t* w);

/*
 * 1 if moe_layer_forward runs problem p as one decode-sized kernel, 0 if
 * through the router, route-and-pack and grouped tensor-core GEMM kernels, -1
 * if p is invalid. Host only, no CUDA call. The one-kernel path takes
 * token-choice batches of T <= 4 tokens with bf16 or FP8 E4M3 experts (not
 * MXFP4) whose routing tables and staged rows fit its shared memory.
 * With T tokens an expert holds at most T rows ("Part 12", "What happens when
 * many users share the GPU?": each token reads its own experts' weights, and
 * the bytes, not the arithmetic, set the time at small batch; "Mixture of
 * Experts Explained", "Why batching erodes the advantage"). A 128-row tensor
 * tile would then be almost all padding, and the launches and hand-offs
 * between kernels cost as much as the router. So one cooperative kernel (one
 * CTA per SM) computes the router, top-K, routing, the gate/up rows and SwiGLU,
 * then, after a grid-wide barrier, the down rows and the weighted combine;
 * each touched weight row is streamed from HBM once. Products are exact and
 * sums fp32 on the tensor cores (mma.sync, the token rows padded to 16); h is
 * rounded to bf16, or fp16 for FP8 experts, as on the GEMM path. Same inputs,
 * outputs, workspace and status codes; the output is the same from run to run.
 * The grid barriers use two words at byte 128 of the workspace's first 256
 * bytes (zeroed with the error word; the kernel leaves them at zero).
 */
int32_t moe_layer_small_batch(const moe_problem_t* p);

/*
 * MXFP4 experts: the weight-side preparation the expert GEMMs need, computed
 * from the E8M0 block scales alone ("AI Infrastructure series, Part 12 of
 * 24", on shipping gpt-oss experts as MXFP4). For every weight row R with
 * block exponents E_b: its reference exponent E_R = max_b E_b - 6 (NaN
 * scales 0xFF left out; clamped to 1..254), stored as the fp32 scale
 * 2^(E_R - 127); and for every block its table index clamp(E_b - E_R, -15,
 * 6) + 15, four blocks (128 elements, one K step of the GEMM) per 32-bit
 * word, stored K-step-major so that one K step of 256 rows is one
 * contiguous 1 KB. A call without a prepared buffer computes the same for
 * the experts it uses, into its workspace.
 *
 * moe_mxfp4_prep_bytes: the buffer size for problem p (host only; 0 if p is
 * invalid or not MXFP4). It depends on n_experts, n_shared, d_model, ffn and
 * shared_ffn, not on T.
 *
 * moe_mxfp4_prepare: fills `prep` (device memory, 256-byte aligned,
 * prep_bytes >= moe_mxfp4_prep_bytes(p), owned by the caller) from the block
 * scales in w (w_gate_scale, w_up_scale, w_down_scale and, when n_shared >
 * 0, the ws_*_scale arrays; every expert, used or not); asynchronous on
 * `stream`. Returns MOE_ERR_INVALID_ARG (p not MXFP4, w or a scale array
 * NULL), MOE_ERR_WORKSPACE (prep misaligned or too small) or MOE_ERR_CUDA.
 * Set w->mx_prep = prep for later calls.
 */
size_t moe_mxfp4_prep_bytes(const moe_problem_t* p);
moe_status_t moe_mxfp4_prepare(const moe_problem_t* p, const moe_weights_t* w, void* prep,
                               size_t prep_bytes, void* stream);

/*
 * Synchronises `stream`, then reads and clears the device error word in `ws`
 * (a workspace previously passed to moe_permute, moe_grouped_swiglu or
 * moe_layer_forward). Returns MOE_OK, MOE_ERR_TIMEOUT, MOE_ERR_DEVICE_BOUNDS,
 * MOE_ERR_RANGE (in that order of precedence when several are recorded), or
 * MOE_ERR_CUDA if the stream itself reports an error.
 */
moe_status_t moe_get_device_status(void* ws, void* stream);

/*
 * Failure-detection test hook (no counterpart on the pages): launches one warp
 * that waits on an mbarrier nothing arrives at, through the same bounded wait
 * the GEMM pipeline uses, with a limit of timeout_us microseconds (1..10^6).
 * The wait gives up and records a timeout in the error word of `ws` (any
 * workspace, >= 256 bytes); moe_get_device_status then returns MOE_ERR_TIMEOUT
 * and the CUDA context stays usable.
 */
moe_status_t moe_debug_stall_wait(void* ws, size_t ws_bytes, uint32_t timeout_us, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_B300_H */
