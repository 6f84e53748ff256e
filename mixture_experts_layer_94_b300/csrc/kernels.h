// kernels.h — host-side launch functions of libmoe's kernels (internal).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"
#include "common.cuh"

namespace moe {

struct RouterArgs {
  int64_t T;
  int32_t d, N, K, score_fn, renormalize;
  int32_t n_groups, topk_groups;  // group-limited routing when n_groups > 1
  const void* hidden;  // [T][d] fp32 or bf16
  const float* w_router;
  const float* router_bias;
  const float* sel_bias;
  int32_t* topk_idx;
  float* topk_w;
  float* logits;       // optional [T][N] output
  float* partial;      // scratch [splits][T][N]
  __nv_bfloat16* w3;   // scratch for the tensor-core path: [np][3 * d_pad]
  int32_t splits, d_slice;  // filled by launch_router
  float* scores_t;     // expert choice: write S transposed [N][T] instead of a top-K
};

// Expert choice: every expert picks the C tokens with the largest score from
// scores_t [N][T]; writes row_token / row_w [N][C], offsets [N+1], counts [N].
cudaError_t launch_expert_choice_select(const float* scores_t, int64_t T, int32_t N, int32_t C,
                                        int32_t* row_token, float* row_w, int32_t* offsets, int32_t* counts,
                                        cudaStream_t s);

// How the router computes its logits.
//  tensor == false: CUDA-core kernel, token tiles x `splits` d slices of
//    `d_slice` inputs (np = N rounded to a power of two when N <= 32).
//  tensor == true (bf16 hidden): tcgen05 GEMM of hidden [T, d] with the router
//    matrix split exactly into three bf16 parts (hi + mid + lo = the fp32
//    value), K = 3 parts x `dslices` slices of `kb_per_slice` 64-wide blocks;
//    splits = 3 * dslices partial logits, MMA N = np (multiple of 16).
struct RouterPlan {
  bool tensor;
  bool merged;  // tensor path: the three parts share each tile (np <= kRouterMergedMaxNp)
  int64_t token_tiles;
  int32_t splits;
  int32_t d_slice;
  int32_t np;
  int32_t dslices, kb_per_slice, nkb_d, d_pad;
};
RouterPlan router_plan(int64_t T, int32_t d, int32_t N, bool hidden_bf16);
cudaError_t launch_router(const RouterArgs& a, bool hidden_bf16, cudaStream_t s);

// bf16 row-major matrix [rows][inner] as a TMA tensor map: box [box_rows][64],
// 128-byte swizzle, zero fill out of bounds. False if the driver refuses it.
bool make_tmap_bf16(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t rows, uint32_t box_rows);

struct PermuteArgs {
  int64_t T;
  int32_t d, N, K, C;  // C = number of 32-token chunks
  int32_t capacity;    // copies an expert keeps (token order); INT32_MAX: no cap
  const int32_t* row_token;  // gather only: the token of each packed row (expert choice)
  const int32_t* topk_idx;
  const void* hidden;
  bool hidden_bf16;
  int32_t* chunk_counts;  // [N][C] scratch; holds per-chunk bases after the scan
  int32_t* counts;        // [N]
  int32_t* offsets;       // [N+1]
  int32_t* perm_src;      // [T*K]
  int32_t* inv_row;       // [T*K]
  void* x_perm;           // [T*K][d] in the activation format (bf16, or fp16 when act_f16)
  float* zero_rows;       // [T][d] fp32 to clear, or nullptr
  void* x_act;            // [T][d] copy of hidden in the activation format, or nullptr
  bool act_f16;           // activations for FP8-weight experts: fp16 rows
  // FP8 / MXFP4 experts in the fused layer: when xq is set the gather writes
  // the two-term E4M3 split of each packed row (xq [2 rows][d], sx [rows])
  // instead of x_perm, and of every token's row for the shared experts
  // (xq_sh [2T][d], sx_sh [T]) when xq_sh is set; see launch_gather_quant.
  uint8_t* xq;
  float* sx;
  uint8_t* xq_sh;
  float* sx_sh;
  uint32_t* err;
  // Optional: also build the GEMM schedule (as launch_schedule) from the new
  // offsets; skipped when groups == nullptr.
  GroupDesc* groups;
  int32_t* ts_gu;
  int32_t* ts_dn;
  int32_t S, F, Fs, tile_rows;
};
cudaError_t launch_permute(const PermuteArgs& a, cudaStream_t s);
// Only the row gather (+ the accumulator clear / activation copy), for rows already
// placed: token of row r = row_token[r], rows = offsets[N].
cudaError_t launch_gather(const PermuteArgs& a, int64_t rows, cudaStream_t s);
// Token choice with at least this many packed rows copies (and splits) each
// hidden row once, token-major, into its K packed rows instead of gathering
// each packed row from hidden.
constexpr int64_t kTokenMajorMinRows = 8192;
// Expert capacity ceil(c * T * K / N) of a problem; INT32_MAX when dropless.
int32_t expert_capacity(const moe_problem_t& p);

struct ScheduleArgs {
  int32_t N, S, F, Fs, d;
  int32_t tile_rows;       // rows per GEMM tile: 128, or 256 for CTA pairs
  int64_t T;
  const int32_t* offsets;  // [N+1]
  GroupDesc* groups;       // [N+S]
  int32_t* tile_start_gu;  // [N+S+1]
  int32_t* tile_start_dn;  // [N+S+1]
};
cudaError_t launch_schedule(const ScheduleArgs& a, cudaStream_t s);

enum GemmPhase { kPhaseGateUp = 0, kPhaseDown = 1, kPhaseRouter = 2 };
enum GemmEpilogue { kEpiSwiGLU = 0, kEpiScatter = 1, kEpiStoreY = 2, kEpiLogits = 3 };

struct GemmArgs {
  const GroupDesc* groups;
  const int32_t* tile_start;  // [G+1]
  int32_t phase_dn;           // 1 for the down GEMM (always m fastest), 0 for gate/up (the groups' order_gu)
  int32_t G;
  int32_t n_ext[2];      // output columns of a group, per kind (gate/up: F, Fs; down: d)
  int32_t n_tiles[2];    // output column tiles of a group, per kind
  int32_t k_blocks[2];   // kBK-wide K blocks, per kind
  int32_t w_rows[2];     // rows one group occupies in its stacked weight matrix, per kind
  __nv_bfloat16* h[2];   // SwiGLU epilogue output, per kind
  int64_t ldh[2];
  float* out_acc;        // scatter epilogue: fp32 [T][d]
  const int32_t* perm_src;
  const float* topk_w;
  int32_t top_k;
  __nv_bfloat16* y;      // store epilogue: bf16 [rows][d] (routed groups)
  __nv_bfloat16* y_sh;   // store epilogue, shared groups: bf16 [S*T][d] (nullptr: y)
  const float* row_w;    // scatter epilogue, expert choice: perm_src is the row's token, row_w its weight
  int32_t d;
  uint32_t* err;
  // FP8 / MXFP4 expert weights: fp32 scale of each weight row, per kind
  // (gate/up phase: w_scale = gate rows, u_scale = up rows; down phase:
  // w_scale = rows of W_down). MXFP4: the row's reference scale 2^(E_row - 127).
  const float* w_scale[2];
  const float* u_scale[2];
  // FP8 / MXFP4 experts: the scale of each activation row, per kind (the
  // token rows of the gate/up phase, the h rows of the down phase).
  const float* a_scale[2];
  // Router phase: one group of all T tokens; tile = (m block, split) with
  // split = part * r_dslices + slice, or, when r_merged, split = slice and
  // the tile adds all three parts into one accumulator.
  int32_t r_tiles, r_m_tiles, r_dslices, r_kb_per_slice, r_nkb_d, r_d_pad, r_np, r_N;
  int32_t r_merged;
  uint32_t r_idesc;
  int64_t r_T;
  float* r_partial;       // [splits][T][N]: 3 * r_dslices, or r_dslices when merged
};

struct GemmMaps {
  CUtensorMap a[2];   // activations per kind
  CUtensorMap b[2];   // weights per kind (gate for the gate/up phase)
  CUtensorMap bu[2];  // up weights per kind (gate/up phase only)
  CUtensorMap bh[2];  // gate/up phase on pairs: gate weights in 64-row boxes (half tiles)
  CUtensorMap uh[2];  // ... and up weights
};

// Tensor maps of the FP8-weight grouped GEMM: activations (two-term E4M3
// rows, see act_quant.cu) per kind with boxes of 16, 32, 64 and 128 rows (a
// tile loads the smallest box that holds its 2 x tokens rows); weight codes
// per kind with 128-row boxes: w = gate (gate/up phase) or down rows, u = up.
// All boxes are 128 bytes of K wide, 128-byte swizzled.
constexpr int kF8XBoxes = 4;     // box rows 16 << i
constexpr int kF8TileRows = 64;  // tokens per tile of the FP8-weight GEMM
struct F8Maps {
  CUtensorMap x[2][kF8XBoxes];
  CUtensorMap w[2];
  CUtensorMap u[2];
  CUtensorMap kw[2];  // MXFP4: block-table indices of the w / u rows (see launch_mx_prep)
  CUtensorMap ku[2];
};

// An activation matrix for the FP8-weight GEMMs: src fp16 [rows][K] ->
// dst uint8 [2*rows][K] (row 2r = hi, 2r+1 = lo E4M3 terms) and scale fp32
// [rows], with src[r] ~= scale[r] * (hi + lo). K % 8 == 0.
// The row gather of the fused layer with the activation split folded in:
// packed row r's token row of hidden, rounded to fp16 as the gather stores it,
// split into xq / sx; then `shared_rows` token rows in order into xq_sh /
// sx_sh. Also clears zero_rows and reports an fp16 overflow, as the gather.
cudaError_t launch_gather_quant(const PermuteArgs& a, int64_t rows, int64_t shared_rows, cudaStream_t s);
cudaError_t launch_act_quant(const void* src, int64_t rows, int32_t K, uint8_t* dst, float* scale,
                             cudaStream_t s);
// ---------------------------------------------------------------- decode-sized batches in one kernel
// decode_layer.cu: router, top-K, routing, gate/up + SwiGLU, down and the
// weighted combine of a token-choice batch of at most kDecodeMaxTokens tokens
// in one cooperative launch of one 512-thread CTA per SM.
// Storage format of the expert matrices on this path.
enum DecodeFormat { kDecodeBf16 = 0, kDecodeE4M3 = 1 };
constexpr int kDecodeThreads = 512;
constexpr int kDecodeMaxTokens = 4;
constexpr int kDecodeMaxSplits = 128;     // router partials (slices of d)
constexpr int kDecodeMaxGrid = 256;       // workspace bound on the grid (SMs)
constexpr size_t kDecodeMaxSmem = 200u << 10;
constexpr size_t kDecodeSyncOffset = 128;  // grid-barrier counters: bytes into the workspace's error block

struct DecodePlan {
  bool ok;            // the problem fits the kernel (token choice, T <= 4, shared memory)
  int grid, rsplits, r_slice;
  int x_stride;       // shared-memory row stride of the token rows (elements)
  int z_len;          // elements of the zero row
  int h_stride, hs_stride;  // row strides of h and of the shared experts' h (elements, padded)
  int hsm_stride;           // shared-memory row stride of the staged h rows (elements)
  size_t smem_x_bytes, smem_bytes;
};
DecodePlan decode_plan(const moe_problem_t& p, int sms);
// Floats of the down phase's per-group results (workspace).
size_t decode_ybuf_floats(const moe_problem_t& p);
// 16-bit elements of the kernel's h rows (routed, or shared), padded rows.
size_t decode_h_elems(const moe_problem_t& p, bool shared);

struct DecodeArgs {
  int64_t T;
  int32_t d, N, K, F, S, Fs;
  int32_t score_fn, renormalize, n_groups, topk_groups;
  int32_t capacity;            // copies an expert keeps (token order); INT32_MAX: no cap
  int32_t fmt;                 // DecodeFormat of the expert weights
  const void* hidden;          // [T][d] bf16 or fp32
  bool hidden_bf16;
  const float* w_router;       // [d][N]
  const float* router_bias;    // [N] or null (added to every logit)
  const float* sel_bias;       // [N] or null (selection only, sigmoid)
  const void* w_gate;          // [N][F][d] (bf16 or E4M3 codes)
  const void* w_up;
  const void* w_down;          // [N][d][F]
  const void* s_gate;          // shared: [S][Fs][d], [S][Fs][d], [S][d][Fs]
  const void* s_up;
  const void* s_down;
  const void* w_gate_scale;    // FP8: fp32 per weight row
  const void* w_up_scale;
  const void* w_down_scale;
  const void* s_gate_scale;
  const void* s_up_scale;
  const void* s_down_scale;
  __nv_bfloat16* out;          // [T][d]
  int32_t* topk_idx;           // [T][K]
  float* topk_w;               // [T][K]
  int32_t* counts;             // [N] or null
  float* router_part;          // [rsplits][T][N]
  void* h;                     // [T*K][h_stride] 16-bit activation format
  void* h_sh;                  // [S*T][hs_stride]
  float* bnd_val;              // [grid*16 + 1][2][64] halves of gate/up groups split between warps
  uint32_t* bnd_cnt;           // [grid*16 + 1]
  float* ybuf;                 // [d/8][entries][2][64] down groups' results
  uint32_t* blk_cnt;           // [d/8] steps done per output block
  uint32_t* sync;              // two zeroed words (barrier count, exit count)
  uint32_t* err;
  int32_t grid, rsplits, r_slice, x_stride, z_len, h_stride, hs_stride, hsm_stride;
  size_t smem_x_bytes, smem_bytes;
};
cudaError_t launch_decode_layer(const DecodeArgs& a, cudaStream_t s);

// uint8 row-major matrix [rows][inner] as a TMA tensor map: box
// [box_rows][128 bytes], 128-byte swizzle, zero fill out of bounds. The row
// pitch (`inner` bytes) must be a multiple of 16.
bool make_tmap_u8(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t rows, uint32_t box_rows);

// fp16 row-major matrix as a TMA tensor map, box [box_rows][64], 128-byte swizzle.
bool make_tmap_f16(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t rows, uint32_t box_rows);

// Grouped GEMM with FP8 E4M3 weights on two-term E4M3 activations: tiles of
// kF8TileRows tokens x 256 weight rows (the schedule built with tile_rows =
// kF8TileRows), one CTA each.
cudaError_t launch_grouped_gemm_fp8(int phase, int epilogue, const F8Maps& maps, const GemmArgs& a,
                                    int64_t tile_bound, cudaStream_t s);
// The same GEMMs for MXFP4 experts: F8Maps::w / u map the packed code
// matrices ([rows][K/2] bytes, 128-row boxes of 64 bytes, 64-byte swizzle).
cudaError_t launch_grouped_gemm_mxfp4(int phase, int epilogue, const F8Maps& maps, const GemmArgs& a,
                                      int64_t tile_bound, cudaStream_t s);
// Per-call preparation of an MXFP4 weight matrix with E8M0 block scales
// bscale [rows][nblk]: each row's reference exponent E_row = (its largest
// block exponent, NaN scales aside) - 6, clamped to 1..254, written as the
// fp32 row scale 2^(E_row - 127); and, for K block kb (128 elements = blocks
// 4kb .. 4kb+3), kidx[kb][row] = four bytes, byte c = the table index of
// block 4kb + c: clamp(E_block - E_row, -kMxIdxBias, 6) + kMxIdxBias (0 past
// the row's last block). Rows of experts whose offsets show no routed rows
// are skipped (offsets may be NULL: all rows).
constexpr int kMxIdxBias = 15;
// Shared memory the preparation of one row group may take: 128 rows of
// nblk block scales (nblk <= 1024, i.e. K <= kMxMaxK elements).
constexpr int kMxMaxK = 32768;
constexpr size_t kMxPrepMaxSmem = 128 * 4 * 257;
cudaError_t launch_mx_prep(const uint8_t* bscale, int64_t rows, int32_t rows_per_expert, int32_t nblk,
                           int32_t kblocks, const int32_t* offsets, float* row_scale, uint32_t* kidx,
                           cudaStream_t s);
// uint32 matrix [kblocks][rows] (an MXFP4 block-index array) as a TMA tensor
// map with a box of 128 rows of one K block; no swizzle, zero fill out of
// bounds. rows % 4 == 0.
bool make_tmap_mx_index(CUtensorMap* m, const uint32_t* ptr, uint64_t rows, uint64_t kblocks);
// uint8 matrix [rows][inner] with a box of [box_rows][64 bytes], 64-byte swizzle.
bool make_tmap_u8_64(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t rows, uint32_t box_rows);

// Upper bound on the tile count (host, from sizes only), used for the grid.
int64_t gemm_tile_bound(int phase, int64_t routed_rows, int32_t N, int32_t S, int64_t T,
                        int32_t F, int32_t Fs, int32_t d, int32_t tile_rows);
// pair = 1: 128-row tiles, one CTA each; pair = 2: 256-row tiles on 2-CTA
// clusters (the down-phase weight maps then use 128-row boxes).
cudaError_t launch_grouped_gemm(int phase, int epilogue, int pair, const GemmMaps& maps, const GemmArgs& a,
                                int64_t tile_bound, cudaStream_t s);

cudaError_t launch_finalize(const float* acc, __nv_bfloat16* out, int64_t n, cudaStream_t s);
// out[t] = bf16(sum_k topk_w[t][k] * y_perm[inv_row[t][k]] + sum_s shared_out[s][t]),
// fp32 in slot order; slots with inv_row < 0 are skipped; shared_out [S][T][d]
// or nullptr.
cudaError_t launch_combine(int64_t T, int32_t K, int32_t d, const __nv_bfloat16* y_perm,
                           const int32_t* inv_row, const float* topk_w,
                           const __nv_bfloat16* shared_out, int32_t S, __nv_bfloat16* out, cudaStream_t s);

}  // namespace moe
