// moe_api.cu — the C ABI (include/moe.h): argument validation, workspace
// layout, TMA tensor maps and the launch sequence of each entry point.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/moe.h"
#include "common.cuh"
#include "kernels.h"

using namespace moe;

namespace {

constexpr int64_t kInt32Max = 2147483647;

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Where the MXFP4 preparation arrays of a weight set sit (in the workspace
// for a per-call preparation, or in a buffer moe_mxfp4_prepare filled):
// every weight row's reference scale (fp32) and block-table index words.
struct MxOffsets {
  size_t rs_gate, rs_up, rs_down, rs_sgate, rs_sup, rs_sdown;
  size_t ki_gate, ki_up, ki_down, ki_sgate, ki_sup, ki_sdown;
};

// Lays the MXFP4 preparation arrays out with `take` (routed experts; the
// shared ones too when `shared`).
template <class Take>
MxOffsets mx_offsets(const moe_problem_t& p, bool shared, Take&& take) {
  MxOffsets o{};
  const size_t kb_d = (p.d_model + 127) / 128, kb_f = (p.ffn + 127) / 128;
  o.rs_gate = take((size_t)p.n_experts * p.ffn * 4);
  o.rs_up = take((size_t)p.n_experts * p.ffn * 4);
  o.rs_down = take((size_t)p.n_experts * p.d_model * 4);
  o.ki_gate = take((size_t)p.n_experts * p.ffn * kb_d * 4);
  o.ki_up = take((size_t)p.n_experts * p.ffn * kb_d * 4);
  o.ki_down = take((size_t)p.n_experts * p.d_model * kb_f * 4);
  if (shared) {
    const size_t kb_fs = (p.shared_ffn + 127) / 128;
    o.rs_sgate = take((size_t)p.n_shared * p.shared_ffn * 4);
    o.rs_sup = take((size_t)p.n_shared * p.shared_ffn * 4);
    o.rs_sdown = take((size_t)p.n_shared * p.d_model * 4);
    o.ki_sgate = take((size_t)p.n_shared * p.shared_ffn * kb_d * 4);
    o.ki_sup = take((size_t)p.n_shared * p.shared_ffn * kb_d * 4);
    o.ki_sdown = take((size_t)p.n_shared * p.d_model * kb_fs * 4);
  }
  return o;
}

struct Layout {
  size_t err, chunk, groups, ts_gu, ts_dn, router, router_w3, ec_scores, ec_token, ec_w;
  size_t topk_idx, topk_w, counts, offsets, perm_src, inv_row, x_perm, x_act, h, h_sh, out_acc, done;
  size_t y_rows, y_sh;  // token choice with a large accumulator: the down GEMM's stored rows (see stored_combine)
  size_t dec_part, dec_bnd_val, dec_bnd_cnt, dec_ybuf, dec_blk, dec_h, dec_h_sh;  // decode-sized batches
  size_t xq, sx, hq, sh, xq_sh, sx_sh, hq_sh, sh_sh;  // FP8 / MXFP4 experts: two-term E4M3 activations + row scales
  MxOffsets mx;  // MXFP4 experts: the per-call preparation of the weights in use
  size_t total;
};

// Tokens each expert takes under expert-choice routing: min(ceil(c T K / N), T),
// c = capacity_factor or 1.
int64_t ec_capacity(const moe_problem_t& p) {
  const double c = p.capacity_factor > 0.0 ? p.capacity_factor : 1.0;
  const double cap = ceil(c * (double)p.T * (double)p.top_k / (double)p.n_experts);
  return cap >= (double)p.T ? p.T : (int64_t)cap;
}

bool is_fp8(const moe_problem_t& p) { return p.expert_dtype == MOE_EXPERT_FP8_E4M3; }

// The fused layer adds every expert row into an fp32 [T][d] accumulator with
// atomics from the down GEMM's epilogue. Once that accumulator outgrows a good
// share of the 126 MB L2, those read-modify-writes go to DRAM (K + S of them
// per output element); token-choice layers then store the unweighted rows in
// bf16 and sum each token's K rows (and shared rows) in a deterministic
// combine instead.
constexpr int64_t kAtomicAccMaxBytes = 96ll << 20;
bool stored_combine(const moe_problem_t& p) {
  return p.routing == MOE_ROUTING_TOKEN_CHOICE && p.T * (int64_t)p.d_model * 4 > kAtomicAccMaxBytes;
}
bool is_mx(const moe_problem_t& p) { return p.expert_dtype == MOE_EXPERT_MXFP4; }
// FP8 and MXFP4 experts both run on the 8-bit tensor path (fp16 activations
// between calls, two-term E4M3 activations inside the GEMMs).
bool is_lowp(const moe_problem_t& p) { return is_fp8(p) || is_mx(p); }

// The shared experts read every token's hidden row in the activation format
// (bf16 for bf16 experts, fp16 for FP8 experts): a copy unless hidden is
// already in it.
bool needs_act_copy(const moe_problem_t& p) {
  return p.n_shared > 0 && (is_lowp(p) || p.hidden_dtype == MOE_F32);
}

// Token-choice batches of at most kDecodeMaxTokens tokens with bf16 or FP8
// experts run as one kernel (decode_layer.cu) when its routing tables and
// staged rows fit the kernel's shared memory: each expert then holds at most
// T rows, and a 128-row GEMM tile would be almost all padding. MXFP4 experts,
// expert choice and larger batches run on the grouped GEMMs. The decision
// takes no CUDA call: the shared memory is sized for a grid of at least
// kDecodePlanSms CTAs (the real grid only needs less).
constexpr int kDecodePlanSms = 100;
bool decode_fused(const moe_problem_t& p) {
  if (p.routing != MOE_ROUTING_TOKEN_CHOICE || p.T < 1 || p.T > kDecodeMaxTokens || is_mx(p)) return false;
  return decode_plan(p, kDecodePlanSms).ok;
}

Layout make_layout(const moe_problem_t& p, int call) {
  Layout L{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align256(off + bytes);
    return o;
  };
  const int64_t T = p.T, TK = p.T * p.top_k;
  const int64_t C = (T + kTokensPerChunk - 1) / kTokensPerChunk;
  const int G = p.n_experts + p.n_shared;
  L.err = take(256);
  L.chunk = take((size_t)p.n_experts * C * 4);
  L.groups = take((size_t)G * sizeof(GroupDesc));
  L.ts_gu = take((size_t)(G + 1) * 4);
  L.ts_dn = take((size_t)(G + 1) * 4);
  if (call == MOE_CALL_ROUTER || call == MOE_CALL_LAYER_FORWARD) {
    const RouterPlan rp = router_plan(T, p.d_model, p.n_experts, p.hidden_dtype == MOE_BF16);
    L.router = take((size_t)rp.splits * T * p.n_experts * 4);
    if (rp.tensor) L.router_w3 = take((size_t)rp.np * 3 * rp.d_pad * 2);
    if (p.routing == MOE_ROUTING_EXPERT_CHOICE) L.ec_scores = take((size_t)p.n_experts * T * 4);
  }
  const int64_t ec_rows = p.routing == MOE_ROUTING_EXPERT_CHOICE ? (int64_t)p.n_experts * ec_capacity(p) : 0;
  const int64_t rows = TK > ec_rows ? TK : ec_rows;  // packed rows of the layer
  if (call == MOE_CALL_LAYER_FORWARD && ec_rows > 0) {
    L.ec_token = take((size_t)ec_rows * 4);
    L.ec_w = take((size_t)ec_rows * 4);
  }
  if (is_mx(p) && (call == MOE_CALL_LAYER_FORWARD || call == MOE_CALL_GROUPED_SWIGLU))
    L.mx = mx_offsets(p, call == MOE_CALL_LAYER_FORWARD && p.n_shared > 0, take);
  if (is_lowp(p) && (call == MOE_CALL_LAYER_FORWARD || call == MOE_CALL_GROUPED_SWIGLU)) {
    L.xq = take((size_t)2 * rows * p.d_model);
    L.sx = take((size_t)rows * 4);
    L.hq = take((size_t)2 * rows * p.ffn);
    L.sh = take((size_t)rows * 4);
    if (call == MOE_CALL_LAYER_FORWARD && p.n_shared > 0) {
      L.xq_sh = take((size_t)2 * T * p.d_model);
      L.sx_sh = take((size_t)T * 4);
      L.hq_sh = take((size_t)2 * p.n_shared * T * p.shared_ffn);
      L.sh_sh = take((size_t)p.n_shared * T * 4);
    }
  }
  if (call == MOE_CALL_LAYER_FORWARD) {
    L.topk_idx = take((size_t)TK * 4);
    L.topk_w = take((size_t)TK * 4);
    L.counts = take((size_t)p.n_experts * 4);
    L.offsets = take((size_t)(p.n_experts + 1) * 4);
    L.perm_src = take((size_t)TK * 4);
    L.inv_row = take((size_t)TK * 4);
    // FP8 / MXFP4 experts: the gather writes the E4M3 split directly (set_gather_quant)
    if (!is_lowp(p)) {
      L.x_perm = take((size_t)rows * p.d_model * 2);
      if (needs_act_copy(p)) L.x_act = take((size_t)T * p.d_model * 2);
    }
    L.h = take((size_t)rows * p.ffn * 2);
    if (p.n_shared > 0) L.h_sh = take((size_t)p.n_shared * T * p.shared_ffn * 2);
    L.out_acc = take((size_t)T * p.d_model * 4);
    L.done = take(4);
    if (T <= kDecodeMaxTokens) {
      L.dec_part = take((size_t)kDecodeMaxSplits * T * p.n_experts * 4);
      L.dec_bnd_val = take((size_t)(kDecodeMaxGrid * (kDecodeThreads / 32) + 1) * 128 * 4);
      L.dec_bnd_cnt = take((size_t)(kDecodeMaxGrid * (kDecodeThreads / 32) + 1) * 4);
      L.dec_ybuf = take(decode_ybuf_floats(p) * 4);
      L.dec_blk = take((size_t)(p.d_model / 8) * 4);
      L.dec_h = take(decode_h_elems(p, false) * 2);
      if (p.n_shared > 0) L.dec_h_sh = take(decode_h_elems(p, true) * 2);
    }
    if (stored_combine(p)) {
      L.y_rows = take((size_t)TK * p.d_model * 2);
      if (p.n_shared > 0) L.y_sh = take((size_t)p.n_shared * T * p.d_model * 2);
    }
  }
  L.total = off;
  return L;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

namespace moe {
// Expert capacity C = ceil(c * T * K / N) ("Chapter 19", §19.6.1), computed in
// double; INT32_MAX when c == 0 (dropless).
int32_t expert_capacity(const moe_problem_t& p) {
  if (!(p.capacity_factor > 0.0)) return 2147483647;
  const double c = ceil(p.capacity_factor * (double)p.T * (double)p.top_k / (double)p.n_experts);
  return c >= 2147483647.0 ? 2147483647 : (int32_t)c;
}
}  // namespace moe

namespace {

// ---------------------------------------------------------------- TMA maps
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool have_encode() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

bool make_map(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t rows, uint32_t box_rows) {
  return moe::make_tmap_bf16(m, ptr, inner, rows, box_rows);
}

}  // namespace

namespace moe {
// bf16 matrix [rows][inner] (row stride = inner elements), box [box_rows][64],
// 128-byte swizzle, zero fill out of bounds.
bool make_tmap_bf16(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t rows, uint32_t box_rows) {
  if (!have_encode()) return false;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kBK, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp16 matrix, same geometry as make_tmap_bf16.
bool make_tmap_f16(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t rows, uint32_t box_rows) {
  if (!have_encode()) return false;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kBK, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}


// uint8 matrix [rows][inner], box [box_rows][128 bytes], 128-byte swizzle,
// zero fill out of bounds.
bool make_tmap_u8(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t rows, uint32_t box_rows) {
  if (!have_encode() || (inner % 16) != 0) return false;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {inner};
  const cuuint32_t box[2] = {128u, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// uint8 matrix [rows][inner], box [box_rows][64 bytes], 64-byte swizzle (the
// 16-byte chunk c of box row R lands at chunk c ^ ((R >> 1) & 3)), zero fill
// out of bounds.
bool make_tmap_u8_64(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t rows, uint32_t box_rows) {
  if (!have_encode() || (inner % 16) != 0) return false;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {inner};
  const cuuint32_t box[2] = {64u, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tmap_mx_index(CUtensorMap* m, const uint32_t* ptr, uint64_t rows, uint64_t kblocks) {
  if (!have_encode() || (rows % 4) != 0) return false;
  const cuuint64_t dims[2] = {rows, kblocks};
  const cuuint64_t strides[1] = {rows * 4};
  const cuuint32_t box[2] = {128u, 1u};
  const cuuint32_t estr[2] = {1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint32_t*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace moe

namespace {

moe_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

#define MOE_TRY(expr)                          \
  do {                                         \
    const moe_status_t _st = (expr);           \
    if (_st != MOE_OK) return _st;             \
  } while (0)
#define MOE_TRY_CUDA(expr)                     \
  do {                                         \
    if ((expr) != cudaSuccess) return MOE_ERR_CUDA; \
  } while (0)

moe_status_t check_ws(const moe_problem_t* p, int call, void* ws, size_t ws_bytes, Layout* L) {
  *L = make_layout(*p, call);
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0 || ws_bytes < L->total) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

// 256-row tiles on CTA pairs once the mean expert group fills one; decode
// shapes (a few rows per expert) keep 128-row tiles on single CTAs.
int32_t gemm_pair(int64_t routed_rows, int32_t N) { return routed_rows >= (int64_t)256 * N ? 2 : 1; }

// Rows per tile of the GEMM schedule: 128 (single CTAs) or 256 (CTA pairs)
// for bf16 experts, kF8TileRows tokens for the FP8-weight kernel.
int32_t gemm_tile_rows(const moe_problem_t& p, int64_t routed_rows) {
  return is_lowp(p) ? kF8TileRows : kBM * gemm_pair(routed_rows, p.n_experts);
}

// The two GEMM phases over groups already described in the workspace.
struct GemmPlan {
  int32_t pair;
  bool fp8;               // FP8 or MXFP4 weights (+ the scales below), fp16 activations
  bool mx;                // MXFP4: *_scale are E8M0 block scales; rs_* the rows' reference scales
  bool mx_prepared;       // MXFP4: rs_* / ki_* were filled by moe_mxfp4_prepare (no per-call preparation)
  bool x_quantized;       // FP8 / MXFP4: xq / sx (and xq_sh / sx_sh) were written by the gather
  int32_t N, S, F, Fs, d, K;
  int64_t T, routed_rows;
  const void* x_routed;   // [routed_rows][d] bf16
  const void* x_shared;   // [T][d] bf16 (S > 0)
  const void* wg;         // [N][F][d]
  const void* wu;
  const void* wd;         // [N][d][F]
  const void* sg;         // [S][Fs][d]
  const void* su;
  const void* sd;         // [S][d][Fs]
  const void* wg_scale;   // FP8: fp32 [N][F], [N][F], [N][d]; MXFP4: E8M0 [N][F][d/32], [N][F][d/32], [N][d][F/32]
  const void* wu_scale;
  const void* wd_scale;
  const void* sg_scale;   // the same for the shared experts
  const void* su_scale;
  const void* sd_scale;
  float* rs_gate;         // MXFP4: reference scale of each weight row, [N][F], [N][F], [N][d]
  float* rs_up;
  float* rs_down;
  float* rs_sgate;        // shared: [S][Fs], [S][Fs], [S][d]
  float* rs_sup;
  float* rs_sdown;
  uint32_t* ki_gate;      // MXFP4: block-table indices, [d/128][N F], [d/128][N F], [F/128][N d]
  uint32_t* ki_up;
  uint32_t* ki_down;
  uint32_t* ki_sgate;     // shared: [d/128][S Fs], [d/128][S Fs], [Fs/128][S d]
  uint32_t* ki_sup;
  uint32_t* ki_sdown;
  const int32_t* offsets; // MXFP4: routed rows per expert (experts without rows are skipped)
  __nv_bfloat16* h;       // [routed_rows][F] (fp16 bits when fp8)
  __nv_bfloat16* h_sh;    // [S*T][Fs] (fp16 bits when fp8)
  uint8_t* xq;            // FP8: two-term E4M3 activations [2 rows][K] and their row scales
  float* sx;
  uint8_t* hq;
  float* sh;
  uint8_t* xq_sh;
  float* sx_sh;
  uint8_t* hq_sh;
  float* sh_sh;
  int epilogue;           // kEpiScatter or kEpiStoreY
  float* out_acc;
  const int32_t* perm_src;
  const float* topk_w;
  const float* row_w;
  __nv_bfloat16* y;
  __nv_bfloat16* y_sh;    // store epilogue, shared experts' rows (nullptr: y)
  const GroupDesc* groups;
  const int32_t* ts_gu;
  const int32_t* ts_dn;
  uint32_t* err;
};

// The MXFP4 preparation arrays of a plan at `base` (routed experts; shared
// ones too when `shared`).
void set_mx_arrays(GemmPlan* g, void* base, const MxOffsets& o, bool shared) {
  g->rs_gate = at<float>(base, o.rs_gate);
  g->rs_up = at<float>(base, o.rs_up);
  g->rs_down = at<float>(base, o.rs_down);
  g->ki_gate = at<uint32_t>(base, o.ki_gate);
  g->ki_up = at<uint32_t>(base, o.ki_up);
  g->ki_down = at<uint32_t>(base, o.ki_down);
  if (shared) {
    g->rs_sgate = at<float>(base, o.rs_sgate);
    g->rs_sup = at<float>(base, o.rs_sup);
    g->rs_sdown = at<float>(base, o.rs_sdown);
    g->ki_sgate = at<uint32_t>(base, o.ki_sgate);
    g->ki_sup = at<uint32_t>(base, o.ki_sup);
    g->ki_sdown = at<uint32_t>(base, o.ki_sdown);
  }
}

// A buffer's layout of the preparation moe_mxfp4_prepare writes (offsets
// from its start, 256-byte aligned) and its size.
MxOffsets prep_offsets(const moe_problem_t& p, size_t* total) {
  size_t off = 0;
  const MxOffsets o = mx_offsets(p, p.n_shared > 0, [&](size_t bytes) {
    const size_t at_ = off;
    off = align256(off + bytes);
    return at_;
  });
  if (total) *total = off;
  return o;
}

// The plan's MXFP4 arrays: the caller's prepared buffer when the weights
// carry one, else the workspace (prepared by this call).
void set_mx_plan(GemmPlan* g, const moe_problem_t& p, const moe_weights_t* w, void* ws, const Layout& L,
                 bool shared) {
  if (w && w->mx_prep) {
    set_mx_arrays(g, const_cast<void*>(w->mx_prep), prep_offsets(p, nullptr), shared);
    g->mx_prepared = true;
  } else {
    set_mx_arrays(g, ws, L.mx, shared);
  }
}

// FP8 / MXFP4 experts in the fused layer: the gather writes the two-term E4M3
// split of the packed rows (and of the shared experts' token rows) directly;
// no x_perm or activation copy is needed.
void set_gather_quant(PermuteArgs* pa, void* ws, const Layout& L, bool shared) {
  pa->xq = at<uint8_t>(ws, L.xq);
  pa->sx = at<float>(ws, L.sx);
  if (shared) {
    pa->xq_sh = at<uint8_t>(ws, L.xq_sh);
    pa->sx_sh = at<float>(ws, L.sx_sh);
  }
  pa->x_perm = nullptr;
  pa->x_act = nullptr;
}

// While the stream is being captured into a CUDA graph, an external record
// keeps the event a real record node of the graph; otherwise a plain record.
cudaError_t record_event(cudaEvent_t e, cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  const cudaError_t q = cudaStreamIsCapturing(s, &cs);
  if (q != cudaSuccess) return q;
  return cs == cudaStreamCaptureStatusActive ? cudaEventRecordWithFlags(e, s, cudaEventRecordExternal)
                                             : cudaEventRecord(e, s);
}

moe_status_t run_gemms_fp8(const GemmPlan& g, cudaStream_t s, cudaEvent_t* ev_after_gateup);

moe_status_t run_gemms(const GemmPlan& g, cudaStream_t s, cudaEvent_t* ev_after_gateup = nullptr) {
  if (g.fp8) return run_gemms_fp8(g, s, ev_after_gateup);
  if (!have_encode()) return MOE_ERR_CUDA;
  const bool sh = g.S > 0;
  GemmMaps m{};
  bool ok = make_map(&m.a[0], g.x_routed, g.d, g.routed_rows, kBM) &&
            make_map(&m.b[0], g.wg, g.d, (uint64_t)g.N * g.F, kBNGateUp) &&
            make_map(&m.bu[0], g.wu, g.d, (uint64_t)g.N * g.F, kBNGateUp);
  if (ok && sh)
    ok = make_map(&m.a[1], g.x_shared, g.d, g.T, kBM) &&
         make_map(&m.b[1], g.sg, g.d, (uint64_t)g.S * g.Fs, kBNGateUp) &&
         make_map(&m.bu[1], g.su, g.d, (uint64_t)g.S * g.Fs, kBNGateUp);
  if (!ok) return MOE_ERR_CUDA;
  // pairs: the half tiles' gate and up rows in 64-row boxes
  if (ok && g.pair == 2)
    ok = make_map(&m.bh[0], g.wg, g.d, (uint64_t)g.N * g.F, kBNGateUp / 2) &&
         make_map(&m.uh[0], g.wu, g.d, (uint64_t)g.N * g.F, kBNGateUp / 2) &&
         (!sh || (make_map(&m.bh[1], g.sg, g.d, (uint64_t)g.S * g.Fs, kBNGateUp / 2) &&
                  make_map(&m.uh[1], g.su, g.d, (uint64_t)g.S * g.Fs, kBNGateUp / 2)));
  if (!ok) return MOE_ERR_CUDA;
  if (g.pair != 2) {
    m.bh[0] = m.b[0];
    m.uh[0] = m.bu[0];
  }
  if (!sh) {
    m.a[1] = m.a[0];
    m.b[1] = m.b[0];
    m.bu[1] = m.bu[0];
    m.bh[1] = m.bh[0];
    m.uh[1] = m.uh[0];
  } else if (g.pair != 2) {
    m.bh[1] = m.b[1];
    m.uh[1] = m.bu[1];
  }
  GemmArgs a{};
  a.groups = g.groups;
  a.G = g.N + g.S;
  a.err = g.err;
  a.d = g.d;
  a.top_k = g.K;

  // gate/up + SwiGLU
  a.tile_start = g.ts_gu;
  a.phase_dn = 0;
  a.n_ext[0] = g.F;
  a.n_ext[1] = sh ? g.Fs : g.F;
  a.k_blocks[0] = a.k_blocks[1] = (g.d + kBK - 1) / kBK;
  a.w_rows[0] = g.F;
  a.w_rows[1] = sh ? g.Fs : g.F;
  a.h[0] = g.h;
  a.h[1] = sh ? g.h_sh : g.h;
  a.ldh[0] = g.F;
  a.ldh[1] = sh ? g.Fs : g.F;
  const int32_t rows = kBM * g.pair;
  int64_t bound = gemm_tile_bound(kPhaseGateUp, g.routed_rows, g.N, g.S, g.T, g.F, g.Fs, g.d, rows);
  MOE_TRY(cuda_status(launch_grouped_gemm(kPhaseGateUp, kEpiSwiGLU, g.pair, m, a, bound, s)));
  if (ev_after_gateup) MOE_TRY(cuda_status(record_event(ev_after_gateup[0], s)));

  // down (+ weighted scatter-add or plain store)
  GemmMaps md{};
  const uint32_t down_box = kBNDown / g.pair;  // a pair loads half the down rows per CTA
  ok = make_map(&md.a[0], g.h, g.F, g.routed_rows, kBM) &&
       make_map(&md.b[0], g.wd, g.F, (uint64_t)g.N * g.d, down_box);
  if (ok && sh)
    ok = make_map(&md.a[1], g.h_sh, g.Fs, (uint64_t)g.S * g.T, kBM) &&
         make_map(&md.b[1], g.sd, g.Fs, (uint64_t)g.S * g.d, down_box);
  if (!ok) return MOE_ERR_CUDA;
  if (!sh) {
    md.a[1] = md.a[0];
    md.b[1] = md.b[0];
  }
  md.bu[0] = md.b[0];
  md.bu[1] = md.b[1];
  md.bh[0] = md.uh[0] = md.b[0];
  md.bh[1] = md.uh[1] = md.b[1];
  a.tile_start = g.ts_dn;
  a.phase_dn = 1;
  a.n_ext[0] = a.n_ext[1] = g.d;
  a.k_blocks[0] = (g.F + kBK - 1) / kBK;
  a.k_blocks[1] = sh ? (g.Fs + kBK - 1) / kBK : a.k_blocks[0];
  a.w_rows[0] = a.w_rows[1] = g.d;
  a.out_acc = g.out_acc;
  a.perm_src = g.perm_src;
  a.topk_w = g.topk_w;
  a.row_w = g.row_w;
  a.y = g.y;
  a.y_sh = g.y_sh;
  bound = gemm_tile_bound(kPhaseDown, g.routed_rows, g.N, g.S, g.T, g.F, g.Fs, g.d, rows);
  MOE_TRY(cuda_status(launch_grouped_gemm(kPhaseDown, g.epilogue, g.pair, md, a, bound, s)));
  if (ev_after_gateup) MOE_TRY(cuda_status(record_event(ev_after_gateup[1], s)));
  return MOE_OK;
}

// The activation maps of one kind (two-term E4M3 rows): boxes of 16, 32, 64
// and 128 rows.
bool make_x_maps(CUtensorMap (&m)[kF8XBoxes], const void* ptr, uint64_t inner, uint64_t rows) {
  for (int i = 0; i < kF8XBoxes; ++i)
    if (!make_tmap_u8(&m[i], ptr, inner, rows, 16u << i)) return false;
  return true;
}

// The code maps of one weight matrix: FP8 rows of K bytes in 128-byte boxes,
// MXFP4 rows of K/2 bytes in 64-byte boxes; 128 rows per box.
bool make_code_map(CUtensorMap* m, const void* ptr, uint64_t K, uint64_t rows, bool mx) {
  return mx ? make_tmap_u8_64(m, ptr, K / 2, rows, 128) : make_tmap_u8(m, ptr, K, rows, 128);
}

// The two GEMM phases for FP8 or MXFP4 experts: each phase's activations are
// first split into two-term E4M3 rows (act_quant.cu); MXFP4 weight matrices
// first get their rows' reference scales and block-table indices
// (launch_mx_prep).
moe_status_t run_gemms_fp8(const GemmPlan& g, cudaStream_t s, cudaEvent_t* ev_after_gateup) {
  if (!have_encode()) return MOE_ERR_CUDA;
  const bool sh = g.S > 0, mx = g.mx;
  auto f32 = [](const void* p) { return static_cast<const float*>(p); };
  auto u8 = [](const void* p) { return static_cast<const uint8_t*>(p); };
  const int32_t kb_d = (g.d + 127) / 128, kb_f = (g.F + 127) / 128, kb_fs = (g.Fs + 127) / 128;
  if (mx && !g.mx_prepared) {
    const int64_t nf = (int64_t)g.N * g.F, nd = (int64_t)g.N * g.d;
    MOE_TRY(cuda_status(launch_mx_prep(u8(g.wg_scale), nf, g.F, g.d / 32, kb_d, g.offsets, g.rs_gate, g.ki_gate, s)));
    MOE_TRY(cuda_status(launch_mx_prep(u8(g.wu_scale), nf, g.F, g.d / 32, kb_d, g.offsets, g.rs_up, g.ki_up, s)));
    MOE_TRY(cuda_status(launch_mx_prep(u8(g.wd_scale), nd, g.d, g.F / 32, kb_f, g.offsets, g.rs_down, g.ki_down, s)));
    if (sh) {
      const int64_t sf = (int64_t)g.S * g.Fs, sd = (int64_t)g.S * g.d;
      MOE_TRY(cuda_status(launch_mx_prep(u8(g.sg_scale), sf, g.Fs, g.d / 32, kb_d, nullptr, g.rs_sgate, g.ki_sgate, s)));
      MOE_TRY(cuda_status(launch_mx_prep(u8(g.su_scale), sf, g.Fs, g.d / 32, kb_d, nullptr, g.rs_sup, g.ki_sup, s)));
      MOE_TRY(cuda_status(launch_mx_prep(u8(g.sd_scale), sd, g.d, g.Fs / 32, kb_fs, nullptr, g.rs_sdown, g.ki_sdown, s)));
    }
  }
  if (!g.x_quantized) {
    MOE_TRY(cuda_status(launch_act_quant(g.x_routed, g.routed_rows, g.d, g.xq, g.sx, s)));
    if (sh) MOE_TRY(cuda_status(launch_act_quant(g.x_shared, g.T, g.d, g.xq_sh, g.sx_sh, s)));
  }
  F8Maps m{};
  bool ok = make_x_maps(m.x[0], g.xq, g.d, 2 * (uint64_t)g.routed_rows) &&
            make_code_map(&m.w[0], g.wg, g.d, (uint64_t)g.N * g.F, mx) &&
            make_code_map(&m.u[0], g.wu, g.d, (uint64_t)g.N * g.F, mx);
  if (ok && sh)
    ok = make_x_maps(m.x[1], g.xq_sh, g.d, 2 * (uint64_t)g.T) &&
         make_code_map(&m.w[1], g.sg, g.d, (uint64_t)g.S * g.Fs, mx) &&
         make_code_map(&m.u[1], g.su, g.d, (uint64_t)g.S * g.Fs, mx);
  if (ok && mx)
    ok = make_tmap_mx_index(&m.kw[0], g.ki_gate, (uint64_t)g.N * g.F, kb_d) &&
         make_tmap_mx_index(&m.ku[0], g.ki_up, (uint64_t)g.N * g.F, kb_d) &&
         (!sh || (make_tmap_mx_index(&m.kw[1], g.ki_sgate, (uint64_t)g.S * g.Fs, kb_d) &&
                  make_tmap_mx_index(&m.ku[1], g.ki_sup, (uint64_t)g.S * g.Fs, kb_d)));
  if (!ok) return MOE_ERR_CUDA;
  if (!sh) {
    for (int i = 0; i < kF8XBoxes; ++i) m.x[1][i] = m.x[0][i];
    m.w[1] = m.w[0];
    m.u[1] = m.u[0];
    m.kw[1] = m.kw[0];
    m.ku[1] = m.ku[0];
  }
  auto launch = [&](int phase, int epi, const F8Maps& maps, const GemmArgs& args, int64_t bound) {
    return mx ? launch_grouped_gemm_mxfp4(phase, epi, maps, args, bound, s)
              : launch_grouped_gemm_fp8(phase, epi, maps, args, bound, s);
  };
  GemmArgs a{};
  a.groups = g.groups;
  a.G = g.N + g.S;
  a.err = g.err;
  a.d = g.d;
  a.top_k = g.K;

  // gate/up + SwiGLU (K advances 128 codes per stage)
  a.tile_start = g.ts_gu;
  a.phase_dn = 0;
  a.n_ext[0] = g.F;
  a.n_ext[1] = sh ? g.Fs : g.F;
  a.k_blocks[0] = a.k_blocks[1] = kb_d;
  a.w_rows[0] = g.F;
  a.w_rows[1] = sh ? g.Fs : g.F;
  a.h[0] = g.h;
  a.h[1] = sh ? g.h_sh : g.h;
  a.ldh[0] = g.F;
  a.ldh[1] = sh ? g.Fs : g.F;
  if (mx) {
    a.w_scale[0] = g.rs_gate;
    a.u_scale[0] = g.rs_up;
    a.w_scale[1] = sh ? g.rs_sgate : g.rs_gate;
    a.u_scale[1] = sh ? g.rs_sup : g.rs_up;
  } else {
    a.w_scale[0] = f32(g.wg_scale);
    a.u_scale[0] = f32(g.wu_scale);
    a.w_scale[1] = sh ? f32(g.sg_scale) : a.w_scale[0];
    a.u_scale[1] = sh ? f32(g.su_scale) : a.u_scale[0];
  }
  a.a_scale[0] = g.sx;
  a.a_scale[1] = sh ? g.sx_sh : g.sx;
  int64_t bound = gemm_tile_bound(kPhaseGateUp, g.routed_rows, g.N, g.S, g.T, g.F, g.Fs, g.d, kF8TileRows);
  MOE_TRY(cuda_status(launch(kPhaseGateUp, kEpiSwiGLU, m, a, bound)));
  if (ev_after_gateup) MOE_TRY(cuda_status(record_event(ev_after_gateup[0], s)));

  // down (+ weighted scatter-add or plain store)
  MOE_TRY(cuda_status(launch_act_quant(g.h, g.routed_rows, g.F, g.hq, g.sh, s)));
  if (sh) MOE_TRY(cuda_status(launch_act_quant(g.h_sh, (int64_t)g.S * g.T, g.Fs, g.hq_sh, g.sh_sh, s)));
  F8Maps md{};
  ok = make_x_maps(md.x[0], g.hq, g.F, 2 * (uint64_t)g.routed_rows) &&
       make_code_map(&md.w[0], g.wd, g.F, (uint64_t)g.N * g.d, mx);
  if (ok && sh)
    ok = make_x_maps(md.x[1], g.hq_sh, g.Fs, 2 * (uint64_t)g.S * g.T) &&
         make_code_map(&md.w[1], g.sd, g.Fs, (uint64_t)g.S * g.d, mx);
  if (ok && mx)
    ok = make_tmap_mx_index(&md.kw[0], g.ki_down, (uint64_t)g.N * g.d, kb_f) &&
         (!sh || make_tmap_mx_index(&md.kw[1], g.ki_sdown, (uint64_t)g.S * g.d, kb_fs));
  if (!ok) return MOE_ERR_CUDA;
  if (!sh) {
    for (int i = 0; i < kF8XBoxes; ++i) md.x[1][i] = md.x[0][i];
    md.w[1] = md.w[0];
    md.kw[1] = md.kw[0];
  }
  md.u[0] = md.w[0];
  md.u[1] = md.w[1];
  md.ku[0] = md.kw[0];
  md.ku[1] = md.kw[1];
  a.tile_start = g.ts_dn;
  a.phase_dn = 1;
  a.n_ext[0] = a.n_ext[1] = g.d;
  a.k_blocks[0] = kb_f;
  a.k_blocks[1] = sh ? kb_fs : kb_f;
  a.w_rows[0] = a.w_rows[1] = g.d;
  if (mx) {
    a.w_scale[0] = g.rs_down;
    a.w_scale[1] = sh ? g.rs_sdown : g.rs_down;
  } else {
    a.w_scale[0] = f32(g.wd_scale);
    a.w_scale[1] = sh ? f32(g.sd_scale) : a.w_scale[0];
  }
  a.u_scale[0] = a.u_scale[1] = nullptr;
  a.a_scale[0] = g.sh;
  a.a_scale[1] = sh ? g.sh_sh : g.sh;
  a.out_acc = g.out_acc;
  a.perm_src = g.perm_src;
  a.topk_w = g.topk_w;
  a.row_w = g.row_w;
  a.y = g.y;
  a.y_sh = g.y_sh;
  bound = gemm_tile_bound(kPhaseDown, g.routed_rows, g.N, g.S, g.T, g.F, g.Fs, g.d, kF8TileRows);
  MOE_TRY(cuda_status(launch(kPhaseDown, g.epilogue, md, a, bound)));
  if (ev_after_gateup) MOE_TRY(cuda_status(record_event(ev_after_gateup[1], s)));
  return MOE_OK;
}

}  // namespace

extern "C" {

const char* moe_status_string(int32_t status) {
  switch (status) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG: invalid argument";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED: problem not supported by this build";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE: workspace missing, misaligned or too small";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA: a CUDA call or kernel launch failed";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT: a device pipeline wait timed out";
    case MOE_ERR_DEVICE_BOUNDS: return "MOE_ERR_DEVICE_BOUNDS: an input index was out of range";
    case MOE_ERR_RANGE: return "MOE_ERR_RANGE: an fp16 activation of the FP8 / MXFP4 path overflowed";
    default: return "MOE_ERR_UNKNOWN: unrecognised status";
  }
}

moe_status_t moe_problem_check(const moe_problem_t* p) {
  if (!p) return MOE_ERR_INVALID_ARG;
  if (p->T < 0 || p->d_model <= 0 || (p->d_model % 8) != 0) return MOE_ERR_INVALID_ARG;
  if (p->n_experts < 1 || p->top_k < 1 || p->top_k > p->n_experts) return MOE_ERR_INVALID_ARG;
  if (p->ffn <= 0 || (p->ffn % 8) != 0) return MOE_ERR_INVALID_ARG;
  if (p->n_shared < 0) return MOE_ERR_INVALID_ARG;
  if (p->n_shared > 0 && (p->shared_ffn <= 0 || (p->shared_ffn % 8) != 0)) return MOE_ERR_INVALID_ARG;
  if (p->score_fn != MOE_SCORE_SOFTMAX && p->score_fn != MOE_SCORE_SIGMOID) return MOE_ERR_INVALID_ARG;
  if (p->renormalize != 0 && p->renormalize != 1) return MOE_ERR_INVALID_ARG;
  if (p->hidden_dtype != MOE_F32 && p->hidden_dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
  if (p->n_groups < 0) return MOE_ERR_INVALID_ARG;
  if (!(p->capacity_factor >= 0.0) || p->capacity_factor > 1e30) return MOE_ERR_INVALID_ARG;  // NaN fails too
  if (p->routing != MOE_ROUTING_TOKEN_CHOICE && p->routing != MOE_ROUTING_EXPERT_CHOICE) return MOE_ERR_INVALID_ARG;
  if (p->routing == MOE_ROUTING_EXPERT_CHOICE && p->n_groups > 1) return MOE_ERR_UNSUPPORTED;
  if (p->expert_dtype != MOE_EXPERT_BF16 && p->expert_dtype != MOE_EXPERT_FP8_E4M3 &&
      p->expert_dtype != MOE_EXPERT_MXFP4)
    return MOE_ERR_INVALID_ARG;
  if (p->expert_dtype == MOE_EXPERT_MXFP4) {  // 32-element scale blocks; code rows in 16-byte units
    if ((p->d_model % 32) != 0 || (p->ffn % 32) != 0) return MOE_ERR_INVALID_ARG;
    if (p->n_shared > 0 && (p->shared_ffn % 32) != 0) return MOE_ERR_INVALID_ARG;
    // a weight row's block scales are staged whole in shared memory
    if (p->d_model > kMxMaxK || p->ffn > kMxMaxK || (p->n_shared > 0 && p->shared_ffn > kMxMaxK))
      return MOE_ERR_UNSUPPORTED;
  }
  if (p->expert_dtype == MOE_EXPERT_FP8_E4M3) {  // 16-byte rows of codes for the TMA boxes
    if ((p->d_model % 16) != 0 || (p->ffn % 16) != 0) return MOE_ERR_INVALID_ARG;
    if (p->n_shared > 0 && (p->shared_ffn % 16) != 0) return MOE_ERR_INVALID_ARG;
  }
  if (p->n_groups > 1) {
    if (p->n_experts % p->n_groups != 0 || p->topk_groups < 1 || p->topk_groups > p->n_groups)
      return MOE_ERR_INVALID_ARG;
    if (p->top_k > p->topk_groups * (p->n_experts / p->n_groups)) return MOE_ERR_INVALID_ARG;
  }
  if (p->n_experts > kMaxExperts || p->top_k > kMaxTopK || p->n_shared > kMaxShared) return MOE_ERR_UNSUPPORTED;
  if (p->T * p->top_k > kInt32Max || p->T * (p->n_shared > 0 ? p->n_shared : 1) > kInt32Max)
    return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

size_t moe_workspace_bytes(const moe_problem_t* p, int32_t call) {
  if (moe_problem_check(p) != MOE_OK) return 0;
  if (call != MOE_CALL_PERMUTE && call != MOE_CALL_GROUPED_SWIGLU && call != MOE_CALL_LAYER_FORWARD &&
      call != MOE_CALL_ROUTER)
    return 0;
  return make_layout(*p, call).total;
}

moe_status_t moe_router_topk(const moe_problem_t* p, const void* hidden, const float* w_router,
                             const float* router_bias, const float* sel_bias, int32_t* topk_idx, float* topk_w,
                             float* logits_opt, void* ws, size_t ws_bytes, void* stream) {
  MOE_TRY(moe_problem_check(p));
  if (p->routing != MOE_ROUTING_TOKEN_CHOICE) return MOE_ERR_INVALID_ARG;
  if (sel_bias && p->score_fn == MOE_SCORE_SOFTMAX) return MOE_ERR_UNSUPPORTED;
  Layout L;
  MOE_TRY(check_ws(p, MOE_CALL_ROUTER, ws, ws_bytes, &L));
  if (p->T == 0) return MOE_OK;
  if (!hidden || !w_router || !topk_idx || !topk_w) return MOE_ERR_INVALID_ARG;
  if (!aligned16(hidden) || !aligned16(w_router)) return MOE_ERR_INVALID_ARG;
  RouterArgs a{p->T, p->d_model, p->n_experts, p->top_k, p->score_fn, p->renormalize,
               p->n_groups, p->topk_groups, hidden, w_router, router_bias, sel_bias, topk_idx, topk_w, logits_opt,
               at<float>(ws, L.router), at<__nv_bfloat16>(ws, L.router_w3), 0, 0};
  return cuda_status(launch_router(a, p->hidden_dtype == MOE_BF16, static_cast<cudaStream_t>(stream)));
}

int64_t moe_expert_choice_capacity(const moe_problem_t* p) {
  if (moe_problem_check(p) != MOE_OK) return -1;
  return ec_capacity(*p);
}

moe_status_t moe_expert_choice_select(const moe_problem_t* p, const void* hidden, const float* w_router,
                                      const float* router_bias, int32_t* row_token, float* row_w,
                                      int32_t* offsets, void* ws, size_t ws_bytes, void* stream) {
  MOE_TRY(moe_problem_check(p));
  if (p->routing != MOE_ROUTING_EXPERT_CHOICE) return MOE_ERR_INVALID_ARG;
  Layout L;
  MOE_TRY(check_ws(p, MOE_CALL_ROUTER, ws, ws_bytes, &L));
  if (p->T == 0) return MOE_OK;
  if (!hidden || !w_router || !row_token || !row_w || !offsets) return MOE_ERR_INVALID_ARG;
  if (!aligned16(hidden) || !aligned16(w_router)) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  RouterArgs a{p->T, p->d_model, p->n_experts, p->top_k, p->score_fn, p->renormalize, 0, 0,
               hidden, w_router, router_bias, nullptr, nullptr, nullptr, nullptr,
               at<float>(ws, L.router), at<__nv_bfloat16>(ws, L.router_w3), 0, 0, at<float>(ws, L.ec_scores)};
  MOE_TRY(cuda_status(launch_router(a, p->hidden_dtype == MOE_BF16, s)));
  return cuda_status(launch_expert_choice_select(a.scores_t, p->T, p->n_experts, (int32_t)ec_capacity(*p),
                                                 row_token, row_w, offsets, nullptr, s));
}

moe_status_t moe_permute(const moe_problem_t* p, const int32_t* topk_idx, const void* hidden, int32_t* counts,
                         int32_t* offsets, int32_t* perm_src, int32_t* inv_row, void* x_perm, void* ws,
                         size_t ws_bytes, void* stream) {
  MOE_TRY(moe_problem_check(p));
  if (p->routing != MOE_ROUTING_TOKEN_CHOICE) return MOE_ERR_INVALID_ARG;
  if (!counts || !offsets) return MOE_ERR_INVALID_ARG;
  if (p->T > 0 && (!topk_idx || !hidden || !perm_src || !inv_row || !x_perm)) return MOE_ERR_INVALID_ARG;
  if (p->T > 0 && (!aligned16(hidden) || !aligned16(x_perm))) return MOE_ERR_INVALID_ARG;
  Layout L;
  MOE_TRY(check_ws(p, MOE_CALL_PERMUTE, ws, ws_bytes, &L));
  PermuteArgs a{};
  a.T = p->T;
  a.d = p->d_model;
  a.N = p->n_experts;
  a.K = p->top_k;
  a.C = (int32_t)((p->T + kTokensPerChunk - 1) / kTokensPerChunk);
  a.capacity = expert_capacity(*p);
  a.topk_idx = topk_idx;
  a.hidden = hidden;
  a.hidden_bf16 = p->hidden_dtype == MOE_BF16;
  a.chunk_counts = at<int32_t>(ws, L.chunk);
  a.counts = counts;
  a.offsets = offsets;
  a.perm_src = perm_src;
  a.inv_row = inv_row;
  a.x_perm = x_perm;
  a.act_f16 = is_lowp(*p);
  a.err = at<uint32_t>(ws, L.err);
  return cuda_status(launch_permute(a, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace {

// The scale arrays a low-precision expert format needs: fp32 row scales
// (16-byte aligned) for FP8, E8M0 block-scale bytes for MXFP4.
bool scales_ok(const moe_problem_t& p, const void* a, const void* b, const void* c) {
  if (!is_lowp(p)) return true;
  if (!a || !b || !c) return false;
  return is_mx(p) || (aligned16(a) && aligned16(b) && aligned16(c));
}

moe_status_t grouped_swiglu_impl(const moe_problem_t* p, const void* x_perm, const int32_t* offsets,
                                 const void* w_gate, const void* sg, const void* w_up, const void* su,
                                 const void* w_down, const void* sd, void* h_perm, void* y_perm, void* ws,
                                 size_t ws_bytes, void* stream) {
  MOE_TRY(moe_problem_check(p));
  const bool fp8 = is_lowp(*p);
  if (!offsets || !w_gate || !w_up || !w_down) return MOE_ERR_INVALID_ARG;
  if (!scales_ok(*p, sg, su, sd)) return MOE_ERR_INVALID_ARG;
  if (!aligned16(w_gate) || !aligned16(w_up) || !aligned16(w_down)) return MOE_ERR_INVALID_ARG;
  // packed rows: T*K copies (token choice) or N*C picks (expert choice)
  const int64_t rows =
      p->routing == MOE_ROUTING_EXPERT_CHOICE ? (int64_t)p->n_experts * ec_capacity(*p) : p->T * p->top_k;
  if (rows > 0 && (!x_perm || !h_perm || !y_perm)) return MOE_ERR_INVALID_ARG;
  if (rows > 0 && (!aligned16(x_perm) || !aligned16(h_perm) || !aligned16(y_perm))) return MOE_ERR_INVALID_ARG;
  moe_problem_t q = *p;
  q.n_shared = 0;
  Layout L;
  MOE_TRY(check_ws(&q, MOE_CALL_GROUPED_SWIGLU, ws, ws_bytes, &L));
  if (rows == 0) return MOE_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int32_t tile_rows = gemm_tile_rows(q, rows);
  const int32_t pair = tile_rows == 2 * kBM ? 2 : 1;
  ScheduleArgs sa{q.n_experts, 0, q.ffn, 0, q.d_model, tile_rows, q.T, offsets, at<GroupDesc>(ws, L.groups),
                  at<int32_t>(ws, L.ts_gu), at<int32_t>(ws, L.ts_dn)};
  MOE_TRY(cuda_status(launch_schedule(sa, s)));
  GemmPlan g{};
  g.pair = pair;
  g.fp8 = fp8;
  g.mx = is_mx(q);
  g.wg_scale = sg;
  g.wu_scale = su;
  g.wd_scale = sd;
  g.offsets = offsets;
  if (fp8) {
    g.xq = at<uint8_t>(ws, L.xq);
    g.sx = at<float>(ws, L.sx);
    g.hq = at<uint8_t>(ws, L.hq);
    g.sh = at<float>(ws, L.sh);
  }
  if (g.mx) set_mx_plan(&g, q, nullptr, ws, L, false);
  g.N = q.n_experts;
  g.S = 0;
  g.F = q.ffn;
  g.Fs = 0;
  g.d = q.d_model;
  g.K = q.top_k;
  g.T = q.T;
  g.routed_rows = rows;
  g.x_routed = x_perm;
  g.wg = w_gate;
  g.wu = w_up;
  g.wd = w_down;
  g.h = static_cast<__nv_bfloat16*>(h_perm);
  g.epilogue = kEpiStoreY;
  g.y = static_cast<__nv_bfloat16*>(y_perm);
  g.groups = at<GroupDesc>(ws, L.groups);
  g.ts_gu = at<int32_t>(ws, L.ts_gu);
  g.ts_dn = at<int32_t>(ws, L.ts_dn);
  g.err = at<uint32_t>(ws, L.err);
  return run_gemms(g, s);
}

}  // namespace

extern "C" {

moe_status_t moe_grouped_swiglu(const moe_problem_t* p, const void* x_perm, const int32_t* offsets,
                                const void* w_gate, const void* w_up, const void* w_down, void* h_perm,
                                void* y_perm, void* ws, size_t ws_bytes, void* stream) {
  if (p && is_lowp(*p)) return MOE_ERR_INVALID_ARG;
  return grouped_swiglu_impl(p, x_perm, offsets, w_gate, nullptr, w_up, nullptr, w_down, nullptr, h_perm, y_perm,
                             ws, ws_bytes, stream);
}

moe_status_t moe_grouped_swiglu_fp8(const moe_problem_t* p, const void* x_perm, const int32_t* offsets,
                                    const void* w_gate, const float* w_gate_scale, const void* w_up,
                                    const float* w_up_scale, const void* w_down, const float* w_down_scale,
                                    void* h_perm, void* y_perm, void* ws, size_t ws_bytes, void* stream) {
  if (p && !is_fp8(*p)) return MOE_ERR_INVALID_ARG;
  return grouped_swiglu_impl(p, x_perm, offsets, w_gate, w_gate_scale, w_up, w_up_scale, w_down, w_down_scale,
                             h_perm, y_perm, ws, ws_bytes, stream);
}

moe_status_t moe_grouped_swiglu_mxfp4(const moe_problem_t* p, const void* x_perm, const int32_t* offsets,
                                      const void* w_gate, const void* w_gate_bscale, const void* w_up,
                                      const void* w_up_bscale, const void* w_down, const void* w_down_bscale,
                                      void* h_perm, void* y_perm, void* ws, size_t ws_bytes, void* stream) {
  if (p && !is_mx(*p)) return MOE_ERR_INVALID_ARG;
  return grouped_swiglu_impl(p, x_perm, offsets, w_gate, w_gate_bscale, w_up, w_up_bscale, w_down,
                             w_down_bscale, h_perm, y_perm, ws, ws_bytes, stream);
}

moe_status_t moe_combine(const moe_problem_t* p, const void* y_perm, const int32_t* inv_row, const float* topk_w,
                         const void* shared_out, void* out, void* stream) {
  MOE_TRY(moe_problem_check(p));
  if (p->routing != MOE_ROUTING_TOKEN_CHOICE) return MOE_ERR_INVALID_ARG;
  if (p->T == 0) return MOE_OK;
  if (!y_perm || !inv_row || !topk_w || !out) return MOE_ERR_INVALID_ARG;
  if (!aligned16(y_perm) || !aligned16(out) || (shared_out && !aligned16(shared_out))) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_combine(p->T, p->top_k, p->d_model, static_cast<const __nv_bfloat16*>(y_perm),
                                    inv_row, topk_w, static_cast<const __nv_bfloat16*>(shared_out), 1,
                                    static_cast<__nv_bfloat16*>(out), static_cast<cudaStream_t>(stream)));
}

namespace {

moe_status_t record(cudaEvent_t* ev, int i, cudaStream_t s) {
  if (!ev) return MOE_OK;
  return cuda_status(record_event(ev[i], s));
}

moe_status_t layer_forward_impl(const moe_problem_t* p, const moe_weights_t* w, const void* hidden, void* out,
                                int32_t* topk_idx_opt, float* topk_w_opt, int32_t* counts_opt, void* ws,
                                size_t ws_bytes, cudaEvent_t* ev, void* stream) {
  MOE_TRY(moe_problem_check(p));
  if (!w || !w->w_router || !w->w_gate || !w->w_up || !w->w_down) return MOE_ERR_INVALID_ARG;
  if (p->n_shared > 0 && (!w->ws_gate || !w->ws_up || !w->ws_down)) return MOE_ERR_INVALID_ARG;
  if (w->sel_bias && p->score_fn == MOE_SCORE_SOFTMAX) return MOE_ERR_UNSUPPORTED;
  if (!aligned16(w->w_gate) || !aligned16(w->w_up) || !aligned16(w->w_down)) return MOE_ERR_INVALID_ARG;
  if (p->n_shared > 0 && (!aligned16(w->ws_gate) || !aligned16(w->ws_up) || !aligned16(w->ws_down)))
    return MOE_ERR_INVALID_ARG;
  if (p->T > 0 && (!hidden || !out || !aligned16(hidden) || !aligned16(out))) return MOE_ERR_INVALID_ARG;
  const bool fp8 = is_lowp(*p);
  if (!scales_ok(*p, w->w_gate_scale, w->w_up_scale, w->w_down_scale)) return MOE_ERR_INVALID_ARG;
  if (p->n_shared > 0 && !scales_ok(*p, w->ws_gate_scale, w->ws_up_scale, w->ws_down_scale))
    return MOE_ERR_INVALID_ARG;
  Layout L;
  MOE_TRY(check_ws(p, MOE_CALL_LAYER_FORWARD, ws, ws_bytes, &L));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t T = p->T;
  const int32_t N = p->n_experts, K = p->top_k, S = p->n_shared;
  int32_t* topk_idx = topk_idx_opt ? topk_idx_opt : at<int32_t>(ws, L.topk_idx);
  float* topk_w = topk_w_opt ? topk_w_opt : at<float>(ws, L.topk_w);
  int32_t* counts = counts_opt ? counts_opt : at<int32_t>(ws, L.counts);
  int32_t* offsets = at<int32_t>(ws, L.offsets);
  uint32_t* err = at<uint32_t>(ws, L.err);
  const bool hbf16 = p->hidden_dtype == MOE_BF16;

  if (T == 0) {  // no tokens: counts are all zero
    PermuteArgs pa{};
    pa.N = N;
    pa.K = K;
    pa.capacity = 2147483647;
    pa.chunk_counts = at<int32_t>(ws, L.chunk);
    pa.counts = counts;
    pa.offsets = offsets;
    pa.err = err;
    return cuda_status(launch_permute(pa, s));
  }

  if (p->routing == MOE_ROUTING_EXPERT_CHOICE) {
    if (topk_idx_opt || topk_w_opt) return MOE_ERR_INVALID_ARG;
    if (w->sel_bias) return MOE_ERR_UNSUPPORTED;
    if (!aligned16(w->w_router)) return MOE_ERR_INVALID_ARG;
    const int32_t C = (int32_t)ec_capacity(*p);
    const int64_t rows = (int64_t)N * C;
    // 1. router logits and per-token scores, then every expert picks its C tokens
    MOE_TRY(record(ev, 0, s));
    RouterArgs ra{T, p->d_model, N, K, p->score_fn, p->renormalize, 0, 0, hidden, w->w_router, w->router_bias,
                  nullptr, nullptr, nullptr, nullptr, at<float>(ws, L.router), at<__nv_bfloat16>(ws, L.router_w3),
                  0, 0, at<float>(ws, L.ec_scores)};
    MOE_TRY(cuda_status(launch_router(ra, hbf16, s)));
    int32_t* row_token = at<int32_t>(ws, L.ec_token);
    float* row_w = at<float>(ws, L.ec_w);
    MOE_TRY(cuda_status(launch_expert_choice_select(ra.scores_t, T, N, C, row_token, row_w, offsets,
                                                    counts_opt, s)));
    MOE_TRY(record(ev, 1, s));
    // 2. pack the picked rows (+ clear the accumulator, bf16 copy of an fp32 hidden)
    PermuteArgs pa{};
    pa.T = T;
    pa.d = p->d_model;
    pa.N = N;
    pa.K = K;
    pa.hidden = hidden;
    pa.hidden_bf16 = hbf16;
    pa.offsets = offsets;
    pa.row_token = row_token;
    pa.x_perm = fp8 ? nullptr : at<void>(ws, L.x_perm);
    pa.zero_rows = at<float>(ws, L.out_acc);
    pa.x_act = !fp8 && needs_act_copy(*p) ? at<void>(ws, L.x_act) : nullptr;
    pa.act_f16 = fp8;
    pa.err = err;
    if (fp8) set_gather_quant(&pa, ws, L, S > 0);
    MOE_TRY(cuda_status(fp8 ? launch_gather_quant(pa, rows, S > 0 ? T : 0, s) : launch_gather(pa, rows, s)));
    MOE_TRY(record(ev, 2, s));
    // 3. GEMM schedule over the N full expert groups and the shared experts
    const int32_t tile_rows = gemm_tile_rows(*p, rows);
    const int32_t pair = tile_rows == 2 * kBM ? 2 : 1;
    ScheduleArgs sa{N, S, p->ffn, p->shared_ffn, p->d_model, tile_rows, T, offsets,
                    at<GroupDesc>(ws, L.groups), at<int32_t>(ws, L.ts_gu), at<int32_t>(ws, L.ts_dn)};
    MOE_TRY(cuda_status(launch_schedule(sa, s)));
    MOE_TRY(record(ev, 3, s));
    // 4-5. grouped SwiGLU GEMMs; the down epilogue adds S[t][e] * y to the row's token
    GemmPlan g{};
    g.pair = pair;
    g.N = N;
    g.S = S;
    g.F = p->ffn;
    g.Fs = p->shared_ffn;
    g.d = p->d_model;
    g.K = K;
    g.T = T;
    g.routed_rows = rows;
    g.x_routed = pa.x_perm;
    g.x_shared = pa.x_act ? pa.x_act : hidden;
    g.wg = w->w_gate;
    g.wu = w->w_up;
    g.wd = w->w_down;
    g.sg = w->ws_gate;
    g.su = w->ws_up;
    g.sd = w->ws_down;
  g.fp8 = fp8;
  g.wg_scale = w->w_gate_scale;
  g.wu_scale = w->w_up_scale;
  g.wd_scale = w->w_down_scale;
  g.sg_scale = w->ws_gate_scale;
  g.su_scale = w->ws_up_scale;
  g.sd_scale = w->ws_down_scale;
  g.mx = is_mx(*p);
  g.offsets = offsets;
  if (g.mx) set_mx_plan(&g, *p, w, ws, L, S > 0);
  if (fp8) {
    g.x_quantized = true;  // by the gather
    g.xq = at<uint8_t>(ws, L.xq);
    g.sx = at<float>(ws, L.sx);
    g.hq = at<uint8_t>(ws, L.hq);
    g.sh = at<float>(ws, L.sh);
    if (S > 0) {
      g.xq_sh = at<uint8_t>(ws, L.xq_sh);
      g.sx_sh = at<float>(ws, L.sx_sh);
      g.hq_sh = at<uint8_t>(ws, L.hq_sh);
      g.sh_sh = at<float>(ws, L.sh_sh);
    }
  }
    g.h = at<__nv_bfloat16>(ws, L.h);
    g.h_sh = S > 0 ? at<__nv_bfloat16>(ws, L.h_sh) : nullptr;
    g.epilogue = kEpiScatter;
    g.out_acc = at<float>(ws, L.out_acc);
    g.perm_src = row_token;
    g.row_w = row_w;
    g.groups = at<GroupDesc>(ws, L.groups);
    g.ts_gu = at<int32_t>(ws, L.ts_gu);
    g.ts_dn = at<int32_t>(ws, L.ts_dn);
    g.err = err;
    MOE_TRY(run_gemms(g, s, ev ? ev + 4 : nullptr));
    MOE_TRY(cuda_status(launch_finalize(g.out_acc, static_cast<__nv_bfloat16*>(out), T * p->d_model, s)));
    return record(ev, 6, s);
  }

  if (decode_fused(*p)) {
    // decode-sized batch: the whole layer in one cooperative kernel
    if (!aligned16(w->w_router)) return MOE_ERR_INVALID_ARG;
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (sms > kDecodeMaxGrid) sms = kDecodeMaxGrid;
    const DecodePlan pl = decode_plan(*p, sms);
    if (!pl.ok) return MOE_ERR_UNSUPPORTED;
    DecodeArgs da{};
    da.T = T;
    da.d = p->d_model;
    da.N = N;
    da.K = K;
    da.F = p->ffn;
    da.S = S;
    da.Fs = p->shared_ffn;
    da.score_fn = p->score_fn;
    da.renormalize = p->renormalize;
    da.n_groups = p->n_groups;
    da.topk_groups = p->topk_groups;
    da.capacity = expert_capacity(*p);
    da.fmt = is_fp8(*p) ? kDecodeE4M3 : kDecodeBf16;
    da.hidden = hidden;
    da.hidden_bf16 = hbf16;
    da.w_router = w->w_router;
    da.router_bias = w->router_bias;
    da.sel_bias = w->sel_bias;
    da.w_gate = w->w_gate;
    da.w_up = w->w_up;
    da.w_down = w->w_down;
    da.s_gate = w->ws_gate;
    da.s_up = w->ws_up;
    da.s_down = w->ws_down;
    da.w_gate_scale = w->w_gate_scale;
    da.w_up_scale = w->w_up_scale;
    da.w_down_scale = w->w_down_scale;
    da.s_gate_scale = w->ws_gate_scale;
    da.s_up_scale = w->ws_up_scale;
    da.s_down_scale = w->ws_down_scale;
    da.out = static_cast<__nv_bfloat16*>(out);
    da.topk_idx = topk_idx;
    da.topk_w = topk_w;
    da.counts = counts;
    da.router_part = at<float>(ws, L.dec_part);
    da.h = at<void>(ws, L.dec_h);
    da.h_sh = S > 0 ? at<void>(ws, L.dec_h_sh) : nullptr;
    da.bnd_val = at<float>(ws, L.dec_bnd_val);
    da.bnd_cnt = at<uint32_t>(ws, L.dec_bnd_cnt);
    da.ybuf = at<float>(ws, L.dec_ybuf);
    da.blk_cnt = at<uint32_t>(ws, L.dec_blk);
    da.sync = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(ws) + L.err + kDecodeSyncOffset);
    da.err = err;
    da.grid = pl.grid;
    da.rsplits = pl.rsplits;
    da.r_slice = pl.r_slice;
    da.x_stride = pl.x_stride;
    da.z_len = pl.z_len;
    da.h_stride = pl.h_stride;
    da.hs_stride = pl.hs_stride;
    da.hsm_stride = pl.hsm_stride;
    da.smem_x_bytes = pl.smem_x_bytes;
    da.smem_bytes = pl.smem_bytes;
    MOE_TRY(record(ev, 0, s));
    MOE_TRY(cuda_status(launch_decode_layer(da, s)));
    for (int i = 1; i <= 6; ++i) MOE_TRY(record(ev, i, s));
    return MOE_OK;
  }

  // 1. router, scoring, top-K, gate weights
  MOE_TRY(record(ev, 0, s));
  if (!aligned16(w->w_router)) return MOE_ERR_INVALID_ARG;
  RouterArgs ra{T, p->d_model, N, K, p->score_fn, p->renormalize, p->n_groups, p->topk_groups, hidden, w->w_router,
                w->router_bias, w->sel_bias, topk_idx, topk_w, nullptr, at<float>(ws, L.router),
                at<__nv_bfloat16>(ws, L.router_w3), 0, 0};
  MOE_TRY(cuda_status(launch_router(ra, hbf16, s)));
  MOE_TRY(record(ev, 1, s));

  // 2. route and pack (+ clear the fp32 accumulator, + bf16 copy of an fp32 hidden for shared experts)
  PermuteArgs pa{};
  pa.T = T;
  pa.d = p->d_model;
  pa.N = N;
  pa.K = K;
  pa.C = (int32_t)((T + kTokensPerChunk - 1) / kTokensPerChunk);
  pa.capacity = expert_capacity(*p);
  pa.topk_idx = topk_idx;
  pa.hidden = hidden;
  pa.hidden_bf16 = hbf16;
  pa.chunk_counts = at<int32_t>(ws, L.chunk);
  pa.counts = counts;
  pa.offsets = offsets;
  pa.perm_src = at<int32_t>(ws, L.perm_src);
  pa.inv_row = at<int32_t>(ws, L.inv_row);
  const bool combine = stored_combine(*p);
  pa.x_perm = fp8 ? nullptr : at<void>(ws, L.x_perm);
  pa.zero_rows = combine ? nullptr : at<float>(ws, L.out_acc);
  pa.x_act = !fp8 && needs_act_copy(*p) ? at<void>(ws, L.x_act) : nullptr;
  pa.act_f16 = fp8;
  pa.err = err;
  if (fp8) set_gather_quant(&pa, ws, L, S > 0);
  // 3. the GEMM schedule (routed experts from offsets, then the shared
  //    experts) is built by the same kernel that finishes the prefix sums
  const int32_t tile_rows = gemm_tile_rows(*p, T * K);
  const int32_t pair = tile_rows == 2 * kBM ? 2 : 1;
  pa.groups = at<GroupDesc>(ws, L.groups);
  pa.ts_gu = at<int32_t>(ws, L.ts_gu);
  pa.ts_dn = at<int32_t>(ws, L.ts_dn);
  pa.S = S;
  pa.F = p->ffn;
  pa.Fs = p->shared_ffn;
  pa.tile_rows = tile_rows;
  MOE_TRY(cuda_status(launch_permute(pa, s)));
  MOE_TRY(record(ev, 2, s));
  MOE_TRY(record(ev, 3, s));

  // 4-5. grouped SwiGLU GEMMs with the fused weighted scatter-add
  GemmPlan g{};
  g.pair = pair;
  g.N = N;
  g.S = S;
  g.F = p->ffn;
  g.Fs = p->shared_ffn;
  g.d = p->d_model;
  g.K = K;
  g.T = T;
  g.routed_rows = T * K;
  g.x_routed = pa.x_perm;
  g.x_shared = pa.x_act ? pa.x_act : hidden;
  g.wg = w->w_gate;
  g.wu = w->w_up;
  g.wd = w->w_down;
  g.sg = w->ws_gate;
  g.su = w->ws_up;
  g.sd = w->ws_down;
  g.fp8 = fp8;
  g.wg_scale = w->w_gate_scale;
  g.wu_scale = w->w_up_scale;
  g.wd_scale = w->w_down_scale;
  g.sg_scale = w->ws_gate_scale;
  g.su_scale = w->ws_up_scale;
  g.sd_scale = w->ws_down_scale;
  g.mx = is_mx(*p);
  g.offsets = offsets;
  if (g.mx) set_mx_plan(&g, *p, w, ws, L, S > 0);
  if (fp8) {
    g.x_quantized = true;  // by the gather
    g.xq = at<uint8_t>(ws, L.xq);
    g.sx = at<float>(ws, L.sx);
    g.hq = at<uint8_t>(ws, L.hq);
    g.sh = at<float>(ws, L.sh);
    if (S > 0) {
      g.xq_sh = at<uint8_t>(ws, L.xq_sh);
      g.sx_sh = at<float>(ws, L.sx_sh);
      g.hq_sh = at<uint8_t>(ws, L.hq_sh);
      g.sh_sh = at<float>(ws, L.sh_sh);
    }
  }
  g.h = at<__nv_bfloat16>(ws, L.h);
  g.h_sh = S > 0 ? at<__nv_bfloat16>(ws, L.h_sh) : nullptr;
  g.epilogue = combine ? kEpiStoreY : kEpiScatter;
  g.out_acc = at<float>(ws, L.out_acc);
  if (combine) {
    g.y = at<__nv_bfloat16>(ws, L.y_rows);
    g.y_sh = S > 0 ? at<__nv_bfloat16>(ws, L.y_sh) : nullptr;
  }
  g.perm_src = pa.perm_src;
  g.topk_w = topk_w;
  g.groups = at<GroupDesc>(ws, L.groups);
  g.ts_gu = at<int32_t>(ws, L.ts_gu);
  g.ts_dn = at<int32_t>(ws, L.ts_dn);
  g.err = err;
  MOE_TRY(run_gemms(g, s, ev ? ev + 4 : nullptr));

  // 6. fp32 -> bf16, or the gate-weighted sum of the stored rows
  if (combine)
    MOE_TRY(cuda_status(launch_combine(T, K, p->d_model, g.y, pa.inv_row, topk_w, g.y_sh, S,
                                       static_cast<__nv_bfloat16*>(out), s)));
  else
    MOE_TRY(cuda_status(launch_finalize(g.out_acc, static_cast<__nv_bfloat16*>(out), T * p->d_model, s)));
  return record(ev, 6, s);
}

}  // namespace

moe_status_t moe_layer_forward(const moe_problem_t* p, const moe_weights_t* w, const void* hidden, void* out,
                               int32_t* topk_idx_opt, float* topk_w_opt, int32_t* counts_opt, void* ws,
                               size_t ws_bytes, void* stream) {
  return layer_forward_impl(p, w, hidden, out, topk_idx_opt, topk_w_opt, counts_opt, ws, ws_bytes, nullptr,
                            stream);
}

moe_status_t moe_layer_forward_profiled(const moe_problem_t* p, const moe_weights_t* w, const void* hidden,
                                        void* out, void* ws, size_t ws_bytes, void* const* stage_events,
                                        void* stream) {
  if (!stage_events) return MOE_ERR_INVALID_ARG;
  cudaEvent_t ev[MOE_LAYER_STAGES + 1];
  for (int i = 0; i <= MOE_LAYER_STAGES; ++i) {
    if (!stage_events[i]) return MOE_ERR_INVALID_ARG;
    ev[i] = static_cast<cudaEvent_t>(stage_events[i]);
  }
  return layer_forward_impl(p, w, hidden, out, nullptr, nullptr, nullptr, ws, ws_bytes, ev, stream);
}

size_t moe_mxfp4_prep_bytes(const moe_problem_t* p) {
  if (moe_problem_check(p) != MOE_OK || !is_mx(*p)) return 0;
  size_t total = 0;
  prep_offsets(*p, &total);
  return total;
}

moe_status_t moe_mxfp4_prepare(const moe_problem_t* p, const moe_weights_t* w, void* prep, size_t prep_bytes,
                               void* stream) {
  MOE_TRY(moe_problem_check(p));
  if (!is_mx(*p) || !w || !prep) return MOE_ERR_INVALID_ARG;
  const bool sh = p->n_shared > 0;
  if (!w->w_gate_scale || !w->w_up_scale || !w->w_down_scale) return MOE_ERR_INVALID_ARG;
  if (sh && (!w->ws_gate_scale || !w->ws_up_scale || !w->ws_down_scale)) return MOE_ERR_INVALID_ARG;
  size_t total = 0;
  const MxOffsets o = prep_offsets(*p, &total);
  if ((reinterpret_cast<uintptr_t>(prep) & 255u) != 0 || prep_bytes < total) return MOE_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  auto u8 = [](const void* q) { return static_cast<const uint8_t*>(q); };
  const int32_t d = p->d_model, F = p->ffn, Fs = p->shared_ffn;
  const int32_t kb_d = (d + 127) / 128, kb_f = (F + 127) / 128, kb_fs = (Fs + 127) / 128;
  const int64_t nf = (int64_t)p->n_experts * F, nd = (int64_t)p->n_experts * d;
  MOE_TRY(cuda_status(launch_mx_prep(u8(w->w_gate_scale), nf, F, d / 32, kb_d, nullptr, at<float>(prep, o.rs_gate),
                                     at<uint32_t>(prep, o.ki_gate), s)));
  MOE_TRY(cuda_status(launch_mx_prep(u8(w->w_up_scale), nf, F, d / 32, kb_d, nullptr, at<float>(prep, o.rs_up),
                                     at<uint32_t>(prep, o.ki_up), s)));
  MOE_TRY(cuda_status(launch_mx_prep(u8(w->w_down_scale), nd, d, F / 32, kb_f, nullptr, at<float>(prep, o.rs_down),
                                     at<uint32_t>(prep, o.ki_down), s)));
  if (sh) {
    const int64_t sf = (int64_t)p->n_shared * Fs, sd = (int64_t)p->n_shared * d;
    MOE_TRY(cuda_status(launch_mx_prep(u8(w->ws_gate_scale), sf, Fs, d / 32, kb_d, nullptr,
                                       at<float>(prep, o.rs_sgate), at<uint32_t>(prep, o.ki_sgate), s)));
    MOE_TRY(cuda_status(launch_mx_prep(u8(w->ws_up_scale), sf, Fs, d / 32, kb_d, nullptr,
                                       at<float>(prep, o.rs_sup), at<uint32_t>(prep, o.ki_sup), s)));
    MOE_TRY(cuda_status(launch_mx_prep(u8(w->ws_down_scale), sd, d, Fs / 32, kb_fs, nullptr,
                                       at<float>(prep, o.rs_sdown), at<uint32_t>(prep, o.ki_sdown), s)));
  }
  return MOE_OK;
}

int32_t moe_layer_forward_kernel_count(const moe_problem_t* p, const moe_weights_t* w) {
  if (moe_problem_check(p) != MOE_OK) return 0;
  if (p->T == 0) return 1;  // the histogram scan that writes zero counts
  // route and pack: histogram, scan (+ schedule), scatter -- one kernel for at
  // most 32 chunks of 32 tokens -- then the gather; gate/up GEMM, down GEMM, finalise
  // router: split + router GEMM (tensor-core logits) or one CUDA-core logits
  // kernel, then top-K
  const int router = router_plan(p->T, p->d_model, p->n_experts, p->hidden_dtype == MOE_BF16).tensor ? 3 : 2;
  // FP8 / MXFP4 experts: the two-term E4M3 split of the down GEMM's
  // activations h (and the shared experts' h); x's is folded into the gather
  // (+ MXFP4 without a prepared buffer: the preparation of gate, up and
  // down, and of the shared experts')
  const bool prep = is_mx(*p) && !(w && w->mx_prep);
  const int quant = (is_lowp(*p) ? (p->n_shared > 0 ? 2 : 1) : 0) + (prep ? (p->n_shared > 0 ? 6 : 3) : 0);
  if (p->routing == MOE_ROUTING_EXPERT_CHOICE) return router + 3 + 3 + quant;  // + select, gather, schedule
  const int route = (p->T + kTokensPerChunk - 1) / kTokensPerChunk <= 32 ? 2 : 4;
  // routing without the row copy; gate/up and down (+ finalise) on the CUDA cores
  if (decode_fused(*p)) return 1;  // the whole layer in one kernel

  return router + route + 3 + quant;
}

int32_t moe_layer_small_batch(const moe_problem_t* p) {
  if (moe_problem_check(p) != MOE_OK) return -1;
  return decode_fused(*p) ? 1 : 0;
}

moe_status_t moe_get_device_status(void* ws, void* stream) {
  if (!ws) return MOE_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  uint32_t word = 0;
  if (cudaMemcpy(&word, ws, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  if (word != 0) {
    if (cudaMemsetAsync(ws, 0, sizeof word, s) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  }
  if (word & kErrTimeout) return MOE_ERR_TIMEOUT;
  if (word & kErrBounds) return MOE_ERR_DEVICE_BOUNDS;
  if (word & kErrRange) return MOE_ERR_RANGE;
  return MOE_OK;
}

}  // extern "C"
