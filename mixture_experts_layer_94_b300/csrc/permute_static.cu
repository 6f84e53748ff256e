// permute_static.cu — route and pack for callers that cannot allocate device
// memory.
//
// Some callers of this library are not allowed to allocate GPU memory on the
// path that routes tokens: an inference server that reserves all device memory
// up front and accounts for every byte, a plug-in that runs inside a host
// framework which owns the allocator, or a latency-critical loop where
// cudaMalloc's implicit device synchronisation and unpredictable cost are not
// acceptable. moe_permute needs a caller-provided workspace for its per-chunk
// expert counts; this variant keeps that scratch in a fixed array compiled into
// the library instead, so the caller passes only inputs and outputs.
//
// The array below is reserved on every GPU that loads the library and stays
// there until the process exits. Every call on a device uses the same array.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/moe.h"
#include "common.cuh"
#include "kernels.h"

namespace {

// Word 0 is the device error word the route-and-pack kernels report into; the
// per-chunk counts start 256 bytes in, keeping them 256-byte aligned.
constexpr int kErrWords = 64;
static __device__ __align__(256) int32_t g_permute_scratch[kErrWords + MOE_PERMUTE_STATIC_MAX_CHUNK_COUNTS];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
struct ScratchAddr {
  CUcontext ctx;  // the context the address was looked up in
  void* addr;
};
ScratchAddr g_scratch_addr[kMaxDevices];

// cuCtxGetCurrent through the runtime's driver entry point (no libcuda link).
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<CtxGetCurrentFn>(nullptr);
    return reinterpret_cast<CtxGetCurrentFn>(f);
  }();
  return fn;
}

// The device address of g_permute_scratch on `dev`. In host code the array's
// name is only a host-side stand-in, so the address is looked up with the
// device current and cached per device, together with the context it was
// looked up in; a call from another context (a non-primary context on the
// same device) looks it up again. Runs after the caller's cudaGetDevice, so
// the device's primary context is current unless the caller made another one
// current.
moe_status_t scratch_address(int dev, void** out) {
  CtxGetCurrentFn get = ctx_get_current();
  CUcontext ctx = nullptr;
  if (!get || get(&ctx) != CUDA_SUCCESS) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  ScratchAddr& c = g_scratch_addr[dev];
  if (!c.addr || c.ctx != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_permute_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
    c.addr = p;
    c.ctx = ctx;
  }
  *out = c.addr;
  return MOE_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" moe_status_t moe_permute_static(const moe_problem_t* p, const int32_t* topk_idx, const void* hidden,
                                           int32_t* counts, int32_t* offsets, int32_t* perm_src, int32_t* inv_row,
                                           void* x_perm, void* stream) {
  const moe_status_t st = moe_problem_check(p);
  if (st != MOE_OK) return st;
  if (p->routing != MOE_ROUTING_TOKEN_CHOICE) return MOE_ERR_INVALID_ARG;
  const int64_t chunks = (p->T + moe::kTokensPerChunk - 1) / moe::kTokensPerChunk;
  if ((int64_t)p->n_experts * chunks > MOE_PERMUTE_STATIC_MAX_CHUNK_COUNTS) return MOE_ERR_UNSUPPORTED;
  if (!counts || !offsets) return MOE_ERR_INVALID_ARG;
  if (p->T > 0 && (!topk_idx || !hidden || !perm_src || !inv_row || !x_perm)) return MOE_ERR_INVALID_ARG;
  if (p->T > 0 && (!aligned16(hidden) || !aligned16(x_perm))) return MOE_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
  void* base = nullptr;
  const moe_status_t sa = scratch_address(dev, &base);
  if (sa != MOE_OK) return sa;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The error word must start at zero; the counts need no clearing (every
  // entry the kernels read is written earlier in the same call).
  if (cudaMemsetAsync(base, 0, sizeof(uint32_t), s) != cudaSuccess) return MOE_ERR_CUDA;
  moe::PermuteArgs a{};
  a.T = p->T;
  a.d = p->d_model;
  a.N = p->n_experts;
  a.K = p->top_k;
  a.C = (int32_t)chunks;
  a.capacity = moe::expert_capacity(*p);
  a.topk_idx = topk_idx;
  a.hidden = hidden;
  a.hidden_bf16 = p->hidden_dtype == MOE_BF16;
  a.chunk_counts = static_cast<int32_t*>(base) + kErrWords;
  a.counts = counts;
  a.offsets = offsets;
  a.perm_src = perm_src;
  a.inv_row = inv_row;
  a.x_perm = x_perm;
  // FP8 and MXFP4 experts read fp16 packed rows, bf16 experts bf16 ones
  // (the rows moe_permute writes for the same problem).
  a.act_f16 = p->expert_dtype == MOE_EXPERT_FP8_E4M3 || p->expert_dtype == MOE_EXPERT_MXFP4;
  a.err = static_cast<uint32_t*>(base);
  return moe::launch_permute(a, s) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
