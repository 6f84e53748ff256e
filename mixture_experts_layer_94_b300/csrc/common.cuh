// common.cuh — shared device helpers of libmoe (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

// Bits of the device error word (first 4 bytes of every workspace).
constexpr uint32_t kErrTimeout = 1u;  // a bounded pipeline wait gave up
constexpr uint32_t kErrBounds = 2u;   // an input index was out of range
constexpr uint32_t kErrRange = 4u;    // an fp16 activation (FP8-weight experts) overflowed

// Bound on any single pipeline wait. The longest legitimate wait in this
// library is one output tile of MMA work (well under a millisecond), so two
// seconds only ever trips on a genuine stall.
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;

constexpr int kTokensPerChunk = 32;  // route-and-pack chunk: one warp, one token per lane
constexpr int kMaxExperts = 256;
constexpr int kMaxTopK = 32;
constexpr int kMaxShared = 8;

// GEMM tiling shared by host and device.
constexpr int kBM = 128;        // rows of the activation tile (MMA M)
constexpr int kBK = 64;         // K elements per pipeline stage (128 B of bf16 = one swizzle atom)
// Router GEMM: the three bf16 parts of the router matrix share a tile when
// their columns (3 x np rows of 128 B) fit the 32 KB B stage of a 1-CTA tile.
constexpr int kRouterMergedMaxNp = 80;
static_assert(3 * kRouterMergedMaxNp * kBK * 2 <= 256 * kBK * 2, "merged router parts exceed a 1-CTA B stage");
static_assert(kRouterMergedMaxNp % 16 == 0, "each part's rows must start on a 1 KB swizzle atom");
constexpr int kBNGateUp = 128;  // gate columns per tile (the up tile adds another 128 -> MMA N = 256)
constexpr int kBNDown = 256;    // output columns per down-projection tile (MMA N = 256)

// One GEMM group: a routed expert (kind 0) or a shared expert (kind 1).
struct GroupDesc {
  int32_t kind;       // 0 routed, 1 shared
  int32_t index;      // expert index within its kind
  int32_t a_row0;     // first row of the group in its activation matrix
  int32_t rows;       // rows of the group
  int32_t m_tiles;    // ceil(rows / kBM)
  int32_t h_row0;     // first row in the group's h / y matrix
  // Tile order of the group in the gate/up GEMM: 0 m fastest (the tiles of
  // one weight column block run together), 1 n fastest (the tiles of one row
  // block run together: for a group whose rows outweigh its weights, so that
  // each row block is read from DRAM once). The down GEMM runs m fastest.
  int32_t order_gu;
  int32_t pad;
};

// Programmatic dependent launch. Every kernel of the library is launched with
// programmatic stream serialisation (launch() below): the next kernel in the
// stream may start once every CTA of this one has called pdl_trigger(), and
// it runs only its own setup until pdl_wait() returns, which is when the
// previous grid has completed and its memory writes are visible. Every kernel
// calls pdl_wait() before its first global-memory access and before any exit,
// so a grid completes only after its predecessor did and the chain stays
// transitive (a kernel may read what any earlier kernel of the stream wrote).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Launches kern<<<grid, block, smem, s>>>(args...) with programmatic stream
// serialisation (see pdl_wait); `extra` adds one more launch attribute (a
// cluster shape) when its id is not cudaLaunchAttributeIgnore.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_attr(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                               const cudaLaunchAttribute& extra, Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (extra.id != cudaLaunchAttributeIgnore) attr[cfg.numAttrs++] = extra;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                          Args&&... args) {
  cudaLaunchAttribute none{};
  none.id = cudaLaunchAttributeIgnore;
  return launch_attr(kern, grid, block, smem, s, none, static_cast<Args&&>(args)...);
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + __expf(-z)); }

}  // namespace moe
