// combine.cu — back to token order.
//
// finalize: out = bf16(out_acc), the last step of the fused layer whose
//   down-projection epilogue already scatter-added w_{t,k} * y into out_acc.
// combine:  the deterministic gate-weighted sum ("Chapter 19:
//   Mixture-of-Experts Models", §19.3.2 and the §19.2 flowchart "Sum with gate
//   weights"): out[t] = bf16(sum_k w[t][k] * y_perm[inv_row[t*K+k]] +
//   sum_s shared[s][t]), fp32 accumulation in slot order, then shared expert
//   order. The step-wise API's last step, and the fused layer's when its fp32
//   accumulator would not fit in L2 (the down epilogue then stores rows).
// Both are HBM-bound streams: 16-byte vector loads and stores, one thread per
// 8 output elements, grid-stride over the whole output.
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

__global__ void __launch_bounds__(256) finalize_kernel(const float* __restrict__ acc,
                                                       __nv_bfloat16* __restrict__ out, int64_t nvec) {
  pdl_trigger();
  pdl_wait();
  for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < nvec; v += (int64_t)gridDim.x * blockDim.x) {
    const float4 a = reinterpret_cast<const float4*>(acc)[2 * v];
    const float4 b = reinterpret_cast<const float4*>(acc)[2 * v + 1];
    reinterpret_cast<uint4*>(out)[v] =
        make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w), pack_bf16x2(b.x, b.y), pack_bf16x2(b.z, b.w));
  }
}

__device__ __forceinline__ void add_bf16x8(float (&acc)[8], const uint4 v, float w) {
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&u[j]);
    const float2 f = __bfloat1622float2(b);
    acc[2 * j] = fmaf(w, f.x, acc[2 * j]);
    acc[2 * j + 1] = fmaf(w, f.y, acc[2 * j + 1]);
  }
}

__global__ void __launch_bounds__(256) combine_kernel(int64_t T, int32_t K, int32_t d,
                                                      const __nv_bfloat16* __restrict__ y_perm,
                                                      const int32_t* __restrict__ inv_row,
                                                      const float* __restrict__ topk_w,
                                                      const __nv_bfloat16* __restrict__ shared_out, int32_t S,
                                                      __nv_bfloat16* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  const int64_t vpr = d / 8;  // 16-byte vectors per row
  const int64_t total = T * vpr;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = i / vpr, v = i - t * vpr;
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.f;
    // Four slots' rows in flight at a time; the sum stays in slot order.
    for (int k0 = 0; k0 < K; k0 += 4) {
      uint4 y[4];
      float w[4];
      bool ok[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int k = k0 + j;
        const int64_t r = k < K ? __ldg(inv_row + t * K + k) : -1;
        ok[j] = r >= 0;  // r < 0: dropped by its expert's capacity
        if (ok[j]) {
          w[j] = __ldg(topk_w + t * K + k);
          y[j] = reinterpret_cast<const uint4*>(y_perm + r * d)[v];
        }
      }
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (ok[j]) add_bf16x8(acc, y[j], w[j]);
    }
    for (int sx = 0; sx < S; ++sx)
      add_bf16x8(acc, reinterpret_cast<const uint4*>(shared_out + ((int64_t)sx * T + t) * d)[v], 1.f);
    reinterpret_cast<uint4*>(out + t * d)[v] =
        make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]),
                   pack_bf16x2(acc[6], acc[7]));
  }
}

int grid_for(int64_t work, int threads) {
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t blocks = (work + threads - 1) / threads;
  const int64_t cap = (int64_t)sms * 8;
  return (int)(blocks < cap ? (blocks < 1 ? 1 : blocks) : cap);
}

}  // namespace

cudaError_t launch_finalize(const float* acc, __nv_bfloat16* out, int64_t n, cudaStream_t s) {
  const int64_t nvec = n / 8;
  if (nvec == 0) return cudaSuccess;
  if (const cudaError_t le_ = launch(finalize_kernel, grid_for(nvec, 256), 256, 0, s, acc, out, nvec); le_ != cudaSuccess) return le_;
  return cudaSuccess;
}

cudaError_t launch_combine(int64_t T, int32_t K, int32_t d, const __nv_bfloat16* y_perm, const int32_t* inv_row,
                           const float* topk_w, const __nv_bfloat16* shared_out, int32_t S, __nv_bfloat16* out,
                           cudaStream_t s) {
  const int64_t work = T * (d / 8);
  if (work == 0) return cudaSuccess;
  return launch(combine_kernel, grid_for(work, 256), 256, 0, s, T, K, d, y_perm, inv_row, topk_w, shared_out,
                shared_out ? S : 0, out);
}

}  // namespace moe
