// Router of the MoE layer: fp32 logits, sigmoid gate scores, noaux_tc grouped top-k
// selection and renormalised combine weights (the DeepSeek-V3-style sigmoid router with
// noaux_tc and routed_scaling_factor of "Show HN: Menjalankan GLM 5.2 di komputer lambat",
// section "Fitur utama yang diimplementasikan").
#include <math.h>

#include "kernels.h"
#include "route_dev.cuh"

namespace moe {

namespace {

constexpr int kRouterThreads = 256;
constexpr int kRouterTokens = 8;   // tokens per CTA in the logits kernel

template <int XDT, int WDT>
__global__ void __launch_bounds__(kRouterThreads)
router_logits_kernel(const void* __restrict__ x, const void* __restrict__ wr,
                     float* __restrict__ logits, int T, int E, int H) {
  const int e = blockIdx.x;
  const int t0 = blockIdx.y * kRouterTokens;
  const int nt = min(kRouterTokens, T - t0);
  float acc[kRouterTokens];
#pragma unroll
  for (int i = 0; i < kRouterTokens; ++i) acc[i] = 0.f;
  for (int h = threadIdx.x; h < H; h += kRouterThreads) {
    const float w = load_act<WDT>(wr, (size_t)e * H + h);
#pragma unroll
    for (int i = 0; i < kRouterTokens; ++i)
      if (i < nt) acc[i] = fmaf(w, load_act<XDT>(x, (size_t)(t0 + i) * H + h), acc[i]);
  }
  __shared__ float red[kRouterTokens][kRouterThreads / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int i = 0; i < kRouterTokens; ++i) {
    float v = acc[i];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) red[i][warp] = v;
  }
  __syncthreads();
  if (threadIdx.x < nt) {
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < kRouterThreads / 32; ++w) v += red[threadIdx.x][w];
    logits[(size_t)(t0 + threadIdx.x) * E + e] = v;
  }
}

constexpr int kSelWarps = 4;
constexpr int kMaxE = 1024;

// One warp per token.
__global__ void __launch_bounds__(kSelWarps * 32)
select_kernel(const float* __restrict__ logits, const float* __restrict__ bias, int T, int E,
              int n_group, int topk_group, int top_k, float rsf, int32_t* __restrict__ ids,
              float* __restrict__ weights, int32_t* __restrict__ counts, int* status) {
  __shared__ float sb[kSelWarps][kMaxE];   // biased scores; -inf once taken or excluded
  __shared__ float ss[kSelWarps][kMaxE];   // unbiased sigmoid scores
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kSelWarps + warp;
  if (t >= T) return;
  const int id = select_token(logits + (size_t)t * E, bias, E, n_group, topk_group, top_k, rsf,
                              sb[warp], ss[warp], ids + (size_t)t * top_k,
                              weights + (size_t)t * top_k, status);
  if (lane < top_k) atomicAdd(&counts[id], 1);
}

}  // namespace

cudaError_t launch_router_logits(const void* x, int act_dtype, const void* router_w,
                                 int router_dtype, float* logits, int T, int E, int H,
                                 cudaStream_t s) {
  dim3 grid(E, (T + kRouterTokens - 1) / kRouterTokens);
  if (act_dtype == MOE_DT_F32 && router_dtype == MOE_DT_F32)
    router_logits_kernel<MOE_DT_F32, MOE_DT_F32><<<grid, kRouterThreads, 0, s>>>(x, router_w, logits, T, E, H);
  else if (act_dtype == MOE_DT_BF16 && router_dtype == MOE_DT_F32)
    router_logits_kernel<MOE_DT_BF16, MOE_DT_F32><<<grid, kRouterThreads, 0, s>>>(x, router_w, logits, T, E, H);
  else if (act_dtype == MOE_DT_F32 && router_dtype == MOE_DT_BF16)
    router_logits_kernel<MOE_DT_F32, MOE_DT_BF16><<<grid, kRouterThreads, 0, s>>>(x, router_w, logits, T, E, H);
  else
    router_logits_kernel<MOE_DT_BF16, MOE_DT_BF16><<<grid, kRouterThreads, 0, s>>>(x, router_w, logits, T, E, H);
  return cudaGetLastError();
}

cudaError_t launch_select(const float* logits, const float* bias, int T, int E, int n_group,
                          int topk_group, int top_k, float rsf, int32_t* ids, float* weights,
                          int32_t* counts, int* status, cudaStream_t s) {
  if (E > kMaxE || n_group > 32 || top_k > 32) return cudaErrorInvalidValue;
  select_kernel<<<(T + kSelWarps - 1) / kSelWarps, kSelWarps * 32, 0, s>>>(
      logits, bias, T, E, n_group, topk_group, top_k, rsf, ids, weights, counts, status);
  return cudaGetLastError();
}

}  // namespace moe
