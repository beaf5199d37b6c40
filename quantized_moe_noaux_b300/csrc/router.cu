// Router of the MoE layer: fp32 logits, sigmoid gate scores, noaux_tc grouped top-k
// selection and renormalised combine weights (the DeepSeek-V3-style sigmoid router with
// noaux_tc and routed_scaling_factor of "Show HN: Menjalankan GLM 5.2 di komputer lambat",
// section "Fitur utama yang diimplementasikan").
#include <math.h>

#include "kernels.h"

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

// Warp-wide argmax of (value, index): larger value wins, equal values go to the lower index.
__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int oi = __shfl_xor_sync(0xffffffffu, i, o);
    if (ov > v || (ov == v && oi < i)) {
      v = ov;
      i = oi;
    }
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
  float* b = sb[warp];
  float* s = ss[warp];
  for (int e = lane; e < E; e += 32) {
    const float sc = sigmoidf_acc(logits[(size_t)t * E + e]);
    s[e] = sc;
    b[e] = sc + bias[e];
  }
  __syncwarp();
  // group score: sum of the two largest biased scores of the group
  const int G = E / n_group;
  float gscore = -INFINITY;
  if (lane < n_group) {
    float m1 = -INFINITY, m2 = -INFINITY;
    for (int i = 0; i < G; ++i) {
      const float v = b[lane * G + i];
      if (v > m1) {
        m2 = m1;
        m1 = v;
      } else if (v > m2) {
        m2 = v;
      }
    }
    gscore = m1 + m2;
  }
  // keep the topk_group best groups (ties -> lower group index)
  unsigned kept = 0;
  for (int r = 0; r < topk_group; ++r) {
    float v = gscore;
    int gi = lane < n_group ? lane : 0x7fffffff;
    warp_argmax(v, gi);
    kept |= 1u << gi;
    if (lane == gi) gscore = -INFINITY;
  }
  // top_k experts among kept groups (ties -> lower expert index)
  float wsum = 0.f;
  int my_id = -1;
  float my_s = 0.f;
  for (int j = 0; j < top_k; ++j) {
    float v = -INFINITY;
    int vi = 0x7fffffff;
    for (int e = lane; e < E; e += 32) {
      const float be = ((kept >> (e / G)) & 1u) ? b[e] : -INFINITY;
      if (be > v) {
        v = be;
        vi = e;
      }
    }
    warp_argmax(v, vi);
    if (vi < 0 || vi >= E) {   // fewer candidates than top_k: host validation forbids it
      raise_status(status, MOE_ERR_DEVICE_CHECK);
      vi = 0;
    }
    const float sv = s[vi];
    wsum += sv;
    if (lane == j) {
      my_id = vi;
      my_s = sv;
    }
    __syncwarp();
    if (lane == 0) b[vi] = -INFINITY;
    __syncwarp();
  }
  if (lane < top_k) {
    ids[(size_t)t * top_k + lane] = my_id;
    weights[(size_t)t * top_k + lane] = my_s / wsum * rsf;
    atomicAdd(&counts[my_id], 1);
  }
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
