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

// Tiled router GEMM for larger batches: a CTA computes a 64-token x 64-expert block of
// logits, staging 32-column slices of x and W_r in shared memory (fp32), so each router
// row is read once per 64 tokens; 256 threads, a 4 x 4 block each (tokens 4 ty.., experts
// 4 tx..) read with one 16-byte shared load per operand, fp32 FMA in ascending column
// order.
constexpr int kRgM = 64, kRgN = 64, kRgK = 32;

template <int DT>
__device__ __forceinline__ void load8(const void* base, size_t i, float (&v)[8]) {
  if constexpr (DT == MOE_DT_F32) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(base) + i));
    const float4 b = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(base) + i) + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  } else {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(static_cast<const unsigned short*>(base) + i));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      v[2 * q] = __uint_as_float(w[q] << 16);
      v[2 * q + 1] = __uint_as_float(w[q] & 0xFFFF0000u);
    }
  }
}

template <int XDT, int WDT>
__global__ void __launch_bounds__(256)
router_gemm_kernel(const void* __restrict__ x, const void* __restrict__ wr, float* __restrict__ logits,
                   int T, int E, int H) {
  __shared__ __align__(16) float xs[kRgK][kRgM + 4];
  __shared__ __align__(16) float ws[kRgK][kRgN + 4];
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int t0 = blockIdx.y * kRgM, e0 = blockIdx.x * kRgN;
  // loader: row lr (token or expert) of the tile, 8 consecutive columns at lk
  const int lr = tid >> 2, lk = (tid & 3) * 8;
  const bool xok = t0 + lr < T, wok = e0 + lr < E;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  float xv[8], wv[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) xv[q] = wv[q] = 0.f;
  if (xok) load8<XDT>(x, (size_t)(t0 + lr) * H + lk, xv);
  if (wok) load8<WDT>(wr, (size_t)(e0 + lr) * H + lk, wv);
  for (int k0 = 0; k0 < H; k0 += kRgK) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      xs[lk + q][lr] = xv[q];
      ws[lk + q][lr] = wv[q];
    }
    __syncthreads();
    if (k0 + kRgK < H) {   // prefetch the next slice while this one is multiplied
      if (xok) load8<XDT>(x, (size_t)(t0 + lr) * H + k0 + kRgK + lk, xv);
      if (wok) load8<WDT>(wr, (size_t)(e0 + lr) * H + k0 + kRgK + lk, wv);
    }
#pragma unroll
    for (int k = 0; k < kRgK; ++k) {
      const float4 av = *reinterpret_cast<const float4*>(&xs[k][4 * ty]);
      const float4 bv = *reinterpret_cast<const float4*>(&ws[k][4 * tx]);
      const float a[4] = {av.x, av.y, av.z, av.w}, b[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = t0 + 4 * ty + i;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = e0 + 4 * tx + j;
      if (e < E) logits[(size_t)t * E + e] = acc[i][j];
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
  const int id = select_token(logits + (size_t)t * E, bias, E, n_group, topk_group, top_k, rsf,
                              sb[warp], ss[warp], ids + (size_t)t * top_k,
                              weights + (size_t)t * top_k, status);
  if (lane < top_k) atomicAdd(&counts[id], 1);
}

}  // namespace

cudaError_t launch_router_logits(const void* x, int act_dtype, const void* router_w,
                                 int router_dtype, float* logits, int T, int E, int H,
                                 cudaStream_t s) {
  if (T >= 128 && H % kRgK == 0) {
    dim3 g((E + kRgN - 1) / kRgN, (T + kRgM - 1) / kRgM);
    if (act_dtype == MOE_DT_F32 && router_dtype == MOE_DT_F32)
      router_gemm_kernel<MOE_DT_F32, MOE_DT_F32><<<g, 256, 0, s>>>(x, router_w, logits, T, E, H);
    else if (act_dtype == MOE_DT_BF16 && router_dtype == MOE_DT_F32)
      router_gemm_kernel<MOE_DT_BF16, MOE_DT_F32><<<g, 256, 0, s>>>(x, router_w, logits, T, E, H);
    else if (act_dtype == MOE_DT_F32 && router_dtype == MOE_DT_BF16)
      router_gemm_kernel<MOE_DT_F32, MOE_DT_BF16><<<g, 256, 0, s>>>(x, router_w, logits, T, E, H);
    else
      router_gemm_kernel<MOE_DT_BF16, MOE_DT_BF16><<<g, 256, 0, s>>>(x, router_w, logits, T, E, H);
    return cudaGetLastError();
  }
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
