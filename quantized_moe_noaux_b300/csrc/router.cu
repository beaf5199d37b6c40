// Router of the MoE layer: fp32 logits, sigmoid gate scores, noaux_tc grouped top-k
// selection and renormalised combine weights (the DeepSeek-V3-style sigmoid router with
// noaux_tc and routed_scaling_factor of "Show HN: Menjalankan GLM 5.2 di komputer lambat",
// section "Fitur utama yang diimplementasikan").
#include <math.h>

#include "kernels.h"
#include "ptx.cuh"
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

// Router logits on the tensor cores for bf16 activations (mma.sync m16n8k16, bf16
// operands, fp32 accumulate). W_r arrives as NS bf16 planes whose sum is W_r exactly: one
// plane for a bf16 router; hi + mid + lo for an fp32 router (split once when the layer is
// created). Every product x * plane is then exact in fp32. The tensor core's internal
// fp32 accumulation is not round-to-nearest, so each MMA starts from zero on one k16 step
// and the step's sum is added to the running fp32 sum with ordinary (RN) additions. A CTA (4 warps, 32 x 32 each) computes
// 64 tokens x 64 experts over one K split of H / S columns, staged 64 columns at a time
// with cp.async (two buffers); with S > 1 splits the partial sums go to [S][T][E] and
// router_split_sum_kernel adds them in split order, so the result is deterministic.
constexpr int kRmBM = 64, kRmBN = 64, kRmBK = 64, kRmLd = kRmBK + 8;   // 144-byte smem rows

template <int NS>
struct RmSmem {
  uint16_t x[2][kRmBM][kRmLd];
  uint16_t w[2][NS][kRmBN][kRmLd];
};

template <int NS>
__global__ void __launch_bounds__(128)
router_mma_kernel(const uint16_t* __restrict__ x, const uint16_t* __restrict__ wp, float* __restrict__ out,
                  int T, int E, int H, int kchunk) {
  extern __shared__ __align__(16) uint8_t rm_smem[];
  RmSmem<NS>& S = *reinterpret_cast<RmSmem<NS>*>(rm_smem);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int wm = warp >> 1, wn = warp & 1;
  const int t0 = blockIdx.y * kRmBM, e0 = blockIdx.x * kRmBN;
  const int kbeg = blockIdx.z * kchunk, nk = kchunk / kRmBK;
  // 16-byte chunk c = tid & 7 of rows tid / 8 + 16 i; rows past T or E are zero-filled
  auto load_stage = [&](int buf, int k0) {
    const int c = tid & 7;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = (tid >> 3) + 16 * i, t = t0 + r;
      ptx::cp_async16(&S.x[buf][r][8 * c], x + (size_t)min(t, T - 1) * H + k0 + 8 * c, t < T ? 16u : 0u);
    }
#pragma unroll
    for (int p = 0; p < NS; ++p)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int r = (tid >> 3) + 16 * i, e = e0 + r;
        ptx::cp_async16(&S.w[buf][p][r][8 * c], wp + ((size_t)p * E + min(e, E - 1)) * H + k0 + 8 * c,
                        e < E ? 16u : 0u);
      }
  };
  float acc[2][4][4];
#pragma unroll
  for (int mi = 0; mi < 2; ++mi)
#pragma unroll
    for (int ni = 0; ni < 4; ++ni)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[mi][ni][q] = 0.f;
  load_stage(0, kbeg);
  ptx::cp_async_commit();
  for (int ks = 0; ks < nk; ++ks) {
    const int buf = ks & 1;
    if (ks + 1 < nk) load_stage(buf ^ 1, kbeg + (ks + 1) * kRmBK);
    ptx::cp_async_commit();
    ptx::cp_async_wait<1>();
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < kRmBK; kk += 16) {
      uint32_t a[2][4];
#pragma unroll
      for (int mi = 0; mi < 2; ++mi)
        ptx::ldmatrix_x4(a[mi], &S.x[buf][32 * wm + 16 * mi + (lane & 15)][kk + 8 * (lane >> 4)]);
#pragma unroll
      for (int nj = 0; nj < 2; ++nj) {   // two n8 blocks per ldmatrix.x4
        uint32_t b[NS][4];
#pragma unroll
        for (int p = 0; p < NS; ++p)
          ptx::ldmatrix_x4(b[p], &S.w[buf][p][32 * wn + 16 * nj + (lane & 7) + ((lane >> 4) << 3)]
                                       [kk + 8 * ((lane >> 3) & 1)]);
#pragma unroll
        for (int mi = 0; mi < 2; ++mi)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            // each k16 step starts from zero: the MMA's internal accumulation then only
            // rounds relative to this step's own products; the step is added in fp32 (RN)
            float th[4] = {0.f, 0.f, 0.f, 0.f};
            ptx::mma_16816_bf16(th, a[mi], b[0][2 * h], b[0][2 * h + 1]);
            if constexpr (NS == 3) {
              float tl[4] = {0.f, 0.f, 0.f, 0.f};
              ptx::mma_16816_bf16(tl, a[mi], b[1][2 * h], b[1][2 * h + 1]);
              ptx::mma_16816_bf16(tl, a[mi], b[2][2 * h], b[2][2 * h + 1]);
#pragma unroll
              for (int q = 0; q < 4; ++q) th[q] += tl[q];
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[mi][2 * nj + h][q] += th[q];
          }
      }
    }
    __syncthreads();
  }
  // accumulator element q of block (mi, ni): row g (+8 for q >= 2), columns 2 tq, 2 tq + 1
  const int g = lane >> 2, tq = lane & 3;
  float* dst = out + (size_t)blockIdx.z * T * E;
#pragma unroll
  for (int mi = 0; mi < 2; ++mi)
#pragma unroll
    for (int ni = 0; ni < 4; ++ni)
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int t = t0 + 32 * wm + 16 * mi + g + 8 * hr, e = e0 + 32 * wn + 8 * ni + 2 * tq;
        if (t < T && e < E)
          *reinterpret_cast<float2*>(dst + (size_t)t * E + e) =
              make_float2(acc[mi][ni][2 * hr], acc[mi][ni][2 * hr + 1]);
      }
}

// logits = sum of the S partial blocks, added in split order.
__global__ void router_split_sum_kernel(const float4* __restrict__ part, float4* __restrict__ logits, int n4,
                                        int S) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += gridDim.x * blockDim.x) {
    float4 v = part[i];
    for (int z = 1; z < S; ++z) {
      const float4 u = part[(size_t)z * n4 + i];
      v.x += u.x;
      v.y += u.y;
      v.z += u.z;
      v.w += u.w;
    }
    logits[i] = v;
  }
}

// hi, mid, lo bf16 planes of an fp32 matrix: hi = bf16(w), mid = bf16(w - hi),
// lo = bf16(w - hi - mid); each difference is exact (Sterbenz) and hi + mid + lo = w for
// every normal w (24 significant bits in three 8-bit pieces).
__global__ void router_split_kernel(const float* __restrict__ w, uint16_t* __restrict__ planes, size_t n) {
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const float v = w[i];
    const __nv_bfloat16 hi = __float2bfloat16_rn(v);
    const float r1 = v - __bfloat162float(hi);
    const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
    const float r2 = r1 - __bfloat162float(mid);
    const __nv_bfloat16 lo = __float2bfloat16_rn(r2);
    planes[i] = __bfloat16_as_ushort(hi);
    planes[n + i] = __bfloat16_as_ushort(mid);
    planes[2 * n + i] = __bfloat16_as_ushort(lo);
  }
}

constexpr int kSelWarps = 4;
constexpr int kMaxE = 1024;

// One warp per token.
__global__ void __launch_bounds__(kSelWarps * 32)
select_kernel(const float* __restrict__ logits, const float* __restrict__ bias, int T, int E,
              int n_group, int topk_group, int top_k, float rsf, float top_p, int32_t* __restrict__ ids,
              float* __restrict__ weights, int32_t* __restrict__ counts, int* status) {
  __shared__ float sb[kSelWarps][kMaxE];   // biased scores; -inf once taken or excluded
  __shared__ float ss[kSelWarps][kMaxE];   // unbiased sigmoid scores
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kSelWarps + warp;
  if (t >= T) return;
  const int id = select_token(logits + (size_t)t * E, bias, E, n_group, topk_group, top_k, rsf, top_p,
                              sb[warp], ss[warp], ids + (size_t)t * top_k,
                              weights + (size_t)t * top_k, status);
  if (lane < top_k && id >= 0) atomicAdd(&counts[id], 1);
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
                          int topk_group, int top_k, float rsf, float top_p, int32_t* ids, float* weights,
                          int32_t* counts, int* status, cudaStream_t s) {
  if (E > kMaxE || n_group > 32 || top_k > 32) return cudaErrorInvalidValue;
  select_kernel<<<(T + kSelWarps - 1) / kSelWarps, kSelWarps * 32, 0, s>>>(
      logits, bias, T, E, n_group, topk_group, top_k, rsf, top_p, ids, weights, counts, status);
  return cudaGetLastError();
}

// Split count of the tensor-core router: the smallest divisor S of H / 64 that gives at least
// two CTAs per SM, keeping S * tiles <= 4 * n_sm (the partial buffer's capacity).
static int router_mma_splits(int T, int E, int H, int n_sm) {
  const long tiles = (long)((T + kRmBM - 1) / kRmBM) * ((E + kRmBN - 1) / kRmBN);
  const int nkb = H / kRmBK;
  int best = 1;
  for (int d = 1; d <= nkb; ++d) {
    if (nkb % d) continue;
    if (d * tiles > 4L * n_sm) break;
    best = d;
    if (d * tiles >= 2L * n_sm) break;
  }
  return best;
}

size_t router_mma_partial_floats(int n_sm) { return (size_t)4 * n_sm * kRmBM * kRmBN; }

bool router_mma_supported(int act_dtype, int H, int E) {
  return act_dtype == MOE_DT_BF16 && H % kRmBK == 0 && E % 4 == 0;
}

cudaError_t router_mma_init() {
  cudaError_t e = cudaFuncSetAttribute(router_mma_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)sizeof(RmSmem<1>));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(router_mma_kernel<3>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sizeof(RmSmem<3>));
  return e;
}

cudaError_t launch_router_split(const float* w, uint16_t* planes, size_t n, cudaStream_t s) {
  router_split_kernel<<<592, 256, 0, s>>>(w, planes, n);
  return cudaGetLastError();
}

cudaError_t launch_router_mma(const void* x, const uint16_t* planes, int n_planes, float* logits, float* partial,
                              int T, int E, int H, int n_sm, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  const int S = router_mma_splits(T, E, H, n_sm);
  const dim3 grid((E + kRmBN - 1) / kRmBN, (T + kRmBM - 1) / kRmBM, S);
  float* out = S == 1 ? logits : partial;
  const uint16_t* xb = static_cast<const uint16_t*>(x);
  if (n_planes == 3)
    router_mma_kernel<3><<<grid, 128, sizeof(RmSmem<3>), s>>>(xb, planes, out, T, E, H, H / S);
  else
    router_mma_kernel<1><<<grid, 128, sizeof(RmSmem<1>), s>>>(xb, planes, out, T, E, H, H / S);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || S == 1) return e;
  const int n4 = T * E / 4;
  router_split_sum_kernel<<<(n4 + 255) / 256, 256, 0, s>>>(reinterpret_cast<const float4*>(partial),
                                                          reinterpret_cast<float4*>(logits), n4, S);
  return cudaGetLastError();
}

}  // namespace moe
