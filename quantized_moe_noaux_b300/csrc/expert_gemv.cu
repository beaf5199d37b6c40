// Generic batch-union expert kernels (any T, any weight format): one CTA per
// (16 output rows, expert, chunk of kTokChunk tokens routed to that expert).
//   up:   h[pair, r] = SiLU(W_g[r] . x_t) * (W_u[r] . x_t)       (SwiGLU gate/up)
//   down: out_acc[t, r] += w[t, slot] * (W_d[r] . h[pair])       (down + weighted combine)
// Weights are dequantised on use from their packed codes (dequant-on-use of the packed
// int4 container, "Show HN: Menjalankan GLM 5.2 di komputer lambat", section "Fitur utama
// yang diimplementasikan"; NVFP4 blocks per "NVIDIA stellt neues GLM-5.2 NVFP4 Modell
// vor", section "Technische Details und Quantisierungsansatz").
#include "kernels.h"

namespace moe {

namespace {

constexpr int kThreads = 256;
constexpr int kRowsPerCta = 16;   // 8 warps x 2 rows

__device__ __forceinline__ uint4 ld_stream(const uint8_t* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

struct TokenChunk {
  int ntok;
  int tok[kTokChunk];    // token index
  int pair[kTokChunk];   // row of the h buffer
  int ent[kTokChunk];    // token*top_k + slot (routed) or -1 (shared)
  int widx;              // weight index
  bool routed;
};

__device__ __forceinline__ bool resolve_item(const ExpertGemvArgs& a, TokenChunk& c) {
  int e, chunk;
  if (a.items) {
    if ((int)blockIdx.y >= __ldg(a.meta)) return false;
    const int it = __ldg(a.items + blockIdx.y);
    e = it >> 16;
    chunk = it & 0xffff;
  } else {
    e = a.E;
    chunk = blockIdx.y;
  }
  c.routed = e < a.E;
  c.widx = c.routed ? e : a.expert_base;
  if (c.routed) {
    const int off = __ldg(a.offsets + e);
    const int cnt = __ldg(a.offsets + e + 1) - off;
    c.ntok = min(kTokChunk, cnt - chunk * kTokChunk);
    if (c.ntok <= 0) return false;
#pragma unroll
    for (int i = 0; i < kTokChunk; ++i) {
      const int p = off + chunk * kTokChunk + min(i, c.ntok - 1);
      const int ent = __ldg(a.entries + p);
      c.ent[i] = ent;
      c.tok[i] = ent / a.top_k;
      c.pair[i] = p;
    }
  } else {
    c.ntok = min(kTokChunk, a.T - chunk * kTokChunk);
    if (c.ntok <= 0) return false;
#pragma unroll
    for (int i = 0; i < kTokChunk; ++i) {
      const int t = chunk * kTokChunk + min(i, c.ntok - 1);
      c.ent[i] = -1;
      c.tok[i] = t;
      c.pair[i] = a.T * a.top_k + t;
    }
  }
  return c.ntok > 0;
}

template <int FMT, int XDT>
__global__ void __launch_bounds__(kThreads)
expert_up_kernel(ExpertGemvArgs a) {
  using F = WFmt<FMT>;
  extern __shared__ float xs[];   // [kTokChunk][H]
  TokenChunk c;
  if (!resolve_item(a, c)) return;
  const int H = a.H, I = a.I;
  for (int i = 0; i < c.ntok; ++i)
    for (int h = threadIdx.x; h < H; h += kThreads)
      xs[i * H + h] = load_act<XDT>(a.x, (size_t)c.tok[i] * H + h);
  __syncthreads();

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const size_t rcb = row_code_bytes(FMT, H), rsb = row_scale_bytes(FMT, H);
  const uint8_t* codes = a.w.gu_codes + (size_t)c.widx * 2 * I * rcb;
  const uint8_t* scales = a.w.gu_scales ? a.w.gu_scales + (size_t)c.widx * 2 * I * rsb : nullptr;
  const float ts = (FMT == MOE_W_NVFP4) ? __ldg(a.w.gu_tscale + c.widx) : 1.f;
  const int nchunks = (int)(rcb / 16);

  for (int rr = 0; rr < kRowsPerCta / 8; ++rr) {
    const int r = blockIdx.x * kRowsPerCta + rr * 8 + warp;
    float ag[kTokChunk], au[kTokChunk];
#pragma unroll
    for (int i = 0; i < kTokChunk; ++i) ag[i] = au[i] = 0.f;
    for (int ch = lane; ch < nchunks; ch += 32) {
      float wg[F::EPC], wu[F::EPC];
      F::decode(ld_stream(codes + (size_t)r * rcb + ch * 16), scales + (size_t)r * rsb, ch, ts, wg);
      F::decode(ld_stream(codes + (size_t)(r + I) * rcb + ch * 16), scales + (size_t)(r + I) * rsb,
                ch, ts, wu);
#pragma unroll
      for (int i = 0; i < kTokChunk; ++i) {
        if (i < c.ntok) {
          const float* xr = xs + i * H + ch * F::EPC;
#pragma unroll
          for (int j = 0; j < F::EPC; ++j) {
            ag[i] = fmaf(wg[j], xr[j], ag[i]);
            au[i] = fmaf(wu[j], xr[j], au[i]);
          }
        }
      }
    }
#pragma unroll
    for (int i = 0; i < kTokChunk; ++i) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        ag[i] += __shfl_xor_sync(0xffffffffu, ag[i], o);
        au[i] += __shfl_xor_sync(0xffffffffu, au[i], o);
      }
    }
    if (lane == 0) {
      for (int i = 0; i < c.ntok; ++i) {
        const float hv = (a.identity_act ? ag[i] : siluf_acc(ag[i])) * au[i];
        a.h[(size_t)c.pair[i] * I + r] = hv;
        if (a.h_amax && c.routed) atomicMax(a.h_amax, __float_as_uint(fabsf(hv)));
      }
    }
  }
}

template <int FMT>
__global__ void __launch_bounds__(kThreads)
expert_down_kernel(ExpertGemvArgs a) {
  using F = WFmt<FMT>;
  extern __shared__ float hs[];   // [kTokChunk][I]
  TokenChunk c;
  if (!resolve_item(a, c)) return;
  const int H = a.H, I = a.I;
  for (int i = 0; i < c.ntok; ++i)
    for (int k = threadIdx.x; k < I; k += kThreads) hs[i * I + k] = a.h[(size_t)c.pair[i] * I + k];
  __syncthreads();

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const size_t rcb = row_code_bytes(FMT, I), rsb = row_scale_bytes(FMT, I);
  const uint8_t* codes = a.w.d_codes + (size_t)c.widx * H * rcb;
  const uint8_t* scales = a.w.d_scales ? a.w.d_scales + (size_t)c.widx * H * rsb : nullptr;
  const float ts = (FMT == MOE_W_NVFP4) ? __ldg(a.w.d_tscale + c.widx) : 1.f;
  const int nchunks = (int)(rcb / 16);

  for (int rr = 0; rr < kRowsPerCta / 8; ++rr) {
    const int r = blockIdx.x * kRowsPerCta + rr * 8 + warp;
    float acc[kTokChunk];
#pragma unroll
    for (int i = 0; i < kTokChunk; ++i) acc[i] = 0.f;
    for (int ch = lane; ch < nchunks; ch += 32) {
      float wv[F::EPC];
      F::decode(ld_stream(codes + (size_t)r * rcb + ch * 16), scales + (size_t)r * rsb, ch, ts, wv);
#pragma unroll
      for (int i = 0; i < kTokChunk; ++i) {
        if (i < c.ntok) {
          const float* hr = hs + i * I + ch * F::EPC;
#pragma unroll
          for (int j = 0; j < F::EPC; ++j) acc[i] = fmaf(wv[j], hr[j], acc[i]);
        }
      }
    }
#pragma unroll
    for (int i = 0; i < kTokChunk; ++i)
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc[i] += __shfl_xor_sync(0xffffffffu, acc[i], o);
    if (lane == 0) {
      for (int i = 0; i < c.ntok; ++i) {
        const float wt = c.routed ? __ldg(a.weights + c.ent[i]) : 1.f;
        atomicAdd(a.out_acc + (size_t)c.tok[i] * H + r, wt * acc[i]);
      }
    }
  }
}

template <typename K>
cudaError_t launch_with_smem(K kernel, dim3 grid, size_t smem, cudaStream_t s,
                             const ExpertGemvArgs& a) {
  kernel<<<grid, kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

template <typename K>
cudaError_t allow_smem(K kernel) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDynSmem);
}

}  // namespace

cudaError_t expert_kernels_init() {
  cudaError_t e = cudaSuccess;
  const cudaError_t r[] = {
      allow_smem(expert_up_kernel<MOE_W_INT4_G32, MOE_DT_F32>),
      allow_smem(expert_up_kernel<MOE_W_INT4_G32, MOE_DT_BF16>),
      allow_smem(expert_up_kernel<MOE_W_NVFP4, MOE_DT_F32>),
      allow_smem(expert_up_kernel<MOE_W_NVFP4, MOE_DT_BF16>),
      allow_smem(expert_up_kernel<MOE_W_BF16, MOE_DT_F32>),
      allow_smem(expert_up_kernel<MOE_W_BF16, MOE_DT_BF16>),
      allow_smem(expert_up_kernel<MOE_W_INT8_ROW, MOE_DT_F32>),
      allow_smem(expert_up_kernel<MOE_W_INT8_ROW, MOE_DT_BF16>),
      allow_smem(expert_up_kernel<MOE_W_INT4_ROW, MOE_DT_F32>),
      allow_smem(expert_up_kernel<MOE_W_INT4_ROW, MOE_DT_BF16>),
      allow_smem(expert_up_kernel<MOE_W_INT2_ROW, MOE_DT_F32>),
      allow_smem(expert_up_kernel<MOE_W_INT2_ROW, MOE_DT_BF16>),
      allow_smem(expert_down_kernel<MOE_W_INT4_G32>),
      allow_smem(expert_down_kernel<MOE_W_NVFP4>),
      allow_smem(expert_down_kernel<MOE_W_BF16>),
      allow_smem(expert_down_kernel<MOE_W_INT8_ROW>),
      allow_smem(expert_down_kernel<MOE_W_INT4_ROW>),
      allow_smem(expert_down_kernel<MOE_W_INT2_ROW>)};
  for (cudaError_t x : r)
    if (x != cudaSuccess) e = x;
  return e;
}

cudaError_t launch_expert_up(const ExpertGemvArgs& a, cudaStream_t s) {
  dim3 grid(a.I / kRowsPerCta, a.max_items);
  const size_t smem = (size_t)kTokChunk * a.H * sizeof(float);
  const bool xf = a.x_dtype == MOE_DT_F32;
  switch (a.fmt) {
    case MOE_W_INT4_G32:
      return xf ? launch_with_smem(expert_up_kernel<MOE_W_INT4_G32, MOE_DT_F32>, grid, smem, s, a)
                : launch_with_smem(expert_up_kernel<MOE_W_INT4_G32, MOE_DT_BF16>, grid, smem, s, a);
    case MOE_W_NVFP4:
      return xf ? launch_with_smem(expert_up_kernel<MOE_W_NVFP4, MOE_DT_F32>, grid, smem, s, a)
                : launch_with_smem(expert_up_kernel<MOE_W_NVFP4, MOE_DT_BF16>, grid, smem, s, a);
    case MOE_W_BF16:
      return xf ? launch_with_smem(expert_up_kernel<MOE_W_BF16, MOE_DT_F32>, grid, smem, s, a)
                : launch_with_smem(expert_up_kernel<MOE_W_BF16, MOE_DT_BF16>, grid, smem, s, a);
    case MOE_W_INT8_ROW:
      return xf ? launch_with_smem(expert_up_kernel<MOE_W_INT8_ROW, MOE_DT_F32>, grid, smem, s, a)
                : launch_with_smem(expert_up_kernel<MOE_W_INT8_ROW, MOE_DT_BF16>, grid, smem, s, a);
    case MOE_W_INT4_ROW:
      return xf ? launch_with_smem(expert_up_kernel<MOE_W_INT4_ROW, MOE_DT_F32>, grid, smem, s, a)
                : launch_with_smem(expert_up_kernel<MOE_W_INT4_ROW, MOE_DT_BF16>, grid, smem, s, a);
    case MOE_W_INT2_ROW:
      return xf ? launch_with_smem(expert_up_kernel<MOE_W_INT2_ROW, MOE_DT_F32>, grid, smem, s, a)
                : launch_with_smem(expert_up_kernel<MOE_W_INT2_ROW, MOE_DT_BF16>, grid, smem, s, a);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_expert_down(const ExpertGemvArgs& a, cudaStream_t s) {
  dim3 grid(a.H / kRowsPerCta, a.max_items);
  const size_t smem = (size_t)kTokChunk * a.I * sizeof(float);
  switch (a.fmt) {
    case MOE_W_INT4_G32: return launch_with_smem(expert_down_kernel<MOE_W_INT4_G32>, grid, smem, s, a);
    case MOE_W_NVFP4: return launch_with_smem(expert_down_kernel<MOE_W_NVFP4>, grid, smem, s, a);
    case MOE_W_BF16: return launch_with_smem(expert_down_kernel<MOE_W_BF16>, grid, smem, s, a);
    case MOE_W_INT8_ROW: return launch_with_smem(expert_down_kernel<MOE_W_INT8_ROW>, grid, smem, s, a);
    case MOE_W_INT4_ROW: return launch_with_smem(expert_down_kernel<MOE_W_INT4_ROW>, grid, smem, s, a);
    case MOE_W_INT2_ROW: return launch_with_smem(expert_down_kernel<MOE_W_INT2_ROW>, grid, smem, s, a);
  }
  return cudaErrorInvalidValue;
}

}  // namespace moe
