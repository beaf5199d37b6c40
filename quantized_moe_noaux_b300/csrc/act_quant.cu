// NVFP4 activation quantiser and the output conversion.
//
// NVFP4 layers feed their routed experts NVFP4 activations: E2M1 elements with an E4M3
// scale per 16 consecutive elements and one fp32 scale per tensor ("NVIDIA stellt neues
// GLM-5.2 NVFP4 Modell vor", section "Technische Details und Quantisierungsansatz"). The
// tensor scale is taken per call: ts = amax / (6 * 448). Each block's scale is
// E4M3_rne_satfinite((amax16 / 6) / ts) and each element's code is
// E2M1_rne_satfinite(v / (scale * ts)); every quotient and product that decides a code is a
// correctly rounded fp32 operation in exactly that order (no contraction into FMAs).
#include "kernels.h"

namespace moe {

namespace {

constexpr int kThreads = 256;

template <int DT>
__global__ void __launch_bounds__(kThreads)
amax_kernel(const void* __restrict__ src, size_t n, unsigned int* amax_bits) {
  float m = 0.f;
  for (size_t i = (size_t)blockIdx.x * kThreads + threadIdx.x; i < n; i += (size_t)gridDim.x * kThreads)
    m = fmaxf(m, fabsf(load_act<DT>(src, i)));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  __shared__ float red[kThreads / 32];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kThreads / 32; ++w) m = fmaxf(m, red[w]);
    atomicMax(amax_bits, __float_as_uint(m));   // non-negative floats order as their bits
  }
}

// One thread per 16-element block; writes the dequantised values (code * scale * ts).
template <int DT>
__global__ void __launch_bounds__(kThreads)
nvfp4_quant_kernel(const void* __restrict__ src, float* __restrict__ dst, size_t nblocks,
                   const unsigned int* __restrict__ amax_bits) {
  const float amax = __uint_as_float(__ldg(amax_bits));
  const float ts = __fdiv_rn(amax, 2688.0f);
  for (size_t b = (size_t)blockIdx.x * kThreads + threadIdx.x; b < nblocks;
       b += (size_t)gridDim.x * kThreads) {
    float v[16], c[16], sb;
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = load_act<DT>(src, b * 16 + i);
    nvfp4_block(v, ts, sb, c);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float out = __fmul_rn(__fmul_rn(c[i], sb), ts);
      dst[b * 16 + i] = out;
    }
  }
}

// Q8_0-style int8 activations (the integer-dot kernels' activations of "Show HN: Menjalankan
// GLM 5.2 di komputer lambat", section "Fitur utama yang diimplementasikan"): one thread per
// 32-element block; step d = fp16_rn(amax / 127), code = clamp(rint(v / d), -127, 127) (d = 0
// gives 0), both quotients correctly rounded fp32 operations; writes code * d (exact in fp32).
template <int DT>
__global__ void __launch_bounds__(kThreads)
q8_0_quant_kernel(const void* __restrict__ src, float* dst, size_t nblocks) {
  for (size_t b = (size_t)blockIdx.x * kThreads + threadIdx.x; b < nblocks;
       b += (size_t)gridDim.x * kThreads) {
    float v[32], amax = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      v[i] = load_act<DT>(src, b * 32 + i);
      amax = fmaxf(amax, fabsf(v[i]));
    }
    const float d = __half2float(__float2half_rn(__fdiv_rn(amax, 127.0f)));
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const float q = d != 0.f ? fminf(fmaxf(rintf(__fdiv_rn(v[i], d)), -127.f), 127.f) : 0.f;
      dst[b * 32 + i] = q * d;
    }
  }
}

// out = acc in the output type, 8 elements per thread step (n is a multiple of 8: H is).
template <int DT>
__global__ void __launch_bounds__(kThreads)
finalize_kernel(const float* __restrict__ acc, void* __restrict__ out, size_t n) {
  for (size_t i = ((size_t)blockIdx.x * kThreads + threadIdx.x) * 8; i < n; i += (size_t)gridDim.x * kThreads * 8) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(acc + i));
    const float4 b = __ldg(reinterpret_cast<const float4*>(acc + i) + 1);
    if constexpr (DT == MOE_DT_F32) {
      reinterpret_cast<float4*>(static_cast<float*>(out) + i)[0] = a;
      reinterpret_cast<float4*>(static_cast<float*>(out) + i)[1] = b;
    } else {
      const __nv_bfloat162 p0 = __floats2bfloat162_rn(a.x, a.y), p1 = __floats2bfloat162_rn(a.z, a.w);
      const __nv_bfloat162 p2 = __floats2bfloat162_rn(b.x, b.y), p3 = __floats2bfloat162_rn(b.z, b.w);
      uint4 o;
      o.x = *reinterpret_cast<const uint32_t*>(&p0);
      o.y = *reinterpret_cast<const uint32_t*>(&p1);
      o.z = *reinterpret_cast<const uint32_t*>(&p2);
      o.w = *reinterpret_cast<const uint32_t*>(&p3);
      *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(out) + i) = o;
    }
  }
}

int grid_for(size_t n) {
  size_t g = (n + kThreads - 1) / kThreads;
  return (int)(g < 148 * 16 ? (g ? g : 1) : 148 * 16);
}

}  // namespace

cudaError_t launch_amax(const void* src, int src_dtype, size_t n, unsigned int* amax_bits,
                        cudaStream_t s) {
  if (src_dtype == MOE_DT_F32)
    amax_kernel<MOE_DT_F32><<<grid_for(n), kThreads, 0, s>>>(src, n, amax_bits);
  else
    amax_kernel<MOE_DT_BF16><<<grid_for(n), kThreads, 0, s>>>(src, n, amax_bits);
  return cudaGetLastError();
}

cudaError_t launch_q8_0_quant(const void* src, int src_dtype, float* dst, size_t n, cudaStream_t s) {
  const size_t nb = n / 32;
  if (nb == 0) return cudaSuccess;
  if (src_dtype == MOE_DT_F32)
    q8_0_quant_kernel<MOE_DT_F32><<<grid_for(nb), kThreads, 0, s>>>(src, dst, nb);
  else
    q8_0_quant_kernel<MOE_DT_BF16><<<grid_for(nb), kThreads, 0, s>>>(src, dst, nb);
  return cudaGetLastError();
}

cudaError_t launch_nvfp4_quant(const void* src, int src_dtype, float* dst, size_t n,
                               const unsigned int* amax_bits, cudaStream_t s) {
  const size_t nb = n / 16;
  if (src_dtype == MOE_DT_F32)
    nvfp4_quant_kernel<MOE_DT_F32><<<grid_for(nb), kThreads, 0, s>>>(src, dst, nb, amax_bits);
  else
    nvfp4_quant_kernel<MOE_DT_BF16><<<grid_for(nb), kThreads, 0, s>>>(src, dst, nb, amax_bits);
  return cudaGetLastError();
}

cudaError_t launch_finalize(const float* out_acc, void* out, int act_dtype, size_t n,
                            cudaStream_t s) {
  if (act_dtype == MOE_DT_F32)
    finalize_kernel<MOE_DT_F32><<<grid_for(n / 8), kThreads, 0, s>>>(out_acc, out, n);
  else
    finalize_kernel<MOE_DT_BF16><<<grid_for(n / 8), kThreads, 0, s>>>(out_acc, out, n);
  return cudaGetLastError();
}

}  // namespace moe
