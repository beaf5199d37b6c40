// Shared device helpers of the MoE layer kernels: storage decoders, element loads,
// the device status word and the per-forward parameter block.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe_layer.h"

namespace moe {

// ------------------------------------------------------------------ status word
// Sticky device-side status: the first failing check wins (atomicCAS from MOE_OK).
__device__ __forceinline__ void raise_status(int* status, int code) {
  if (status) atomicCAS(status, MOE_OK, code);
}

// ------------------------------------------------------------- element decoders
__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16) {
  return __uint_as_float(bits16 << 16);
}

// int4 two's-complement nibble -> float
__device__ __forceinline__ float int4_to_float(uint32_t nib) {
  return (float)((int)(nib ^ 8u) - 8);
}

// FP4 E2M1 nibble -> float: 1 sign, 2 exponent bits (bias 1), 1 mantissa bit,
// exponent field 0 is subnormal with step 0.5.
__device__ __forceinline__ float e2m1_to_float(uint32_t nib) {
  uint32_t e = (nib >> 1) & 3u, m = nib & 1u;
  uint32_t mag = e ? (((e + 126u) << 23) | (m << 22)) : (m ? 0x3F000000u : 0u);
  return __uint_as_float(mag | ((nib & 8u) << 28));
}

// FP8 E4M3 byte -> float (bias 7, subnormal step 2^-9). Scale bytes are non-negative
// finite in this layer; the NaN pattern is not special-cased.
__device__ __forceinline__ float e4m3_to_float(uint32_t b) {
  uint32_t e = (b >> 3) & 15u, m = b & 7u;
  float mag = e ? __uint_as_float(((e + 120u) << 23) | (m << 20)) : (float)m * 0.001953125f;
  return (b & 0x80u) ? -mag : mag;
}

// Load element i of an activation row stored as fp32 or bf16.
template <int DT>
__device__ __forceinline__ float load_act(const void* base, size_t i) {
  if constexpr (DT == MOE_DT_F32) {
    return __ldg(reinterpret_cast<const float*>(base) + i);
  } else {
    return bf16_bits_to_float(__ldg(reinterpret_cast<const unsigned short*>(base) + i));
  }
}

// 8 consecutive activation elements from element index i (a multiple of 8): one 16-byte load
// for bf16, two for fp32.
template <int DT>
__device__ __forceinline__ void load8_act(const void* base, size_t i, float (&v)[8]) {
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

template <int DT>
__device__ __forceinline__ void store_act(void* base, size_t i, float v) {
  if constexpr (DT == MOE_DT_F32) {
    reinterpret_cast<float*>(base)[i] = v;
  } else {
    reinterpret_cast<__nv_bfloat16*>(base)[i] = __float2bfloat16_rn(v);
  }
}

__device__ __forceinline__ float sigmoidf_acc(float z) { return 1.0f / (1.0f + expf(-z)); }
__device__ __forceinline__ float siluf_acc(float z) { return z / (1.0f + expf(-z)); }

// ------------------------------------------------------- NVFP4 activation blocks
// One 16-element block of an NVFP4 activation with tensor scale ts ("NVIDIA stellt neues
// GLM-5.2 NVFP4 Modell vor", section "Technische Details und Quantisierungsansatz": E2M1
// elements with an FP8 E4M3 scale per 16 elements): block scale sb =
// E4M3_rne_satfinite((amax16 / 6) / ts), element code c[i] = E2M1_rne_satfinite(v[i] /
// (sb * ts)), each quotient and product a correctly rounded fp32 operation in that order.
// The dequantised element is c[i] * sb * ts. ts = 0 gives sb = 0 and all-zero codes.
// nvfp4_block_bits gives the storage: the E4M3 byte of sb and the E2M1 nibble of each c[i].
__device__ __forceinline__ void nvfp4_block_bits(const float (&v)[16], float ts, uint32_t& sbyte,
                                                 uint32_t (&nib)[16]) {
  float bmax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) bmax = fmaxf(bmax, fabsf(v[i]));
  sbyte = 0u;
  if (ts != 0.f) {
    const float ratio = __fdiv_rn(__fdiv_rn(bmax, 6.0f), ts);
    sbyte = __nv_cvt_float_to_fp8(ratio, __NV_SATFINITE, __NV_E4M3);
  }
  const float denom = __fmul_rn(e4m3_to_float(sbyte), ts);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    nib[i] = 0u;
    if (denom != 0.f)
      nib[i] = __nv_cvt_float_to_fp4(__fdiv_rn(v[i], denom), __NV_E2M1, cudaRoundNearest) & 15u;
  }
}

__device__ __forceinline__ void nvfp4_block(const float (&v)[16], float ts, float& sb, float (&c)[16]) {
  uint32_t sbyte, nib[16];
  nvfp4_block_bits(v, ts, sbyte, nib);
  sb = e4m3_to_float(sbyte);
#pragma unroll
  for (int i = 0; i < 16; ++i) c[i] = e2m1_to_float(nib[i]);
}

// ------------------------------------------------------------ weight formats
// A weight row is read in 16-byte chunks. Per chunk:
//   int4_g32: 32 elements, one fp16 scale (the chunk is exactly one g32 group)
//   nvfp4:    32 elements, two E4M3 scales (two 16-element blocks), tensor scale
//   bf16:      8 elements, no scale
template <int FMT>
struct WFmt;

template <>
struct WFmt<MOE_W_INT4_G32> {
  static constexpr int EPC = 32;             // elements per 16-byte chunk
  static constexpr int SCALE_BYTES_PER_CHUNK = 2;
  __device__ __forceinline__ static void decode(uint4 d, const uint8_t* srow, int chunk,
                                                float /*tscale*/, float (&w)[EPC]) {
    float s = __half2float(__ldg(reinterpret_cast<const __half*>(srow) + chunk));
    uint32_t words[4] = {d.x, d.y, d.z, d.w};
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
      for (int i = 0; i < 8; ++i) w[q * 8 + i] = int4_to_float((words[q] >> (4 * i)) & 15u) * s;
  }
};

template <>
struct WFmt<MOE_W_NVFP4> {
  static constexpr int EPC = 32;
  static constexpr int SCALE_BYTES_PER_CHUNK = 2;
  __device__ __forceinline__ static void decode(uint4 d, const uint8_t* srow, int chunk,
                                                float tscale, float (&w)[EPC]) {
    float s0 = e4m3_to_float(__ldg(srow + 2 * chunk)) * tscale;
    float s1 = e4m3_to_float(__ldg(srow + 2 * chunk + 1)) * tscale;
    uint32_t words[4] = {d.x, d.y, d.z, d.w};
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
      for (int i = 0; i < 8; ++i)
        w[q * 8 + i] = e2m1_to_float((words[q] >> (4 * i)) & 15u) * (q < 2 ? s0 : s1);
  }
};

template <>
struct WFmt<MOE_W_BF16> {
  static constexpr int EPC = 8;
  static constexpr int SCALE_BYTES_PER_CHUNK = 0;
  __device__ __forceinline__ static void decode(uint4 d, const uint8_t*, int, float,
                                                float (&w)[EPC]) {
    uint32_t words[4] = {d.x, d.y, d.z, d.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      w[2 * q] = __uint_as_float(words[q] << 16);
      w[2 * q + 1] = __uint_as_float(words[q] & 0xFFFF0000u);
    }
  }
};

// Per-row integer formats (one fp32 scale per row): int8 16, int4 32, int2 64 elements per
// 16-byte chunk, two's complement fields from the low bits up.
template <int BITS>
struct WFmtRow {
  static constexpr int EPC = 128 / BITS;
  __device__ __forceinline__ static void decode(uint4 d, const uint8_t* srow, int, float, float (&w)[EPC]) {
    const float s = __ldg(reinterpret_cast<const float*>(srow));
    const uint32_t words[4] = {d.x, d.y, d.z, d.w};
    constexpr int per = 32 / BITS;
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
      for (int i = 0; i < per; ++i) {
        const int v = (int)(words[q] << (32 - BITS * (i + 1))) >> (32 - BITS);   // sign-extended field
        w[q * per + i] = (float)v * s;
      }
  }
};
template <>
struct WFmt<MOE_W_INT8_ROW> : WFmtRow<8> {};
template <>
struct WFmt<MOE_W_INT4_ROW> : WFmtRow<4> {};
template <>
struct WFmt<MOE_W_INT2_ROW> : WFmtRow<2> {};

__host__ __device__ inline bool is_row_format(int fmt) {
  return fmt == MOE_W_INT8_ROW || fmt == MOE_W_INT4_ROW || fmt == MOE_W_INT2_ROW;
}

// Bytes of one stored weight row of K input elements (codes) and of its scales.
__host__ __device__ inline size_t row_code_bytes(int fmt, int K) {
  return fmt == MOE_W_BF16       ? (size_t)K * 2
         : fmt == MOE_W_INT8_ROW ? (size_t)K
         : fmt == MOE_W_INT2_ROW ? (size_t)K / 4
                                 : (size_t)K / 2;
}
__host__ __device__ inline size_t row_scale_bytes(int fmt, int K) {
  return fmt == MOE_W_INT4_G32 ? (size_t)K / 32 * 2
         : fmt == MOE_W_NVFP4  ? (size_t)K / 16
         : is_row_format(fmt)  ? 4
                               : 0;
}

// ----------------------------------------------------------- work decomposition
// Token chunk processed by one generic expert CTA.
constexpr int kTokChunk = 4;
// Work item: expert index (E = shared) in the high half, token chunk in the low half.
__host__ __device__ inline int pack_item(int e, int chunk) { return (e << 16) | chunk; }

// Device view of the expert weights (one format).
struct ExpertWeights {
  const uint8_t* gu_codes;   // [n, 2I, row_code_bytes(H)]
  const uint8_t* gu_scales;  // [n, 2I, row_scale_bytes(H)]
  const float* gu_tscale;    // [n] (NVFP4)
  const uint8_t* d_codes;    // [n, H, row_code_bytes(I)]
  const uint8_t* d_scales;
  const float* d_tscale;
};

}  // namespace moe
