// Epilogue of one grouped-GEMM tile (weight rows x expert-sorted token columns), shared by
// the fp16 and the block-scaled FP4 kernels. Run by warps 0-3: warp w reads TMEM lanes
// 32w..32w+31 of the tile's accumulator, 32 columns at a time, and every warp goes its own
// way (no barrier between them), so a warp can leave at any tile when the CTA aborts.
//   gate/up: accumulator row 32w + l is gate row 64 mt + 16 w + l (l < 16) or the up row of
//     the same h column (l >= 16; the weight stores put the rows of a tile in this order);
//     h = SiLU(gate) * up for every token column c < n ("SwiGLU" of the expert FFN), written
//     as fp16, or as fp32 together with the amax of the routed rows when h is quantised to
//     NVFP4 next.
//   down: y row row0 + c of the expert-sorted output (a routed entry below T * top_k, else
//     shared-expert token row0 + c - T * top_k) for every token column c < n; plain
//     coalesced stores (a warp writes 128 consecutive bytes of one row per column), the
//     weighted combine of the rows follows in one ordered pass (combine_kernel).
// sc_out multiplies the accumulator first (the fp32 tensor scales of NVFP4 operands, else 1).
#pragma once

#include "kernels.h"
#include "ptx.cuh"

namespace moe {

template <bool H32, int EPI>
__device__ __forceinline__ void gemm_tile_epilogue(uint32_t lane_addr, int N, int n, int row0, int mt,
                                                   float sc_out, const GemmParams& p) {
  const int warp = (threadIdx.x >> 5) & 3, lane = threadIdx.x & 31;
  const int Tk = p.T * p.top_k;
  float hmax = 0.f;
  for (int c0 = 0; c0 < N; c0 += 32) {
    float v[32];
    ptx::tmem_ld32(lane_addr + (uint32_t)c0, v);
    if (EPI == 0) {
      // lanes 0-15 hold gate rows, 16-31 the matching up rows: swap halves so that each
      // lane owns 16 token columns of one h column
      const bool upl = lane >= 16;
      const int hcol = 64 * mt + 16 * warp + (lane & 15);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float send = upl ? v[j] : v[16 + j];
        const float recv = __shfl_xor_sync(0xffffffffu, send, 16);
        const float g = (upl ? recv : v[j]) * sc_out;
        const float u = (upl ? v[16 + j] : recv) * sc_out;
        const int c = c0 + j + (upl ? 16 : 0);
        if (c < n) {
          const float hv = (p.identity_act ? g : siluf_acc(g)) * u;
          const size_t idx = (size_t)(row0 + c) * p.I + hcol;
          if (H32) {
            p.h32[idx] = hv;
            if (row0 + c < Tk) hmax = fmaxf(hmax, fabsf(hv));
          } else {
            p.h16[idx] = __float2half_rn(hv);
          }
        }
      }
    } else {
      float* yrow = p.y + (size_t)(row0 + c0) * p.H + 128 * mt + 32 * warp + lane;
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (c0 + j < n) yrow[(size_t)j * p.H] = v[j] * sc_out;
    }
  }
  if (EPI == 0 && H32) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) hmax = fmaxf(hmax, __shfl_xor_sync(0xffffffffu, hmax, o));
    if (lane == 0 && hmax > 0.f) atomicMax(p.h_amax, __float_as_uint(hmax));
  }
}

}  // namespace moe
