// Grouped expert GEMMs of NVFP4 layers on the block-scaled FP4 tensor cores ("NVIDIA stellt
// neues GLM-5.2 NVFP4 Modell vor", section "Technische Details und Quantisierungsansatz":
// E2M1 elements with one FP8 E4M3 scale per 16 elements and an fp32 tensor scale). Both
// operands stay in their 4-bit storage all the way into the tensor core: tcgen05.mma
// kind::mxf4nvf4 multiplies E2M1 codes block-scaled by their E4M3 scales and accumulates in
// fp32; the two fp32 tensor scales multiply the accumulator in the epilogue.
//
// A tile is D = W[128 rows, K] . X[n <= 128 tokens, K]^T of one expert (weight rows on the
// MMA's M side, the expert's tokens on N, as in the fp16 kernel), K walked in stages of 256
// elements: one 128-byte row of packed codes per weight row and per token, four MMAs of
// K = 64 each. Persistent CTAs walk the tiles (item, 128-row block) round-robin; warp roles:
//   warp 4    TMA of the stage's 128 x 128-byte weight codes (128-byte swizzle) and one bulk
//             copy of its 2 KB of weight scales, already in the MMA's scale order
//   warp 5    TMA of the stage's n x 128-byte activation codes (boxes of 32, 64 or 128 rows)
//   warp 6    activation scales: the 16 scale bytes per token of the stage, from the
//             row-major scale matrix (four stages per load round), into the MMA's order
//   warp 7    copies both scale blocks shared -> TMEM (tcgen05.cp, in issue order with the
//             MMAs that read them), issues the four MMAs, releases the stage by commit
//   warps 0-3 epilogue of the previous tile from the other TMEM accumulator
//             (gemm_tile_epilogue: SwiGLU h rows, or the weighted combine)
// TMEM: two 128-column accumulators and, per pipeline stage, 16 columns of weight scales and
// 16 of activation scales (the stage's smem slot and TMEM slot are released together).
// Every wait has a time limit (GemmParams::wait_ns); a time-out sets MOE_ERR_TIMEOUT, the
// CTA stops issuing work, lets copies and MMAs in flight land, frees its TMEM and exits.
#include <cuda.h>

#include "gemm_epi.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kF4WarpW = 4;
constexpr int kF4WarpB = 5;
constexpr int kF4WarpSF = 6;
constexpr int kF4WarpMma = 7;
constexpr int kF4Threads = 8 * 32;
constexpr int kF4BM = 128;
constexpr int kF4BN = kFp4MaxN;
constexpr int kF4BK = 256;                // K elements per stage (128 bytes of codes per row)
constexpr int kF4Stages = 5;
constexpr int kF4A = kF4BM * 128;         // 16 KB of weight codes
constexpr int kF4B = kF4BN * 128;         // 16 KB of activation codes
constexpr int kF4SF = 4 * 512;            // 4 MMAs x (32 rows x 16 bytes) of scales
constexpr int kF4AccCols = 128;
constexpr int kF4SfCols = 32;             // per stage: 4 x 4 weight-scale + 4 x 4 activation-scale
constexpr uint32_t kF4TmemCols = 512;
static_assert(kF4BN == 128, "one 512-byte scale block covers 128 token rows");
static_assert(2 * kF4AccCols + kF4Stages * kF4SfCols <= (int)kF4TmemCols, "TMEM budget");

struct F4Smem {
  uint8_t a[kF4Stages][kF4A];
  uint8_t b[kF4Stages][kF4B];
  uint8_t sfa[kF4Stages][kF4SF];
  uint8_t sfb[kF4Stages][kF4SF];
  uint64_t full[kF4Stages];
  uint64_t empty[kF4Stages];
  uint64_t tmem_full[2];
  uint64_t tmem_empty[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
};

constexpr size_t kF4SmemBytes = sizeof(F4Smem) + 1024;   // + alignment slack
static_assert(kF4SmemBytes <= 227 * 1024, "FP4 GEMM shared memory over the per-CTA limit");

__device__ __forceinline__ void f4_abort(F4Smem& S, int* status) {
  atomicExch(&S.abort, 1);
  raise_status(status, MOE_ERR_TIMEOUT);
}

__device__ __forceinline__ bool f4_aborted(const F4Smem& S) { return *(volatile const int*)&S.abort != 0; }

template <int EPI>
__global__ void __launch_bounds__(kF4Threads, 1)
moe_gemm_fp4_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_b32,
                    const __grid_constant__ CUtensorMap tm_b64, const __grid_constant__ CUtensorMap tm_b128,
                    const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  F4Smem& S = *reinterpret_cast<F4Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int MT = p.mtiles;
  const int n_items = __ldg(p.n_items);
  const int skip = p.item_skip ? __ldg(p.item_skip) : 0;
  const int ntiles = n_items * MT;
  if ((int)blockIdx.x >= ntiles) return;   // no tile for this CTA (uniform)
  const int NK = p.K / kF4BK;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned long long lim = p.wait_ns;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kF4Stages; ++s) {
      ptx::mbar_init(&S.full[s], 3);    // weight copy (+ tx), activation copy (+ tx), scale stager
      ptx::mbar_init(&S.empty[s], 1);   // tcgen05.commit
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&S.tmem_full[b], 1);
      ptx::mbar_init(&S.tmem_empty[b], 4);
    }
    ptx::mbar_init(&S.mma_done, 1);
    ptx::fence_mbar_init();
    S.abort = 0;
  }
  if (warp == kF4WarpMma) {
    ptx::tmem_alloc(&S.tmem_base, kF4TmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = S.tmem_base;

  if (warp == kF4WarpW) {
    // ------------------------------------------------------------ weight producer
    if (lane == 0) {
      ptx::prefetch_tmap(&tm_w);
      int kg = 0;
      bool stop = false;
      for (int t = blockIdx.x; t < ntiles && !stop && !f4_aborted(S); t += gridDim.x) {
        const int4 it = __ldg(p.items + skip + t / MT);
        const int e = it.x - p.e_sub, mt = t % MT;
        const int wrow = e * p.rows_per_expert + kF4BM * mt;
        const uint8_t* sf = p.wsf + ((size_t)e * MT + mt) * (size_t)NK * kF4SF;
        for (int ks = 0; ks < NK; ++ks, ++kg) {
          const int s = kg % kF4Stages;
          if (kg >= kF4Stages && !ptx::mbar_wait_ns(&S.empty[s], ((kg / kF4Stages) - 1) & 1, lim)) {
            f4_abort(S, p.status);
            stop = true;
            break;
          }
          ptx::mbar_arrive_expect_tx(&S.full[s], kF4A + kF4SF);
          ptx::tma_load_2d(S.a[s], &tm_w, ks * 128, wrow, &S.full[s]);
          ptx::bulk_g2s(S.sfa[s], sf + (size_t)ks * kF4SF, kF4SF, &S.full[s], ptx::policy_evict_first());
        }
      }
    }
  } else if (warp == kF4WarpB) {
    // ---------------------------------------------------- activation code producer
    if (lane == 0) {
      ptx::prefetch_tmap(&tm_b32);
      ptx::prefetch_tmap(&tm_b64);
      ptx::prefetch_tmap(&tm_b128);
      int kg = 0;
      bool stop = false;
      for (int t = blockIdx.x; t < ntiles && !stop && !f4_aborted(S); t += gridDim.x) {
        const int4 it = __ldg(p.items + skip + t / MT);
        const int row0 = it.y, n = it.z;
        // the shortest box that covers the tile; rows past it are not read by the MMA's N
        const CUtensorMap* tm = n <= 32 ? &tm_b32 : n <= 64 ? &tm_b64 : &tm_b128;
        const uint32_t box_bytes = (n <= 32 ? 32u : n <= 64 ? 64u : 128u) * 128u;
        for (int ks = 0; ks < NK; ++ks, ++kg) {
          const int s = kg % kF4Stages;
          if (kg >= kF4Stages && !ptx::mbar_wait_ns(&S.empty[s], ((kg / kF4Stages) - 1) & 1, lim)) {
            f4_abort(S, p.status);
            stop = true;
            break;
          }
          ptx::mbar_arrive_expect_tx(&S.full[s], box_bytes);
          ptx::tma_load_2d(S.b[s], tm, ks * 128, row0, &S.full[s]);
        }
      }
    }
  } else if (warp == kF4WarpSF) {
    // --------------------------------------------------- activation scale stager
    // Lane l owns token rows l, 32 + l, 64 + l, 96 + l of the tile; a round loads their 16
    // scale bytes for up to four stages, then fills each stage's block: MMA kk's 512 bytes
    // hold, at 16 r + 4 q, the four scale bytes (K blocks 16 ks + 4 kk ..) of token row
    // 32 q + r. Rows at or past n get zero scales.
    const int sf_row = p.K / 16;
    int kg = 0;
    bool stop = false;
    for (int t = blockIdx.x; t < ntiles && !stop; t += gridDim.x) {
      if (__any_sync(0xffffffffu, f4_aborted(S))) break;
      const int4 it = __ldg(p.items + skip + t / MT);
      const int row0 = it.y, n = it.z;
      for (int ks0 = 0; ks0 < NK && !stop; ks0 += 4) {
        uint4 v[4][4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int r = lane + 32 * q;
            v[j][q] = make_uint4(0u, 0u, 0u, 0u);
            if (ks0 + j < NK && r < n)
              v[j][q] = __ldg(reinterpret_cast<const uint4*>(p.asf + (size_t)(row0 + r) * sf_row) + ks0 + j);
          }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (ks0 + j >= NK) break;
          const int s = kg % kF4Stages;
          const bool ok = kg < kF4Stages || ptx::mbar_wait_ns(&S.empty[s], ((kg / kF4Stages) - 1) & 1, lim);
          if (!__all_sync(0xffffffffu, ok)) {
            if (lane == 0) f4_abort(S, p.status);
            stop = true;
            break;
          }
          uint32_t* dst = reinterpret_cast<uint32_t*>(S.sfb[s]) + lane * 4;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            dst[q] = v[j][q].x;
            dst[128 + q] = v[j][q].y;
            dst[256 + q] = v[j][q].z;
            dst[384 + q] = v[j][q].w;
          }
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&S.full[s]);
          ++kg;
        }
      }
    }
  } else if (warp == kF4WarpMma) {
    // ------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int kg = 0, tc = 0;
      bool stop = false;
      for (int t = blockIdx.x; t < ntiles && !stop && !f4_aborted(S); t += gridDim.x, ++tc) {
        const int4 it = __ldg(p.items + skip + t / MT);
        const int N = ((it.z + 15) / 16) * 16;
        const uint32_t idesc = ptx::fp4_idesc(kF4BM, N);
        const int buf = tc & 1;
        if (tc >= 2 && !ptx::mbar_wait_ns(&S.tmem_empty[buf], ((tc >> 1) - 1) & 1, lim)) {
          f4_abort(S, p.status);
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(buf * kF4AccCols);
        for (int ks = 0; ks < NK; ++ks, ++kg) {
          const int s = kg % kF4Stages;
          if (!ptx::mbar_wait_ns(&S.full[s], (kg / kF4Stages) & 1, lim)) {
            f4_abort(S, p.status);
            stop = true;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t sf = tmem + (uint32_t)(2 * kF4AccCols + s * kF4SfCols);
          const uint32_t a0 = ptx::smem_u32(S.a[s]), b0 = ptx::smem_u32(S.b[s]);
          const uint32_t sa = ptx::smem_u32(S.sfa[s]), sb = ptx::smem_u32(S.sfb[s]);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            ptx::tc_cp_32x128b_x4(sf + 4 * kk, ptx::kmajor_desc(sa + 512 * kk, 128, 128));
            ptx::tc_cp_32x128b_x4(sf + 16 + 4 * kk, ptx::kmajor_desc(sb + 512 * kk, 128, 128));
          }
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            ptx::tc_mma_fp4(d, ptx::sw128_desc(a0 + 32 * kk), ptx::sw128_desc(b0 + 32 * kk), idesc, sf + 4 * kk,
                            sf + 16 + 4 * kk, (ks | kk) != 0 ? 1u : 0u);
          ptx::tc_commit(&S.empty[s]);
        }
        if (stop) break;
        ptx::tc_commit(&S.tmem_full[buf]);
      }
    }
  } else {
    // ------------------------------------------------------ epilogue (warps 0-3)
    int tc = 0;
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++tc) {
      const int4 it = __ldg(p.items + skip + t / MT);
      const int e = it.x, row0 = it.y, n = it.z, mt = t % MT;
      const int N = ((n + 15) / 16) * 16;
      const int buf = tc & 1;
      const bool ok = ptx::mbar_wait_ns(&S.tmem_full[buf], (tc >> 1) & 1, lim);
      if (!ok) f4_abort(S, p.status);
      if (__any_sync(0xffffffffu, !ok || f4_aborted(S))) break;
      ptx::tc_fence_after();
      const float sc_out = __ldg(p.w_tscale + e) * __fdiv_rn(__uint_as_float(__ldg(p.act_amax)), 2688.0f);
      gemm_tile_epilogue<true, EPI>(tmem + (uint32_t)(buf * kF4AccCols) + ((uint32_t)(32 * warp) << 16), N, n, row0,
                                    mt, sc_out, p);
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&S.tmem_empty[buf]);
    }
  }

  // ---------------------------------------------------------------------- teardown
  ptx::tc_fence_before();
  __syncthreads();
  if (f4_aborted(S) && threadIdx.x == 0) {
    // copies and MMAs issued before the abort complete on their own; give them time to land
    for (int i = 0; i < 2000; ++i) __nanosleep(1000);
  }
  if (warp == kF4WarpMma) {
    if (f4_aborted(S) && lane == 0) {
      ptx::tc_commit(&S.mma_done);
      ptx::mbar_wait_ns(&S.mma_done, 0, 100000000ull);
    }
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kF4TmemCols);
  }
}

// Row of the row-major store held by row r of 128-row tile mt of the FP4 weight store: the
// gate/up tiles interleave 16 gate rows and the 16 up rows of the same h columns per warp
// quarter (the pairing gemm_tile_epilogue reads), the down tiles keep the row order.
__device__ __forceinline__ int fp4_src_row(int r, int mt, bool gate_up, int I) {
  if (!gate_up) return 128 * mt + r;
  const int w = r >> 5, l = r & 31;
  return l < 16 ? 64 * mt + 16 * w + l : I + 64 * mt + 16 * w + (l - 16);
}

// FP4 weight store, written once at layer creation from the row-major NVFP4 store (codes
// [rows][K/2], low nibble = even element; E4M3 scales [rows][K/16]):
//   codes  [n_exp * rows][K/2]: the same bytes, rows in tile order (fp4_src_row);
//   scales per (expert, 128-row tile, 256-column stage) 2048 bytes: MMA kk's 512 bytes
//          hold at 16 r + 4 q + c the scale of tile row 32 q + r for columns
//          256 ks + 64 kk + 16 c .. + 15 (the order tcgen05.cp puts into TMEM).
__global__ void fp4_pack_kernel(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ scales, int K,
                                int n_exp, int rows, int I, int gate_up, uint8_t* __restrict__ dcodes,
                                uint8_t* __restrict__ dsf) {
  const size_t row_bytes = (size_t)K / 2, sf_bytes = (size_t)K / 16;
  const size_t chunks = row_bytes / 16;
  const size_t n_code = (size_t)n_exp * rows * chunks;
  const int MT = rows / 128, NK = K / 256;
  const size_t n_sf = (size_t)n_exp * MT * NK * 4 * 32;
  for (size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x; idx < n_code + n_sf;
       idx += (size_t)gridDim.x * blockDim.x) {
    if (idx < n_code) {
      const size_t drow = idx / chunks, ch = idx % chunks;
      const int e = (int)(drow / rows), r = (int)(drow % rows);
      const size_t srow = (size_t)e * rows + fp4_src_row(r % 128, r / 128, gate_up != 0, I);
      *reinterpret_cast<uint4*>(dcodes + drow * row_bytes + ch * 16) =
          *reinterpret_cast<const uint4*>(codes + srow * row_bytes + ch * 16);
    } else {
      size_t j = idx - n_code;
      const int r = (int)(j % 32);
      j /= 32;
      const int kk = (int)(j % 4);
      j /= 4;
      const int ks = (int)(j % NK);
      j /= NK;
      const int mt = (int)(j % MT);
      const int e = (int)(j / MT);
      uint32_t w[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const size_t srow = (size_t)e * rows + fp4_src_row(32 * q + r, mt, gate_up != 0, I);
        const uint8_t* src = scales + srow * sf_bytes + 16 * ks + 4 * kk;
        w[q] = (uint32_t)src[0] | ((uint32_t)src[1] << 8) | ((uint32_t)src[2] << 16) | ((uint32_t)src[3] << 24);
      }
      uint8_t* dst = dsf + ((((size_t)e * MT + mt) * NK + ks) * 4 + kk) * 512 + (size_t)r * 16;
      *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

// One 16-element NVFP4 block -> 8 bytes of packed codes (element 2j in the low nibble of
// byte j) and its E4M3 scale byte.
__device__ __forceinline__ void fp4_block_store(const float (&v)[16], float ts, uint8_t* codes8, uint8_t* sbyte) {
  uint32_t sb, nib[16];
  nvfp4_block_bits(v, ts, sb, nib);
  uint32_t w[2] = {0u, 0u};
#pragma unroll
  for (int i = 0; i < 16; ++i) w[i >> 3] |= nib[i] << (4 * (i & 7));
  *reinterpret_cast<uint2*>(codes8) = make_uint2(w[0], w[1]);
  *sbyte = (uint8_t)sb;
}

// Activation rows of the FP4 gate/up GEMM: sorted row q (< T * top_k) is token
// entries[q] / top_k quantised to NVFP4 with the per-call tensor scale ts = amax / 2688:
// codes [q][H/2], scales [q][H/16]. One CTA per sorted row.
template <int XDT>
__global__ void __launch_bounds__(256)
quant_gather_fp4_kernel(const void* __restrict__ x, int H, const int32_t* __restrict__ entries, int top_k,
                        const unsigned int* __restrict__ amax_bits, uint8_t* __restrict__ codes,
                        uint8_t* __restrict__ sf) {
  const int q = blockIdx.x;
  const int tok = __ldg(entries + q) / top_k;
  const float ts = __fdiv_rn(__uint_as_float(__ldg(amax_bits)), 2688.0f);
  for (int b = threadIdx.x; b < H / 16; b += 256) {
    float v[16];
    {
      float v0[8], v1[8];
      load8_act<XDT>(x, (size_t)tok * H + 16 * b, v0);
      load8_act<XDT>(x, (size_t)tok * H + 16 * b + 8, v1);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        v[j] = v0[j];
        v[8 + j] = v1[j];
      }
    }
    fp4_block_store(v, ts, codes + (size_t)q * (H / 2) + 8 * b, sf + (size_t)q * (H / 16) + b);
  }
}

// h of the FP4 down GEMM: the fp32 routed h rows [T * top_k][I] quantised with the per-call
// tensor scale (amax of all routed h / 2688) into codes [.][I/2] and scales [.][I/16].
__global__ void __launch_bounds__(256)
quant_h_fp4_kernel(const float* __restrict__ h, size_t nblocks, const unsigned int* __restrict__ amax_bits,
                   uint8_t* __restrict__ codes, uint8_t* __restrict__ sf) {
  const float ts = __fdiv_rn(__uint_as_float(__ldg(amax_bits)), 2688.0f);
  for (size_t b = (size_t)blockIdx.x * 256 + threadIdx.x; b < nblocks; b += (size_t)gridDim.x * 256) {
    float v[16];
    const float4* src = reinterpret_cast<const float4*>(h + b * 16);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float4 f = src[j];
      v[4 * j] = f.x;
      v[4 * j + 1] = f.y;
      v[4 * j + 2] = f.z;
      v[4 * j + 3] = f.w;
    }
    fp4_block_store(v, ts, codes + 8 * b, sf + b);
  }
}

template <int EPI>
cudaError_t launch_fp4_t(const Fp4Maps& m, const GemmParams& p, int grid, cudaStream_t s) {
  moe_gemm_fp4_kernel<EPI><<<grid, kF4Threads, kF4SmemBytes, s>>>(
      *reinterpret_cast<const CUtensorMap*>(&m.w), *reinterpret_cast<const CUtensorMap*>(&m.act[0]),
      *reinterpret_cast<const CUtensorMap*>(&m.act[1]), *reinterpret_cast<const CUtensorMap*>(&m.act[2]), p);
  return cudaGetLastError();
}

size_t grid_for(size_t n) {
  size_t g = (n + 255) / 256;
  if (g > 148 * 16) g = 148 * 16;
  return g ? g : 1;
}

}  // namespace

bool fp4_gemm_supported(int H, int I) { return H % 256 == 0 && I % 256 == 0 && H >= 256 && I >= 256; }

cudaError_t fp4_gemm_init() {
  cudaError_t e0 = cudaFuncSetAttribute(moe_gemm_fp4_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)kF4SmemBytes);
  cudaError_t e1 = cudaFuncSetAttribute(moe_gemm_fp4_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)kF4SmemBytes);
  return e0 != cudaSuccess ? e0 : e1;
}

size_t fp4_scale_bytes(int rows, int K, int n_exp) { return (size_t)n_exp * rows * (K / 16); }

cudaError_t launch_fp4_pack(const uint8_t* codes, const uint8_t* scales, int K, int n_exp, int rows, int I,
                            bool gate_up, uint8_t* dcodes, uint8_t* dsf, cudaStream_t s) {
  fp4_pack_kernel<<<148 * 8, 256, 0, s>>>(codes, scales, K, n_exp, rows, I, gate_up ? 1 : 0, dcodes, dsf);
  return cudaGetLastError();
}

cudaError_t launch_quant_gather_fp4(const void* x, int act_dtype, int H, const int32_t* entries, int Tk, int top_k,
                                    const unsigned int* amax_bits, uint8_t* codes, uint8_t* sf, cudaStream_t s) {
  if (Tk <= 0) return cudaSuccess;
  if (act_dtype == MOE_DT_F32)
    quant_gather_fp4_kernel<MOE_DT_F32><<<Tk, 256, 0, s>>>(x, H, entries, top_k, amax_bits, codes, sf);
  else
    quant_gather_fp4_kernel<MOE_DT_BF16><<<Tk, 256, 0, s>>>(x, H, entries, top_k, amax_bits, codes, sf);
  return cudaGetLastError();
}

cudaError_t launch_quant_h_fp4(const float* h, size_t n, const unsigned int* amax_bits, uint8_t* codes, uint8_t* sf,
                               cudaStream_t s) {
  const size_t nb = n / 16;
  if (nb == 0) return cudaSuccess;
  quant_h_fp4_kernel<<<(int)grid_for(nb), 256, 0, s>>>(h, nb, amax_bits, codes, sf);
  return cudaGetLastError();
}

cudaError_t launch_gemm_fp4(int epi, const Fp4Maps& m, const GemmParams& p, int max_tiles, int n_sm, cudaStream_t s) {
  if (max_tiles <= 0) return cudaSuccess;
  const int grid = max_tiles < n_sm ? max_tiles : n_sm;
  return epi == 0 ? launch_fp4_t<0>(m, p, grid, s) : launch_fp4_t<1>(m, p, grid, s);
}

}  // namespace moe
