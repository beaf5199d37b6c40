// Grouped expert GEMMs of NVFP4 layers on the block-scaled FP4 tensor cores ("NVIDIA stellt
// neues GLM-5.2 NVFP4 Modell vor", section "Technische Details und Quantisierungsansatz":
// E2M1 elements with one FP8 E4M3 scale per 16 elements and an fp32 tensor scale). Both
// operands stay in their 4-bit storage all the way into the tensor core: tcgen05.mma
// kind::mxf4nvf4 multiplies E2M1 codes block-scaled by their E4M3 scales and accumulates in
// fp32; the two fp32 tensor scales multiply the accumulator in the epilogue.
//
// A tile is D = W[128 rows, K] . X[n <= 160 tokens, K]^T of one expert (weight rows on the
// MMA's M side, the expert's tokens on N, as in the fp16 kernel), K walked in stages of 256
// elements: one 128-byte row of packed codes per weight row and per token, four MMAs of
// K = 64 each. Persistent CTAs walk the tiles (item, 128-row block) round-robin; warp roles:
//   warp 8     TMA of the stage's 128 x 128-byte weight codes (128-byte swizzle) and one bulk
//              copy of its 2 KB of weight scales (laid out per MMA as 32 x 16 bytes)
//   warp 9     TMA of the stage's n x 128-byte activation codes (boxes of 32, 64, 128 or 160
//              rows)
//   warps 4-7  scales into TMEM: warp 4 + q writes lanes 32q..32q+31 of the stage's scale
//              slot with tcgen05.st, the same values in every lane quarter (the block-scaled
//              MMA reads the scales of row 32 j + l from lane l, column j): the weight scales
//              from shared memory, the activation scales (16 bytes per token and stage) from
//              the row-major scale matrix, loaded four stages per round
//   warp 10    issues the four MMAs of a stage once its operands and scales are in place and
//              releases both rings' stages by commit (4 MMAs and 2 commits per stage: the
//              single issuing thread is the kernel's narrowest resource)
//   warps 0-3  epilogue of the previous tile from the other TMEM accumulator
//              (gemm_tile_epilogue: SwiGLU h rows, or the weighted combine)
// Rings: weights 6 stages, activations 4; the activation stage's TMEM scale slot is freed
// with it (by the commit of the MMAs that read it). TMEM: two 160-column accumulators and
// four 48-column scale slots (16 weight-scale + 4 x 8 activation-scale columns).
// Every wait has a time limit (GemmParams::wait_ns); a time-out sets MOE_ERR_TIMEOUT, the
// CTA stops issuing work, lets copies and MMAs in flight land, frees its TMEM and exits.
#include <cuda.h>

#include "gemm_epi.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kF4WarpSc = 4;              // warps 4-7: scales into TMEM
constexpr int kF4WarpW = 8;
constexpr int kF4WarpB = 9;
constexpr int kF4WarpMma = 10;
constexpr int kF4Threads = 11 * 32;
constexpr int kF4BM = 128;
constexpr int kF4BN = kFp4MaxN;
constexpr int kF4BK = 256;                // K elements per stage (128 bytes of codes per row)
constexpr int kF4WStages = 6;             // weight ring
constexpr int kF4BStages = 4;             // activation ring = TMEM scale slots
constexpr int kF4A = kF4BM * 128;         // 16 KB of weight codes
constexpr int kF4B = kF4BN * 128;         // 20 KB of activation codes
constexpr int kF4SFA = 4 * 512;           // 4 MMAs x (32 rows x 16 bytes) of weight scales
constexpr int kF4AccCols = 160;
constexpr int kF4SlotCols = 48;           // 4 MMAs x 4 weight-scale + 4 MMAs x 8 activation-scale
constexpr int kF4NB = kF4BN / 32;         // activation-scale columns used per MMA (5)
constexpr uint32_t kF4TmemCols = 512;
static_assert(kF4BN % 32 == 0 && kF4NB <= 8, "activation scale columns per MMA");
static_assert(2 * kF4AccCols + kF4BStages * kF4SlotCols <= (int)kF4TmemCols, "TMEM budget");

struct F4Smem {
  uint8_t a[kF4WStages][kF4A];
  uint8_t b[kF4BStages][kF4B];
  uint8_t sfa[kF4WStages][kF4SFA];
  uint64_t full_w[kF4WStages];
  uint64_t empty_w[kF4WStages];
  uint64_t full_b[kF4BStages];
  uint64_t empty_b[kF4BStages];
  uint64_t sf_full[kF4BStages];
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
                    const __grid_constant__ CUtensorMap tm_b160, const GemmParams p) {
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
    for (int s = 0; s < kF4WStages; ++s) {
      ptx::mbar_init(&S.full_w[s], 1);    // weight copies (+ tx)
      ptx::mbar_init(&S.empty_w[s], 1);   // tcgen05.commit
    }
    for (int s = 0; s < kF4BStages; ++s) {
      ptx::mbar_init(&S.full_b[s], 1);    // activation copy (+ tx)
      ptx::mbar_init(&S.empty_b[s], 1);   // tcgen05.commit
      ptx::mbar_init(&S.sf_full[s], 4);   // the four scale warps
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
        const uint8_t* sf = p.wsf + ((size_t)e * MT + mt) * (size_t)NK * kF4SFA;
        for (int ks = 0; ks < NK; ++ks, ++kg) {
          const int s = kg % kF4WStages;
          if (kg >= kF4WStages && !ptx::mbar_wait_ns(&S.empty_w[s], ((kg / kF4WStages) - 1) & 1, lim)) {
            f4_abort(S, p.status);
            stop = true;
            break;
          }
          ptx::mbar_arrive_expect_tx(&S.full_w[s], kF4A + kF4SFA);
          ptx::tma_load_2d(S.a[s], &tm_w, ks * 128, wrow, &S.full_w[s]);
          ptx::bulk_g2s(S.sfa[s], sf + (size_t)ks * kF4SFA, kF4SFA, &S.full_w[s], ptx::policy_evict_first());
        }
      }
    }
  } else if (warp == kF4WarpB) {
    // ---------------------------------------------------- activation code producer
    if (lane == 0) {
      ptx::prefetch_tmap(&tm_b32);
      ptx::prefetch_tmap(&tm_b64);
      ptx::prefetch_tmap(&tm_b128);
      ptx::prefetch_tmap(&tm_b160);
      int kg = 0;
      bool stop = false;
      for (int t = blockIdx.x; t < ntiles && !stop && !f4_aborted(S); t += gridDim.x) {
        const int4 it = __ldg(p.items + skip + t / MT);
        const int row0 = it.y, n = it.z;
        // the shortest box that covers the tile; rows past it are not read by the MMA's N
        const CUtensorMap* tm = n <= 32 ? &tm_b32 : n <= 64 ? &tm_b64 : n <= 128 ? &tm_b128 : &tm_b160;
        const uint32_t box_bytes = (n <= 32 ? 32u : n <= 64 ? 64u : n <= 128 ? 128u : 160u) * 128u;
        for (int ks = 0; ks < NK; ++ks, ++kg) {
          const int s = kg % kF4BStages;
          if (kg >= kF4BStages && !ptx::mbar_wait_ns(&S.empty_b[s], ((kg / kF4BStages) - 1) & 1, lim)) {
            f4_abort(S, p.status);
            stop = true;
            break;
          }
          ptx::mbar_arrive_expect_tx(&S.full_b[s], box_bytes);
          ptx::tma_load_2d(S.b[s], tm, ks * 128, row0, &S.full_b[s]);
        }
      }
    }
  } else if (warp >= kF4WarpSc && warp < kF4WarpSc + 4) {
    // ------------------------------------------------------- scales into TMEM
    // Lane l holds, per MMA kk of the stage, the four scale bytes (K blocks 16 ks + 4 kk ..)
    // of weight rows 32 j + l (j < 4; column 4 kk + j of the slot) and of token rows
    // 32 c + l (c < 5; column 16 + 8 kk + c). Token rows at or past n get zero scales.
    const uint32_t lane_base = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)(2 * kF4AccCols);
    const int sf_row = p.K / 16;
    int kg = 0;
    bool stop = false;
    for (int t = blockIdx.x; t < ntiles && !stop; t += gridDim.x) {
      if (__any_sync(0xffffffffu, f4_aborted(S))) break;
      const int4 it = __ldg(p.items + skip + t / MT);
      const int row0 = it.y, n = it.z;
      for (int ks0 = 0; ks0 < NK && !stop; ks0 += 4) {
        uint4 v[4][kF4NB];
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
          for (int c = 0; c < kF4NB; ++c) {
            const int r = lane + 32 * c;
            v[j][c] = make_uint4(0u, 0u, 0u, 0u);
            if (ks0 + j < NK && r < n)
              v[j][c] = __ldg(reinterpret_cast<const uint4*>(p.asf + (size_t)(row0 + r) * sf_row) + ks0 + j);
          }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (ks0 + j >= NK) break;
          const int sw = kg % kF4WStages, sb = kg % kF4BStages;
          // the weight scales have landed; the slot's previous MMAs have completed
          const bool ok = ptx::mbar_wait_ns(&S.full_w[sw], (kg / kF4WStages) & 1, lim) &&
                          (kg < kF4BStages || ptx::mbar_wait_ns(&S.empty_b[sb], ((kg / kF4BStages) - 1) & 1, lim));
          if (!__all_sync(0xffffffffu, ok)) {
            if (lane == 0) f4_abort(S, p.status);
            stop = true;
            break;
          }
          uint32_t lo[16], hi[32];
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint4 a = *reinterpret_cast<const uint4*>(S.sfa[sw] + kk * 512 + lane * 16);
            lo[4 * kk] = a.x;
            lo[4 * kk + 1] = a.y;
            lo[4 * kk + 2] = a.z;
            lo[4 * kk + 3] = a.w;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              uint32_t w = 0u;
              if (c < kF4NB) w = kk == 0 ? v[j][c].x : kk == 1 ? v[j][c].y : kk == 2 ? v[j][c].z : v[j][c].w;
              hi[8 * kk + c] = w;
            }
          }
          const uint32_t col = lane_base + (uint32_t)(sb * kF4SlotCols);
          ptx::tmem_st16(col, lo);
          ptx::tmem_st32(col + 16, hi);
          ptx::tmem_wait_st();
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&S.sf_full[sb]);
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
          const int sw = kg % kF4WStages, sb = kg % kF4BStages;
          if (!ptx::mbar_wait_ns(&S.full_w[sw], (kg / kF4WStages) & 1, lim) ||
              !ptx::mbar_wait_ns(&S.full_b[sb], (kg / kF4BStages) & 1, lim) ||
              !ptx::mbar_wait_ns(&S.sf_full[sb], (kg / kF4BStages) & 1, lim)) {
            f4_abort(S, p.status);
            stop = true;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t sf = tmem + (uint32_t)(2 * kF4AccCols + sb * kF4SlotCols);
          const uint32_t a0 = ptx::smem_u32(S.a[sw]), b0 = ptx::smem_u32(S.b[sb]);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            ptx::tc_mma_fp4(d, ptx::sw128_desc(a0 + 32 * kk), ptx::sw128_desc(b0 + 32 * kk), idesc, sf + 4 * kk,
                            sf + 16 + 8 * kk, (ks | kk) != 0 ? 1u : 0u);
          ptx::tc_commit(&S.empty_w[sw]);
          ptx::tc_commit(&S.empty_b[sb]);
        }
        if (stop) break;
        ptx::tc_commit(&S.tmem_full[buf]);
      }
    }
  } else if (warp < 4) {
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

// NVFP4 activation of each token, once per call: x [T, H] quantised with the per-call
// tensor scale ts = amax / 2688 into codes [T][H/2] and scales [T][H/16]. One thread per
// 16-element block.
template <int XDT>
__global__ void __launch_bounds__(256)
quant_tokens_fp4_kernel(const void* __restrict__ x, size_t nblocks, const unsigned int* __restrict__ amax_bits,
                        uint8_t* __restrict__ codes, uint8_t* __restrict__ sf) {
  const float ts = __fdiv_rn(__uint_as_float(__ldg(amax_bits)), 2688.0f);
  for (size_t b = (size_t)blockIdx.x * 256 + threadIdx.x; b < nblocks; b += (size_t)gridDim.x * 256) {
    float v[16];
    {
      float v0[8], v1[8];
      load8_act<XDT>(x, 16 * b, v0);
      load8_act<XDT>(x, 16 * b + 8, v1);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        v[j] = v0[j];
        v[8 + j] = v1[j];
      }
    }
    fp4_block_store(v, ts, codes + 8 * b, sf + b);
  }
}

// Activation rows of the FP4 gate/up GEMM: sorted row q (< T * top_k) is a copy of token
// entries[q] / top_k's codes [q][H/2] and scales [q][H/16]. One CTA per sorted row.
__global__ void __launch_bounds__(256)
gather_fp4_rows_kernel(const uint8_t* __restrict__ tok_codes, const uint8_t* __restrict__ tok_sf, int H,
                       const int32_t* __restrict__ entries, int top_k, uint8_t* __restrict__ codes,
                       uint8_t* __restrict__ sf, int32_t* __restrict__ inv, const int32_t* __restrict__ n_routed) {
  const int q = blockIdx.x;
  if (q >= __ldg(n_routed)) return;   // past the routed rows (adaptive top-p)
  const int ent = __ldg(entries + q);
  const int tok = ent / top_k;
  if (threadIdx.x == 0) inv[ent] = q;   // sorted row of each (token, slot)
  const int nc = H / 32, ns = H / 256;   // 16-byte words of codes and of scales per row
  const uint4* sc = reinterpret_cast<const uint4*>(tok_codes + (size_t)tok * (H / 2));
  const uint4* ss = reinterpret_cast<const uint4*>(tok_sf + (size_t)tok * (H / 16));
  uint4* dc = reinterpret_cast<uint4*>(codes + (size_t)q * (H / 2));
  uint4* ds = reinterpret_cast<uint4*>(sf + (size_t)q * (H / 16));
  for (int i = threadIdx.x; i < nc + ns; i += 256) {
    if (i < nc) dc[i] = __ldg(sc + i);
    else ds[i - nc] = __ldg(ss + (i - nc));
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

size_t grid_for(size_t n) {
  size_t g = (n + 255) / 256;
  if (g > 148 * 16) g = 148 * 16;
  return g ? g : 1;
}

template <int EPI>
cudaError_t launch_fp4_t(const Fp4Maps& m, const GemmParams& p, int grid, cudaStream_t s) {
  moe_gemm_fp4_kernel<EPI><<<grid, kF4Threads, kF4SmemBytes, s>>>(
      *reinterpret_cast<const CUtensorMap*>(&m.w), *reinterpret_cast<const CUtensorMap*>(&m.act[0]),
      *reinterpret_cast<const CUtensorMap*>(&m.act[1]), *reinterpret_cast<const CUtensorMap*>(&m.act[2]),
      *reinterpret_cast<const CUtensorMap*>(&m.act[3]), p);
  return cudaGetLastError();
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

cudaError_t launch_quant_gather_fp4(const void* x, int act_dtype, int H, int T, const int32_t* entries, int top_k,
                                    const unsigned int* amax_bits, uint8_t* tok_codes, uint8_t* tok_sf,
                                    uint8_t* codes, uint8_t* sf, int32_t* inv, const int32_t* n_routed,
                                    cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  const size_t nb = (size_t)T * H / 16;
  if (act_dtype == MOE_DT_F32)
    quant_tokens_fp4_kernel<MOE_DT_F32><<<(int)grid_for(nb), 256, 0, s>>>(x, nb, amax_bits, tok_codes, tok_sf);
  else
    quant_tokens_fp4_kernel<MOE_DT_BF16><<<(int)grid_for(nb), 256, 0, s>>>(x, nb, amax_bits, tok_codes, tok_sf);
  gather_fp4_rows_kernel<<<T * top_k, 256, 0, s>>>(tok_codes, tok_sf, H, entries, top_k, codes, sf, inv, n_routed);
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
