// Grouped expert GEMMs of the MoE layer on the tcgen05 tensor cores (the batch-union path
// for more than a handful of tokens: "Batch-union MoE" in "Show HN: Menjalankan GLM 5.2 di
// komputer lambat", section "Fitur utama yang diimplementasikan": each selected expert's
// weights are read once per call and applied to every token routed to it).
//
// A tile is D = W[128 rows, K] . X[N tokens, K]^T of one expert: weight rows on the MMA's M
// side, the expert's tokens (<= 256 rows of an expert-sorted activation matrix) on the N
// side, so a lightly loaded expert still fills the tensor core's M dimension. The quantised
// weights stay quantised in HBM and are dequantised on use (the packed int4
// "dequant-on-use" of the same section; NVFP4 blocks per "NVIDIA stellt neues GLM-5.2 NVFP4
// Modell vor", section "Technische Details und Quantisierungsansatz").
//
// Persistent CTAs (one per SM) walk the tiles (item, 128-row block) in a static round-robin
// order; warp roles:
//   warp 18    bulk copy of the packed weights: 128 rows x 256 columns of codes and their
//              scales per copy (18 KB, laid out at layer creation for conflict-free reads)
//   warps 4-15 dequantise 64 columns per K stage into an fp16 tile in the 128-byte swizzle
//              layout the MMA reads (int4 * fp16 scale rounded once to fp16; E2M1 * E4M3 is
//              exact in fp16, the fp32 tensor scales are applied in the epilogue); three
//              groups of 4 warps, one per ring slot, a thread converts one row of its stage
//   warp 16    TMA: the N x 64 fp16 activation tile of the same K stage (one box of 32, 64,
//              128 or 256 rows)
//   warp 17    issues tcgen05.mma kind::f16 (M=128, N, K=16) x 4 per stage into one of two
//              TMEM accumulators (256 columns each) and releases stages with tcgen05.commit
//   warps 0-3  epilogue of the previous tile while the next one runs (gemm_tile_epilogue):
//     gate/up: M rows pair 16 gate with 16 up rows per warp; h = SiLU(gate) * up is
//              written to the expert-sorted h matrix (fp16, or fp32 for NVFP4 layers
//              whose h is quantised next);
//     down:    the expert-sorted output rows y (fp32), combined per token afterwards.
// A separately stored bf16 shared expert (the NVFP4 layers keep it unquantised) is
// converted to fp16 once at layer creation (exact for its range, gate/up rows stored in tile
// order) and runs through the same kernel with each stage's 128-row weight tile loaded by
// one TMA box straight into the MMA's layout (kWF16).
// Every wait is bounded; a time-out sets MOE_ERR_TIMEOUT, the CTA stops issuing work, lets
// copies and MMAs in flight land, frees its TMEM and exits.
#include <cuda.h>

#include "gemm_epi.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kEpiWarps = 4;      // warps 0-3
constexpr int kDqWarp0 = 4;       // warps 4-15: three groups of 4, one per A/B ring slot
constexpr int kDqGroups = 3;
constexpr int kDqWarps = 4 * kDqGroups;
constexpr int kWarpB = kDqWarp0 + kDqWarps;
constexpr int kWarpMma = kWarpB + 1;
constexpr int kWarpW = kWarpB + 2;
constexpr int kGThreads = (kWarpW + 1) * 32;
constexpr int kBM = 128;          // weight rows per tile (MMA M)
constexpr int kBN = 256;          // max tokens per tile (MMA N)
constexpr int kBK = 64;           // K per stage: one 128-byte swizzle atom of fp16
constexpr int kSub = 4;           // K stages per packed weight group (256 columns)
constexpr int kABStages = 3;
constexpr int kWStages = 3;
constexpr int kAStage = kBM * kBK * 2;     // 16 KB fp16 weight tile
constexpr int kBStage = kBN * kBK * 2;     // 32 KB fp16 activation tile
constexpr int kGroupCodes = kBM * 128;     // 16 KB: 128 rows x 256 4-bit codes
constexpr int kGroupBytes = kGroupCodes + kBM * 16;   // + 2 KB of scales
constexpr int kBoxRows = 16;
constexpr int kAccCols = 256;
constexpr uint32_t kTmemCols = 2 * kAccCols;

struct GSmem {
  uint8_t a[kABStages][kAStage];
  uint8_t b[kABStages][kBStage];
  uint8_t w[kWStages][kGroupBytes];
  uint64_t full_ab[kABStages];
  uint64_t empty_ab[kABStages];
  uint64_t full_w[kWStages];
  uint64_t empty_w[kWStages];
  uint64_t tmem_full[2];
  uint64_t tmem_empty[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
};

constexpr size_t kGSmemBytes = sizeof(GSmem) + 1024;   // + alignment slack
static_assert(kGSmemBytes <= 227 * 1024, "grouped GEMM shared memory over the per-CTA limit");

// Wait on an mbarrier phase for at most limit_ns, adding the cycles spent to `acc`
// (profiling trace); false on time-out.
__device__ __forceinline__ bool wait_bar_t(uint64_t* bar, uint32_t parity, unsigned long long& acc,
                                           unsigned long long limit_ns) {
  const unsigned long long t0 = clock64();
  const bool ok = ptx::mbar_wait_ns(bar, parity, limit_ns);
  acc += clock64() - t0;
  return ok;
}

__device__ __forceinline__ void set_abort(GSmem& S, int* status) {
  atomicExch(&S.abort, 1);
  raise_status(status, MOE_ERR_TIMEOUT);
}

__device__ __forceinline__ bool aborted(const GSmem& S) { return *(volatile const int*)&S.abort != 0; }

__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 u2h(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

// Packed code word (see gemm_pack_kernel): element 2i at bits 4i..4i+3, element 2i+1 at bits
// 16+4i..; pair i (elements 2i, 2i+1) is (w >> 4i) & 0x000F000F.
// int4 (two's complement): (nibble ^ 8) in the mantissa of 1024 is 1032 + code exactly;
// subtracting 1032 is exact; the product with the fp16 scale is rounded once.
__device__ __forceinline__ uint4 dq_int4x8(uint32_t w, __half2 s2) {
  const __half2 k1032 = __float2half2_rn(1032.f);
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t p = ((w >> (4 * i)) & 0x000F000Fu) ^ 0x64086408u;
    o[i] = h2u(__hmul2(__hsub2(u2h(p), k1032), s2));
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// E2M1 x 8 -> fp16 x 8 times the block scale. The nibble's exponent and mantissa bits placed
// at fp16 bits 9-11 (sign at 15) give the E2M1 value times 2^-14 (its subnormal included);
// both products are exact in fp16.
__device__ __forceinline__ uint4 dq_e2m1x8(uint32_t w, __half2 s2) {
  const __half2 k2p14 = __float2half2_rn(16384.f);
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t p = (w >> (4 * i)) & 0x000F000Fu;
    const uint32_t bits = ((p & 0x00070007u) << 9) | ((p & 0x00080008u) << 12);
    o[i] = h2u(__hmul2(__hmul2(u2h(bits), k2p14), s2));
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// Non-negative E4M3 byte -> fp16 (exact): its 7 magnitude bits at fp16 bits 7-13 give the
// value times 2^-8 (subnormals included).
__device__ __forceinline__ __half e4m3_to_half(uint32_t b) {
  const __half v = __ushort_as_half((unsigned short)((b & 0x7Fu) << 7));
  return __hmul(v, __float2half(256.f));
}

template <int WFMT, int EPI>
__global__ void __launch_bounds__(kGThreads, 1)
moe_gemm_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_b32,
                const __grid_constant__ CUtensorMap tm_b64, const __grid_constant__ CUtensorMap tm_b128,
                const __grid_constant__ CUtensorMap tm_b256, const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  GSmem& S = *reinterpret_cast<GSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int MT = p.mtiles;
  const int n_items = __ldg(p.n_items);
  const int skip = p.item_skip ? __ldg(p.item_skip) : 0;
  const int ntiles = n_items * MT;
  if ((int)blockIdx.x >= ntiles) return;   // no tile for this CTA (uniform)
  const int NK = p.K / kBK;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned long long t_start = clock64();
  // optional per-CTA trace (cycles): [0] kernel, [1] MMA waiting operands, [2] MMA waiting
  // an accumulator, [3] dequant waiting weights, [4] dequant waiting a free stage, [5]
  // activation producer waiting, [6] weight producer waiting, [7] epilogue waiting, [8]
  // epilogue busy, [9] tiles, [10] dequant loop
  unsigned long long* tr = p.trace ? p.trace + (size_t)blockIdx.x * 64 + p.trace_base : nullptr;
  unsigned long long w0 = 0, w1 = 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kABStages; ++s) {
      // B producer (+ tx) and one dequant group (4 warps), or the two TMA producers (fp16
      // weights)
      ptx::mbar_init(&S.full_ab[s], WFMT == kWF16 ? 2 : 1 + 4);
      ptx::mbar_init(&S.empty_ab[s], 1);   // tcgen05.commit
    }
    for (int s = 0; s < kWStages; ++s) {
      ptx::mbar_init(&S.full_w[s], 1);
      ptx::mbar_init(&S.empty_w[s], kDqWarps);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&S.tmem_full[b], 1);
      ptx::mbar_init(&S.tmem_empty[b], kEpiWarps);
    }
    ptx::mbar_init(&S.mma_done, 1);
    ptx::fence_mbar_init();
    S.abort = 0;
  }
  if (warp == kWarpMma) {
    ptx::tmem_alloc(&S.tmem_base, kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = S.tmem_base;

  if (warp == kWarpW) {
    // ------------------------------------------------------------ weight producer
    if (lane == 0) {
      if (WFMT == kWF16) ptx::prefetch_tmap(&tm_w);
      int kg = 0, wg = 0;
      for (int t = blockIdx.x; t < ntiles && !aborted(S); t += gridDim.x) {
        const int4 it = __ldg(p.items + skip + t / MT);
        const int e = it.x, mt = t % MT;
        if (WFMT == kWF16) {
          // fp16 weight tiles straight into the MMA's A stages
          for (int ks = 0; ks < NK; ++ks, ++kg) {
            const int s = kg % kABStages;
            if (kg >= kABStages && !wait_bar_t(&S.empty_ab[s], ((kg / kABStages) - 1) & 1, w0, p.wait_ns)) {
              set_abort(S, p.status);
              break;
            }
            ptx::mbar_arrive_expect_tx(&S.full_ab[s], kAStage);
            ptx::tma_load_2d(S.a[s], &tm_w, ks * kBK, (e - p.e_sub) * p.rows_per_expert + kBM * mt, &S.full_ab[s]);
          }
        } else {
          // expert -> packed-store index: through the HBM cache's slot table when the
          // experts live in host memory
          const int widx = p.slot_of ? __ldg(p.slot_of + e) : e - p.e_sub;
          const uint8_t* src = p.wpack + ((size_t)widx * MT + mt) * (size_t)(NK / kSub) * kGroupBytes;
          for (int g = 0; g < NK / kSub; ++g, ++wg) {
            const int s = wg % kWStages;
            if (wg >= kWStages && !wait_bar_t(&S.empty_w[s], ((wg / kWStages) - 1) & 1, w0, p.wait_ns)) {
              set_abort(S, p.status);
              break;
            }
            ptx::mbar_arrive_expect_tx(&S.full_w[s], kGroupBytes);
            ptx::bulk_g2s(S.w[s], src + (size_t)g * kGroupBytes, kGroupBytes, &S.full_w[s],
                          ptx::policy_evict_first());
          }
        }
      }
      if (tr) tr[6] = w0;
    }
  } else if (warp == kWarpB) {
    // ------------------------------------------------------- activation producer
    if (lane == 0) {
      ptx::prefetch_tmap(&tm_b32);
      ptx::prefetch_tmap(&tm_b64);
      ptx::prefetch_tmap(&tm_b128);
      ptx::prefetch_tmap(&tm_b256);
      int kg = 0;
      for (int t = blockIdx.x; t < ntiles && !aborted(S); t += gridDim.x) {
        const int4 it = __ldg(p.items + skip + t / MT);
        const int row0 = it.y, n = it.z;
        // one TMA box per stage, the shortest of 32/64/128/256 rows that covers the tile
        // (rows past the tile land in the stage buffer but the MMA's N stops short of them)
        const CUtensorMap* tm = n <= 32 ? &tm_b32 : n <= 64 ? &tm_b64 : n <= 128 ? &tm_b128 : &tm_b256;
        const uint32_t box_bytes = (n <= 32 ? 32u : n <= 64 ? 64u : n <= 128 ? 128u : 256u) * 128u;
        for (int ks = 0; ks < NK; ++ks, ++kg) {
          const int s = kg % kABStages;
          if (kg >= kABStages && !wait_bar_t(&S.empty_ab[s], ((kg / kABStages) - 1) & 1, w0, p.wait_ns)) {
            set_abort(S, p.status);
            break;
          }
          ptx::mbar_arrive_expect_tx(&S.full_ab[s], box_bytes);
          ptx::tma_load_2d(S.b[s], tm, ks * kBK, row0, &S.full_ab[s]);
        }
      }
      if (tr) tr[5] = w0;
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int kg = 0, tc = 0;
      for (int t = blockIdx.x; t < ntiles && !aborted(S); t += gridDim.x, ++tc) {
        const int4 it = __ldg(p.items + skip + t / MT);
        const int N = ((it.z + kBoxRows - 1) / kBoxRows) * kBoxRows;
        const uint32_t idesc = ptx::f16_idesc(kBM, N, false);
        const int buf = tc & 1;
        if (tc >= 2 && !wait_bar_t(&S.tmem_empty[buf], ((tc >> 1) - 1) & 1, w1, p.wait_ns)) {
          set_abort(S, p.status);
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(buf * kAccCols);
        for (int ks = 0; ks < NK; ++ks, ++kg) {
          const int s = kg % kABStages;
          if (!wait_bar_t(&S.full_ab[s], (kg / kABStages) & 1, w0, p.wait_ns)) {
            set_abort(S, p.status);
            break;
          }
          ptx::tc_fence_after();
          const uint32_t a0 = ptx::smem_u32(S.a[s]), b0 = ptx::smem_u32(S.b[s]);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            ptx::tc_mma_f16(d, ptx::sw128_desc(a0 + 32 * kk), ptx::sw128_desc(b0 + 32 * kk), idesc,
                            (ks | kk) != 0 ? 1u : 0u);
          ptx::tc_commit(&S.empty_ab[s]);
        }
        ptx::tc_commit(&S.tmem_full[buf]);
      }
      if (tr) {
        tr[1] = w0;
        tr[2] = w1;
        tr[9] = tc;
      }
    }
  } else if (warp >= kDqWarp0) {
    // ------------------------------------------------ dequantisers (warps 4-15)
    // Group j of 4 warps takes the K stages of ring slot j (kg mod 3 == j); a thread
    // converts one whole 64-column row of its stage, then fences once for the tensor core.
    // Within a packed weight group (4 K stages) a dequant group waits for the weights
    // before its first stage (kq <= 2) and releases them after its last (kq >= 1).
    if (WFMT != kWF16) {
      const int dq = threadIdx.x - kDqWarp0 * 32;
      const int grp = dq >> 7, r = dq & (kBM - 1);
      uint8_t* const arow_base = &S.a[0][0] + (r >> 3) * 1024 + (r & 7) * 128;
      unsigned long long w0d = 0, w1d = 0;
      int kg = 0, wg = 0;
      bool stop = false;
      for (int t = blockIdx.x; t < ntiles && !stop; t += gridDim.x) {
        for (int ks = 0; ks < NK; ++ks, ++kg) {
          const int kq = ks % kSub, ws = wg % kWStages;
          const int s = kg % kABStages;
          if (s == grp) {
            if (kq <= kSub - 2 && !wait_bar_t(&S.full_w[ws], (wg / kWStages) & 1, w0d, p.wait_ns)) set_abort(S, p.status);
            if (kg >= kABStages && !wait_bar_t(&S.empty_ab[s], ((kg / kABStages) - 1) & 1, w1d, p.wait_ns))
              set_abort(S, p.status);
            if (__any_sync(0xffffffffu, aborted(S))) {   // warp-uniform exit
              stop = true;
              break;
            }
            uint8_t* arow = arow_base + s * kAStage;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int slot = (kq * 2 + h) * kBM + r;
              const uint4 q = *reinterpret_cast<const uint4*>(S.w[ws] + slot * 16);
              const uint32_t sc = *reinterpret_cast<const unsigned short*>(S.w[ws] + kGroupCodes + slot * 2);
              uint4 o[4];
              if (WFMT == MOE_W_INT4_G32) {
                const __half2 s2 = __half2half2(__ushort_as_half((unsigned short)sc));
                o[0] = dq_int4x8(q.x, s2);
                o[1] = dq_int4x8(q.y, s2);
                o[2] = dq_int4x8(q.z, s2);
                o[3] = dq_int4x8(q.w, s2);
              } else {
                const __half2 s0 = __half2half2(e4m3_to_half(sc & 0xFFu));
                const __half2 s1 = __half2half2(e4m3_to_half(sc >> 8));
                o[0] = dq_e2m1x8(q.x, s0);
                o[1] = dq_e2m1x8(q.y, s0);
                o[2] = dq_e2m1x8(q.z, s1);
                o[3] = dq_e2m1x8(q.w, s1);
              }
#pragma unroll
              for (int j = 0; j < 4; ++j)
                *reinterpret_cast<uint4*>(arow + (((4 * h + j) ^ (r & 7)) << 4)) = o[j];
            }
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              ptx::mbar_arrive(&S.full_ab[s]);
              if (kq >= 1) ptx::mbar_arrive(&S.empty_w[ws]);   // this group's last stage here
            }
          }
          if (kq == kSub - 1) ++wg;
        }
      }
      if (tr && threadIdx.x == kDqWarp0 * 32) {
        tr[3] = w0d;
        tr[4] = w1d;
        tr[10] = clock64() - t_start;
      }
    }
  } else {
    // ------------------------------------------------------ epilogue (warps 0-3)
    int tc = 0;
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++tc) {
      const int4 it = __ldg(p.items + skip + t / MT);
      const int e = it.x, row0 = it.y, n = it.z, mt = t % MT;
      const int N = ((n + kBoxRows - 1) / kBoxRows) * kBoxRows;
      const int buf = tc & 1;
      if (!wait_bar_t(&S.tmem_full[buf], (tc >> 1) & 1, w0, p.wait_ns)) set_abort(S, p.status);
      if (__any_sync(0xffffffffu, aborted(S))) break;
      const unsigned long long t_busy = clock64();
      ptx::tc_fence_after();
      float sc_out = 1.f;
      if (WFMT == MOE_W_NVFP4)
        sc_out = __ldg(p.w_tscale + e) * __fdiv_rn(__uint_as_float(__ldg(p.act_amax)), 2688.0f);
      const uint32_t lane_addr = tmem + (uint32_t)(buf * kAccCols) + ((uint32_t)(32 * warp) << 16);
      gemm_tile_epilogue<WFMT == MOE_W_NVFP4, EPI>(lane_addr, N, n, row0, mt, sc_out, p);
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&S.tmem_empty[buf]);
      w1 += clock64() - t_busy;
    }
    if (tr && threadIdx.x == 0) {
      tr[7] = w0;
      tr[8] = w1;
    }
  }

  // ---------------------------------------------------------------------- teardown
  ptx::tc_fence_before();
  __syncthreads();
  if (tr && threadIdx.x == 0) tr[0] = clock64() - t_start;
  if (aborted(S) && threadIdx.x == 0) {
    // copies and MMAs issued before the abort complete on their own; give them time to land
    for (int i = 0; i < 2000; ++i) __nanosleep(1000);
  }
  if (warp == kWarpMma) {
    if (aborted(S) && lane == 0) {
      ptx::tc_commit(&S.mma_done);
      ptx::mbar_wait_ns(&S.mma_done, 0, 100000000ull);
    }
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

// Packed weights of the grouped GEMM, written once at layer creation from the row-major
// store (codes [rows][K/2], scales [rows][K/16 bytes]). Per (expert, 128-row tile, 256-column
// group), 18432 bytes: codes [k-stage 4][half 2][row 128][16 B] then scales
// [k-stage 4][half 2][row 128][2 B], so the dequantising thread of (row, half) reads 16
// consecutive bytes and its neighbours the next ones. The 16 bytes hold the 32 codes of
// columns 64 kq + 32 h .. of the row; word j holds columns 8j..8j+7 with column 8j + 2i in
// bits 4i..4i+3 and 8j + 2i + 1 in bits 16 + 4i... Scale bytes: int4 the fp16 scale of the
// 32 columns; NVFP4 the two E4M3 scales of its 16-column blocks. Gate/up tiles take gate rows
// 64 mt + 16 w + l and the matching up rows at tile rows 32 w + l and 32 w + 16 + l.
__global__ void gemm_pack_kernel(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ scales, int K,
                                 int n_exp, int rows_per_expert, int I, int gate_up, int mtiles,
                                 uint8_t* __restrict__ dst) {
  const int ngroups = K / 256;
  const size_t total = (size_t)n_exp * mtiles * ngroups * (kSub * 2 * kBM);   // (row, half, kq) entries
  const size_t sbytes = (size_t)K / 16;                                        // scale bytes per row
  for (size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += (size_t)gridDim.x * blockDim.x) {
    const int slot = (int)(idx % (kSub * 2 * kBM));           // (kq * 2 + h) * 128 + r
    const size_t grp = idx / (kSub * 2 * kBM);                // (e * mtiles + mt) * ngroups + g
    const int g = (int)(grp % ngroups);
    const int mt = (int)((grp / ngroups) % mtiles);
    const int e = (int)(grp / ((size_t)ngroups * mtiles));
    const int r = slot % kBM, h = (slot / kBM) & 1, kq = slot / (2 * kBM);
    int row;
    if (gate_up) {
      const int w = r >> 5, l = r & 31;
      row = (l < 16) ? 64 * mt + 16 * w + l : I + 64 * mt + 16 * w + (l - 16);
    } else {
      row = kBM * mt + r;
    }
    const size_t grow = (size_t)e * rows_per_expert + row;
    const int col0 = 256 * g + 64 * kq + 32 * h;
    const uint8_t* src = codes + grow * (K / 2) + col0 / 2;
    uint32_t words[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t w = 0;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t b = src[4 * j + i];   // columns 8j + 2i (low nibble), 8j + 2i + 1 (high)
        w |= (b & 15u) << (4 * i);
        w |= (b >> 4) << (16 + 4 * i);
      }
      words[j] = w;
    }
    uint8_t* out = dst + grp * kGroupBytes;
    *reinterpret_cast<uint4*>(out + (size_t)slot * 16) = make_uint4(words[0], words[1], words[2], words[3]);
    const uint8_t* ssrc = scales + grow * sbytes + col0 / 16;   // int4: fp16 of group col0/32
    out[kGroupCodes + (size_t)slot * 2] = ssrc[0];
    out[kGroupCodes + (size_t)slot * 2 + 1] = ssrc[1];
  }
}

// Items of the grouped GEMMs: chunks of <= `chunk` consecutive expert-sorted rows of one
// expert: the routed experts in id order, then the shared expert (index E) over all T
// tokens. n_items[0] = routed items, n_items[1] = shared items, n_items[2] = both.
__global__ void gemm_items_kernel(const int32_t* __restrict__ offsets, int E, int T, int top_k, int chunk,
                                  int4* __restrict__ items, int32_t* __restrict__ n_items) {
  // one warp: lane owns a contiguous run of experts; a warp scan gives its first item slot
  const int lane = threadIdx.x & 31;
  if (threadIdx.x >= 32) return;
  const int per = (E + 31) / 32;
  const int x0 = min(E, lane * per), x1 = min(E, x0 + per);
  int mine = 0;
  for (int x = x0; x < x1; ++x) mine += (offsets[x + 1] - offsets[x] + chunk - 1) / chunk;
  int incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  int pos = incl - mine;
  for (int x = x0; x < x1; ++x) {
    const int o = offsets[x], c = offsets[x + 1] - o;
    for (int j = 0; j < c; j += chunk) items[pos++] = make_int4(x, o + j, min(chunk, c - j), 0);
  }
  const int nr = __shfl_sync(0xffffffffu, incl, 31);
  const int nsh = (T + chunk - 1) / chunk;
  for (int j = lane; j < nsh; j += 32)
    items[nr + j] = make_int4(E, T * top_k + chunk * j, min(chunk, T - chunk * j), 0);
  if (lane == 0) {
    n_items[0] = nr;
    n_items[1] = nsh;
    n_items[2] = nr + nsh;
  }
}

// bf16 [rows][K] -> fp16. With gate_up, output row 128 mt + 32 w + l takes gate row
// 64 mt + 16 w + l (l < 16) or up row I + 64 mt + 16 w + (l - 16), the row order of the
// grouped GEMM's gate/up tiles, so one 128-row TMA box loads a whole tile.
__global__ void bf16_to_f16_kernel(const uint16_t* __restrict__ src, __half* __restrict__ dst, size_t rows, int K,
                                   int gate_up, int I) {
  const size_t n = rows * (size_t)K;
  for (size_t i = (size_t)blockIdx.x * 256 + threadIdx.x; i < n; i += (size_t)gridDim.x * 256) {
    const size_t r = i / K, c = i % K;
    size_t sr = r;
    if (gate_up) {
      const int mt = (int)(r / 128), w = (int)(r % 128) / 32, l = (int)(r % 32);
      sr = l < 16 ? 64 * mt + 16 * w + l : I + 64 * mt + 16 * w + (l - 16);
    }
    dst[i] = __float2half_rn(__uint_as_float((uint32_t)src[sr * K + c] << 16));
  }
}

// Expert-sorted activation rows for the gate/up GEMM: row q < T*k is the token of entry q,
// row T*k + t is token t (shared expert). x is converted to fp16, except that NVFP4 layers
// quantise the routed rows (q < T*k) to NVFP4 with the per-call tensor scale
// ts = amax / 2688: such a row holds code * block scale (exact in fp16) and ts is applied
// in the GEMM epilogue. The shared expert always reads the unquantised x.
template <int XDT, bool FP4>
__global__ void __launch_bounds__(256)
gather_act_kernel(const void* __restrict__ x, int H, const int32_t* __restrict__ entries, int Tk, int top_k,
                  int first_row, __half* __restrict__ dst, const __half* __restrict__ xq16,
                  int32_t* __restrict__ inv, const int32_t* __restrict__ n_routed) {
  const int q = first_row + (int)blockIdx.x;
  if (q < Tk && q >= __ldg(n_routed)) return;   // past the routed rows (adaptive top-p)
  const int ent = q < Tk ? __ldg(entries + q) : 0;
  const int tok = q < Tk ? ent / top_k : q - Tk;
  if (q < Tk && threadIdx.x == 0) inv[ent] = q;   // sorted row of each (token, slot)
  __half* drow = dst + (size_t)q * H;
  if (!FP4 || q >= Tk) {
    for (int i = threadIdx.x * 8; i < H; i += 256 * 8) {
      float v[8];
      load8_act<XDT>(x, (size_t)tok * H + i, v);
      uint4 o;
      o.x = h2u(__floats2half2_rn(v[0], v[1]));
      o.y = h2u(__floats2half2_rn(v[2], v[3]));
      o.z = h2u(__floats2half2_rn(v[4], v[5]));
      o.w = h2u(__floats2half2_rn(v[6], v[7]));
      *reinterpret_cast<uint4*>(drow + i) = o;
    }
  } else {
    // routed rows of an NVFP4 layer: copies of the token's quantised row
    const uint4* srow = reinterpret_cast<const uint4*>(xq16 + (size_t)tok * H);
    for (int i = threadIdx.x; i < H / 8; i += 256) reinterpret_cast<uint4*>(drow)[i] = __ldg(srow + i);
  }
}

// NVFP4 activations, once per token: each 16-element block as code * block scale in fp16
// (one thread per block; the tensor scale comes from the amax of all tokens).
template <int XDT>
__global__ void __launch_bounds__(256)
quant_tokens_fp4_kernel(const void* __restrict__ x, size_t nblocks, const unsigned int* __restrict__ amax_bits,
                        __half* __restrict__ xq16) {
  const float ts = __fdiv_rn(__uint_as_float(__ldg(amax_bits)), 2688.0f);
  for (size_t b = (size_t)blockIdx.x * 256 + threadIdx.x; b < nblocks; b += (size_t)gridDim.x * 256) {
    float v[16], c[16], sb;
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
    nvfp4_block(v, ts, sb, c);
    uint32_t o[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) o[j] = h2u(__floats2half2_rn(c[2 * j] * sb, c[2 * j + 1] * sb));
    uint4* d = reinterpret_cast<uint4*>(xq16 + 16 * b);
    d[0] = make_uint4(o[0], o[1], o[2], o[3]);
    d[1] = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

// NVFP4 h: quantise the fp32 routed h rows with the per-call tensor scale (amax of all routed
// h) into code * block scale in fp16.
__global__ void __launch_bounds__(256)
quant_h_kernel(const float* __restrict__ h, size_t nblocks, const unsigned int* __restrict__ amax_bits,
               __half* __restrict__ dst) {
  const float ts = __fdiv_rn(__uint_as_float(__ldg(amax_bits)), 2688.0f);
  for (size_t b = (size_t)blockIdx.x * 256 + threadIdx.x; b < nblocks; b += (size_t)gridDim.x * 256) {
    float v[16], c[16], sb;
    const float4* src = reinterpret_cast<const float4*>(h + b * 16);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float4 f = src[j];
      v[4 * j] = f.x;
      v[4 * j + 1] = f.y;
      v[4 * j + 2] = f.z;
      v[4 * j + 3] = f.w;
    }
    nvfp4_block(v, ts, sb, c);
    uint32_t o[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) o[j] = h2u(__floats2half2_rn(c[2 * j] * sb, c[2 * j + 1] * sb));
    uint4* d = reinterpret_cast<uint4*>(dst + b * 16);
    d[0] = make_uint4(o[0], o[1], o[2], o[3]);
    d[1] = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

// ----------------------------------------------------------------- tensor maps

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

template <int WFMT, int EPI>
cudaError_t launch_gemm_t(const GemmMaps& m, const GemmParams& p, int grid, cudaStream_t s) {
  moe_gemm_kernel<WFMT, EPI><<<grid, kGThreads, kGSmemBytes, s>>>(
      *reinterpret_cast<const CUtensorMap*>(&m.codes), *reinterpret_cast<const CUtensorMap*>(&m.act[0]),
      *reinterpret_cast<const CUtensorMap*>(&m.act[1]), *reinterpret_cast<const CUtensorMap*>(&m.act[2]),
      *reinterpret_cast<const CUtensorMap*>(&m.act[3]), p);
  return cudaGetLastError();
}

template <int WFMT, int EPI>
cudaError_t init_gemm_one() {
  return cudaFuncSetAttribute(moe_gemm_kernel<WFMT, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)kGSmemBytes);
}

}  // namespace

static_assert(sizeof(CUtensorMap) == sizeof(TensorMapBytes), "tensor map storage size");

bool make_tmap_2d(TensorMapBytes* out, const void* base, int elem_bytes, uint64_t inner, uint64_t rows,
                  uint32_t box_inner, uint32_t box_rows, bool swizzle128) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {inner * (uint64_t)elem_bytes};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t es[2] = {1, 1};
  const CUtensorMapDataType dt = elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  return fn(reinterpret_cast<CUtensorMap*>(out), dt, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool gemm_supported(int H, int I) { return H % 256 == 0 && I % 256 == 0 && H >= 256 && I >= 256; }

int gemm_max_items(int T, int top_k, int E, bool routed, bool shared, int chunk) {
  const long tk = (long)T * top_k;
  return (int)((routed ? tk / chunk + (tk < E ? tk : E) + 1 : 0) + (shared ? (T + chunk - 1) / chunk : 0));
}

cudaError_t gemm_kernels_init() {
  cudaError_t e = cudaSuccess;
  const cudaError_t r[] = {init_gemm_one<MOE_W_INT4_G32, 0>(), init_gemm_one<MOE_W_INT4_G32, 1>(),
                           init_gemm_one<MOE_W_NVFP4, 0>(),    init_gemm_one<MOE_W_NVFP4, 1>(),
                           init_gemm_one<kWF16, 0>(),          init_gemm_one<kWF16, 1>()};
  for (cudaError_t x : r)
    if (x != cudaSuccess) e = x;
  return e;
}

cudaError_t launch_gemm_items(const int32_t* offsets, int E, int T, int top_k, int chunk, int4* items,
                              int32_t* n_items, cudaStream_t s) {
  if (chunk < 16 || chunk > kBN) return cudaErrorInvalidValue;
  gemm_items_kernel<<<1, 32, 0, s>>>(offsets, E, T, top_k, chunk, items, n_items);
  return cudaGetLastError();
}

cudaError_t launch_bf16_to_f16(const void* src, void* dst, size_t rows, int K, bool gate_up, int I,
                               cudaStream_t s) {
  const size_t n = rows * (size_t)K;
  size_t g = (n + 255) / 256;
  if (g > 148 * 16) g = 148 * 16;
  bf16_to_f16_kernel<<<(int)(g ? g : 1), 256, 0, s>>>(static_cast<const uint16_t*>(src), static_cast<__half*>(dst),
                                                      rows, K, gate_up ? 1 : 0, I);
  return cudaGetLastError();
}

cudaError_t launch_gather_act(const void* x, int act_dtype, bool nvfp4, int H, const int32_t* entries, int Tk,
                              int top_k, int rows, __half* dst, const unsigned int* amax_bits, __half* xq16,
                              int32_t* inv, const int32_t* n_routed, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  const bool xf = act_dtype == MOE_DT_F32;
  if (nvfp4) {
    const int T = rows - Tk;
    const size_t nb = (size_t)T * H / 16;
    size_t g = (nb + 255) / 256;
    if (g > 148 * 16) g = 148 * 16;
    if (nb > 0) {
      if (xf) quant_tokens_fp4_kernel<MOE_DT_F32><<<(int)g, 256, 0, s>>>(x, nb, amax_bits, xq16);
      else quant_tokens_fp4_kernel<MOE_DT_BF16><<<(int)g, 256, 0, s>>>(x, nb, amax_bits, xq16);
    }
    if (xf)
      gather_act_kernel<MOE_DT_F32, true><<<rows, 256, 0, s>>>(x, H, entries, Tk, top_k, 0, dst, xq16, inv, n_routed);
    else
      gather_act_kernel<MOE_DT_BF16, true><<<rows, 256, 0, s>>>(x, H, entries, Tk, top_k, 0, dst, xq16, inv, n_routed);
  } else {
    if (xf)
      gather_act_kernel<MOE_DT_F32, false><<<rows, 256, 0, s>>>(x, H, entries, Tk, top_k, 0, dst, nullptr, inv,
                                                                n_routed);
    else
      gather_act_kernel<MOE_DT_BF16, false><<<rows, 256, 0, s>>>(x, H, entries, Tk, top_k, 0, dst, nullptr, inv,
                                                                 n_routed);
  }
  return cudaGetLastError();
}

cudaError_t launch_gather_shared_rows(const void* x, int act_dtype, int H, int Tk, int T, __half* dst,
                                      cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  if (act_dtype == MOE_DT_F32)
    gather_act_kernel<MOE_DT_F32, false><<<T, 256, 0, s>>>(x, H, nullptr, Tk, 1, Tk, dst, nullptr, nullptr, nullptr);
  else
    gather_act_kernel<MOE_DT_BF16, false><<<T, 256, 0, s>>>(x, H, nullptr, Tk, 1, Tk, dst, nullptr, nullptr, nullptr);
  return cudaGetLastError();
}

namespace {

// Weighted combine of the grouped path ("routed_scaling_factor"-scaled routing weights times
// each selected expert's output, plus the shared expert): out[t] = sum over routed slots j in
// ascending order of w[t, j] * y[inv[t k + j]], then + y[T k + t], in fp32, converted once to
// the activation dtype. A fixed order, so repeated calls give identical outputs. Slots the
// adaptive top-p dropped (id -1) are skipped.
template <int DT>
__global__ void __launch_bounds__(256)
combine_kernel(const float* __restrict__ y, const int32_t* __restrict__ inv, const int32_t* __restrict__ ids,
               const float* __restrict__ w, int T, int top_k, int H, void* __restrict__ out) {
  const int t = blockIdx.x;
  const int Tk = T * top_k;
  for (int h = threadIdx.x * 4; h < H; h += 256 * 4) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < top_k; ++j) {
      if (__ldg(ids + (size_t)t * top_k + j) < 0) continue;
      const float wj = __ldg(w + (size_t)t * top_k + j);
      const float4 v = __ldg(reinterpret_cast<const float4*>(y + (size_t)__ldg(inv + (size_t)t * top_k + j) * H + h));
      acc.x += wj * v.x;
      acc.y += wj * v.y;
      acc.z += wj * v.z;
      acc.w += wj * v.w;
    }
    const float4 sh = __ldg(reinterpret_cast<const float4*>(y + (size_t)(Tk + t) * H + h));
    acc.x += sh.x;
    acc.y += sh.y;
    acc.z += sh.z;
    acc.w += sh.w;
    if constexpr (DT == MOE_DT_F32) {
      *reinterpret_cast<float4*>(static_cast<float*>(out) + (size_t)t * H + h) = acc;
    } else {
      const __nv_bfloat162 p0 = __floats2bfloat162_rn(acc.x, acc.y), p1 = __floats2bfloat162_rn(acc.z, acc.w);
      uint2 o;
      o.x = *reinterpret_cast<const uint32_t*>(&p0);
      o.y = *reinterpret_cast<const uint32_t*>(&p1);
      *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(out) + (size_t)t * H + h) = o;
    }
  }
}

}  // namespace

cudaError_t launch_combine(const float* y, const int32_t* inv, const int32_t* ids, const float* weights, int T,
                           int top_k, int H, void* out, int act_dtype, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  if (act_dtype == MOE_DT_F32)
    combine_kernel<MOE_DT_F32><<<T, 256, 0, s>>>(y, inv, ids, weights, T, top_k, H, out);
  else
    combine_kernel<MOE_DT_BF16><<<T, 256, 0, s>>>(y, inv, ids, weights, T, top_k, H, out);
  return cudaGetLastError();
}

cudaError_t launch_quant_h(const float* h, size_t n, const unsigned int* amax_bits, __half* dst, cudaStream_t s) {
  const size_t nb = n / 16;
  if (nb == 0) return cudaSuccess;
  size_t g = (nb + 255) / 256;
  if (g > 148 * 16) g = 148 * 16;
  quant_h_kernel<<<(int)g, 256, 0, s>>>(h, nb, amax_bits, dst);
  return cudaGetLastError();
}

cudaError_t launch_gemm(int wfmt, int epi, const GemmMaps& m, const GemmParams& p, int max_tiles, int n_sm,
                        cudaStream_t s) {
  if (max_tiles <= 0) return cudaSuccess;
  const int grid = max_tiles < n_sm ? max_tiles : n_sm;
  if (wfmt == MOE_W_INT4_G32)
    return epi == 0 ? launch_gemm_t<MOE_W_INT4_G32, 0>(m, p, grid, s) : launch_gemm_t<MOE_W_INT4_G32, 1>(m, p, grid, s);
  if (wfmt == MOE_W_NVFP4)
    return epi == 0 ? launch_gemm_t<MOE_W_NVFP4, 0>(m, p, grid, s) : launch_gemm_t<MOE_W_NVFP4, 1>(m, p, grid, s);
  if (wfmt == kWF16)
    return epi == 0 ? launch_gemm_t<kWF16, 0>(m, p, grid, s) : launch_gemm_t<kWF16, 1>(m, p, grid, s);
  return cudaErrorInvalidValue;
}

size_t gemm_pack_bytes(int rows_per_expert, int K, int n_exp) {
  return (size_t)n_exp * (rows_per_expert / kBM) * (K / 256) * kGroupBytes;
}

cudaError_t launch_gemm_pack(const uint8_t* codes, const void* scales, int K, int n_exp, int rows_per_expert,
                             int I, bool gate_up, uint8_t* dst, cudaStream_t s) {
  gemm_pack_kernel<<<148 * 8, 256, 0, s>>>(codes, static_cast<const uint8_t*>(scales), K, n_exp, rows_per_expert, I,
                                          gate_up ? 1 : 0, rows_per_expert / kBM, dst);
  return cudaGetLastError();
}

}  // namespace moe
