// Fused decode-path kernel of the MoE layer (T <= 8 tokens per call), plus the weight repack
// it reads.
//
// One persistent cooperative grid (one CTA per SM) runs the whole layer forward of a decode
// step: router logits, noaux_tc selection and batch-union grouping, the SwiGLU gate/up
// projection of the shared and the selected experts, and the down projection fused with the
// weighted combine ("Show HN: Menjalankan GLM 5.2 di komputer lambat", section "Fitur utama
// yang diimplementasikan": DeepSeek-V3-style router with noaux_tc, routed_scaling_factor and
// a shared expert; packed int4 with dequant-on-use; batch-union MoE). Every selected expert's
// weights are streamed from HBM exactly once.
//
// Weights are repacked at layer creation into 16-row tiles in the register-fragment order of
// the m16n8k16 fp16 MMA. One 32-bit word holds the 8 int4 codes a lane needs for one MMA;
// a shift and four LOP3s turn it into the four fp16 A registers: (code + 8) is placed in the
// mantissa of 1024.0 (rows 0-7: value 1032 + c) or at mantissa bit 4 (rows 8-15: value
// 1152 + 16c). The MMA accumulates in fp32; the per-row bias (1032 or 1152 times the group's
// activation sum) is removed and the fp16 group scale applied once per 32-element group.
// Column layout of the MMA's B operand:
//   MODE 1 (one token): column n of MMA m holds the token's values of group (m/2) mod 8, so the
//     8 groups of a 256-column k-block land in 8 accumulator columns; the operand is built in
//     registers from a compact fp16 copy of the activation (the other columns are zero);
//   MODE 0 (2..8 tokens): column n holds token n, from a fragment-ordered activation panel.
//
// Work per CTA, in order, each item a 16-row x 2048-column panel (18 KB) brought in by the
// producer warp with TMA bulk copies into a ring of slots:
//   consumers: activations staged; router rows e = cta, cta + grid (unrolled vector loads)
//   A  shared-expert gate/up tiles           (no dependency)
//   C1 shared-expert down tiles              (waits until every shared gate/up tile is done)
//   B  selected experts' gate/up tiles       (waits for the routing, in shared memory)
//   C2 selected experts' down tiles          (waits until that expert's gate/up tiles are done)
// Warps: 8 consumers, 1 producer (TMA bulk copies), 1 routing warp. Once a CTA's router
// rows are written, its routing warp waits until every CTA has written its rows, selects
// each token's experts (one warp per token, in turn) and groups the entries, while the
// consumers already run the shared expert (A, C1). Every CTA obtains the same routing from
// the same logits (CTA 0 also writes it out). The producer issues the shared-expert items
// first and the routed items once the routing warp publishes the routing.
// Down tiles add w * y into an fp32 accumulator with atomics; the last CTA to finish its
// down tiles (a ticket counter) converts the whole output to the output type. All
// inter-CTA waits are bounded; on time-out the kernel records MOE_ERR_TIMEOUT, drains its
// own copies in flight and returns.
#include <cstddef>

#include "kernels.h"
#include "ptx.cuh"
#include "route_dev.cuh"

namespace moe {

namespace {

constexpr int kDecThreads = 320;      // 8 consumer warps, 1 producer warp, 1 routing warp
constexpr int kConsumers = 256;
constexpr int kPanelK = 2048;          // columns per item
constexpr int kCodeBytes = 16384;      // 16 rows x 2048 int4
constexpr int kScaleBytes = 2048;      // 16 rows x 64 groups fp16
constexpr int kItemBytes = kCodeBytes + kScaleBytes;
constexpr int kMaxH = 6144;
constexpr int kMaxI = 2048;
constexpr int kMaxE = 256;
constexpr int kMaxK = 16;
constexpr int kMaxActive = 64;         // T * top_k <= 64 on this path
constexpr uint32_t kMbarSpin = 1u << 22;

// Shared memory common to both modes (16-byte aligned: the reduction buffer takes float4
// stores).
struct alignas(16) DecCommon {
  float red[2][8][32][8];              // cross-warp reduction (double-buffered per unit)
  float selb[kMaxE];                   // selection scratch: biased and unbiased scores of one token
  float sels[kMaxE];
  int idsel[8][kMaxK];                 // per token: selected experts and weights
  float wsel[8][kMaxK];
  int cnt[kMaxE];
  int soff[kMaxE];
  int aslot[kMaxE];
  int active[kMaxE];
  int meta_pair[kMaxActive][8];        // per active expert: h row of token n (-1: not routed)
  float meta_w[kMaxActive][8];         // per active expert: combine weight of token n
  int colpair[8];
  float colw[8];
  int n_active;
  int flag;
  int abort;
  int issued;
  int consumed;
};

template <int MODE>
struct DecSmem;

template <>
struct DecSmem<1> {
  static constexpr int kSlots = 8;
  uint8_t slots[kSlots][kItemBytes];
  uint32_t xs[kMaxH / 2];              // compact fp16 pairs of the token's activation
  uint32_t hs[kMaxI / 2];              // compact fp16 pairs of the current h row
  float xsums[kMaxH / 32];             // per 32-element group: sum of the fp16 values
  float hsums[kMaxI / 32];
  uint64_t full[kSlots];
  uint64_t empty[kSlots];
  uint64_t route_bar;
  uint64_t router_bar;
  DecCommon c;
};

template <>
struct DecSmem<0> {
  static constexpr int kSlots = 3;
  uint8_t slots[kSlots][kItemBytes];
  uint2 xpanel[kMaxH / 16 * 32];       // B fragments of x: 8 bytes per lane per MMA
  uint2 hpanel[kMaxI / 16 * 32];       // B fragments of h
  float xsums[kMaxH / 32 * 8];         // per group and column: sum of the fp16 values
  float hsums[kMaxI / 32 * 8];
  uint64_t full[kSlots];
  uint64_t empty[kSlots];
  uint64_t route_bar;
  uint64_t router_bar;
  DecCommon c;
};

static_assert(offsetof(DecSmem<1>, c) % 16 == 0 && offsetof(DecSmem<0>, c) % 16 == 0,
              "vector stores into the common block need 16-byte alignment");
static_assert(offsetof(DecSmem<1>, xs) % 16 == 0 && offsetof(DecSmem<1>, hs) % 16 == 0,
              "vector accesses into the staged activations need 16-byte alignment");
static_assert(offsetof(DecSmem<0>, xsums) % 8 == 0 && offsetof(DecSmem<1>, xsums) % 8 == 0 &&
                  offsetof(DecSmem<0>, hsums) % 8 == 0 && offsetof(DecSmem<1>, hsums) % 8 == 0,
              "float2 reads of the group sums need 8-byte alignment");
static_assert(sizeof(DecSmem<1>) <= 227 * 1024, "decode kernel shared memory over the per-CTA limit");
static_assert(sizeof(DecSmem<0>) <= 227 * 1024, "decode kernel shared memory over the per-CTA limit");

// ------------------------------------------------------------------ helpers

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ float2 half2_to_float2(uint32_t u) {
  return __half22float2(*reinterpret_cast<const __half2*>(&u));
}

// Elementwise fp16x2 product of two registers (round to nearest).
__device__ __forceinline__ uint32_t hmul2_bits(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// One word of codes -> the four fp16 A registers of an m16n8k16 MMA (see file comment).
__device__ __forceinline__ void decode_word(uint32_t w, uint32_t (&a)[4]) {
  const uint32_t w2 = w >> 8;
  a[0] = (w & 0x000F000Fu) ^ 0x64086408u;
  a[1] = (w & 0x00F000F0u) ^ 0x64806480u;
  a[2] = (w2 & 0x000F000Fu) ^ 0x64086408u;
  a[3] = (w2 & 0x00F000F0u) ^ 0x64806480u;
}

// Bounded wait for *p >= target (one thread). Returns false on time-out.
__device__ __forceinline__ bool wait_geq(const uint32_t* p, uint32_t target, uint32_t spin_max) {
  for (uint32_t i = 0; i < spin_max; ++i) {
    if (ptx::ld_acquire(p) >= target) return true;
    __nanosleep(64);
  }
  return false;
}

struct Geo {
  int T, H, I, E, k;
  int NTu, Pu, NTd, Pd;   // tiles and panels per tile: up (gate/up) and down
  int G, c;
};

// Item ranges of this CTA (balanced contiguous split of each segment over the grid).
__device__ __forceinline__ void seg_range(int n, int G, int c, int& b, int& e) {
  b = (int)(((long)n * c) / G);
  e = (int)(((long)n * (c + 1)) / G);
}

// 8 consecutive activation elements at element index idx (bf16 or fp32 storage).
template <int XDT>
__device__ __forceinline__ void load_act8(const void* x, size_t idx, float (&v)[8]) {
  if constexpr (XDT == MOE_DT_F32) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(x) + idx));
    const float4 b = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(x) + idx) + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  } else {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(static_cast<const unsigned short*>(x) + idx));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      v[2 * q] = __uint_as_float(w[q] << 16);
      v[2 * q + 1] = __uint_as_float(w[q] & 0xFFFF0000u);
    }
  }
}

// Sum of the fp16 values held by 4 half2 words.
__device__ __forceinline__ float sum4h2(const uint32_t (&p)[4]) {
  float s = 0.f;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float2 f = half2_to_float2(p[q]);
    s += f.x + f.y;
  }
  return s;
}

// ------------------------------------------------------------- activation staging

// MODE 1: compact fp16 pairs of token 0 and the per-group sums (thread per 32-element group).
template <int XDT>
__device__ void stage_x1(DecSmem<1>& S, const void* x, int H) {
  for (int j = threadIdx.x; j < H / 32; j += kConsumers) {
    float s = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float v[8];
      load_act8<XDT>(x, (size_t)32 * j + 8 * q, v);
      uint32_t p[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) p[i] = pack_half2(v[2 * i], v[2 * i + 1]);
      s += sum4h2(p);
      *reinterpret_cast<uint4*>(&S.xs[16 * j + 4 * q]) = make_uint4(p[0], p[1], p[2], p[3]);
    }
    S.xsums[j] = s;
  }
}

// MODE 0: fragment panel (column n = token n, zero for n >= T) and per-(group, token) sums.
// Element pair (k, k+1), k = 16 m + r, goes to lane (token, (r mod 8) / 2), half r / 8.
template <int XDT>
__device__ void stage_x0(DecSmem<0>& S, const void* x, int T, int H) {
  const int ng = H / 32;
  for (int idx = threadIdx.x; idx < ng * 8; idx += kConsumers) {
    const int j = idx >> 3, tok = idx & 7;
    float s = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {   // 8 elements 32 j + 8 q ..: MMA m = 2 j + q / 2, half q & 1
      uint32_t p[4] = {0u, 0u, 0u, 0u};
      if (tok < T) {
        float v[8];
        load_act8<XDT>(x, (size_t)tok * H + 32 * j + 8 * q, v);
#pragma unroll
        for (int i = 0; i < 4; ++i) p[i] = pack_half2(v[2 * i], v[2 * i + 1]);
        s += sum4h2(p);
      }
      const int m = 2 * j + (q >> 1);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint32_t* e = reinterpret_cast<uint32_t*>(&S.xpanel[m * 32 + tok * 4 + i]);
        e[q & 1] = p[i];
      }
    }
    S.xsums[idx] = s;   // [group j][column tok]
  }
}

// h rows of the current expert (rows S.c.colpair, written by other CTAs: read through L2).
__device__ void stage_h1(DecSmem<1>& S, const __half* h16, int I) {
  const int row = S.c.colpair[0];
  for (int i = threadIdx.x; i < I / 8; i += kConsumers) {
    uint4 u = make_uint4(0u, 0u, 0u, 0u);
    if (row >= 0) u = __ldcg(reinterpret_cast<const uint4*>(h16 + (size_t)row * I) + i);
    *reinterpret_cast<uint4*>(&S.hs[4 * i]) = u;
  }
  ptx::bar_sync(1, kConsumers);
  for (int j = threadIdx.x; j < I / 32; j += kConsumers) {
    float s = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 u = *reinterpret_cast<const uint4*>(&S.hs[16 * j + 4 * q]);
      const uint32_t p[4] = {u.x, u.y, u.z, u.w};
      s += sum4h2(p);
    }
    S.hsums[j] = s;
  }
}

__device__ void stage_h0(DecSmem<0>& S, const __half* h16, int I) {
  const int ng = I / 32;
  for (int idx = threadIdx.x; idx < ng * 8; idx += kConsumers) {
    const int j = idx >> 3, col = idx & 7;
    const int row = S.c.colpair[col];
    float s = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t p[4] = {0u, 0u, 0u, 0u};
      if (row >= 0) {
        const uint4 u = __ldcg(reinterpret_cast<const uint4*>(h16 + (size_t)row * I + 32 * j + 8 * q));
        p[0] = u.x; p[1] = u.y; p[2] = u.z; p[3] = u.w;
        s += sum4h2(p);
      }
      const int m = 2 * j + (q >> 1);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint32_t* e = reinterpret_cast<uint32_t*>(&S.hpanel[m * 32 + col * 4 + i]);
        e[q & 1] = p[i];
      }
    }
    S.hsums[idx] = s;
  }
}

// ------------------------------------------------------- consumer: compute

// One item (16 rows x 2048 columns): warp `w` handles k-block w (256 columns = 16 MMAs).
// m_base = global MMA index of the panel start (p * 128). kb = global k-block index.
// MODE 1: `act` = compact fp16 pairs; lane group g holds the operand of MMAs 2g, 2g+1 only.
// Four independent accumulator chains keep the MMA pipe busy.
__device__ __forceinline__ void compute_item1(const uint32_t* act, const float* sums, const uint8_t* slot,
                                              int m_base, int kb, float (&acc)[4]) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const uint8_t* codes = slot + ((size_t)(4 * w) * 32 + lane) * 16;
  const uint8_t* scl = slot + kCodeBytes + (w * 8 + g) * 32;
  const uint32_t* xb = act + 8 * (m_base + 16 * w + 2 * g) + t;
  const uint32_t b00 = xb[0], b01 = xb[4], b10 = xb[8], b11 = xb[12];
  // the B operand of MMA mi is the lane's x values when its group column is this lane
  // group's (mi / 2 == g), else zero: an fp16 multiply by 1 or 0 (exact) on the FMA pipe,
  // which leaves the ALU pipe to the int4 decode
  uint32_t msk[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) msk[j] = j == g ? 0x3C003C00u : 0u;
  float d[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i) d[i][0] = d[i][1] = d[i][2] = d[i][3] = 0.f;
#pragma unroll
  for (int cc = 0; cc < 4; ++cc) {
    const uint4 q = *reinterpret_cast<const uint4*>(codes + cc * 32 * 16);
    const uint32_t words[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int mi = 4 * cc + i;           // MMA within the k-block; active lane group mi / 2
      uint32_t a[4];
      decode_word(words[i], a);
      const uint32_t bx = hmul2_bits((mi & 1) ? b10 : b00, msk[mi >> 1]);
      const uint32_t by = hmul2_bits((mi & 1) ? b11 : b01, msk[mi >> 1]);
      ptx::mma_16816(d[i], a, bx, by, d[i]);
    }
  }
  float dd[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) dd[r] = (d[0][r] + d[1][r]) + (d[2][r] + d[3][r]);
  const uint2 sraw = *reinterpret_cast<const uint2*>(scl + t * 8);
  const float2 sg = half2_to_float2(sraw.x);   // s[g][j0], s[g][j0+1]
  const float2 su = half2_to_float2(sraw.y);   // s[g+8][j0], s[g+8][j0+1]
  const float2 X = *reinterpret_cast<const float2*>(sums + 8 * kb + 2 * t);
  acc[0] = fmaf(sg.x, fmaf(-1032.f, X.x, dd[0]), acc[0]);
  acc[0] = fmaf(sg.y, fmaf(-1032.f, X.y, dd[1]), acc[0]);
  acc[1] = fmaf(su.x, fmaf(-1152.f, X.x, dd[2]), acc[1]);
  acc[1] = fmaf(su.y, fmaf(-1152.f, X.y, dd[3]), acc[1]);
}

// MODE 0: B fragments from the panel; each group's two MMAs form an independent chain.
__device__ __forceinline__ void compute_item0(const uint2* panel, const float* sums, const uint8_t* slot,
                                              int m_base, int kb, float (&acc)[4]) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int gq = lane >> 2, t = lane & 3;
  const uint8_t* codes = slot + ((size_t)(4 * w) * 32 + lane) * 16;
  const uint8_t* scl = slot + kCodeBytes + (w * 8 + gq) * 32;
  const uint2* bp = panel + (size_t)(m_base + 16 * w) * 32 + lane;
  const uint4 s0 = *reinterpret_cast<const uint4*>(scl);
  const uint4 s1 = *reinterpret_cast<const uint4*>(scl + 16);
  const uint32_t sw[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
  for (int cc = 0; cc < 4; ++cc) {
    const uint4 q = *reinterpret_cast<const uint4*>(codes + cc * 32 * 16);
    const uint32_t words[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int gi = 0; gi < 2; ++gi) {
      const int jl = 2 * cc + gi;   // group within the k-block
      float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        uint32_t a[4];
        decode_word(words[2 * gi + i], a);
        const uint2 b = bp[(4 * cc + 2 * gi + i) * 32];
        ptx::mma_16816(d, a, b.x, b.y, d);
      }
      // scale words per (k-block, row g): [t'][s[g][2t'], s[g][2t'+1], s[g+8][2t'], s[g+8][2t'+1]]
      const float2 sgp = half2_to_float2(sw[2 * (jl >> 1)]);
      const float2 sup = half2_to_float2(sw[2 * (jl >> 1) + 1]);
      const float sgate = (jl & 1) ? sgp.y : sgp.x;
      const float sup1 = (jl & 1) ? sup.y : sup.x;
      const float2 X = *reinterpret_cast<const float2*>(sums + (8 * kb + jl) * 8 + 2 * t);
      acc[0] = fmaf(sgate, fmaf(-1032.f, X.x, d[0]), acc[0]);
      acc[1] = fmaf(sgate, fmaf(-1032.f, X.y, d[1]), acc[1]);
      acc[2] = fmaf(sup1, fmaf(-1152.f, X.x, d[2]), acc[2]);
      acc[3] = fmaf(sup1, fmaf(-1152.f, X.y, d[3]), acc[3]);
    }
  }
}

// Cross-warp reduction of the tile accumulators into red (consumers, then named barrier).
// `half` selects the second 16-row tile of a down pair.
template <int MODE>
__device__ __forceinline__ void stash_acc(DecCommon& C, int rb, int half, float (&acc)[4]) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  if (MODE == 1) {
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {
      acc[0] += __shfl_xor_sync(0xffffffffu, acc[0], o);
      acc[1] += __shfl_xor_sync(0xffffffffu, acc[1], o);
    }
    if ((lane & 3) == 0) {
      C.red[rb][w][lane >> 2][2 * half] = acc[0];
      C.red[rb][w][lane >> 2][2 * half + 1] = acc[1];
    }
  } else {
    *reinterpret_cast<float4*>(&C.red[rb][w][lane][4 * half]) = make_float4(acc[0], acc[1], acc[2], acc[3]);
  }
}

// Value of MMA row r (0..15) for column n after the reduction (rows 8..15 carry a x16 unit).
template <int MODE>
__device__ __forceinline__ float reduced(const DecCommon& C, int rb, int half, int r, int n) {
  float v = 0.f;
  if (MODE == 1) {
#pragma unroll
    for (int w = 0; w < 8; ++w) v += C.red[rb][w][r & 7][2 * half + (r >> 3)];
  } else {
    const int ln = (r & 7) * 4 + (n >> 1);
    const int idx = 4 * half + (r >> 3) * 2 + (n & 1);
#pragma unroll
    for (int w = 0; w < 8; ++w) v += C.red[rb][w][ln][idx];
  }
  return (r >= 8) ? v * 0.0625f : v;
}

// ------------------------------------------------------------------ selection

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Order key of (biased score v, expert e): larger v first, lower e on ties. The float's
// bits are mapped to an unsigned integer with the same order (v = -0 does not occur: a
// sigmoid in (0, 1) plus a bias never rounds to -0); the low word is ~e.
__device__ __forceinline__ unsigned long long sel_key(float v, int e) {
  const uint32_t u = __float_as_uint(v);
  const uint32_t k = u ^ ((uint32_t)((int32_t)u >> 31) | 0x80000000u);
  return ((unsigned long long)k << 32) | (uint32_t)~e;
}

// Bitonic clean-up of an 8-key bitonic sequence into descending order.
__device__ __forceinline__ void bitonic_merge8(unsigned long long (&K)[8]) {
#pragma unroll
  for (int j = 4; j > 0; j >>= 1)
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int l = i ^ j;
      if (l > i && K[i] < K[l]) {
        const unsigned long long t = K[i];
        K[i] = K[l];
        K[l] = t;
      }
    }
}

// One warp: noaux_tc selection of one token with the same result as the sequential picks,
// bit for bit. Each group's score adds its two largest biased scores; the topk_group best
// groups are kept (lower index on ties); the top_k kept experts in the order "larger biased
// score first, lower index on ties" fill the slots; the weights' normaliser adds the picked
// unbiased scores in slot order. Lane l holds experts l*E/32 .. (l+1)*E/32 - 1.
// Fast path (n_group divides 32, top_k <= 8): groups are whole runs of lanes, group top-2
// values merge over those lanes, and the top-8 keys come from a per-lane sort followed by
// five butterfly merges of sorted 8-lists. Otherwise: group scores from shared memory and
// top_k rounds of a warp argmax.
__device__ __forceinline__ void select_warp(DecCommon& C, const float* logits_row, const float* bias, int E,
                                            int n_group, int topk_group, int top_k, float rsf, int* idsel,
                                            float* wsel) {
  constexpr int kE = kMaxE / 32;
  const int lane = threadIdx.x & 31;
  const int epl = E / 32;
  float lg[kE], bi_[kE], s[kE], b[kE];
#pragma unroll
  for (int j = 0; j < kE; ++j) {   // all loads first, so their latencies overlap
    lg[j] = bi_[j] = 0.f;
    if (j < epl) {
      lg[j] = __ldcg(logits_row + lane * epl + j);
      bi_[j] = __ldg(bias + lane * epl + j);
    }
  }
#pragma unroll
  for (int j = 0; j < kE; ++j) {
    s[j] = b[j] = 0.f;
    if (j < epl) {
      s[j] = sigmoidf_acc(lg[j]);
      b[j] = s[j] + bi_[j];
      C.selb[lane * epl + j] = b[j];
      C.sels[lane * epl + j] = s[j];
    }
  }
  __syncwarp();
  const int G = E / n_group;
  int my_e = -1;
  float my_s = 0.f;
  if ((32 % n_group) == 0 && top_k <= 8) {
    // group of lane = lane / lpg; top-2 of the lane's values, then of the group's lanes
    const int lpg = 32 / n_group;
    float m1 = -INFINITY, m2 = -INFINITY;
#pragma unroll
    for (int j = 0; j < kE; ++j) {
      if (j < epl) {
        const float v = b[j];
        if (v > m1) {
          m2 = m1;
          m1 = v;
        } else if (v > m2) {
          m2 = v;
        }
      }
    }
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float o1 = __shfl_xor_sync(0xffffffffu, m1, o), o2 = __shfl_xor_sync(0xffffffffu, m2, o);
      if (o < lpg) {
        const float n1 = fmaxf(m1, o1);
        m2 = fmaxf(fminf(m1, o1), fmaxf(m2, o2));
        m1 = n1;
      }
    }
    const float gs = m1 + m2;
    const int gid = lane / lpg;
    int grank = 0;
#pragma unroll
    for (int g2 = 0; g2 < 32; ++g2) {
      const float w2 = __shfl_sync(0xffffffffu, gs, (g2 * lpg) & 31);
      if (g2 < n_group) grank += (w2 > gs) || (w2 == gs && g2 < gid);
    }
    const bool kept = grank < topk_group;
    unsigned long long K[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) K[j] = (j < epl && kept) ? sel_key(b[j], lane * epl + j) : 0ull;
    // sort the lane's 8 keys (descending bitonic network)
#pragma unroll
    for (int k2 = 2; k2 <= 8; k2 <<= 1)
#pragma unroll
      for (int j2 = k2 >> 1; j2 > 0; j2 >>= 1)
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int l = i ^ j2;
          if (l > i) {
            const bool desc = (i & k2) == 0 || k2 == 8;
            if (desc ? (K[i] < K[l]) : (K[i] > K[l])) {
              const unsigned long long t = K[i];
              K[i] = K[l];
              K[l] = t;
            }
          }
        }
    // top 8 of the union of two sorted lists: max(A[i], B[7-i]) is bitonic, then clean up
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      unsigned long long P[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) P[i] = __shfl_xor_sync(0xffffffffu, K[i], o);
#pragma unroll
      for (int i = 0; i < 8; ++i) K[i] = K[i] > P[7 - i] ? K[i] : P[7 - i];
      bitonic_merge8(K);
    }
    unsigned long long mine = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (lane == j) mine = K[j];
    if (lane < top_k) {
      my_e = (int)~(uint32_t)mine;
      my_s = C.sels[my_e];
    }
  } else {
    // group scores: lane gi scans group gi from a lane-dependent start (spreads the banks)
    float gs = -INFINITY;
    if (lane < n_group) {
      float m1 = -INFINITY, m2 = -INFINITY;
      const float* bg = C.selb + lane * G;
      int i2 = lane % G;
      for (int i = 0; i < G; ++i) {
        const float v = bg[i2];
        if (++i2 == G) i2 = 0;
        if (v > m1) {
          m2 = m1;
          m1 = v;
        } else if (v > m2) {
          m2 = v;
        }
      }
      gs = m1 + m2;
    }
    int grank = 0;
    for (int g2 = 0; g2 < n_group; ++g2) {
      const float w2 = __shfl_sync(0xffffffffu, gs, g2);
      grank += (w2 > gs) || (w2 == gs && g2 < lane);
    }
    const unsigned kept = __ballot_sync(0xffffffffu, lane < n_group && grank < topk_group);
    unsigned cand = 0;
#pragma unroll
    for (int j = 0; j < kE; ++j)
      if (j < epl && ((kept >> ((lane * epl + j) / G)) & 1u)) cand |= 1u << j;
    // top_k argmax rounds; lane r keeps the r-th pick
    for (int r = 0; r < top_k; ++r) {
      float bv = -INFINITY, bs = 0.f;
      int bi = E;   // E: none
#pragma unroll
      for (int j = 0; j < kE; ++j) {
        if ((cand >> j) & 1u) {
          if (bi == E || b[j] > bv) {
            bv = b[j];
            bs = s[j];
            bi = lane * epl + j;
          }
        }
      }
      const float local_s = bs;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (oi != E && (bi == E || ov > bv || (ov == bv && oi < bi))) {
          bv = ov;
          bi = oi;
        }
      }
      const int win = bi < E ? bi / epl : 0;
      const float ws = __shfl_sync(0xffffffffu, local_s, win);
      if (lane == win && bi < E) cand &= ~(1u << (bi - lane * epl));
      if (lane == r) {
        my_e = bi;
        my_s = ws;
      }
    }
  }
  float wsum = 0.f;
  for (int j = 0; j < top_k; ++j) wsum += __shfl_sync(0xffffffffu, my_s, j);
  if (lane < top_k) {
    idsel[lane] = my_e;
    wsel[lane] = my_s / wsum * rsf;
  }
  __syncwarp();
}

}  // namespace

struct DecodeArgs {
  const void* x;
  int T;
  const void* router_w;
  const float* bias;
  int H, I, E, top_k, n_group, topk_group;
  float rsf;
  const uint8_t* up_store;     // [E+1][I/8 tiles][H/2048 panels][18432]
  const uint8_t* down_store;   // [E+1][H/16 tiles][I/2048 panels][18432]
  float* logits;               // [T, E]
  int32_t* ids;
  float* weights;
  int32_t* offsets;
  int32_t* entries;
  __half* h16;                 // [T*k + T, I]
  float* out_acc;              // [T, H], zero between calls
  void* out;
  uint32_t* sync;              // see the kernel
  int* status;
  uint32_t spin_max;
  unsigned long long* trace;   // optional [grid][64] phase timestamps (ns, slots 0..15), or NULL
};

namespace {

// Phase timestamp of this CTA (profiling hook; one thread records).
#define DEC_TRACE(i)                                                            \
  do {                                                                          \
    if (a.trace) a.trace[(size_t)blockIdx.x * 64 + (i)] = global_ns();          \
  } while (0)

// One consumer warp: group the selected (token, slot) entries per expert and publish the
// routing in shared memory (CTA 0 also to global): counts, exclusive scans (entry
// offsets, active slots), the ascending entry lists and each active expert's columns.
template <int MODE>
__device__ void group_in_cta(DecSmem<MODE>& S, const DecodeArgs& a, const Geo& g) {
  DecCommon& C = S.c;
  const int lane = threadIdx.x & 31;
  const int T = g.T, E = g.E, k = g.k;
  // grouping: counts, exclusive scans (entry offsets, active slots), entry lists
  const int n = T * k;
  for (int e = lane; e < E; e += 32) C.cnt[e] = 0;
  __syncwarp();
  for (int f = lane; f < n; f += 32) atomicAdd(&C.cnt[C.idsel[f / k][f % k]], 1);
  __syncwarp();
  const int epl = E / 32;   // lane owns experts lane*epl .. +epl-1 (epl <= kMaxE / 32)
  int cl[kMaxE / 32];
  int local = 0, nact = 0;
#pragma unroll
  for (int i = 0; i < kMaxE / 32; ++i) {
    cl[i] = i < epl ? C.cnt[lane * epl + i] : 0;
    local += cl[i];
    nact += cl[i] > 0;
  }
  int incl = local, inca = nact;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    const int va = __shfl_up_sync(0xffffffffu, inca, o);
    if (lane >= o) {
      incl += v;
      inca += va;
    }
  }
  int run = incl - local, apos = inca - nact;
#pragma unroll
  for (int i = 0; i < kMaxE / 32; ++i) {
    if (i < epl) {
      const int e = lane * epl + i;
      C.soff[e] = run;
      if (g.c == 0) a.offsets[e] = run;
      if (cl[i] > 0) {
        C.aslot[e] = apos;
        C.active[apos++] = e;
      }
      run += cl[i];
    }
  }
  const int na = __shfl_sync(0xffffffffu, inca, 31);
  if (lane == 31 && g.c == 0) a.offsets[E] = run;
  for (int i = lane; i < na * 8; i += 32) {
    C.meta_pair[i >> 3][i & 7] = -1;
    C.meta_w[i >> 3][i & 7] = 0.f;
  }
  __syncwarp();
  const int* flat = &C.idsel[0][0];   // entry f = token * top_k + slot at idsel[token][slot]
  for (int f = lane; f < n; f += 32) {
    const int tok = f / k, slot = f % k;
    const int e = C.idsel[tok][slot];
    int rank = 0;
#pragma unroll 8
    for (int f2 = 0; f2 < f; ++f2) rank += (flat[(f2 / k) * kMaxK + f2 % k] == e);
    const int q = C.soff[e] + rank;
    const int sl = C.aslot[e];
    C.meta_pair[sl][tok] = q;
    C.meta_w[sl][tok] = C.wsel[tok][slot];
    if (g.c == 0) {
      a.entries[q] = f;
      a.ids[f] = e;
      a.weights[f] = C.wsel[tok][slot];
    }
  }
  if (lane == 0) C.n_active = na;
  __syncwarp();
}

template <int MODE, int XDT, int WDT>
__global__ void __launch_bounds__(kDecThreads, 1) moe_decode_kernel(DecodeArgs a) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  DecSmem<MODE>& S = *reinterpret_cast<DecSmem<MODE>*>(smem_raw);
  DecCommon& C = S.c;
  constexpr int kSlots = DecSmem<MODE>::kSlots;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  Geo g;
  g.T = a.T;
  g.H = a.H;
  g.I = a.I;
  g.E = a.E;
  g.k = a.top_k;
  g.NTu = a.I / 8;
  g.Pu = a.H / kPanelK;
  g.NTd = a.H / 16;
  g.Pd = a.I / kPanelK;
  g.G = gridDim.x;
  g.c = blockIdx.x;
  // sync words: [0] CTAs done with router rows, [2] CTAs exited, [4] CTAs done with down
  // tiles; [8..8+E] gate/up tiles done per expert
  uint32_t* up_done = a.sync + 8;
  const int shared_e = a.E;
  const size_t up_tile_bytes = (size_t)g.Pu * kItemBytes;
  const size_t dn_tile_bytes = (size_t)g.Pd * kItemBytes;

  if (tid == 0) {
    for (int s = 0; s < kSlots; ++s) {
      ptx::mbar_init(&S.full[s], 1);
      ptx::mbar_init(&S.empty[s], 8);
    }
    ptx::mbar_init(&S.route_bar, 1);
    ptx::mbar_init(&S.router_bar, 1);
    ptx::fence_mbar_init();
    C.abort = 0;
    C.issued = 0;
    C.consumed = 0;
    C.n_active = 0;
  }
  __syncthreads();

  int a0, a1, c10, c11;
  seg_range(g.NTu, g.G, g.c, a0, a1);    // shared gate/up tiles
  seg_range(g.NTd / 2, g.G, g.c, c10, c11);  // shared down tile pairs
  c10 *= 2;
  c11 *= 2;

  if (warp == 8) {
    // ------------------------------------------------------------- producer warp
    const uint64_t pol = ptx::policy_evict_first();
    int it = 0;
    bool ok = true;
    unsigned long long p_wait = 0;   // cycles waiting for a free slot (profiling)
    // Brings item `it` into slot it % kSlots once the consumers released its previous use.
    auto issue = [&](const uint8_t* src) {
      if (!ok) return;
      const int slot = it % kSlots;
      const unsigned long long t0 = clock64();
      if (it >= kSlots && !ptx::mbar_wait_backoff(&S.empty[slot], ((it / kSlots) - 1) & 1, kMbarSpin, 4, 128))
        ok = false;
      p_wait += clock64() - t0;
      if (ok && *(volatile int*)&C.abort) ok = false;
      if (!ok) return;
      ptx::mbar_arrive_expect_tx(&S.full[slot], kItemBytes);
      ptx::bulk_g2s(S.slots[slot], src, kItemBytes, &S.full[slot], pol);
      ++it;
      *(volatile int*)&C.issued = it;
    };
    if (lane == 0) {
      // the router rows' weight loads go first: after two items the producer waits until this
      // CTA's router rows are done, so the shared-expert prefetch does not delay the routing
      int n_sh = 0;
      for (int tl = a0; tl < a1; ++tl)
        for (int p = 0; p < g.Pu; ++p) {
          if (n_sh++ == 2) ptx::mbar_wait_backoff(&S.router_bar, 0, kMbarSpin, 4, 128);
          issue(a.up_store + ((size_t)shared_e * g.NTu + tl) * up_tile_bytes + (size_t)p * kItemBytes);
        }
      if (n_sh <= 2) ptx::mbar_wait_backoff(&S.router_bar, 0, kMbarSpin, 4, 128);
      for (int tl = c10; tl < c11; ++tl)
        for (int p = 0; p < g.Pd; ++p)
          issue(a.down_store + ((size_t)shared_e * g.NTd + tl) * dn_tile_bytes + (size_t)p * kItemBytes);
      DEC_TRACE(13);
    }
    if (lane == 0) {
      // the routing warp publishes the routing (selection and grouping) through route_bar
      if (!ptx::mbar_wait_backoff(&S.route_bar, 0, kMbarSpin * 16, 4, 256)) {
        ok = false;
        atomicExch(&C.abort, 1);
        raise_status(a.status, MOE_ERR_TIMEOUT);
      }
      DEC_TRACE(14);
      const int na = ok ? C.n_active : 0;
      int b0, b1, c20, c21;
      seg_range(na * g.NTu, g.G, g.c, b0, b1);
      seg_range(na * (g.NTd / 2), g.G, g.c, c20, c21);   // down tile pairs
      c20 *= 2;
      c21 *= 2;
      for (int r = b0; r < b1; ++r) {
        const int e = C.active[r / g.NTu], tl = r % g.NTu;
        for (int p = 0; p < g.Pu; ++p)
          issue(a.up_store + ((size_t)e * g.NTu + tl) * up_tile_bytes + (size_t)p * kItemBytes);
      }
      for (int u = c20; u < c21; ++u) {
        const int e = C.active[u / g.NTd], tl = u % g.NTd;
        for (int p = 0; p < g.Pd; ++p)
          issue(a.down_store + ((size_t)e * g.NTd + tl) * dn_tile_bytes + (size_t)p * kItemBytes);
      }
      if (!ok) {
        atomicExch(&C.abort, 1);
        raise_status(a.status, MOE_ERR_TIMEOUT);
      }
      if (a.trace) {
        a.trace[(size_t)blockIdx.x * 64 + 21] = p_wait;
        a.trace[(size_t)blockIdx.x * 64 + 22] = (unsigned long long)it;
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------- routing warp
    // Waits for every CTA's router rows, selects each token's experts and groups the
    // entries while the consumers work on the shared expert; route_bar publishes the result
    // to the producer and the consumers.
    int ok = 0;
    if (lane == 0) {
      ok = wait_geq(a.sync + 0, (uint32_t)g.G, a.spin_max) ? 1 : 0;
      __threadfence();
      DEC_TRACE(3);
    }
    __syncwarp();
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok) {
      for (int t = 0; t < g.T; ++t)
        select_warp(C, a.logits + (size_t)t * g.E, a.bias, g.E, a.n_group, a.topk_group, g.k, a.rsf, C.idsel[t],
                    C.wsel[t]);
      if (lane == 0) DEC_TRACE(15);
      group_in_cta<MODE>(S, a, g);
      if (lane == 0) DEC_TRACE(23);
    } else if (lane == 0) {
      atomicExch(&C.abort, 1);
      raise_status(a.status, MOE_ERR_TIMEOUT);
      C.n_active = 0;
    }
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(&S.route_bar);
  } else {
    // ------------------------------------------------------------- consumers
    const int T = g.T, H = g.H, E = g.E;
    if (tid == 0) {
      DEC_TRACE(0);
      if (a.trace) a.trace[(size_t)blockIdx.x * 64 + 24] = clock64();
    }
    if constexpr (MODE == 1) {
      stage_x1<XDT>(S, a.x, H);
    } else {
      stage_x0<XDT>(S, a.x, T, H);
    }
    ptx::bar_sync(1, kConsumers);
    if (tid == 0) DEC_TRACE(1);

    // router rows e = c, c + G, ... two at a time: each thread takes 4 consecutive columns
    // per 1024 of both rows, all loads issued together; fp32 FMA, then warp and CTA
    // reductions
    for (int e0 = g.c; e0 < E; e0 += 2 * g.G) {
      const int e1 = e0 + g.G;
      const bool two = e1 < E;
      float racc[2][8];
#pragma unroll
      for (int i = 0; i < 8; ++i) racc[0][i] = racc[1][i] = 0.f;
      float4 wv[2][kMaxH / 1024];
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const int e = rr ? e1 : e0;
#pragma unroll
        for (int q = 0; q < kMaxH / 1024; ++q) {
          const int col = 1024 * q + 4 * tid;
          wv[rr][q] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (col < H && (rr == 0 || two)) {
            if constexpr (WDT == MOE_DT_F32) {
              wv[rr][q] =
                  __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(a.router_w) + (size_t)e * H + col));
            } else {
              const uint2 u = __ldg(reinterpret_cast<const uint2*>(static_cast<const unsigned short*>(a.router_w) +
                                                                   (size_t)e * H + col));
              wv[rr][q] = make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u),
                                      __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u));
            }
          }
        }
      }
#pragma unroll
      for (int q = 0; q < kMaxH / 1024; ++q) {
        const int col = 1024 * q + 4 * tid;
        if (col < H) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            if (i < T) {
              float xv[4];
              if constexpr (XDT == MOE_DT_F32) {
                const float4 f =
                    __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(a.x) + (size_t)i * H + col));
                xv[0] = f.x; xv[1] = f.y; xv[2] = f.z; xv[3] = f.w;
              } else {
                const uint2 u = __ldg(reinterpret_cast<const uint2*>(static_cast<const unsigned short*>(a.x) +
                                                                     (size_t)i * H + col));
                xv[0] = __uint_as_float(u.x << 16);
                xv[1] = __uint_as_float(u.x & 0xFFFF0000u);
                xv[2] = __uint_as_float(u.y << 16);
                xv[3] = __uint_as_float(u.y & 0xFFFF0000u);
              }
#pragma unroll
              for (int rr = 0; rr < 2; ++rr) {
                racc[rr][i] = fmaf(wv[rr][q].x, xv[0], racc[rr][i]);
                racc[rr][i] = fmaf(wv[rr][q].y, xv[1], racc[rr][i]);
                racc[rr][i] = fmaf(wv[rr][q].z, xv[2], racc[rr][i]);
                racc[rr][i] = fmaf(wv[rr][q].w, xv[3], racc[rr][i]);
              }
            }
          }
        }
      }
#pragma unroll
      for (int rr = 0; rr < 2; ++rr)
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          float v = racc[rr][i];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
          if (lane == 0) C.red[0][warp][i][rr] = v;
        }
      ptx::bar_sync(1, kConsumers);
      if (tid < 2 * T) {
        const int rr = tid / T, i = tid % T;
        if (rr == 0 || two) {
          float v = 0.f;
#pragma unroll
          for (int w = 0; w < 8; ++w) v += C.red[0][w][i][rr];
          a.logits[(size_t)i * E + (rr ? e1 : e0)] = v;
        }
      }
      ptx::bar_sync(1, kConsumers);
    }
    // this CTA's router rows are published; the routing warp takes it from here and the
    // consumers start on the shared expert
    if (tid == 0) {
      __threadfence();
      ptx::red_release_add(a.sync + 0, 1u);
      ptx::mbar_arrive(&S.router_bar);
      DEC_TRACE(2);
    }

    float acc[4];
    // profiling counters (cycles, consumer thread 0): waiting for item data, computing items,
    // tile reduction and epilogue, expert transitions
    unsigned long long c_wait = 0, c_comp = 0, c_epi = 0, c_tr = 0;
    int it = 0;          // items consumed
    int it_ok = 0;       // items whose copy this CTA saw complete (contiguous prefix)
    // Wait for item `it`; on time-out or abort the item is skipped and not released, so
    // its slot is never re-armed while a copy may still be in flight.
    auto wait_item = [&](const uint8_t*& slot) -> bool {
      const int s = it % kSlots;
      slot = S.slots[s];
      if (*(volatile int*)&C.abort) return false;
      if (!ptx::mbar_wait_backoff(&S.full[s], (it / kSlots) & 1, kMbarSpin, 16, 32)) {
        atomicExch(&C.abort, 1);
        raise_status(a.status, MOE_ERR_TIMEOUT);
        return false;
      }
      return true;
    };
    auto run_items = [&](int np, bool up) {
      for (int p = 0; p < np; ++p) {
        const uint8_t* slot;
        const unsigned long long t0 = clock64();
        const bool have = wait_item(slot);
        const unsigned long long t1 = clock64();
        c_wait += t1 - t0;
        if (have) {
          if constexpr (MODE == 1) {
            compute_item1(up ? S.xs : S.hs, up ? S.xsums : S.hsums, slot, p * 128, p * 8 + warp, acc);
          } else {
            compute_item0(up ? S.xpanel : S.hpanel, up ? S.xsums : S.hsums, slot, p * 128, p * 8 + warp, acc);
          }
        }
        __syncwarp();
        c_comp += clock64() - t1;
        if (have) {
          if (lane == 0) ptx::mbar_arrive(&S.empty[it % kSlots]);
          if (it_ok == it) ++it_ok;
        }
        ++it;
      }
    };

    // gate/up tiles are counted per expert and published with one release-add per run
    int up_e = -1, up_n = 0;
    auto flush_up = [&]() {
      if (up_n > 0 && tid == 0) ptx::red_release_add(up_done + up_e, (uint32_t)up_n);
      up_n = 0;
    };

    // one thread waits until every gate/up tile of expert e is done; uniform continuation
    auto wait_up = [&](int e) {
      if (tid == 0) {
        const bool ok = !*(volatile int*)&C.abort && wait_geq(up_done + e, (uint32_t)g.NTu, a.spin_max);
        if (!ok) {
          atomicExch(&C.abort, 1);
          raise_status(a.status, MOE_ERR_TIMEOUT);
        }
      }
      ptx::bar_sync(1, kConsumers);
    };

    // One loop over the four phases (A shared gate/up, C1 shared down, B routed gate/up,
    // C2 routed down) so the unrolled item body exists once in the code: the consumer's
    // instruction footprint stays small. Tile results are reduced through a double-buffered
    // block, so one barrier per tile suffices.
    int lo = a0, hi = a1, cur_sl = -2, cur_up = -1, rb = 0, n_act = 0;
#pragma unroll 1
    for (int ph = 0; ph < 4; ++ph) {
      if (ph == 1) {
        lo = c10 / 2;   // down units are pairs of 16-row tiles
        hi = c11 / 2;
      } else if (ph == 2) {
        // the routed phases need the routing warp's result
        if (tid == 0) {
          DEC_TRACE(6);
          C.flag = ptx::mbar_wait_backoff(&S.route_bar, 0, kMbarSpin * 16, 4, 256) ? 1 : 0;
          if (!C.flag) {
            atomicExch(&C.abort, 1);
            raise_status(a.status, MOE_ERR_TIMEOUT);
          }
          DEC_TRACE(7);
        }
        ptx::bar_sync(1, kConsumers);
        n_act = C.flag ? C.n_active : 0;
        seg_range(n_act * g.NTu, g.G, g.c, lo, hi);
      } else if (ph == 3) {
        seg_range(n_act * (g.NTd / 2), g.G, g.c, lo, hi);
      }
      const int up = (ph & 1) == 0;
      const int ntl = up ? g.NTu : g.NTd / 2;
#pragma unroll 1
      for (int u = lo; u < hi; ++u) {
        const int sl = ph < 2 ? -1 : u / ntl;
        const int tl = ph < 2 ? u : u % ntl;
        const int e = sl < 0 ? shared_e : C.active[sl];
        const unsigned long long tt0 = clock64();
        if (sl != cur_sl || up != cur_up) {
          // new expert or new direction: publish finished gate/up tiles, load the columns'
          // h rows and weights, and for down tiles wait for that expert's h and stage it
          flush_up();
          up_e = e;
          ptx::bar_sync(1, kConsumers);
          if (tid < 8) {
            if (sl < 0) {
              C.colpair[tid] = tid < T ? T * g.k + tid : -1;
              C.colw[tid] = tid < T ? 1.f : 0.f;
            } else {
              C.colpair[tid] = C.meta_pair[sl][tid];
              C.colw[tid] = C.meta_w[sl][tid];
            }
          }
          ptx::bar_sync(1, kConsumers);
          if (!up) {
            wait_up(e);
            if (tid == 0 && ph == 1) DEC_TRACE(5);
            if (tid == 0 && ph == 3) DEC_TRACE(9);
            if constexpr (MODE == 1) {
              stage_h1(S, a.h16, g.I);
            } else {
              stage_h0(S, a.h16, g.I);
            }
            ptx::bar_sync(1, kConsumers);
          }
          cur_sl = sl;
          cur_up = up;
        }
        c_tr += clock64() - tt0;
        unsigned long long te0;
        if (up) {
#pragma unroll
          for (int i = 0; i < 4; ++i) acc[i] = 0.f;
          run_items(g.Pu, true);
          te0 = clock64();
          stash_acc<MODE>(C, rb, 0, acc);
        } else {
          // a pair of 16-row down tiles per unit: one barrier for both
#pragma unroll 1
          for (int half = 0; half < 2; ++half) {
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[i] = 0.f;
            run_items(g.Pd, false);
            stash_acc<MODE>(C, rb, half, acc);
          }
          te0 = clock64();
        }
        ptx::bar_sync(1, kConsumers);
        if (up) {
          const int nt = (MODE == 1) ? 8 : 64;
          if (tid < nt) {
            const int r = (MODE == 1) ? tid : (tid >> 3), n = (MODE == 1) ? 0 : (tid & 7);
            const int pr = C.colpair[n];
            if (pr >= 0) {
              const float gate = reduced<MODE>(C, rb, 0, r, n), upv = reduced<MODE>(C, rb, 0, r + 8, n);
              a.h16[(size_t)pr * g.I + tl * 8 + r] = __float2half_rn(siluf_acc(gate) * upv);
            }
          }
          ++up_n;
        } else {
          const int nt = (MODE == 1) ? 32 : 256;
          if (tid < nt) {
            const int half = (MODE == 1) ? (tid >> 4) : (tid >> 7);
            const int r = (MODE == 1) ? (tid & 15) : ((tid & 127) >> 3), n = (MODE == 1) ? 0 : (tid & 7);
            const float wn = C.colw[n];
            if (n < T && wn != 0.f)
              atomicAdd(a.out_acc + (size_t)n * H + (2 * tl + half) * 16 + r, wn * reduced<MODE>(C, rb, half, r, n));
          }
        }
        rb ^= 1;
        c_epi += clock64() - te0;
      }
      if (up) flush_up();
      if (tid == 0) DEC_TRACE(ph == 0 ? 4 : ph == 2 ? 8 : 10);
    }
    // ---- the last CTA to finish its down tiles converts the whole output (every other CTA's
    // atomics are ordered before its ticket by the barrier and fence below)
    ptx::bar_sync(1, kConsumers);
    if (tid == 0) {
      __threadfence();
      const uint32_t ticket = atomicAdd(a.sync + 4, 1u);
      C.flag = ticket == (uint32_t)g.G - 1;
      DEC_TRACE(11);
    }
    ptx::bar_sync(1, kConsumers);
    if (C.flag) {
      __threadfence();
      const int n4 = T * H / 4;
#pragma unroll 4
      for (int i = tid; i < n4; i += kConsumers) {
        const float4 v = __ldcg(reinterpret_cast<const float4*>(a.out_acc) + i);
        reinterpret_cast<float4*>(a.out_acc)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        store_act<XDT>(a.out, 4 * (size_t)i, v.x);
        store_act<XDT>(a.out, 4 * (size_t)i + 1, v.y);
        store_act<XDT>(a.out, 4 * (size_t)i + 2, v.z);
        store_act<XDT>(a.out, 4 * (size_t)i + 3, v.w);
      }
    }
    if (tid == 0) {
      C.consumed = it_ok;
      DEC_TRACE(12);
      if (a.trace) a.trace[(size_t)blockIdx.x * 64 + 25] = clock64();
      if (a.trace) {
        unsigned long long* tr = a.trace + (size_t)blockIdx.x * 64;
        tr[16] = c_wait;
        tr[17] = c_comp;
        tr[18] = c_epi;
        tr[19] = c_tr;
        tr[20] = (unsigned long long)it;
      }
    }
  }
  __syncthreads();
  if (tid == 0) {
    // drain copies this CTA issued but did not see complete (only after an abort): the last
    // issued item of each slot is the only one that can still be in flight
    const int issued = C.issued;
    for (int i = max(C.consumed, issued - kSlots); i < issued; ++i)
      ptx::mbar_wait(&S.full[i % kSlots], (i / kSlots) & 1, kMbarSpin);
    __threadfence();
    const uint32_t old = atomicAdd(a.sync + 2, 1u);
    if (old == (uint32_t)g.G - 1) {
      // last CTA out: reset the counters for the next call
      a.sync[0] = 0;
      a.sync[4] = 0;
      for (int i = 0; i <= g.E; ++i) up_done[i] = 0;
      __threadfence();
      a.sync[2] = 0;
    }
  }
}

// ------------------------------------------------------------------ repack

// Row-major int4-g32 matrix (codes [R][K/2], fp16 scales [R][K/32]) -> 16-row tiles of
// 2048-column panels in MMA fragment order. `up` selects the gate/up row pairing
// (MMA rows 0-7 = gate rows 8i.., rows 8-15 = up rows R/2 + 8i..).
// Per panel: codes [32 chunks of 64 columns][32 lanes][4 words] (word q of lane (g, t) in
// chunk c: the 8 nibbles (g, 2t) (g+8, 2t) (g, 2t+8) (g+8, 2t+8) (g, 2t+1) (g+8, 2t+1)
// (g, 2t+9) (g+8, 2t+9) of MMA 4c+q, low nibble first), then scales [8 k-blocks][8 g][4 t]
// x {s[g][j], s[g][j+1], s[g+8][j], s[g+8][j+1]} with j = 8 * kblock + 2t.
__global__ void repack_kernel(const uint8_t* __restrict__ codes, const __half* __restrict__ scales,
                              int R, int K, int up, uint8_t* __restrict__ dst) {
  const int ntile = R / 16, np = K / kPanelK;
  const size_t words_per_panel = kCodeBytes / 4;
  const size_t total_words = (size_t)ntile * np * words_per_panel;
  const size_t total_scl = (size_t)ntile * np * (kScaleBytes / 8);   // 8-byte scale quads
  auto row_of = [&](int tile, int m) -> int {
    if (!up) return tile * 16 + m;
    const int half = R / 2;
    return (m < 8) ? tile * 8 + m : half + tile * 8 + (m - 8);
  };
  auto nib = [&](int row, int kk) -> uint32_t {
    const uint8_t b = codes[(size_t)row * (K / 2) + (kk >> 1)];
    return (kk & 1) ? (b >> 4) : (b & 15u);
  };
  for (size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total_words + total_scl;
       idx += (size_t)gridDim.x * blockDim.x) {
    if (idx < total_words) {
      const size_t tp = idx / words_per_panel;          // tile * np + panel
      const int wi = (int)(idx % words_per_panel);      // word within the panel
      const int tile = (int)(tp / np), p = (int)(tp % np);
      const int q = wi & 3, lane = (wi >> 2) & 31, c = wi >> 7;
      const int gq = lane >> 2, t = lane & 3;
      const int k0 = p * kPanelK + 64 * c + 16 * q;
      const int rA = row_of(tile, gq), rB = row_of(tile, gq + 8);
      const uint32_t w = nib(rA, k0 + 2 * t) | (nib(rB, k0 + 2 * t) << 4) | (nib(rA, k0 + 2 * t + 8) << 8) |
                         (nib(rB, k0 + 2 * t + 8) << 12) | (nib(rA, k0 + 2 * t + 1) << 16) |
                         (nib(rB, k0 + 2 * t + 1) << 20) | (nib(rA, k0 + 2 * t + 9) << 24) |
                         (nib(rB, k0 + 2 * t + 9) << 28);
      reinterpret_cast<uint32_t*>(dst + tp * kItemBytes)[wi] = w;
    } else {
      const size_t si = idx - total_words;
      const size_t tp = si / (kScaleBytes / 8);
      const int qi = (int)(si % (kScaleBytes / 8));     // (kb, g, t) quad
      const int tile = (int)(tp / np), p = (int)(tp % np);
      const int t = qi & 3, gq = (qi >> 2) & 7, kb = qi >> 5;
      const int grp = (p * kPanelK) / 32 + 8 * kb + 2 * t;
      const int rA = row_of(tile, gq), rB = row_of(tile, gq + 8);
      __half* o = reinterpret_cast<__half*>(dst + tp * kItemBytes + kCodeBytes) + (size_t)qi * 4;
      o[0] = scales[(size_t)rA * (K / 32) + grp];
      o[1] = scales[(size_t)rA * (K / 32) + grp + 1];
      o[2] = scales[(size_t)rB * (K / 32) + grp];
      o[3] = scales[(size_t)rB * (K / 32) + grp + 1];
    }
  }
}

template <int MODE, int XDT, int WDT>
cudaError_t launch_decode_t(const DecodeArgs& a, int grid, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kDecThreads);
  cfg.dynamicSmemBytes = sizeof(DecSmem<MODE>);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, moe_decode_kernel<MODE, XDT, WDT>, a);
}

template <int MODE, int XDT, int WDT>
cudaError_t init_one() {
  return cudaFuncSetAttribute(moe_decode_kernel<MODE, XDT, WDT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)sizeof(DecSmem<MODE>));
}

}  // namespace

size_t decode_tile_bytes(int R, int K) { return (size_t)(R / 16) * (K / kPanelK) * kItemBytes; }

bool decode_supported(int H, int I, int E, int top_k, int T) {
  return H % kPanelK == 0 && I % kPanelK == 0 && H <= kMaxH && I <= kMaxI && E <= kMaxE && E % 32 == 0 &&
         T >= 1 && T <= 8 && T * top_k <= kMaxActive && top_k <= kMaxK;
}

size_t decode_smem_bytes() {
  return sizeof(DecSmem<0>) > sizeof(DecSmem<1>) ? sizeof(DecSmem<0>) : sizeof(DecSmem<1>);
}

cudaError_t decode_occupancy(int* blocks_per_sm) {
  int b0 = 0, b1 = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b0, moe_decode_kernel<0, MOE_DT_BF16, MOE_DT_F32>,
                                                                kDecThreads, sizeof(DecSmem<0>));
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b1, moe_decode_kernel<1, MOE_DT_BF16, MOE_DT_F32>, kDecThreads,
                                                      sizeof(DecSmem<1>));
  *blocks_per_sm = b0 < b1 ? b0 : b1;
  return e;
}

cudaError_t launch_repack(const uint8_t* codes, const void* scales, int R, int K, bool up, uint8_t* dst,
                          cudaStream_t s) {
  repack_kernel<<<148 * 8, 256, 0, s>>>(codes, static_cast<const __half*>(scales), R, K, up ? 1 : 0, dst);
  return cudaGetLastError();
}

cudaError_t decode_kernels_init() {
  cudaError_t e = cudaSuccess;
  const cudaError_t r[] = {init_one<0, MOE_DT_F32, MOE_DT_F32>(), init_one<0, MOE_DT_BF16, MOE_DT_F32>(),
                           init_one<0, MOE_DT_F32, MOE_DT_BF16>(), init_one<0, MOE_DT_BF16, MOE_DT_BF16>(),
                           init_one<1, MOE_DT_F32, MOE_DT_F32>(), init_one<1, MOE_DT_BF16, MOE_DT_F32>(),
                           init_one<1, MOE_DT_F32, MOE_DT_BF16>(), init_one<1, MOE_DT_BF16, MOE_DT_BF16>()};
  for (cudaError_t x : r)
    if (x != cudaSuccess) e = x;
  return e;
}

cudaError_t launch_decode_fused(const DecodeLaunch& d, int act_dtype, int router_dtype, int grid,
                                cudaStream_t s) {
  DecodeArgs a;
  a.x = d.x;
  a.T = d.T;
  a.router_w = d.router_w;
  a.bias = d.bias;
  a.H = d.H;
  a.I = d.I;
  a.E = d.E;
  a.top_k = d.top_k;
  a.n_group = d.n_group;
  a.topk_group = d.topk_group;
  a.rsf = d.rsf;
  a.up_store = d.up_store;
  a.down_store = d.down_store;
  a.logits = d.logits;
  a.ids = d.ids;
  a.weights = d.weights;
  a.offsets = d.offsets;
  a.entries = d.entries;
  a.h16 = static_cast<__half*>(d.h16);
  a.out_acc = d.out_acc;
  a.out = d.out;
  a.sync = d.sync;
  a.status = d.status;
  a.spin_max = d.spin_max;
  a.trace = d.trace;
  const bool xf = act_dtype == MOE_DT_F32, wf = router_dtype == MOE_DT_F32;
  if (a.T == 1) {
    if (xf) return wf ? launch_decode_t<1, MOE_DT_F32, MOE_DT_F32>(a, grid, s) : launch_decode_t<1, MOE_DT_F32, MOE_DT_BF16>(a, grid, s);
    return wf ? launch_decode_t<1, MOE_DT_BF16, MOE_DT_F32>(a, grid, s) : launch_decode_t<1, MOE_DT_BF16, MOE_DT_BF16>(a, grid, s);
  }
  if (xf) return wf ? launch_decode_t<0, MOE_DT_F32, MOE_DT_F32>(a, grid, s) : launch_decode_t<0, MOE_DT_F32, MOE_DT_BF16>(a, grid, s);
  return wf ? launch_decode_t<0, MOE_DT_BF16, MOE_DT_F32>(a, grid, s) : launch_decode_t<0, MOE_DT_BF16, MOE_DT_BF16>(a, grid, s);
}

}  // namespace moe
