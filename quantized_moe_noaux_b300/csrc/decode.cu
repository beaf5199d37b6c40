// Fused decode-path kernel of the MoE layer (T <= 8 tokens per call) on the tcgen05 tensor
// cores, with the dequantised weights staged in tensor memory.
//
// One persistent cooperative grid (one CTA per SM) runs the whole layer forward of a decode
// step: router logits, noaux_tc selection and batch-union grouping, the SwiGLU gate/up
// projection of the shared and the selected experts, and the down projection with the
// weighted combine ("Show HN: Menjalankan GLM 5.2 di komputer lambat", section "Fitur utama
// yang diimplementasikan": DeepSeek-V3-style router with noaux_tc, routed_scaling_factor and
// a shared expert; packed int4 with dequant-on-use; batch-union MoE). Every selected expert's
// weights are streamed from HBM exactly once.
//
// Weights are read from the packed store of the grouped GEMM: per (expert, 128-row tile,
// 256-column group) one 18 KB item (codes, then fp16 scales). Gate/up tiles pair 16 gate rows
// with the matching 16 up rows in each 32-row quarter.
//
// A unit of work is (expert, 128-row tile, K split); each CTA walks its share of four
// segments in order: shared gate/up, routed gate/up (after the routing is known), shared
// down, routed down. Warp roles:
//   warp 12     producer: one TMA bulk copy per item into a ring of shared-memory slots;
// (segment order: shared gate/up, routed gate/up, shared down, routed down)
//   warps 4-11  decoders: every item is split over the 8 warps (row quarter = warp mod 4,
//               column half = the warp's half of the group); a thread turns its row's 128
//               int4 codes into fp16 (code times the fp16 group scale, rounded once) and
//               stores them to tensor memory (a ring of three 128-column A slots);
//   warp 13     lane 0 issues tcgen05.mma kind::f16 (M=128 weight rows with A read from
//               tensor memory, N=16 columns: the tokens, K=16) into one of two accumulators;
//   warp 15     stages the h rows each down unit multiplies into one of two shared-memory
//               panels, once all gate/up tiles of that expert are done;
//   warps 0-11  router rows at the start;
//   warps 0-3   then the epilogue of each unit: the accumulator
//               rows go to a K-split partial buffer; the last split of a gate/up tile to
//               arrive computes h = SiLU(gate) * up (fp16); the last unit of a 128-row block
//               of the output to arrive computes out = sum_j w_j y_j + y_shared in a fixed
//               order (the combine is deterministic);
//   warps 0-3   routing, between the router rows and the first epilogue: once every CTA's
//               router rows are written, block-parallel selection of each token's experts
//               and grouping of the entries (every CTA gets the same result);
//   warp 14     spare.
// The activations (B operand) live in shared memory as [K/8][T][8] fp16 panels: an 8 x 16 B
// core matrix starting at a chunk holds the T tokens of that chunk in its first T rows (the
// other rows read the next chunk; those accumulator columns are ignored).
// All waits are bounded; on time-out the kernel records MOE_ERR_TIMEOUT, stops issuing work,
// lets its copies and MMAs in flight land, frees its tensor memory and returns.
#include <cstddef>

#include "kernels.h"
#include "ptx.cuh"
#include "route_dev.cuh"

namespace moe {

namespace {

constexpr int kEpiWarps = 4;           // warps 0-3
constexpr int kDecWarp0 = 4;           // warps 4-11
constexpr int kWarpProd = 12;
constexpr int kWarpMma = 13;
constexpr int kWarpRoute = 14;
constexpr int kWarpStage = 15;
constexpr int kWorkWarps = 12;         // warps 0-11 share the router rows
constexpr int kDecThreads = 16 * 32;
constexpr int kTileM = 128;            // weight rows per unit (MMA M)
constexpr int kGroupK = 256;           // K columns per item
constexpr int kItemCodes = 16384;      // 128 rows x 256 int4
constexpr int kItemBytes = 18432;      // + 128 rows x 8 fp16 scales
constexpr int kASlots = 3;             // tensor-memory A slots of 128 columns
constexpr int kDCol0 = kASlots * 128;  // two 16-column accumulators after the A slots
constexpr int kN = 16;                 // MMA N (tokens; T <= 8 columns used)
constexpr uint32_t kTmemCols = 512;
constexpr int kMaxT = 8;
constexpr int kMaxH = 8192;
constexpr int kMaxI = 4096;
constexpr int kMaxE = 256;
constexpr int kMaxK = 16;
constexpr int kMaxActive = 64;         // T * top_k <= 64 on this path
constexpr int kMaxSlots = 12;          // shared-memory ring slots
constexpr int kMaxKsu = 8;             // K splits of a gate/up tile
constexpr int kMaxKsd = 4;             // K splits of a down tile
constexpr int kPanelPad = 512;         // bytes after a panel that the last core matrices may touch
constexpr int kSmemLimit = 227 * 1024;

// Fixed part of the shared memory (the ring and the panels follow at runtime offsets).
struct alignas(16) DecFixed {
  float selb[kMaxE];                   // selection scratch: biased and unbiased scores of one token
  float sels[kMaxE];
  int idsel[kMaxT][kMaxK];             // per token: selected experts and weights (slot order)
  float wsel[kMaxT][kMaxK];
  int cnt[kMaxE];
  int soff[kMaxE];
  int aslot[kMaxE];
  int active[kMaxE];                   // active expert a (routed units use slot 1 + a)
  int meta_j[kMaxActive][kMaxT];       // per active expert and token: selection slot (-1 none)
  float red[kWorkWarps][2][kMaxT];     // router-row reduction
  // one-token mode (CUDA-core dot products): unit results handed to the epilogue, the half
  // sums of a unit, and per 32-column group the sums of the activation values that meet
  // the 1032 + c and the 1152 + 16 c decoded forms (x, and the two h panels)
  float gscore[32];                    // block selection: group scores, kept flags, picks
  int gkept[32];
  int pick[kMaxK];
  float dsm[2][2][kTileM];             // [accumulator buffer][column half][row]
  float xsum[kMaxH / 32][2];
  float hsum[2][kMaxI / 32][2];
  uint64_t full[kMaxSlots];
  uint64_t empty[kMaxSlots];
  uint64_t afull[kASlots];
  uint64_t aempty[kASlots];
  uint64_t dfull[2];
  uint64_t dempty[2];
  uint64_t hfree[2];
  uint64_t hready[2];
  uint64_t route_bar;
  uint64_t router_bar;

  uint64_t fin_bar;
  uint32_t tmem_base;
  int n_active;
  int abort;
  int issued;
  int consumed;
  int flag;      // epilogue: this unit arrived last
  int ep_stop;   // epilogue: uniform stop decision
  int ep_nact;   // epilogue: active experts, read once by thread 0
};

struct DecodeArgs {
  const void* x;
  int T;
  const void* router_w;
  const float* bias;
  int H, I, E, top_k, n_group, topk_group;
  float rsf;
  float top_p;                 // adaptive expert top-p (0 < top_p < 1), else every slot kept
  int identity_act;            // test-only: h = gate * up (no SiLU)
  const uint8_t* pack_up;      // [E+1][I/64 tiles][H/256 groups][18432]
  const uint8_t* pack_dn;      // [E+1][H/128 tiles][I/256 groups][18432]
  float* logits;               // [T, E]
  int32_t* ids;
  float* weights;
  int32_t* offsets;
  int32_t* entries;
  __half* h16;                 // [(1 + active) * T][I]: h of slot s, token t at row s * T + t
  float* gu_part;              // gate/up K-split partials [slot][tile][split][T][128]
  float* y_part;               // down K-split outputs [T][top_k + 1][split][H]
  void* out;
  uint32_t* sync;              // [0] CTAs done with router rows, [2] CTAs exited; up_done, up_cnt, dn_cnt
  int* status;
  unsigned long long wait_ns;  // time limit of the waits on other CTAs
  unsigned long long* trace;   // optional [grid][64] phase timestamps (ns), or NULL
  int ns;                      // ring slots
  int off_ring, off_x, off_h0, off_h1;   // shared-memory offsets
  int ksu, ksd;                // K splits of gate/up and down units
};

// Sync-word layout: [0] CTAs done with router rows, [2] CTAs exited, [3] set when a CTA
// aborted, [4] selection published; then per-slot gate/up tiles done, per (slot, tile)
// K-split arrivals, per 128-row block down arrivals, and the published selection.
constexpr int kSyncUpDone = 8;                          // [1 + kMaxActive] tiles done per slot
constexpr int kSyncUpCnt = kSyncUpDone + 1 + kMaxActive;   // [(1 + kMaxActive) * NTu] split arrivals
__host__ __device__ inline int sync_dn_cnt(int ntu) { return kSyncUpCnt + (1 + kMaxActive) * ntu; }
// published selection: [kMaxT * kMaxK] expert ids, then as many weights (fp32 bits)
__host__ __device__ inline int sync_route(int ntu) { return sync_dn_cnt(ntu) + kMaxH / kTileM; }

// ------------------------------------------------------------------ helpers

__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 u2h(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// One word of packed codes (column 8j + 2i in bits 4i..4i+3, 8j + 2i + 1 in bits 16+4i..)
// -> four fp16x2 (columns 8j..8j+7 in order) of code * scale. (nibble ^ 8) placed in the
// mantissa of 1024 is 1032 + code; placed at mantissa bit 4 it is 1152 + 16 code. Both are
// turned into the code exactly (a subtraction, or x 1/16 - 72 in one fused step); the
// product with the scale is rounded once.
__device__ __forceinline__ void dq_word(uint32_t w, __half2 s2, uint32_t* o) {
  const __half2 k1032 = __float2half2_rn(1032.f);
  const __half2 k16 = __float2half2_rn(0.0625f);
  const __half2 km72 = __float2half2_rn(-72.f);
  const uint32_t w2 = w >> 8;
  const uint32_t p0 = (w & 0x000F000Fu) ^ 0x64086408u;
  const uint32_t p1 = (w & 0x00F000F0u) ^ 0x64806480u;
  const uint32_t p2 = (w2 & 0x000F000Fu) ^ 0x64086408u;
  const uint32_t p3 = (w2 & 0x00F000F0u) ^ 0x64806480u;
  o[0] = h2u(__hmul2(__hsub2(u2h(p0), k1032), s2));
  o[1] = h2u(__hmul2(__hfma2(u2h(p1), k16, km72), s2));
  o[2] = h2u(__hmul2(__hsub2(u2h(p2), k1032), s2));
  o[3] = h2u(__hmul2(__hfma2(u2h(p3), k16, km72), s2));
}

// acc + (fp16 half of a) * (fp16 half of x) with one fp32 rounding (the product is exact).
__device__ __forceinline__ float fma_f16f32(uint32_t a, uint32_t x, float acc, bool hi) {
  const unsigned short ah = hi ? (unsigned short)(a >> 16) : (unsigned short)(a & 0xFFFFu);
  const unsigned short xh = hi ? (unsigned short)(x >> 16) : (unsigned short)(x & 0xFFFFu);
  asm("fma.rn.f32.f16 %0, %1, %2, %0;" : "+f"(acc) : "h"(ah), "h"(xh));
  return acc;
}

// Time limit of the waits inside a CTA (mbarrier phases) and of the final drains.
constexpr unsigned long long kLocalWaitNs = 2000000000ull;

// Wait for an mbarrier phase; false when the CTA's abort flag is set or after limit_ns.
// (try_wait itself may suspend the thread for a while, so the bound is a time, not a count.)
__device__ __forceinline__ bool bar_wait(uint64_t* bar, uint32_t parity, const int* abort_flag,
                                         unsigned long long limit_ns) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (;;) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if (abort_flag && *(volatile const int*)abort_flag) return false;
    if (global_ns() - t0 > limit_ns) return false;
  }
}

// Wait for *p >= target, written by other CTAs (each calling thread polls with acquire
// loads); false when the abort flag is set or after limit_ns.
__device__ __forceinline__ bool geq_wait(const uint32_t* p, uint32_t target, const int* abort_flag,
                                         unsigned long long limit_ns) {
  if (ptx::ld_acquire(p) >= target) return true;
  const unsigned long long t0 = global_ns();
  for (;;) {
    __nanosleep(128);
    if (ptx::ld_acquire(p) >= target) return true;
    if (*(volatile const int*)abort_flag) return false;
    if (global_ns() - t0 > limit_ns) return false;
  }
}

// Balanced contiguous split of n units over G CTAs.
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

// ------------------------------------------------------------------ selection

// noaux_tc selection of one token by the four epilogue warps (128 threads, named barrier 2),
// with the same result as the sequential picks, bit for bit: s = sigmoid(logit), b = s +
// bias; a group's score adds its two largest b (a thread scans each group); the
// topk_group best groups are kept (lower index on ties); an expert of a kept group takes
// slot r when exactly r kept experts rank above it (larger b first, lower index on ties);
// the normaliser adds the picked unbiased scores in slot order. Adaptive top-p as in
// select_token (route_dev.cuh), sums in the same order: a slot stays while the s of the
// slots ranked above it (larger s, lower id on ties) sum below top_p times the total;
// dropped slots get id -1 and weight 0, the kept weights are renormalised.
__device__ void select_block(DecFixed& C, const float* logits_row, const float* bias, int E, int n_group,
                             int topk_group, int top_k, float rsf, float top_p, int* idsel, float* wsel) {
  const int tid = threadIdx.x;
  for (int e = tid; e < E; e += 128) {
    const float sc = sigmoidf_acc(__ldcg(logits_row + e));
    C.sels[e] = sc;
    C.selb[e] = sc + __ldg(bias + e);
  }
  ptx::bar_sync(2, 128);
  const int G = E / n_group;
  if (tid < n_group) {
    float m1 = -INFINITY, m2 = -INFINITY;
    for (int i = 0; i < G; ++i) {
      const float v = C.selb[tid * G + i];
      if (v > m1) {
        m2 = m1;
        m1 = v;
      } else if (v > m2) {
        m2 = v;
      }
    }
    C.gscore[tid] = m1 + m2;
  }
  ptx::bar_sync(2, 128);
  if (tid < n_group) {
    const float gs = C.gscore[tid];
    int rank = 0;
    for (int g2 = 0; g2 < n_group; ++g2) {
      const float o = C.gscore[g2];
      rank += (o > gs) || (o == gs && g2 < tid);
    }
    C.gkept[tid] = rank < topk_group;
  }
  ptx::bar_sync(2, 128);
  for (int e = tid; e < E; e += 128) {
    if (!C.gkept[e / G]) continue;
    const float v = C.selb[e];
    int rank = 0;
    for (int g2 = 0; g2 < n_group; ++g2) {
      if (!C.gkept[g2]) continue;
      for (int e2 = g2 * G; e2 < (g2 + 1) * G; ++e2) {
        const float o = C.selb[e2];
        rank += (o > v) || (o == v && e2 < e);
      }
    }
    if (rank < top_k) C.pick[rank] = e;
  }
  ptx::bar_sync(2, 128);
  if (tid == 0) {
    float wsum = 0.f;
    for (int j = 0; j < top_k; ++j) wsum += C.sels[C.pick[j]];
    float norm = wsum;
    unsigned keep = (1u << top_k) - 1u;
    if (top_p > 0.f && top_p < 1.f) {
      keep = 0u;
      for (int j = 0; j < top_k; ++j) {
        const float sj = C.sels[C.pick[j]];
        int rank = 0;
        float before = 0.f;
        for (int i = 0; i < top_k; ++i) {
          const float si = C.sels[C.pick[i]];
          const bool above = si > sj || (si == sj && C.pick[i] < C.pick[j]);
          rank += above;
          if (above) before += si;
        }
        if (rank == 0 || before < top_p * wsum) keep |= 1u << j;
      }
      norm = 0.f;
      for (int i = 0; i < top_k; ++i)
        if ((keep >> i) & 1u) norm += C.sels[C.pick[i]];
    }
    for (int j = 0; j < top_k; ++j) {
      const bool kj = (keep >> j) & 1u;
      idsel[j] = kj ? C.pick[j] : -1;
      wsel[j] = kj ? C.sels[C.pick[j]] / norm * rsf : 0.f;
    }
  }
  ptx::bar_sync(2, 128);
}

// Phase timestamp of this CTA (profiling hook; one thread records).
#define DEC_TRACE(i)                                                            \
  do {                                                                          \
    if (a.trace) a.trace[(size_t)blockIdx.x * 64 + (i)] = global_ns();          \
  } while (0)

// One warp: group the selected (token, slot) entries per expert and publish the routing in
// shared memory (CTA 0 also to global): counts, exclusive scans (entry offsets, active
// slots), each active expert's selection slot per token, and the ascending entry lists.
__device__ void group_in_cta(DecFixed& C, const DecodeArgs& a) {
  const int lane = threadIdx.x & 31;
  const int T = a.T, E = a.E, k = a.top_k;
  const bool cta0 = blockIdx.x == 0;
  const int n = T * k;
  for (int e = lane; e < E; e += 32) C.cnt[e] = 0;
  __syncwarp();
  for (int f = lane; f < n; f += 32) {
    const int e = C.idsel[f / k][f % k];
    if (e >= 0) atomicAdd(&C.cnt[e], 1);   // -1: dropped by the adaptive top-p
  }
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
      if (cta0) a.offsets[e] = run;
      if (cl[i] > 0) {
        C.aslot[e] = apos;
        C.active[apos++] = e;
      }
      run += cl[i];
    }
  }
  const int na = __shfl_sync(0xffffffffu, inca, 31);
  if (lane == 31 && cta0) a.offsets[E] = run;
  for (int i = lane; i < na * kMaxT; i += 32) C.meta_j[i / kMaxT][i % kMaxT] = -1;
  __syncwarp();
  const int* flat = &C.idsel[0][0];   // entry f = token * top_k + slot at idsel[token][slot]
  for (int f = lane; f < n; f += 32) {
    const int tok = f / k, slot = f % k;
    const int e = C.idsel[tok][slot];
    if (e >= 0) C.meta_j[C.aslot[e]][tok] = slot;
    if (cta0) {
      if (e >= 0) {
        int rank = 0;
        for (int f2 = 0; f2 < f; ++f2) rank += (flat[(f2 / k) * kMaxK + f2 % k] == e);
        a.entries[C.soff[e] + rank] = f;
      }
      a.ids[f] = e;
      a.weights[f] = C.wsel[tok][slot];
    }
  }
  if (lane == 0) C.n_active = na;
  __syncwarp();
}

// A unit of work: expert slot (0 = shared, 1 + a = active expert a), expert index in the
// packed store, 128-row tile, K split and its item range.
struct Unit {
  int down, slot, e, tile, split, g0, ng;
};

struct Geo {
  int NTu, NGu, NTd, NGd, ksu, ksd;
  int G, c;
  int a0, a1, c10, c11;   // this CTA's shared gate/up and shared down unit ranges
};

// Unit v of segment ph (0 shared gate/up, 1 shared down, 2 routed gate/up, 3 routed down).
__device__ __forceinline__ Unit make_unit(const Geo& g, const DecFixed& C, int ph, int v, int E) {
  Unit u;
  u.down = ph & 1;
  const int nt = u.down ? g.NTd : g.NTu, ks = u.down ? g.ksd : g.ksu, ngr = u.down ? g.NGd : g.NGu;
  const int per = nt * ks;
  const int sl = ph < 2 ? 0 : 1 + v / per;
  const int w = v % per;
  u.slot = sl;
  u.e = sl == 0 ? E : C.active[sl - 1];
  u.tile = w / ks;
  u.split = w % ks;
  u.ng = ngr / ks;
  u.g0 = u.split * u.ng;
  return u;
}

// Execution order of the segments: shared gate/up, routed gate/up (once the routing is
// known), shared down, routed down. The shared down units come after the routed gate/up
// ones so that no CTA idles on the shared expert's h while the routing is already known;
// by the time they run, that h is complete.
__device__ __forceinline__ int seg_at(int step) { return step == 0 ? 0 : step == 1 ? 2 : step == 2 ? 1 : 3; }

__device__ __forceinline__ void seg_of(const Geo& g, int ph, int nact, int& lo, int& hi) {
  if (ph == 0) {
    lo = g.a0;
    hi = g.a1;
  } else if (ph == 1) {
    lo = g.c10;
    hi = g.c11;
  } else if (ph == 2) {
    seg_range(nact * g.NTu * g.ksu, g.G, g.c, lo, hi);
  } else {
    seg_range(nact * g.NTd * g.ksd, g.G, g.c, lo, hi);
  }
}

template <int XDT, int WDT, bool CC>
__global__ void __launch_bounds__(kDecThreads, 1) moe_decode_kernel(DecodeArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  DecFixed& C = *reinterpret_cast<DecFixed*>(smem_raw);
  uint8_t* const ring = smem_raw + a.off_ring;
  uint8_t* const xpanel = smem_raw + a.off_x;
  uint8_t* const hpanel[2] = {smem_raw + a.off_h0, smem_raw + a.off_h1};
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = a.T, H = a.H, I = a.I, E = a.E, k = a.top_k;
  const int ns = a.ns;
  Geo g;
  g.NTu = I / 64;
  g.NGu = H / kGroupK;
  g.NTd = H / kTileM;
  g.NGd = I / kGroupK;
  g.ksu = a.ksu;
  g.ksd = a.ksd;
  g.G = gridDim.x;
  g.c = blockIdx.x;
  seg_range(g.NTu * g.ksu, g.G, g.c, g.a0, g.a1);
  seg_range(g.NTd * g.ksd, g.G, g.c, g.c10, g.c11);
  uint32_t* const up_done = a.sync + kSyncUpDone;
  uint32_t* const up_cnt = a.sync + kSyncUpCnt;
  uint32_t* const dn_cnt = a.sync + sync_dn_cnt(g.NTu);

  if (tid == 0) {
    for (int s = 0; s < ns; ++s) {
      ptx::mbar_init(&C.full[s], 1);
      ptx::mbar_init(&C.empty[s], 8);
    }
    for (int s = 0; s < kASlots; ++s) {
      ptx::mbar_init(&C.afull[s], 8);
      ptx::mbar_init(&C.aempty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      // one-token mode: the 8 decoder warps arrive themselves; tensor mode: one commit
      ptx::mbar_init(&C.dfull[b], CC ? 8 : 1);
      ptx::mbar_init(&C.dempty[b], kEpiWarps);
      ptx::mbar_init(&C.hfree[b], CC ? 8 : 1);
      ptx::mbar_init(&C.hready[b], 1);
    }
    ptx::mbar_init(&C.route_bar, 1);
    ptx::mbar_init(&C.router_bar, 1);

    ptx::mbar_init(&C.fin_bar, 1);
    ptx::fence_mbar_init();
    C.abort = 0;
    C.issued = 0;
    C.consumed = 0;
    C.n_active = 0;
  }
  if (!CC && warp == kWarpMma) {
    ptx::tmem_alloc(&C.tmem_base, kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = CC ? 0u : C.tmem_base;

  auto abort_now = [&]() {
    atomicExch(&C.abort, 1);
    atomicExch(a.sync + 3, 1u);   // the last CTA out then resets every counter
    raise_status(a.status, MOE_ERR_TIMEOUT);
  };
  auto aborted = [&]() { return *(volatile int*)&C.abort != 0; };
  // The routing, once the routing warp published it (bounded wait; 0 active on time-out).
  auto wait_route = [&]() -> int {
    if (!bar_wait(&C.route_bar, 0, &C.abort, kLocalWaitNs)) {
      abort_now();
      return 0;
    }
    return C.n_active;
  };
  // Router rows e = c, c + G, ..., two at a time over warps 0-11: a thread takes 4
  // consecutive columns per 1536 of both rows (fp32 FMA), then warp and CTA reductions.
  // Afterwards this CTA's rows are published to the routing warps of every CTA.
  auto router_rows = [&]() {
    constexpr int kRowVec = (kMaxH + 1535) / 1536;
    for (int e0 = g.c; e0 < E; e0 += 2 * g.G) {
      const int e1 = e0 + g.G;
      const bool two = e1 < E;
      float racc[2][kMaxT];
#pragma unroll
      for (int i = 0; i < kMaxT; ++i) racc[0][i] = racc[1][i] = 0.f;
      float4 wv[2][kRowVec];
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const int e = rr ? e1 : e0;
#pragma unroll
        for (int qq = 0; qq < kRowVec; ++qq) {
          const int col = 1536 * qq + 4 * tid;
          wv[rr][qq] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (col < H && (rr == 0 || two)) {
            if constexpr (WDT == MOE_DT_F32) {
              wv[rr][qq] =
                  __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(a.router_w) + (size_t)e * H + col));
            } else {
              const uint2 uu = __ldg(reinterpret_cast<const uint2*>(static_cast<const unsigned short*>(a.router_w) +
                                                                    (size_t)e * H + col));
              wv[rr][qq] = make_float4(__uint_as_float(uu.x << 16), __uint_as_float(uu.x & 0xFFFF0000u),
                                       __uint_as_float(uu.y << 16), __uint_as_float(uu.y & 0xFFFF0000u));
            }
          }
        }
      }
#pragma unroll
      for (int qq = 0; qq < kRowVec; ++qq) {
        const int col = 1536 * qq + 4 * tid;
        if (col < H) {
#pragma unroll
          for (int i = 0; i < kMaxT; ++i) {
            if (i < T) {
              float xv[4];
              if constexpr (XDT == MOE_DT_F32) {
                const float4 f =
                    __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(a.x) + (size_t)i * H + col));
                xv[0] = f.x; xv[1] = f.y; xv[2] = f.z; xv[3] = f.w;
              } else {
                const uint2 uu = __ldg(reinterpret_cast<const uint2*>(static_cast<const unsigned short*>(a.x) +
                                                                      (size_t)i * H + col));
                xv[0] = __uint_as_float(uu.x << 16);
                xv[1] = __uint_as_float(uu.x & 0xFFFF0000u);
                xv[2] = __uint_as_float(uu.y << 16);
                xv[3] = __uint_as_float(uu.y & 0xFFFF0000u);
              }
#pragma unroll
              for (int rr = 0; rr < 2; ++rr) {
                racc[rr][i] = fmaf(wv[rr][qq].x, xv[0], racc[rr][i]);
                racc[rr][i] = fmaf(wv[rr][qq].y, xv[1], racc[rr][i]);
                racc[rr][i] = fmaf(wv[rr][qq].z, xv[2], racc[rr][i]);
                racc[rr][i] = fmaf(wv[rr][qq].w, xv[3], racc[rr][i]);
              }
            }
          }
        }
      }
#pragma unroll
      for (int rr = 0; rr < 2; ++rr)
#pragma unroll
        for (int i = 0; i < kMaxT; ++i) {
          float v = racc[rr][i];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
          if (lane == 0) C.red[warp][rr][i] = v;
        }
      ptx::bar_sync(1, kWorkWarps * 32);
      if (tid < 2 * T) {
        const int rr = tid / T, i = tid % T;
        if (rr == 0 || two) {
          float v = 0.f;
#pragma unroll
          for (int w = 0; w < kWorkWarps; ++w) v += C.red[w][rr][i];
          a.logits[(size_t)i * E + (rr ? e1 : e0)] = v;
        }
      }
      ptx::bar_sync(1, kWorkWarps * 32);
    }
    if (tid == 0) {
      __threadfence();
      ptx::red_release_add(a.sync + 0, 1u);
      ptx::mbar_arrive(&C.router_bar);
      DEC_TRACE(2);
    }
  };

  if (warp == kWarpProd) {
    // ------------------------------------------------------------- producer
    if (lane == 0) {
      const uint64_t pol = ptx::policy_evict_first();
      int it = 0;
      bool ok = true;
      unsigned long long c_wait = 0;   // profiling: cycles waiting for a free slot
      auto issue = [&](const uint8_t* src) {
        if (!ok) return;
        const int s = it % ns;
        const unsigned long long t0 = clock64();
        // the first two items go out at once; the rest wait until this CTA's router rows are
        // written, so the weight stream does not delay the routing
        if (it == 2 && !bar_wait(&C.router_bar, 0, &C.abort, kLocalWaitNs)) ok = false;
        if (ok && it >= ns && !bar_wait(&C.empty[s], ((it / ns) - 1) & 1, &C.abort, kLocalWaitNs)) ok = false;
        c_wait += clock64() - t0;
        if (ok && aborted()) ok = false;
        if (!ok) return;
        ptx::mbar_arrive_expect_tx(&C.full[s], kItemBytes);
        ptx::bulk_g2s(ring + (size_t)s * kItemBytes, src, kItemBytes, &C.full[s], pol);
        ++it;
        *(volatile int*)&C.issued = it;
      };
      int nact = 0;
      for (int step = 0; step < 4 && ok; ++step) {
        const int ph = seg_at(step);
        if (ph == 2) nact = wait_route();
        int lo, hi;
        seg_of(g, ph, nact, lo, hi);
        for (int v = lo; v < hi && ok; ++v) {
          const Unit u = make_unit(g, C, ph, v, E);
          const uint8_t* base = u.down ? a.pack_dn + ((size_t)u.e * g.NTd + u.tile) * g.NGd * kItemBytes
                                       : a.pack_up + ((size_t)u.e * g.NTu + u.tile) * g.NGu * kItemBytes;
          for (int q = 0; q < u.ng; ++q) issue(base + (size_t)(u.g0 + q) * kItemBytes);
        }
      }
      if (!ok) abort_now();
      DEC_TRACE(13);
      if (a.trace) {
        a.trace[(size_t)blockIdx.x * 64 + 27] = c_wait;
        a.trace[(size_t)blockIdx.x * 64 + 28] = (unsigned long long)it;
      }
    }
  } else if (warp == kWarpRoute) {
    // spare warp (the routing runs on the epilogue warps)
  } else if (warp >= kDecWarp0 && warp < kDecWarp0 + 8) {
    // ------------------------------------------------------------- decoders
    const int dt = tid - kDecWarp0 * 32;       // 0..255
    const int hf = (warp - kDecWarp0) >> 2;    // column half of every item: groups 4 hf .. 4 hf + 3
    const int q = warp & 3, r = 32 * q + lane;  // TMEM lane quarter and weight row
    // activation panel: [H/8][T][8] fp16 (the tensor core reads it)
    {
      const int n = (H / 8) * T;
      for (int idx = dt; idx < n; idx += 256) {
        const int c = idx % T, chunk = idx / T;
        float v[8];
        load_act8<XDT>(a.x, (size_t)c * H + 8 * chunk, v);
        uint4 o;
        o.x = h2u(__floats2half2_rn(v[0], v[1]));
        o.y = h2u(__floats2half2_rn(v[2], v[3]));
        o.z = h2u(__floats2half2_rn(v[4], v[5]));
        o.w = h2u(__floats2half2_rn(v[6], v[7]));
        *reinterpret_cast<uint4*>(xpanel + (size_t)idx * 16) = o;
      }
      ptx::fence_proxy_async_smem();
      ptx::bar_sync(3, 256);
      if constexpr (CC) {
        // per 32-column group: sums of the x values at the 1032 + c and 1152 + 16 c positions
        const uint32_t* xp = reinterpret_cast<const uint32_t*>(xpanel);
        for (int j = dt; j < H / 32; j += 256) {
          float s1 = 0.f, s16 = 0.f;
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const float2 p0 = __half22float2(u2h(xp[16 * j + 4 * w]));
            const float2 p1 = __half22float2(u2h(xp[16 * j + 4 * w + 1]));
            const float2 p2 = __half22float2(u2h(xp[16 * j + 4 * w + 2]));
            const float2 p3 = __half22float2(u2h(xp[16 * j + 4 * w + 3]));
            s1 += (p0.x + p0.y) + (p2.x + p2.y);
            s16 += (p1.x + p1.y) + (p3.x + p3.y);
          }
          C.xsum[j][0] = s1;
          C.xsum[j][1] = s16;
        }
        ptx::bar_sync(3, 256);
      }
    }
    router_rows();
    int it_ok = 0;   // items consumed (for the drain count)
    if constexpr (CC) {
      // ---- one token: every thread computes its row's dot product over its half of each
      // item (groups 4 hf .. 4 hf + 3) with exact products; unit results go to the
      // epilogue through shared memory
      int it = 0, uc = 0, sw = -1, sslot = -1, nact = 0;
      bool ok = true;
      unsigned long long c_full = 0, c_busy = 0, c_hand = 0, c_route = 0, c_hready = 0;
      const unsigned long long c_loop0 = clock64();
      unsigned long long c_ph[4] = {0, 0, 0, 0};
      int rs = 0;           // ring slot of item `it`
      uint32_t rpar = 0;    // its phase parity
      for (int step = 0; step < 4 && ok; ++step) {
        const int ph = seg_at(step);
        c_ph[step] = clock64();
        if (ph == 2) {
          const unsigned long long tr0 = clock64();
          if (lane == 0) nact = wait_route();
          nact = __shfl_sync(0xffffffffu, nact, 0);
          c_route += clock64() - tr0;
        }
        int lo, hi;
        seg_of(g, ph, nact, lo, hi);
        for (int v = lo; v < hi && ok; ++v, ++uc) {
          const Unit u = make_unit(g, C, ph, v, E);
          const uint32_t* act;
          const float(*asum)[2];
          if (u.down) {
            if (u.slot != sslot || sw < 0) {
              // the previous panel is free once every decoder is done with it
              if (sw >= 0) {
                // this warp is done with the previous panel
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&C.hfree[sw & 1]);
              }
              ++sw;
              sslot = u.slot;
              const unsigned long long th0 = clock64();
              if (!bar_wait(&C.hready[sw & 1], (sw >> 1) & 1, &C.abort, kLocalWaitNs)) ok = false;
              c_hready += clock64() - th0;
              if (__any_sync(0xffffffffu, !ok)) {
                ok = false;
                abort_now();
                break;
              }
            }
            act = reinterpret_cast<const uint32_t*>(hpanel[sw & 1]);
            asum = C.hsum[sw & 1];
          } else {
            act = reinterpret_cast<const uint32_t*>(xpanel);
            asum = C.xsum;
          }
          float y = 0.f;
          for (int qi = 0; qi < u.ng; ++qi, ++it) {
            const int s = rs;
            const uint32_t par = rpar;
            if (++rs == ns) {
              rs = 0;
              rpar ^= 1u;
            }
            const unsigned long long t0 = clock64();
            if (!bar_wait(&C.full[s], par, &C.abort, kLocalWaitNs)) ok = false;
            const unsigned long long t1 = clock64();
            c_full += t1 - t0;
            if (__any_sync(0xffffffffu, !ok)) {
              ok = false;
              abort_now();
              break;
            }
            const uint8_t* sl = ring + (size_t)s * kItemBytes;
            const int gbase = (u.g0 + qi) * 8;   // 32-column group index of the item's first group
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              const int gi = 4 * hf + h;
              const uint4 cw = *reinterpret_cast<const uint4*>(sl + ((size_t)gi * kTileM + r) * 16);
              const float sc =
                  __half2float(*reinterpret_cast<const __half*>(sl + kItemCodes + ((size_t)gi * kTileM + r) * 2));
              const uint32_t* xg = act + 16 * (gbase + gi);
              const uint32_t w[4] = {cw.x, cw.y, cw.z, cw.w};
              float a1 = 0.f, a1b = 0.f, a16 = 0.f, a16b = 0.f;
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const uint4 xv = *reinterpret_cast<const uint4*>(xg + 4 * j);
                const uint32_t w2 = w[j] >> 8;
                const uint32_t p0 = (w[j] & 0x000F000Fu) ^ 0x64086408u;
                const uint32_t p1 = (w[j] & 0x00F000F0u) ^ 0x64806480u;
                const uint32_t p2 = (w2 & 0x000F000Fu) ^ 0x64086408u;
                const uint32_t p3 = (w2 & 0x00F000F0u) ^ 0x64806480u;
                a1 = fma_f16f32(p0, xv.x, a1, false);
                a1b = fma_f16f32(p0, xv.x, a1b, true);
                a16 = fma_f16f32(p1, xv.y, a16, false);
                a16b = fma_f16f32(p1, xv.y, a16b, true);
                a1 = fma_f16f32(p2, xv.z, a1, false);
                a1b = fma_f16f32(p2, xv.z, a1b, true);
                a16 = fma_f16f32(p3, xv.w, a16, false);
                a16b = fma_f16f32(p3, xv.w, a16b, true);
              }
              const float c1 = fmaf(-1032.f, asum[gbase + gi][0], a1 + a1b);
              const float c16 = fmaf(-1152.f, asum[gbase + gi][1], a16 + a16b);
              y = fmaf(sc, fmaf(c16, 0.0625f, c1), y);
            }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&C.empty[s]);
            c_busy += clock64() - t1;
            ++it_ok;
          }
          if (!ok) break;
          // unit result: each column half goes to accumulator buffer uc % 2 (once the
          // epilogue released it two units ago); the epilogue adds the halves
          const unsigned long long th = clock64();
          const int db = uc & 1;
          if (uc >= 2 && !bar_wait(&C.dempty[db], ((uc >> 1) - 1) & 1, &C.abort, kLocalWaitNs)) abort_now();
          C.dsm[db][hf][r] = y;
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&C.dfull[db]);
          c_hand += clock64() - th;
          ok = !aborted();
          ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        }
      }
      if (a.trace && tid == kDecWarp0 * 32) {
        unsigned long long* tr = a.trace + (size_t)blockIdx.x * 64;
        tr[16] = c_full;
        tr[17] = c_hand;
        tr[18] = c_busy;
        tr[19] = (unsigned long long)it_ok;
        tr[35] = c_route;
        tr[36] = c_hready;
        tr[37] = clock64() - c_loop0;
        for (int i = 0; i < 4; ++i) tr[38 + i] = c_ph[i] ? c_ph[i] - c_loop0 : 0;
      }
      if (tid == kDecWarp0 * 32) C.consumed = it_ok;
    } else {
    const int ipu_up = g.NGu / g.ksu, ipu_dn = g.NGd / g.ksd;
    int n_items = (g.a1 - g.a0) * ipu_up + (g.c11 - g.c10) * ipu_dn;   // shared items; routed ones later
    bool routed_known = false;
    unsigned long long c_full = 0, c_aempty = 0, c_busy = 0;   // profiling (cycles)
    for (int i = 0;; ++i) {
      if (i >= n_items) {
        if (routed_known) break;
        int nact = 0;
        if (lane == 0) nact = wait_route();
        nact = __shfl_sync(0xffffffffu, nact, 0);
        int lo, hi;
        seg_of(g, 2, nact, lo, hi);
        n_items += (hi - lo) * ipu_up;
        seg_of(g, 3, nact, lo, hi);
        n_items += (hi - lo) * ipu_dn;
        routed_known = true;
        if (i >= n_items) break;
      }
      const int s = i % ns, as = i % kASlots;
      bool ok = !aborted();
      const unsigned long long t0 = clock64();
      if (ok && !bar_wait(&C.full[s], (i / ns) & 1, &C.abort, kLocalWaitNs)) ok = false;
      const unsigned long long t1 = clock64();
      if (ok && i >= kASlots && !bar_wait(&C.aempty[as], ((i / kASlots) - 1) & 1, &C.abort, kLocalWaitNs))
        ok = false;
      const unsigned long long t2 = clock64();
      c_full += t1 - t0;
      c_aempty += t2 - t1;
      if (__any_sync(0xffffffffu, !ok)) {
        abort_now();
        break;
      }
      ptx::tc_fence_after();
      const uint8_t* sl = ring + (size_t)s * kItemBytes;
      const uint32_t tbase = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(128 * as);
#pragma unroll 1
      for (int gp = 2 * hf; gp < 2 * hf + 2; ++gp) {
        uint32_t o[32];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int gi = 2 * gp + h;    // 32-column group within the item
          const uint4 cw = *reinterpret_cast<const uint4*>(sl + ((size_t)gi * kTileM + r) * 16);
          const __half sc = *reinterpret_cast<const __half*>(sl + kItemCodes + ((size_t)gi * kTileM + r) * 2);
          const __half2 s2 = __half2half2(sc);
          dq_word(cw.x, s2, &o[16 * h + 0]);
          dq_word(cw.y, s2, &o[16 * h + 4]);
          dq_word(cw.z, s2, &o[16 * h + 8]);
          dq_word(cw.w, s2, &o[16 * h + 12]);
        }
        ptx::tmem_st32(tbase + (uint32_t)(32 * gp), o);
      }
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        ptx::mbar_arrive(&C.empty[s]);
        ptx::mbar_arrive(&C.afull[as]);
      }
      c_busy += clock64() - t2;
      ++it_ok;
    }
    if (a.trace && tid == kDecWarp0 * 32) {
      unsigned long long* tr = a.trace + (size_t)blockIdx.x * 64;
      tr[16] = c_full;
      tr[17] = c_aempty;
      tr[18] = c_busy;
      tr[19] = (unsigned long long)it_ok;
    }
    // consumed item count (the drain below needs it)
    if (tid == kDecWarp0 * 32) C.consumed = it_ok;
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------- MMA issuer
    if (!CC && lane == 0) {
      constexpr uint32_t idesc = ptx::f16_idesc(kTileM, kN, false);
      const uint32_t lbo = 16u * (uint32_t)T, sbo = 128u;
      const uint64_t dstep = (uint64_t)(2 * T);   // one K step (16 columns = 32 T bytes) in descriptor units
      int it = 0, uc = 0;
      int hsw = -1, hslot = -1;   // down-unit switch index and slot whose h panel is in use
      bool ok = true;
      int nact = 0;
      unsigned long long c_afull = 0, c_dempty = 0, c_stage = 0, c_issue = 0;   // profiling (cycles)
      const unsigned long long c_start = clock64();
      for (int step = 0; step < 4 && ok; ++step) {
        const int ph = seg_at(step);
        if (ph == 2) nact = wait_route();
        int lo, hi;
        seg_of(g, ph, nact, lo, hi);
        for (int v = lo; v < hi && ok; ++v, ++uc) {
          const Unit u = make_unit(g, C, ph, v, E);
          uint32_t panel;
          if (u.down) {
            if (u.slot != hslot || hsw < 0) {
              // a new expert: release the previous panel once its MMAs complete, then wait
              // for the stager to fill panel (switch index) % 2 with this expert's h rows
              const unsigned long long ts0 = clock64();
              if (hsw >= 0) ptx::tc_commit(&C.hfree[hsw & 1]);
              ++hsw;
              hslot = u.slot;
              if (!bar_wait(&C.hready[hsw & 1], (hsw >> 1) & 1, &C.abort, kLocalWaitNs)) {
                ok = false;
                break;
              }
              c_stage += clock64() - ts0;
            }
            panel = ptx::smem_u32(hpanel[hsw & 1]);
          } else {
            panel = ptx::smem_u32(xpanel);
          }
          const int db = uc & 1;
          const unsigned long long tw = clock64();
          if (uc >= 2 && !bar_wait(&C.dempty[db], ((uc >> 1) - 1) & 1, &C.abort, kLocalWaitNs)) {
            ok = false;
            break;
          }
          c_dempty += clock64() - tw;
          ptx::tc_fence_after();
          const uint32_t d = tmem + (uint32_t)(kDCol0 + kN * db);
          for (int qi = 0; qi < u.ng; ++qi, ++it) {
            const int as = it % kASlots;
            const unsigned long long ta = clock64();
            if (!bar_wait(&C.afull[as], (it / kASlots) & 1, &C.abort, kLocalWaitNs)) {
              ok = false;
              break;
            }
            c_afull += clock64() - ta;
            ptx::tc_fence_after();
            const uint32_t a0 = tmem + (uint32_t)(128 * as);
            const uint64_t bd0 = ptx::kmajor_desc(panel + (uint32_t)(u.g0 + qi) * 16u * 32u * (uint32_t)T, lbo, sbo);
            const uint32_t acc0 = qi != 0 ? 1u : 0u;
            const unsigned long long ti = clock64();
#pragma unroll
            for (int jj = 0; jj < 16; ++jj)
              ptx::tc_mma_f16_tmem_a(d, a0 + 8u * jj, bd0 + dstep * (uint64_t)jj, idesc, jj ? 1u : acc0);
            ptx::tc_commit(&C.aempty[as]);
            c_issue += clock64() - ti;
          }
          if (ok) ptx::tc_commit(&C.dfull[db]);
        }
      }
      if (!ok) abort_now();
      DEC_TRACE(14);
      if (a.trace) {
        unsigned long long* tr = a.trace + (size_t)blockIdx.x * 64;
        tr[20] = c_afull;
        tr[21] = c_dempty;
        tr[22] = c_stage;
        tr[23] = (unsigned long long)uc;
        tr[33] = c_issue;
        tr[34] = clock64() - c_start;
      }
    }
  } else if (warp == kWarpStage) {
    // ------------------------------------------------------------- h stager
    // Walks this CTA's down units in order; for each new expert, waits until every MMA that
    // read the panel it will overwrite has completed and until all the expert's gate/up
    // tiles (from every CTA) are done, copies the expert's h rows into the panel
    // ([I/8][T][8] fp16) and signals the MMA issuer.
    int hsw = -1, hslot = -1;
    bool ok = true;
    unsigned long long c_wait = 0;
    for (int ph = 1; ph < 4 && ok; ph += 2) {
      int nact = 0;
      if (ph == 3) {
        if (lane == 0) nact = wait_route();
        nact = __shfl_sync(0xffffffffu, nact, 0);
      }
      int lo, hi;
      seg_of(g, ph, nact, lo, hi);
      for (int v = lo; v < hi && ok; ++v) {
        const Unit u = make_unit(g, C, ph, v, E);
        if (u.slot == hslot && hsw >= 0) continue;
        ++hsw;
        hslot = u.slot;
        const int b = hsw & 1;
        const unsigned long long t0 = clock64();
        bool good = true;
        if (hsw >= 2 && !bar_wait(&C.hfree[b], ((hsw - 2) >> 1) & 1, &C.abort, kLocalWaitNs)) good = false;
        if (good && !geq_wait(up_done + u.slot, (uint32_t)g.NTu, &C.abort, a.wait_ns)) good = false;
        c_wait += clock64() - t0;
        if (__any_sync(0xffffffffu, !good)) {
          if (lane == 0) abort_now();
          ok = false;
          break;
        }
        const int n = (I / 8) * T;
        for (int idx = lane; idx < n; idx += 32) {
          const int c = idx % T, chunk = idx / T;
          const uint4 hv = __ldcg(reinterpret_cast<const uint4*>(a.h16 + ((size_t)u.slot * T + c) * I) + chunk);
          *reinterpret_cast<uint4*>(hpanel[b] + (size_t)idx * 16) = hv;
        }
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if constexpr (CC) {
          // per 32-column group: sums of the h values at the 1032 + c and 1152 + 16 c positions
          const uint32_t* hp = reinterpret_cast<const uint32_t*>(hpanel[b]);
          for (int j = lane; j < I / 32; j += 32) {
            float s1 = 0.f, s16 = 0.f;
#pragma unroll
            for (int w = 0; w < 4; ++w) {
              const float2 p0 = __half22float2(u2h(hp[16 * j + 4 * w]));
              const float2 p1 = __half22float2(u2h(hp[16 * j + 4 * w + 1]));
              const float2 p2 = __half22float2(u2h(hp[16 * j + 4 * w + 2]));
              const float2 p3 = __half22float2(u2h(hp[16 * j + 4 * w + 3]));
              s1 += (p0.x + p0.y) + (p2.x + p2.y);
              s16 += (p1.x + p1.y) + (p3.x + p3.y);
            }
            C.hsum[b][j][0] = s1;
            C.hsum[b][j][1] = s16;
          }
          __syncwarp();
        }
        if (lane == 0) ptx::mbar_arrive(&C.hready[b]);
      }
    }
    if (a.trace && lane == 0) a.trace[(size_t)blockIdx.x * 64 + 32] = c_wait;
  } else {
    // ------------------------------------------------------------- epilogue warps 0-3
    const int q = warp, r = tid;   // TMEM lane quarter q, accumulator row r
    if (tid == 0) {
      DEC_TRACE(0);
      if (a.trace) a.trace[(size_t)blockIdx.x * 64 + 29] = clock64();
    }
    unsigned long long c_dfull = 0, c_epi = 0, c_last = 0;   // profiling (cycles)
    router_rows();
    // routing: once every CTA's router rows are written, select each token's experts
    // (block-parallel), group the entries (warp 0) and publish the result to this CTA
    {
      if (tid == 0) {
        C.ep_stop = geq_wait(a.sync + 0, (uint32_t)g.G, &C.abort, a.wait_ns) ? 0 : 1;
        __threadfence();
        DEC_TRACE(3);
      }
      ptx::bar_sync(2, kEpiWarps * 32);
      if (!C.ep_stop) {
        for (int t = 0; t < T; ++t)
          select_block(C, a.logits + (size_t)t * E, a.bias, E, a.n_group, a.topk_group, k, a.rsf, a.top_p,
                       C.idsel[t], C.wsel[t]);
        if (tid == 0) DEC_TRACE(7);
        if (warp == 0) group_in_cta(C, a);
      } else if (tid == 0) {
        abort_now();
        C.n_active = 0;
      }
      ptx::bar_sync(2, kEpiWarps * 32);
      if (tid == 0) {
        ptx::mbar_arrive(&C.route_bar);
        DEC_TRACE(15);
      }
    }
    // unit epilogues; every stop decision and the routing are taken by thread 0 and
    // shared, so the four warps pass the same named barriers
    const int ksu = g.ksu, ksd = g.ksd;
    int uc = 0, nact = 0;
    bool have_route = false, ok = true;
    auto ep_route = [&]() -> int {
      if (tid == 0) C.ep_nact = wait_route();
      ptx::bar_sync(2, kEpiWarps * 32);
      return C.ep_nact;
    };
    for (int step = 0; step < 4 && ok; ++step) {
      const int ph = seg_at(step);
      if (tid == 0 && step >= 1) DEC_TRACE(3 + step);   // 4: shared gate/up, 5: routed gate/up, 6: shared down done
      if (ph == 2 && !have_route) {
        nact = ep_route();
        have_route = true;
      }
      int lo, hi;
      seg_of(g, ph, nact, lo, hi);
      for (int v = lo; v < hi && ok; ++v, ++uc) {
        const Unit u = make_unit(g, C, ph, v, E);
        const int db = uc & 1;
        const unsigned long long tw = clock64();
        if (!bar_wait(&C.dfull[db], (uc >> 1) & 1, &C.abort, kLocalWaitNs)) abort_now();
        const unsigned long long tb = clock64();
        c_dfull += tb - tw;
        ptx::bar_sync(2, kEpiWarps * 32);
        if (tid == 0) C.ep_stop = aborted() ? 1 : 0;
        ptx::bar_sync(2, kEpiWarps * 32);
        if (C.ep_stop) {
          ok = false;
          break;
        }
        float dv[16];
        if constexpr (CC) {
#pragma unroll
          for (int c = 0; c < 16; ++c) dv[c] = 0.f;
          dv[0] = C.dsm[db][0][r] + C.dsm[db][1][r];
        } else {
          ptx::tc_fence_after();
          ptx::tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(kDCol0 + kN * db), dv);
          ptx::tc_fence_before();
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&C.dempty[db]);
        if (!u.down) {
          // gate/up: K-split partial of this tile, then the last split computes h
          float* part = a.gu_part + ((((size_t)u.slot * g.NTu + u.tile) * ksu + u.split) * T) * kTileM;
#pragma unroll
          for (int c = 0; c < kMaxT; ++c)
            if (c < T) part[(size_t)c * kTileM + r] = dv[c];
          __threadfence();
          ptx::bar_sync(2, kEpiWarps * 32);
          if (tid == 0) {
            const uint32_t old = atomicAdd(up_cnt + u.slot * g.NTu + u.tile, 1u);
            C.flag = old == (uint32_t)(ksu - 1);
            if (C.flag) up_cnt[u.slot * g.NTu + u.tile] = 0;
          }
          ptx::bar_sync(2, kEpiWarps * 32);
          if (C.flag) {
            const unsigned long long tl = clock64();
            __threadfence();
            if (lane < 16) {
              const float* p0 = a.gu_part + (((size_t)u.slot * g.NTu + u.tile) * ksu * T) * kTileM;
#pragma unroll 1
              for (int c = 0; c < T; ++c) {
                // all splits' loads first, then the sums in split order
                float gv[kMaxKsu], uv[kMaxKsu];
#pragma unroll
                for (int sp = 0; sp < kMaxKsu; ++sp) {
                  gv[sp] = uv[sp] = 0.f;
                  if (sp < ksu) {
                    gv[sp] = __ldcg(p0 + ((size_t)sp * T + c) * kTileM + 32 * q + lane);
                    uv[sp] = __ldcg(p0 + ((size_t)sp * T + c) * kTileM + 32 * q + 16 + lane);
                  }
                }
                float gs = 0.f, us = 0.f;
#pragma unroll
                for (int sp = 0; sp < kMaxKsu; ++sp)
                  if (sp < ksu) {
                    gs += gv[sp];
                    us += uv[sp];
                  }
                a.h16[((size_t)u.slot * T + c) * I + 64 * u.tile + 16 * q + lane] =
                    __float2half_rn((a.identity_act ? gs : siluf_acc(gs)) * us);
              }
            }
            __threadfence();
            ptx::bar_sync(2, kEpiWarps * 32);
            if (tid == 0) ptx::red_release_add(up_done + u.slot, 1u);
            c_last += clock64() - tl;
          }
        } else {
          // down: this split's y rows of the unit's tokens, then the last unit of the
          // 128-row block to arrive combines the block's outputs
          if (!have_route) {
            nact = ep_route();
            have_route = true;
          }
          const int row = kTileM * u.tile + r;
#pragma unroll
          for (int c = 0; c < kMaxT; ++c) {
            if (c < T) {
              const int j = u.slot == 0 ? k : C.meta_j[u.slot - 1][c];
              if (j >= 0) a.y_part[(((size_t)c * (k + 1) + j) * ksd + u.split) * H + row] = dv[c];
            }
          }
          __threadfence();
          ptx::bar_sync(2, kEpiWarps * 32);
          if (tid == 0) {
            const uint32_t target = (uint32_t)((nact + 1) * ksd);
            const uint32_t old = atomicAdd(dn_cnt + u.tile, 1u);
            C.flag = old == target - 1;
            if (C.flag) dn_cnt[u.tile] = 0;
          }
          ptx::bar_sync(2, kEpiWarps * 32);
          if (C.flag) {
            const unsigned long long tl = clock64();
            __threadfence();
            for (int c = 0; c < T; ++c) {
              const float* yp = a.y_part + (size_t)c * (k + 1) * ksd * H + row;
              // per selection slot: all its splits' loads first, then the sum in split order;
              // slots in order, the shared expert last
              float acc = 0.f, ysh = 0.f;
              for (int j = 0; j <= k; ++j) {
                if (j < k && C.idsel[c][j] < 0) continue;   // slot dropped by the adaptive top-p
                float yv[kMaxKsd];
#pragma unroll
                for (int sp = 0; sp < kMaxKsd; ++sp)
                  yv[sp] = sp < ksd ? __ldcg(yp + ((size_t)j * ksd + sp) * H) : 0.f;
                float ys = 0.f;
#pragma unroll
                for (int sp = 0; sp < kMaxKsd; ++sp)
                  if (sp < ksd) ys += yv[sp];
                if (j < k)
                  acc = fmaf(C.wsel[c][j], ys, acc);
                else
                  ysh = ys;
              }
              store_act<XDT>(a.out, (size_t)c * H + row, acc + ysh);
            }
            c_last += clock64() - tl;
          }
        }
        c_epi += clock64() - tb;
      }
    }
    if (tid == 0) {
      DEC_TRACE(12);
      if (a.trace) {
        unsigned long long* tr = a.trace + (size_t)blockIdx.x * 64;
        tr[24] = c_dfull;
        tr[25] = c_epi;
        tr[26] = c_last;
        tr[30] = clock64();
        tr[31] = (unsigned long long)uc;
      }
    }
  }

  // ---------------------------------------------------------------------- teardown
  ptx::tc_fence_before();
  __syncthreads();
  if (tid == 0) {
    // after an abort, wait for the copies that may still be in flight (the last ns issued)
    const int issued = C.issued;
    if (issued != C.consumed)
      for (int i = max(0, issued - ns); i < issued; ++i) bar_wait(&C.full[i % ns], (i / ns) & 1, nullptr, kLocalWaitNs);
  }
  if (!CC && warp == kWarpMma) {
    if (aborted() && lane == 0) {
      ptx::tc_commit(&C.fin_bar);
      bar_wait(&C.fin_bar, 0, nullptr, kLocalWaitNs);
    }
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
  if (tid == 0) {
    __threadfence();
    const uint32_t old = atomicAdd(a.sync + 2, 1u);
    if (old == (uint32_t)g.G - 1) {
      // last CTA out: reset the per-call counters for the next call (after a time-out
      // also the K-split and row-block counters that the aborted units left behind)
      a.sync[0] = 0;
      a.sync[4] = 0;
      for (int i = 0; i <= kMaxActive; ++i) up_done[i] = 0;
      if (__ldcg(a.sync + 3)) {
        for (int i = 0; i < (1 + kMaxActive) * g.NTu; ++i) up_cnt[i] = 0;
        for (int i = 0; i < g.NTd; ++i) dn_cnt[i] = 0;
        a.sync[3] = 0;
      }
      __threadfence();
      a.sync[2] = 0;
    }
  }
}

template <int XDT, int WDT, bool CC>
cudaError_t launch_decode_t(const DecodeArgs& a, int grid, size_t smem, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kDecThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, moe_decode_kernel<XDT, WDT, CC>, a);
}

template <int XDT, int WDT>
cudaError_t init_one() {
  cudaError_t e = cudaFuncSetAttribute(moe_decode_kernel<XDT, WDT, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kSmemLimit);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(moe_decode_kernel<XDT, WDT, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemLimit);
  return e;
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Shared-memory layout for T tokens: fixed block, ring, activation panel, h panels.
// Returns the dynamic shared-memory bytes (0 if the ring would have fewer than 2 slots).
size_t decode_layout(int T, int H, int I, DecodeArgs* a) {
  const size_t fixed = align_up(sizeof(DecFixed), 1024);
  const size_t xb = align_up((size_t)H * T * 2 + kPanelPad, 128);
  const size_t hb = align_up((size_t)I * T * 2 + kPanelPad, 128);
  const size_t rest = fixed + xb + 2 * hb;
  if (rest + 2 * (size_t)kItemBytes > (size_t)kSmemLimit) return 0;
  int ns = (int)(((size_t)kSmemLimit - rest) / kItemBytes);
  if (ns > kMaxSlots) ns = kMaxSlots;
  if (a) {
    a->ns = ns;
    a->off_ring = (int)fixed;
    a->off_x = (int)(fixed + (size_t)ns * kItemBytes);
    a->off_h0 = a->off_x + (int)xb;
    a->off_h1 = a->off_h0 + (int)hb;
  }
  return fixed + (size_t)ns * kItemBytes + xb + 2 * hb;
}

int pick_split(int n, const int* cands, int nc) {
  for (int i = 0; i < nc; ++i)
    if (n % cands[i] == 0) return cands[i];
  return 1;
}

// K splits: gate/up units of about 6 items and down units of about 4 at the GLM shape.
// Smaller units balance the CTAs' shares better but cost more per-unit epilogue work
// (partials, fences, counters); at these sizes that work dominates.
int ksu_for(int H) {
  const int c[] = {4, 3, 2};
  return pick_split(H / kGroupK, c, 3);
}

int ksd_for(int I) {
  const int c[] = {2};
  return pick_split(I / kGroupK, c, 1);
}

}  // namespace

bool decode_supported(int H, int I, int E, int top_k, int T) {
  return H % kGroupK == 0 && I % kGroupK == 0 && H <= kMaxH && I <= kMaxI && E <= kMaxE && E % 32 == 0 &&
         T >= 1 && T <= kMaxT && T * top_k <= kMaxActive && top_k <= kMaxK && decode_layout(T, H, I, nullptr) > 0;
}

size_t decode_sync_words(int I) { return (size_t)sync_route(I / 64) + 2 * kMaxT * kMaxK + 8; }

size_t decode_gu_part_floats(int T, int H, int I, int E, int top_k) {
  const int act = T * top_k < E ? T * top_k : E;
  return (size_t)(1 + act) * (I / 64) * ksu_for(H) * T * kTileM;
}

size_t decode_y_part_floats(int T, int H, int I, int top_k) { return (size_t)T * (top_k + 1) * ksd_for(I) * H; }

size_t decode_h16_elems(int T, int I, int E, int top_k) {
  const int act = T * top_k < E ? T * top_k : E;
  return (size_t)(1 + act) * T * I;
}

cudaError_t decode_occupancy(int* blocks_per_sm) {
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, moe_decode_kernel<MOE_DT_BF16, MOE_DT_F32, false>,
                                                       kDecThreads, kSmemLimit);
}

cudaError_t decode_kernels_init() {
  cudaError_t e = cudaSuccess;
  const cudaError_t r[] = {init_one<MOE_DT_F32, MOE_DT_F32>(), init_one<MOE_DT_BF16, MOE_DT_F32>(),
                           init_one<MOE_DT_F32, MOE_DT_BF16>(), init_one<MOE_DT_BF16, MOE_DT_BF16>()};
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
  a.top_p = d.top_p;
  a.identity_act = d.identity_act;
  a.pack_up = d.pack_up;
  a.pack_dn = d.pack_dn;
  a.logits = d.logits;
  a.ids = d.ids;
  a.weights = d.weights;
  a.offsets = d.offsets;
  a.entries = d.entries;
  a.h16 = d.h16;
  a.gu_part = d.gu_part;
  a.y_part = d.y_part;
  a.out = d.out;
  a.sync = d.sync;
  a.status = d.status;
  a.wait_ns = d.wait_ns;
  a.trace = d.trace;
  a.ksu = ksu_for(d.H);
  a.ksd = ksd_for(d.I);
  const size_t smem = decode_layout(d.T, d.H, d.I, &a);
  if (smem == 0) return cudaErrorInvalidValue;
  const bool xf = act_dtype == MOE_DT_F32, wf = router_dtype == MOE_DT_F32;
  // one token: CUDA-core dot products (exact products, fp32 sums); 2..8 tokens: tensor cores
  if (d.T == 1) {
    if (xf) return wf ? launch_decode_t<MOE_DT_F32, MOE_DT_F32, true>(a, grid, smem, s)
                      : launch_decode_t<MOE_DT_F32, MOE_DT_BF16, true>(a, grid, smem, s);
    return wf ? launch_decode_t<MOE_DT_BF16, MOE_DT_F32, true>(a, grid, smem, s)
              : launch_decode_t<MOE_DT_BF16, MOE_DT_BF16, true>(a, grid, smem, s);
  }
  if (xf) return wf ? launch_decode_t<MOE_DT_F32, MOE_DT_F32, false>(a, grid, smem, s)
                    : launch_decode_t<MOE_DT_F32, MOE_DT_BF16, false>(a, grid, smem, s);
  return wf ? launch_decode_t<MOE_DT_BF16, MOE_DT_F32, false>(a, grid, smem, s)
            : launch_decode_t<MOE_DT_BF16, MOE_DT_BF16, false>(a, grid, smem, s);
}

}  // namespace moe
