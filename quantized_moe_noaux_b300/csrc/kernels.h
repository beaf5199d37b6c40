// Host-side launchers of the layer's kernels (internal to libmoe).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace moe {

// Router: logits[T, E] = x[T, H] W_r[E, H]^T in fp32.
// Tensor-core router logits (bf16 activations, H % 64 == 0, E % 4 == 0): W_r as n_planes
// (1 or 3) bf16 planes [n_planes][E][H] summing to W_r; partial: router_mma_partial_floats
// floats of scratch. launch_router_split writes the hi/mid/lo planes of an fp32 W_r [n].
bool router_mma_supported(int act_dtype, int H, int E);
size_t router_mma_partial_floats(int n_sm);
cudaError_t router_mma_init();
cudaError_t launch_router_split(const float* w, uint16_t* planes, size_t n, cudaStream_t s);
cudaError_t launch_router_mma(const void* x, const uint16_t* planes, int n_planes, float* logits, float* partial,
                              int T, int E, int H, int n_sm, cudaStream_t s);
cudaError_t launch_router_logits(const void* x, int act_dtype, const void* router_w,
                                 int router_dtype, float* logits, int T, int E, int H,
                                 cudaStream_t s);

// Selection: sigmoid, bias, group top-2 sums, top-k-group, top-k, adaptive top-p (0 < top_p
// < 1; dropped slots id -1), renormalise x rsf. Also histograms the routed experts into
// counts[E] (zeroed by the caller).
cudaError_t launch_select(const float* logits, const float* bias, int T, int E, int n_group,
                          int topk_group, int top_k, float rsf, float top_p, int32_t* ids, float* weights,
                          int32_t* counts, int* status, cudaStream_t s);

// Grouping: offsets[E+1] (offsets[E] = routed entries), entries (ascending token per
// expert; slots with id -1 have none) and the work list
// (expert, token-chunk) of every active expert, plus the inline shared expert when
// shared_inline != 0. meta[0] = number of work items.
cudaError_t launch_group(const int32_t* ids, const int32_t* counts, int T, int top_k, int E,
                         int shared_inline, int32_t* offsets, int32_t* entries, int32_t* items,
                         int32_t* meta, cudaStream_t s);

struct ExpertGemvArgs {
  ExpertWeights w;
  int fmt;            // weight format of these experts
  int H, I, E, top_k, T;
  const void* x;      // activations feeding gate/up (act dtype, or fp32 if x_f32)
  int x_dtype;        // MOE_DT_F32 | MOE_DT_BF16
  const int32_t* offsets;
  const int32_t* entries;
  const int32_t* items;     // work list, NULL = the shared expert alone (grid covers T)
  const int32_t* meta;      // meta[0] = item count (with items)
  int expert_base;          // weight index of "expert E" (shared) in w (E, or 0 if separate)
  float* h;                 // [T*k + T, I] fp32
  unsigned int* h_amax;     // NVFP4 routed h amax (bits of a non-negative float) or NULL
  const float* weights;     // [T, k]
  float* out_acc;           // [T, H] fp32
  int max_items;
  int identity_act;         // test-only: h = gate * up (no SiLU)
};

// Largest dynamic shared memory a generic expert CTA may use (x or h rows of a token chunk).
constexpr int kMaxDynSmem = 227 * 1024;
cudaError_t expert_kernels_init();   // once per process/device before the first launch
cudaError_t launch_expert_up(const ExpertGemvArgs& a, cudaStream_t s);
cudaError_t launch_expert_down(const ExpertGemvArgs& a, cudaStream_t s);

// NVFP4 activation quantiser: amax over n elements, then per-16-block quantise to
// dequantised fp32 values. src is act dtype (or fp32 when src_dtype = MOE_DT_F32).
cudaError_t launch_amax(const void* src, int src_dtype, size_t n, unsigned int* amax_bits,
                        cudaStream_t s);
cudaError_t launch_nvfp4_quant(const void* src, int src_dtype, float* dst, size_t n,
                               const unsigned int* amax_bits, cudaStream_t s);
// Q8_0-style int8 activations, dequantised to fp32: per 32 elements d = fp16(amax / 127),
// dst = clamp(rint(v / d), -127, 127) * d (dst may alias an fp32 src).
cudaError_t launch_q8_0_quant(const void* src, int src_dtype, float* dst, size_t n, cudaStream_t s);

// ------------------------------------------------------------- fused decode path
// One cooperative kernel per decode step (T <= 8) reading the grouped GEMM's packed int4
// store (shared expert at index E). Scratch per layer (sized for min(max_tokens, 8)
// tokens): sync words (zero at creation, left zero by every call), h rows, gate/up K-split
// partials and down outputs.
bool decode_supported(int H, int I, int E, int top_k, int T);
size_t decode_sync_words(int I);
size_t decode_gu_part_floats(int T, int H, int I, int E, int top_k);
size_t decode_y_part_floats(int T, int H, int I, int top_k);
size_t decode_h16_elems(int T, int I, int E, int top_k);
cudaError_t decode_occupancy(int* blocks_per_sm);
cudaError_t decode_kernels_init();

struct DecodeLaunch {
  const void* x;
  int T;
  const void* router_w;
  const float* bias;
  int H, I, E, top_k, n_group, topk_group;
  float rsf;
  float top_p;                 // adaptive expert top-p (0 < top_p < 1), else off
  int identity_act;            // test-only: h = gate * up (no SiLU)
  const uint8_t* pack_up;      // grouped-GEMM packed gate/up store
  const uint8_t* pack_dn;      // grouped-GEMM packed down store
  float* logits;
  int32_t* ids;
  float* weights;
  int32_t* offsets;
  int32_t* entries;
  __half* h16;
  float* gu_part;
  float* y_part;
  void* out;
  uint32_t* sync;
  int* status;
  unsigned long long wait_ns;  // time limit of the waits on other CTAs
  unsigned long long* trace;   // optional per-CTA phase timestamps, or NULL
};
cudaError_t launch_decode_fused(const DecodeLaunch& d, int act_dtype, int router_dtype, int grid,
                                cudaStream_t s);

// ------------------------------------------------ grouped GEMM path (tcgen05)
// Opaque storage of one CUtensorMap (128 bytes, 64-byte aligned).
struct alignas(64) TensorMapBytes {
  unsigned char b[128];
};
struct GemmMaps {
  TensorMapBytes codes;    // fp16 weights [rows, K], 64 x 128 box, 128-byte swizzle (kWF16 only)
  TensorMapBytes act[4];   // expert-sorted fp16 activations [rows, K], 64 x {32,64,128,256} boxes,
                           // 128-byte swizzle
};
// Weight storage of the grouped GEMM besides MOE_W_INT4_G32 / MOE_W_NVFP4: plain fp16
// rows (a bf16 shared expert converted once at layer creation).
constexpr int kWF16 = 16;

struct GemmParams {
  const int4* items;          // (expert, first sorted row, rows, 0)
  const int32_t* n_items;     // device count of this launch's items
  const int32_t* item_skip;   // device count of items to skip first, or NULL
  int e_sub;                  // subtracted from the item's expert index to index the weights
  const uint8_t* wpack;       // packed weights (int4 / NVFP4), see gemm_pack_kernel
  int mtiles;                 // 128-row tiles per expert
  int K;                      // reduction length (H for gate/up, I for down)
  int rows_per_expert;        // 2I (gate/up) or H (down)
  int H, I, T, top_k;
  __half* h16;                // gate/up output [rows, I] (fp16)
  float* h32;                 // gate/up output [rows, I] (fp32, NVFP4 layers)
  unsigned int* h_amax;       // NVFP4: amax bits of the routed h
  float* y;                   // down output: expert-sorted rows [rows, H] fp32 (combined later)
  const int32_t* entries;     // [T * top_k] token * top_k + slot, grouped by expert
  const float* weights;       // [T * top_k]
  const float* w_tscale;      // NVFP4 per-expert tensor scales of this matrix, or NULL
  const unsigned int* act_amax;   // NVFP4: amax bits of the B activations, or NULL
  int* status;
  unsigned long long wait_ns; // time limit of every wait on another warp's or unit's work
  unsigned long long* trace;  // optional per-CTA profiling trace (64 slots per CTA), or NULL
  int trace_base;             // first slot of this launch's 11
  const int32_t* slot_of;     // packed-store slot of each expert (HBM expert cache), or NULL
  int identity_act;           // test-only: h = gate * up (no SiLU)
  // block-scaled FP4 kernel only
  const uint8_t* wsf;         // weight scales in MMA order (fp4_pack_kernel)
  const uint8_t* asf;         // activation E4M3 scales [rows, K / 16] of the sorted rows
};
bool make_tmap_2d(TensorMapBytes* out, const void* base, int elem_bytes, uint64_t inner, uint64_t rows,
                  uint32_t box_inner, uint32_t box_rows, bool swizzle128);
bool gemm_supported(int H, int I);
// Items of at most `chunk` rows (16..256): the fp16 kernels take 256, the FP4 kernel kFp4MaxN.
int gemm_max_items(int T, int top_k, int E, bool routed, bool shared, int chunk);
cudaError_t gemm_kernels_init();
cudaError_t launch_gemm_items(const int32_t* offsets, int E, int T, int top_k, int chunk, int4* items,
                              int32_t* n_items, cudaStream_t s);
cudaError_t launch_bf16_to_f16(const void* src, void* dst, size_t rows, int K, bool gate_up, int I,
                               cudaStream_t s);
// Expert-sorted fp16 activation rows: row q < Tk is token entries[q] / top_k, row Tk + t is
// token t (shared expert). NVFP4 layers quantise each token once into xq16 [T, H] (code *
// block scale, fp16; the tensor scale from amax_bits) and copy that row for routed rows.
cudaError_t launch_gather_act(const void* x, int act_dtype, bool nvfp4, int H, const int32_t* entries, int Tk,
                              int top_k, int rows, __half* dst, const unsigned int* amax_bits, __half* xq16,
                              int32_t* inv, const int32_t* n_routed, cudaStream_t s);
// out[t] = sum_j w[t, j] y[inv[t k + j]] + y[T k + t] (routed slots in ascending order, fp32),
// in the activation dtype: the combine of the grouped path. inv[t k + j] = sorted row of
// entry t k + j (written by the gather kernels); slots with ids < 0 are skipped.
cudaError_t launch_combine(const float* y, const int32_t* inv, const int32_t* ids, const float* weights, int T,
                           int top_k, int H, void* out, int act_dtype, cudaStream_t s);
cudaError_t launch_quant_h(const float* h, size_t n, const unsigned int* amax_bits, __half* dst, cudaStream_t s);
// fp16 x rows Tk .. Tk + T - 1 of the sorted activation matrix (the shared expert's rows).
cudaError_t launch_gather_shared_rows(const void* x, int act_dtype, int H, int Tk, int T, __half* dst,
                                      cudaStream_t s);
// Persistent launch over n_items x mtiles tiles (max_tiles bounds them; grid <= n_sm).
cudaError_t launch_gemm(int wfmt, int epi, const GemmMaps& m, const GemmParams& p, int max_tiles, int n_sm,
                        cudaStream_t s);
size_t gemm_pack_bytes(int rows_per_expert, int K, int n_exp);
cudaError_t launch_gemm_pack(const uint8_t* codes, const void* scales, int K, int n_exp, int rows_per_expert,
                             int I, bool gate_up, uint8_t* dst, cudaStream_t s);

// ------------------------------------ block-scaled FP4 grouped GEMM (NVFP4 layers)
// Routed experts of NVFP4 layers with a separately stored shared expert: E2M1 weights and
// activations straight into tcgen05.mma kind::mxf4nvf4 (gemm_fp4.cu).
constexpr int kFp4MaxN = 160;       // token rows per tile (item chunk)
struct Fp4Maps {
  TensorMapBytes w;        // weight codes [n_exp * rows, K/2] uint8, 128 x 128 box, 128-byte swizzle
  TensorMapBytes act[4];   // sorted activation codes [rows, K/2] uint8, 128 x {32, 64, 128, 160} boxes
};
bool fp4_gemm_supported(int H, int I);
cudaError_t fp4_gemm_init();
size_t fp4_scale_bytes(int rows, int K, int n_exp);   // bytes of the MMA-ordered weight scales
cudaError_t launch_fp4_pack(const uint8_t* codes, const uint8_t* scales, int K, int n_exp, int rows, int I,
                            bool gate_up, uint8_t* dcodes, uint8_t* dsf, cudaStream_t s);
// NVFP4 codes [T*k, H/2] and E4M3 scales [T*k, H/16] of the sorted routed rows (row q =
// token entries[q] / top_k), tensor scale amax / 2688 from amax_bits; each token is
// quantised once into tok_codes [T, H/2] / tok_sf [T, H/16], then copied to its rows.
cudaError_t launch_quant_gather_fp4(const void* x, int act_dtype, int H, int T, const int32_t* entries, int top_k,
                                    const unsigned int* amax_bits, uint8_t* tok_codes, uint8_t* tok_sf,
                                    uint8_t* codes, uint8_t* sf, int32_t* inv, const int32_t* n_routed,
                                    cudaStream_t s);
cudaError_t launch_quant_h_fp4(const float* h, size_t n, const unsigned int* amax_bits, uint8_t* codes, uint8_t* sf,
                               cudaStream_t s);
cudaError_t launch_gemm_fp4(int epi, const Fp4Maps& m, const GemmParams& p, int max_tiles, int n_sm, cudaStream_t s);

// ------------------------------------------------------------- HBM expert cache
// Slot table of the cache (expert -> slot of the packed store), written by a kernel that
// takes it by value, so the host's table may change as soon as the launch is enqueued.
constexpr int kMaxSlotTable = 1025;   // E <= 1024 routed experts + the shared expert
struct SlotTable {
  int32_t slot[kMaxSlotTable];
};
cudaError_t launch_set_slots(const SlotTable& t, int n, int32_t* dst, cudaStream_t s);

// Debug checks of a routing (ids [T*k], offsets [E+1], entries): sets MOE_ERR_DEVICE_CHECK in
// *status on a violation (ids outside [-1, E), offsets not monotone or not ending at the
// routed count, an entry naming another expert's slot or tokens out of order).
cudaError_t launch_check_routing(const int32_t* ids, const int32_t* offsets, const int32_t* entries, int T,
                                 int top_k, int E, int* status, cudaStream_t s);

// out[T, H] (act dtype) = out_acc
cudaError_t launch_finalize(const float* out_acc, void* out, int act_dtype, size_t n,
                            cudaStream_t s);

}  // namespace moe
