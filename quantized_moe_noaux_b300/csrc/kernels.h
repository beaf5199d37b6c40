// Host-side launchers of the layer's kernels (internal to libmoe).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace moe {

// Router: logits[T, E] = x[T, H] W_r[E, H]^T in fp32.
cudaError_t launch_router_logits(const void* x, int act_dtype, const void* router_w,
                                 int router_dtype, float* logits, int T, int E, int H,
                                 cudaStream_t s);

// Selection: sigmoid, bias, group top-2 sums, top-k-group, top-k, renormalise x rsf.
// Also histograms the chosen experts into counts[E] (zeroed by the caller).
cudaError_t launch_select(const float* logits, const float* bias, int T, int E, int n_group,
                          int topk_group, int top_k, float rsf, int32_t* ids, float* weights,
                          int32_t* counts, int* status, cudaStream_t s);

// Grouping: offsets[E+1], entries[T*k] (ascending token per expert) and the work list
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

// ------------------------------------------------------------- fused decode path
size_t decode_tile_bytes(int R, int K);
bool decode_supported(int H, int I, int E, int top_k, int T);
size_t decode_smem_bytes();
cudaError_t decode_occupancy(int* blocks_per_sm);
cudaError_t decode_kernels_init();
// Repack a row-major int4-g32 matrix [R][K] into decode tiles (up = gate/up row pairing).
cudaError_t launch_repack(const uint8_t* codes, const void* scales, int R, int K, bool up, uint8_t* dst,
                          cudaStream_t s);

struct DecodeLaunch {
  const void* x;
  int T;
  const void* router_w;
  const float* bias;
  int H, I, E, top_k, n_group, topk_group;
  float rsf;
  const uint8_t* up_store;
  const uint8_t* down_store;
  float* logits;
  int32_t* ids;
  float* weights;
  int32_t* offsets;
  int32_t* entries;
  int32_t* active_g;
  int32_t* meta_g;
  void* h16;
  float* out_acc;
  void* out;
  uint32_t* sync;
  int* status;
  uint32_t spin_max;
};
cudaError_t launch_decode_fused(const DecodeLaunch& d, int act_dtype, int router_dtype, int grid,
                                cudaStream_t s);

// out[T, H] (act dtype) = out_acc
cudaError_t launch_finalize(const float* out_acc, void* out, int act_dtype, size_t n,
                            cudaStream_t s);

}  // namespace moe
