// Batch-union grouping of the MoE layer: per-expert offsets (exclusive scan of the
// histogram built by the selection kernel), the per-expert entry lists in ascending token
// order, and the list of (expert, token-chunk) work items, so each selected expert's
// weights are streamed once per call for all tokens routed to it ("Batch-union MoE" in
// "Show HN: Menjalankan GLM 5.2 di komputer lambat", section "Fitur utama yang
// diimplementasikan").
#include "kernels.h"

namespace moe {

namespace {

constexpr int kGroupThreads = 256;

// One CTA per expert: stable compaction of the flat (token, slot) indices that chose it.
__global__ void __launch_bounds__(kGroupThreads)
group_kernel(const int32_t* __restrict__ ids, const int32_t* __restrict__ counts, int T,
             int top_k, int E, int shared_inline, int32_t* __restrict__ offsets,
             int32_t* __restrict__ entries, int32_t* __restrict__ items,
             int32_t* __restrict__ meta) {
  __shared__ int warp_sum[kGroupThreads / 32];
  __shared__ int base_s;
  const int e = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  // offset of this expert = sum of the counts of the experts before it
  int part = 0;
  for (int i = threadIdx.x; i < e; i += kGroupThreads) part += counts[i];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
  if (lane == 0) warp_sum[warp] = part;
  __syncthreads();
  if (threadIdx.x == 0) {
    int b = 0;
    for (int w = 0; w < kGroupThreads / 32; ++w) b += warp_sum[w];
    base_s = b;
    offsets[e] = b;
    if (e == E - 1) offsets[E] = T * top_k;
  }
  __syncthreads();
  int running = base_s;
  const int n = T * top_k;
  if (counts[e] > 0) {
    for (int c0 = 0; c0 < n; c0 += kGroupThreads) {
      const int i = c0 + threadIdx.x;
      const bool hit = i < n && ids[i] == e;
      const unsigned m = __ballot_sync(0xffffffffu, hit);
      __syncthreads();   // warp_sum reuse
      if (lane == 0) warp_sum[warp] = __popc(m);
      __syncthreads();
      int before = 0, total = 0;
#pragma unroll
      for (int w = 0; w < kGroupThreads / 32; ++w) {
        const int c = warp_sum[w];
        before += (w < warp) ? c : 0;
        total += c;
      }
      if (hit) entries[running + before + __popc(m & ((1u << lane) - 1u))] = i;
      running += total;
    }
  }

  // CTA 0 also writes the work list (serial over experts; at most E + T*k/kTokChunk items)
  if (e == 0 && threadIdx.x == 0) {
    int nitems = 0;
    for (int x = 0; x < E; ++x) {
      const int c = counts[x];
      for (int ch = 0; ch * kTokChunk < c; ++ch) items[nitems++] = pack_item(x, ch);
    }
    if (shared_inline)
      for (int ch = 0; ch * kTokChunk < T; ++ch) items[nitems++] = pack_item(E, ch);
    meta[0] = nitems;
  }
}

}  // namespace

cudaError_t launch_group(const int32_t* ids, const int32_t* counts, int T, int top_k, int E,
                         int shared_inline, int32_t* offsets, int32_t* entries, int32_t* items,
                         int32_t* meta, cudaStream_t s) {
  group_kernel<<<E, kGroupThreads, 0, s>>>(ids, counts, T, top_k, E, shared_inline, offsets,
                                           entries, items, meta);
  return cudaGetLastError();
}

}  // namespace moe
