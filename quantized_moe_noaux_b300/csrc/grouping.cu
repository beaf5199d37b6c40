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
    if (e == E - 1) offsets[E] = b + counts[e];   // routed entries (slots with id -1 have none)
  }
  __syncthreads();
  // Each warp owns a contiguous span of the n entries: it counts the span's hits with
  // ballots, a CTA-wide exclusive scan of the 8 counts gives its first position, and a
  // second pass writes the hits in order (entries stay in ascending token order).
  const int n = T * top_k;
  if (counts[e] > 0) {
    const int span = (n + kGroupThreads / 32 - 1) / (kGroupThreads / 32);
    const int i0 = warp * span, i1 = min(n, i0 + span);
    int mine = 0;
    for (int c0 = i0; c0 < i1; c0 += 32) {
      const int i = c0 + lane;
      mine += __popc(__ballot_sync(0xffffffffu, i < i1 && __ldg(ids + i) == e));
    }
    __syncthreads();   // warp_sum reuse
    if (lane == 0) warp_sum[warp] = mine;
    __syncthreads();
    int pos = base_s;
    for (int w = 0; w < warp; ++w) pos += warp_sum[w];
    for (int c0 = i0; c0 < i1; c0 += 32) {
      const int i = c0 + lane;
      const bool hit = i < i1 && __ldg(ids + i) == e;
      const unsigned m = __ballot_sync(0xffffffffu, hit);
      if (hit) entries[pos + __popc(m & ((1u << lane) - 1u))] = i;
      pos += __popc(m);
    }
  }

  // CTA 0's first warp also writes the work list (at most E + T*k/kTokChunk items, plus
  // the inline shared expert's chunks): each lane owns a contiguous run of experts, a warp
  // scan gives every lane its first slot
  if (items && e == 0 && warp == 0) {
    const int per = (E + 31) / 32;
    const int x0 = min(E, lane * per), x1 = min(E, x0 + per);
    int mine = 0;
    for (int x = x0; x < x1; ++x) mine += (counts[x] + kTokChunk - 1) / kTokChunk;
    int incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int pos = incl - mine;
    for (int x = x0; x < x1; ++x)
      for (int ch = 0; ch * kTokChunk < counts[x]; ++ch) items[pos++] = pack_item(x, ch);
    const int total = __shfl_sync(0xffffffffu, incl, 31);
    const int nsh = shared_inline ? (T + kTokChunk - 1) / kTokChunk : 0;
    for (int ch = lane; ch < nsh; ch += 32) items[total + ch] = pack_item(E, ch);
    if (lane == 0) meta[0] = total + nsh;
  }
}

// Debug checks of a call's routing (one CTA): every id in [-1, E); offsets start at 0, never
// decrease and end at the number of routed slots (ids >= 0), at most T * k; each entry of
// expert e's range names a slot whose id is e, tokens strictly ascending within the range.
// A violation sets MOE_ERR_DEVICE_CHECK; reads stay inside the arrays whatever their values.
__global__ void __launch_bounds__(1024)
check_routing_kernel(const int32_t* __restrict__ ids, const int32_t* __restrict__ offsets,
                     const int32_t* __restrict__ entries, int T, int top_k, int E, int* status) {
  __shared__ int bad, routed;
  if (threadIdx.x == 0) {
    bad = 0;
    routed = 0;
  }
  __syncthreads();
  const int n = T * top_k;
  int mine = 0;
  for (int f = threadIdx.x; f < n; f += blockDim.x) {
    const int id = ids[f];
    if (id < -1 || id >= E) bad = 1;
    mine += id >= 0;
  }
  atomicAdd(&routed, mine);
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    if (offsets[e + 1] < offsets[e]) bad = 1;
  __syncthreads();
  const int total = offsets[E];
  if (threadIdx.x == 0 && (offsets[0] != 0 || total != routed || total > n)) bad = 1;
  __syncthreads();
  if (!bad) {
    for (int q = threadIdx.x; q < total; q += blockDim.x) {
      int lo = 0, hi = E - 1;   // expert whose range holds q: last e with offsets[e] <= q
      while (lo < hi) {
        const int mid = (lo + hi + 1) / 2;
        if (offsets[mid] <= q) lo = mid;
        else hi = mid - 1;
      }
      const int ent = entries[q];
      if (ent < 0 || ent >= n || ids[ent] != lo) {
        bad = 1;
      } else if (q > offsets[lo]) {
        const int prev = entries[q - 1];
        if (prev < 0 || prev >= n || prev / top_k >= ent / top_k) bad = 1;
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0 && bad) raise_status(status, MOE_ERR_DEVICE_CHECK);
}

__global__ void set_slots_kernel(const SlotTable t, int n, int32_t* __restrict__ dst) {
  for (int i = threadIdx.x; i < n; i += blockDim.x) dst[i] = t.slot[i];
}

}  // namespace

cudaError_t launch_check_routing(const int32_t* ids, const int32_t* offsets, const int32_t* entries, int T,
                                 int top_k, int E, int* status, cudaStream_t s) {
  if (T <= 0 || top_k <= 0 || E <= 0) return cudaErrorInvalidValue;
  check_routing_kernel<<<1, 1024, 0, s>>>(ids, offsets, entries, T, top_k, E, status);
  return cudaGetLastError();
}

cudaError_t launch_set_slots(const SlotTable& t, int n, int32_t* dst, cudaStream_t s) {
  if (n <= 0 || n > kMaxSlotTable) return cudaErrorInvalidValue;
  set_slots_kernel<<<1, 256, 0, s>>>(t, n, dst);
  return cudaGetLastError();
}

cudaError_t launch_group(const int32_t* ids, const int32_t* counts, int T, int top_k, int E,
                         int shared_inline, int32_t* offsets, int32_t* entries, int32_t* items,
                         int32_t* meta, cudaStream_t s) {
  group_kernel<<<E, kGroupThreads, 0, s>>>(ids, counts, T, top_k, E, shared_inline, offsets,
                                           entries, items, meta);
  return cudaGetLastError();
}

}  // namespace moe
