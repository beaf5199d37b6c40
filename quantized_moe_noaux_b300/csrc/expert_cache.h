// HBM cache of host-resident experts (internal to libmoe).
//
// The routed experts of a cached layer live in pinned host memory, already in the grouped
// GEMM's packed layout; an HBM store of `slots` expert slots holds the ones in use, and the
// GEMM reads an expert through its slot ("Cara kerja eksekusi MoE berbasis streaming disk"
// in "Show HN: Menjalankan GLM 5.2 di komputer lambat": a per-layer LRU cache of experts
// over slower storage, an optional pinned hot store, usage counts that pick the experts to
// pin; "Yönlendirici İleriye Dönük Ön-Getirme" in "Show HN: GLM 5.2 Modelini Yavaş
// Bilgisayarımda Çalıştırmak": the router predicts the next layer's experts, whose loads
// start early; here the slower tier is host memory over the host link, the fast one HBM).
//
// Host logic only: which expert goes into which slot, least recently used eviction of
// experts that are neither needed by the current request nor pinned, the copies (one
// cudaMemcpyAsync per matrix and expert, on the cache's own copy stream), and counters.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

#include "../../include/moe_layer.h"

namespace moe {

class ExpertCache {
 public:
  // Counters (moe_layer_cache_stats order).
  enum { kHits = 0, kMisses, kPrefetched, kPrefetchHits, kBytesH2D, kEvictions, kNumStats };

  ~ExpertCache();

  // n_experts routed experts of up_bytes + dn_bytes packed bytes each, in pinned host
  // memory (host_up / host_dn, owned by the caller); HBM slots dev_up / dev_dn of the same
  // sizes (owned by the caller). Creates the copy stream and events.
  moe_status init(int n_experts, int slots, size_t up_bytes, size_t dn_bytes, const uint8_t* host_up,
                  const uint8_t* host_dn, uint8_t* dev_up, uint8_t* dev_dn);

  // Make every expert with counts[e] > 0 resident. Copies for misses are issued on the copy
  // stream; before the first copy that overwrites a slot, the copy stream waits for the
  // last recorded compute of this layer (note_compute). prefetch = true counts loads as
  // prefetched instead of missed and does not count hits. MOE_ERR_UNSUPPORTED when the
  // request needs more slots than the unpinned part of the cache holds.
  moe_status ensure(const int32_t* counts, bool prefetch);

  // The compute stream waits for every copy issued so far.
  moe_status wait_copies(cudaStream_t compute);
  // Record the end of a compute that reads slots (eviction fences on it).
  moe_status note_compute(cudaStream_t compute);

  // Pin the n experts with the highest usage counts (ties: lower id), loading them if
  // needed; earlier pins are released. MOE_ERR_INVALID_ARG when n leaves fewer than
  // `min_free` unpinned slots.
  moe_status pin_hot(int n, int min_free);

  int slot_of(int e) const { return slot_of_[e]; }
  bool pinned(int e) const { return pinned_[e] != 0; }
  const int64_t* stats() const { return stats_; }
  cudaStream_t copy_stream() const { return copy_; }
  int slots() const { return slots_; }

 private:
  int choose_slot(const std::vector<char>& needed) const;
  moe_status load(int e, int slot, bool& fenced);

  int n_ = 0, slots_ = 0;
  size_t up_bytes_ = 0, dn_bytes_ = 0;
  const uint8_t* host_up_ = nullptr;
  const uint8_t* host_dn_ = nullptr;
  uint8_t* dev_up_ = nullptr;
  uint8_t* dev_dn_ = nullptr;
  std::vector<int> slot_of_;        // [E] slot, -1 if not resident
  std::vector<int> owner_;          // [slots] expert, -1 if free
  std::vector<uint64_t> last_use_;  // [slots] request tick of the last use
  std::vector<char> pinned_;        // [E]
  std::vector<char> prefetched_;    // [E] loaded by a prefetch, not used since
  std::vector<uint64_t> usage_;     // [E] requests that routed to the expert
  uint64_t tick_ = 0;
  int64_t stats_[kNumStats] = {};
  cudaStream_t copy_ = nullptr;
  cudaEvent_t copied_ = nullptr, computed_ = nullptr;
  bool computed_valid_ = false;
};

}  // namespace moe
