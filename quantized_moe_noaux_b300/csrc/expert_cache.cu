// HBM cache of host-resident experts: slot assignment, LRU eviction, pinning, copies.
#include "expert_cache.h"

namespace moe {

ExpertCache::~ExpertCache() {
  if (copy_) cudaStreamSynchronize(copy_);
  if (copied_) cudaEventDestroy(copied_);
  if (computed_) cudaEventDestroy(computed_);
  if (copy_) cudaStreamDestroy(copy_);
}

moe_status ExpertCache::init(int n_experts, int slots, size_t up_bytes, size_t dn_bytes, const uint8_t* host_up,
                             const uint8_t* host_dn, uint8_t* dev_up, uint8_t* dev_dn) {
  n_ = n_experts;
  slots_ = slots;
  up_bytes_ = up_bytes;
  dn_bytes_ = dn_bytes;
  host_up_ = host_up;
  host_dn_ = host_dn;
  dev_up_ = dev_up;
  dev_dn_ = dev_dn;
  slot_of_.assign(n_, -1);
  owner_.assign(slots_, -1);
  last_use_.assign(slots_, 0);
  pinned_.assign(n_, 0);
  prefetched_.assign(n_, 0);
  usage_.assign(n_, 0);
  if (cudaStreamCreateWithFlags(&copy_, cudaStreamNonBlocking) != cudaSuccess ||
      cudaEventCreateWithFlags(&copied_, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&computed_, cudaEventDisableTiming) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

// A free slot, else the least recently used slot whose expert is neither needed by the
// current request nor pinned; -1 if none.
int ExpertCache::choose_slot(const std::vector<char>& needed) const {
  int best = -1;
  for (int s = 0; s < slots_; ++s) {
    const int o = owner_[s];
    if (o < 0) return s;
    if (needed[o] || pinned_[o]) continue;
    if (best < 0 || last_use_[s] < last_use_[best]) best = s;
  }
  return best;
}

moe_status ExpertCache::load(int e, int slot, bool& fenced) {
  // kernels enqueued before this point may still read the slot: the copy waits for them
  if (!fenced && computed_valid_) {
    if (cudaStreamWaitEvent(copy_, computed_, 0) != cudaSuccess) return MOE_ERR_CUDA;
    fenced = true;
  }
  // the slot stops holding its expert before the first byte is overwritten, so a failed
  // copy leaves it free rather than claimed by an expert whose bytes are gone
  const int old = owner_[slot];
  if (old >= 0) {
    slot_of_[old] = -1;
    owner_[slot] = -1;
    prefetched_[old] = 0;
    ++stats_[kEvictions];
  }
  if (cudaMemcpyAsync(dev_up_ + (size_t)slot * up_bytes_, host_up_ + (size_t)e * up_bytes_, up_bytes_,
                      cudaMemcpyHostToDevice, copy_) != cudaSuccess ||
      cudaMemcpyAsync(dev_dn_ + (size_t)slot * dn_bytes_, host_dn_ + (size_t)e * dn_bytes_, dn_bytes_,
                      cudaMemcpyHostToDevice, copy_) != cudaSuccess)
    return MOE_ERR_CUDA;
  owner_[slot] = e;
  slot_of_[e] = slot;
  stats_[kBytesH2D] += (int64_t)(up_bytes_ + dn_bytes_);
  return MOE_OK;
}

moe_status ExpertCache::ensure(const int32_t* counts, bool prefetch) {
  ++tick_;
  std::vector<char> needed(n_, 0);
  for (int e = 0; e < n_; ++e) needed[e] = counts[e] > 0;
  bool fenced = false;
  for (int e = 0; e < n_; ++e) {
    if (!needed[e]) continue;
    if (!prefetch) ++usage_[e];
    int s = slot_of_[e];
    if (s >= 0) {
      if (!prefetch) {
        ++stats_[kHits];
        if (prefetched_[e]) {
          ++stats_[kPrefetchHits];
          prefetched_[e] = 0;
        }
      }
      last_use_[s] = tick_;
      continue;
    }
    s = choose_slot(needed);
    if (s < 0) return MOE_ERR_UNSUPPORTED;   // the request does not fit the unpinned slots
    moe_status st = load(e, s, fenced);
    if (st) return st;
    last_use_[s] = tick_;
    if (prefetch) {
      prefetched_[e] = 1;
      ++stats_[kPrefetched];
    } else {
      ++stats_[kMisses];
    }
  }
  return cudaEventRecord(copied_, copy_) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status ExpertCache::wait_copies(cudaStream_t compute) {
  return cudaStreamWaitEvent(compute, copied_, 0) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status ExpertCache::note_compute(cudaStream_t compute) {
  if (cudaEventRecord(computed_, compute) != cudaSuccess) return MOE_ERR_CUDA;
  computed_valid_ = true;
  return MOE_OK;
}

moe_status ExpertCache::pin_hot(int n, int min_free) {
  if (n < 0 || n > n_ || slots_ - n < min_free) return MOE_ERR_INVALID_ARG;
  // the n most used experts (ties: lower id), by repeated selection of the maximum
  std::vector<char> want(n_, 0);
  for (int r = 0; r < n; ++r) {
    int best = -1;
    for (int e = 0; e < n_; ++e)
      if (!want[e] && (best < 0 || usage_[e] > usage_[best])) best = e;
    want[best] = 1;
  }
  pinned_.assign(n_, 0);
  bool fenced = false;
  ++tick_;
  for (int e = 0; e < n_; ++e) {
    if (!want[e]) continue;
    if (slot_of_[e] < 0) {
      const int s = choose_slot(want);
      if (s < 0) return MOE_ERR_UNSUPPORTED;
      moe_status st = load(e, s, fenced);
      if (st) return st;
      last_use_[s] = tick_;
    }
    pinned_[e] = 1;
  }
  return cudaEventRecord(copied_, copy_) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
