// Drives moe::ExpertCache (the library's expert_cache.cu, compiled unchanged against the
// runtime double in cuda_runtime.h) through a small C interface, for the host-policy tests
// in tests/test_cache_policy.py. Test infrastructure only.
//
// Memory: the "pinned host" store holds, for expert e and matrix m (0 = gate/up, 1 = down),
// a byte pattern unique to (e, m); the "HBM" slots start filled with 0xEE. Copies run at
// once, so slot contents can be compared with the store after every call.
#include "cuda_runtime.h"

#include <stdint.h>
#include <string.h>

#include <vector>

#include "../../quantized_moe_noaux_b300/csrc/expert_cache.h"

struct FakeStream {
  int id;
};
struct FakeEvent {
  int id;
};

namespace {

enum { kCopy = 1, kWait = 2, kRecord = 3, kSync = 4 };
constexpr int kOpInts = 7;   // kind, stream, event, matrix, slot, expert, bytes

struct Harness {
  moe::ExpertCache* cache = nullptr;
  int E = 0, slots = 0;
  size_t up = 0, dn = 0;
  std::vector<uint8_t> host_up, host_dn, dev_up, dev_dn;
  std::vector<int32_t> log;
  std::vector<FakeStream*> streams;
  std::vector<FakeEvent*> events;
  FakeStream compute{100};
  int next_stream = 1, next_event = 1;
  int fail_in = 0;   // the fail_in-th fallible call from now fails; 0: none
};

Harness g;

bool fail_now() {
  if (g.fail_in <= 0) return false;
  return --g.fail_in == 0;
}

void push(int kind, int stream, int event, int matrix, int slot, int expert, long bytes) {
  const int32_t op[kOpInts] = {kind, stream, event, matrix, slot, expert, (int32_t)bytes};
  g.log.insert(g.log.end(), op, op + kOpInts);
}

uint8_t pattern(int e, int m, size_t i) { return (uint8_t)(e * 37 + i * 11 + m * 101 + (i >> 8)); }

// (matrix, index) of p inside one of two arrays of `unit`-byte records, else matrix -1;
// index -2 when p is not at a record boundary.
void locate(const void* p, const uint8_t* a0, const uint8_t* a1, size_t n0, size_t n1, size_t u0,
            size_t u1, int& matrix, int& index) {
  const uint8_t* b = static_cast<const uint8_t*>(p);
  matrix = -1;
  index = -1;
  if (b >= a0 && b < a0 + n0) {
    matrix = 0;
    index = (b - a0) % u0 ? -2 : (int)((b - a0) / u0);
  } else if (b >= a1 && b < a1 + n1) {
    matrix = 1;
    index = (b - a1) % u1 ? -2 : (int)((b - a1) / u1);
  }
}

}  // namespace

cudaError_t cudaStreamCreateWithFlags(cudaStream_t* stream, unsigned int) {
  if (fail_now()) return cudaErrorUnknown;
  *stream = new FakeStream{g.next_stream++};
  g.streams.push_back(*stream);
  return cudaSuccess;
}

cudaError_t cudaEventCreateWithFlags(cudaEvent_t* event, unsigned int) {
  if (fail_now()) return cudaErrorUnknown;
  *event = new FakeEvent{g.next_event++};
  g.events.push_back(*event);
  return cudaSuccess;
}

cudaError_t cudaStreamSynchronize(cudaStream_t stream) {
  push(kSync, stream->id, 0, 0, 0, 0, 0);
  return cudaSuccess;
}

cudaError_t cudaStreamDestroy(cudaStream_t) { return cudaSuccess; }
cudaError_t cudaEventDestroy(cudaEvent_t) { return cudaSuccess; }

cudaError_t cudaMemcpyAsync(void* dst, const void* src, size_t count, cudaMemcpyKind kind,
                            cudaStream_t stream) {
  if (fail_now()) return cudaErrorUnknown;
  int dm, slot, sm, expert;
  locate(dst, g.dev_up.data(), g.dev_dn.data(), g.dev_up.size(), g.dev_dn.size(), g.up, g.dn, dm, slot);
  locate(src, g.host_up.data(), g.host_dn.data(), g.host_up.size(), g.host_dn.size(), g.up, g.dn, sm,
         expert);
  const int matrix = (dm == sm && kind == cudaMemcpyHostToDevice) ? dm : -1;
  if (matrix >= 0 && slot >= 0 && expert >= 0) {
    const size_t cap = matrix == 0 ? g.up : g.dn;
    memcpy(dst, src, count < cap ? count : cap);
  }
  push(kCopy, stream->id, 0, matrix, slot, expert, (long)count);
  return cudaSuccess;
}

cudaError_t cudaStreamWaitEvent(cudaStream_t stream, cudaEvent_t event, unsigned int) {
  if (fail_now()) return cudaErrorUnknown;
  push(kWait, stream->id, event->id, 0, 0, 0, 0);
  return cudaSuccess;
}

cudaError_t cudaEventRecord(cudaEvent_t event, cudaStream_t stream) {
  if (fail_now()) return cudaErrorUnknown;
  push(kRecord, stream->id, event->id, 0, 0, 0, 0);
  return cudaSuccess;
}

extern "C" {

void ch_destroy() {
  delete g.cache;
  g.cache = nullptr;
  for (FakeStream* s : g.streams) delete s;
  for (FakeEvent* e : g.events) delete e;
  g.streams.clear();
  g.events.clear();
  g.log.clear();
}

int ch_create(int E, int slots, long up_bytes, long dn_bytes) {
  ch_destroy();
  g.E = E;
  g.slots = slots;
  g.up = (size_t)up_bytes;
  g.dn = (size_t)dn_bytes;
  g.host_up.resize((size_t)E * g.up);
  g.host_dn.resize((size_t)E * g.dn);
  for (int e = 0; e < E; ++e) {
    for (size_t i = 0; i < g.up; ++i) g.host_up[e * g.up + i] = pattern(e, 0, i);
    for (size_t i = 0; i < g.dn; ++i) g.host_dn[e * g.dn + i] = pattern(e, 1, i);
  }
  g.dev_up.assign((size_t)slots * g.up, 0xEE);
  g.dev_dn.assign((size_t)slots * g.dn, 0xEE);
  g.cache = new moe::ExpertCache();
  return g.cache->init(E, slots, g.up, g.dn, g.host_up.data(), g.host_dn.data(), g.dev_up.data(),
                       g.dev_dn.data());
}

int ch_ensure(const int32_t* counts, int prefetch) { return g.cache->ensure(counts, prefetch != 0); }
int ch_note_compute() { return g.cache->note_compute(&g.compute); }
int ch_wait_copies() { return g.cache->wait_copies(&g.compute); }
int ch_pin_hot(int n, int min_free) { return g.cache->pin_hot(n, min_free); }
int ch_slot_of(int e) { return g.cache->slot_of(e); }
int ch_pinned(int e) { return g.cache->pinned(e) ? 1 : 0; }
int ch_slots() { return g.cache->slots(); }
int ch_copy_stream() { return g.cache->copy_stream()->id; }
int ch_compute_stream() { return g.compute.id; }
int ch_num_stats() { return moe::ExpertCache::kNumStats; }

void ch_stats(int64_t* out) {
  for (int i = 0; i < moe::ExpertCache::kNumStats; ++i) out[i] = g.cache->stats()[i];
}

// Moves up to cap operations (kOpInts ints each) of the log into out, oldest first, and
// drops them from the log; returns how many were moved.
int ch_take_log(int32_t* out, int cap) {
  const int n = (int)(g.log.size() / kOpInts) < cap ? (int)(g.log.size() / kOpInts) : cap;
  memcpy(out, g.log.data(), (size_t)n * kOpInts * sizeof(int32_t));
  g.log.erase(g.log.begin(), g.log.begin() + (size_t)n * kOpInts);
  return n;
}

// 1 when both matrices of `slot` hold expert e's bytes.
int ch_slot_holds(int slot, int e) {
  return memcmp(g.dev_up.data() + slot * g.up, g.host_up.data() + e * g.up, g.up) == 0 &&
         memcmp(g.dev_dn.data() + slot * g.dn, g.host_dn.data() + e * g.dn, g.dn) == 0;
}

void ch_fail_call(int n) { g.fail_in = n; }

}  // extern "C"
