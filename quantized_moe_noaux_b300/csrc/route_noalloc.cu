// Routing entry point that allocates nothing (moe_route_noalloc in include/moe_layer.h).
//
// moe_layer_forward needs a layer handle whose workspace moe_layer_create allocated with
// cudaMalloc. Some callers cannot allocate device memory at the point they need routing:
// code running while a stream is being captured into a CUDA graph (cudaMalloc is not a
// capturable operation), callers inside a host framework that owns the whole device
// memory budget, and runtimes that forbid allocation after start-up. This variant runs the
// same router, selection and grouping kernels with their scratch (logits, per-expert
// histogram, work list, status word) in one file-scope __device__ array of fixed size, so
// it only needs the caller's inputs and outputs.
#include <mutex>

#include "kernels.h"

namespace {

// Scratch limits (elements): T*E logits, E+1 counts, the grouping work list, meta words.
constexpr size_t kLogitsMax = 262144;   // 1 MiB of fp32 logits: T * E <= 262144
constexpr size_t kCountsMax = 1024 + 1;
constexpr size_t kItemsMax = 8192;
constexpr size_t kMetaWords = 16;
constexpr size_t align256(size_t b) { return (b + 255) / 256 * 256; }
constexpr size_t kOffLogits = 0;
constexpr size_t kOffCounts = kOffLogits + align256(kLogitsMax * 4);
constexpr size_t kOffItems = kOffCounts + align256(kCountsMax * 4);
constexpr size_t kOffMeta = kOffItems + align256(kItemsMax * 4);
constexpr size_t kOffStatus = kOffMeta + align256(kMetaWords * 4);
constexpr size_t kScratchBytes = kOffStatus + 256;   // ~1.04 MiB per device

// Every device that loads the library holds this array until the process exits.
static __device__ __align__(256) unsigned char g_route_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned char* g_scratch_addr[kMaxDevices] = {};

// Device address of g_route_scratch on the current device. In host code the symbol is a
// host-side stand-in, so the address is looked up once per device (with that device
// current) and cached.
cudaError_t scratch_on_current_device(unsigned char** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_route_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = static_cast<unsigned char*>(p);
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

long routing_items(int T, int top_k, int E) {
  const long tk = (long)T * top_k;
  return tk / moe::kTokChunk + (tk < E ? tk : E) + 1;
}

}  // namespace

extern "C" moe_status moe_route_noalloc(const void* x, int32_t act_dtype, int32_t T, int32_t H,
                                        const void* router_w, int32_t router_dtype,
                                        const float* bias, int32_t E, int32_t n_group,
                                        int32_t topk_group, int32_t top_k,
                                        float routed_scaling_factor, int32_t* ids, float* weights,
                                        int32_t* offsets, int32_t* entries, void* stream) {
  if (T < 0 || H <= 0 || E <= 0 || n_group <= 0 || topk_group <= 0 || top_k <= 0)
    return MOE_ERR_INVALID_ARG;
  if (act_dtype != MOE_DT_F32 && act_dtype != MOE_DT_BF16) return MOE_ERR_INVALID_ARG;
  if (router_dtype != MOE_DT_F32 && router_dtype != MOE_DT_BF16) return MOE_ERR_INVALID_ARG;
  if (!(routed_scaling_factor > 0.f)) return MOE_ERR_INVALID_ARG;
  if (E > 1024 || E % n_group || n_group > 32) return MOE_ERR_UNSUPPORTED;
  const int G = E / n_group;
  if (G < 2 || topk_group > n_group || top_k > topk_group * G || top_k > 32) return MOE_ERR_UNSUPPORTED;
  // the fixed scratch bounds the problem size
  if ((size_t)T * E > kLogitsMax || routing_items(T, top_k, E) > (long)kItemsMax)
    return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!x || !router_w || !bias || !ids || !weights || !offsets || !entries) return MOE_ERR_INVALID_ARG;
  // the tiled router reads x and W_r 16 bytes at a time; the other buffers hold 4-byte elements
  auto misaligned = [](const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) != 0; };
  if (misaligned(x, 16) || misaligned(router_w, 16) || misaligned(bias, 4) || misaligned(ids, 4) ||
      misaligned(weights, 4) || misaligned(offsets, 4) || misaligned(entries, 4))
    return MOE_ERR_INVALID_ARG;

  unsigned char* base = nullptr;
  if (scratch_on_current_device(&base) != cudaSuccess) return MOE_ERR_CUDA;
  float* logits = reinterpret_cast<float*>(base + kOffLogits);
  int32_t* counts = reinterpret_cast<int32_t*>(base + kOffCounts);
  int32_t* items = reinterpret_cast<int32_t*>(base + kOffItems);
  int32_t* meta = reinterpret_cast<int32_t*>(base + kOffMeta);
  int* status = reinterpret_cast<int*>(base + kOffStatus);
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  // The array keeps the previous call's contents: the histogram and status start at zero.
  if (cudaMemsetAsync(counts, 0, (size_t)(E + 1) * sizeof(int32_t), s) != cudaSuccess ||
      cudaMemsetAsync(status, 0, sizeof(int), s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (moe::launch_router_logits(x, act_dtype, router_w, router_dtype, logits, T, E, H, s) != cudaSuccess ||
      moe::launch_select(logits, bias, T, E, n_group, topk_group, top_k, routed_scaling_factor, 0.f, ids,
                         weights, counts, status, s) != cudaSuccess ||
      moe::launch_group(ids, counts, T, top_k, E, 0, offsets, entries, items, meta, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
