// C ABI of the MoE layer (include/moe_layer.h): layer creation (weight upload and
// workspace sizing), the forward pipeline, routing read-back and status reporting.
#include <atomic>
#include <cstdio>
#include <cstring>
#include <new>
#include <vector>

#include "expert_cache.h"
#include "kernels.h"

using namespace moe;

struct moe_layer {
  moe_config cfg{};
  int device = 0;
  bool shared_inline = false;   // shared expert stored at index E of the routed arrays
  int path = MOE_PATH_AUTO;
  // weights (device)
  void* router_w = nullptr;
  float* bias = nullptr;
  ExpertWeights w{};     // routed experts (+ shared when inline)
  ExpertWeights ws{};    // separately stored shared expert
  // tensor-core router (bf16 activations): W_r as bf16 planes summing to W_r, and the
  // split-K scratch
  const uint16_t* router_planes = nullptr;
  int router_nplanes = 0;
  float* router_part = nullptr;
  // workspace (device)
  float* logits = nullptr;
  int32_t* ids = nullptr;
  float* weights = nullptr;
  int32_t* counts = nullptr;
  int32_t* offsets = nullptr;
  int32_t* entries = nullptr;
  int32_t* items = nullptr;
  int32_t* meta = nullptr;
  float* h = nullptr;
  float* out_acc = nullptr;
  float* xq = nullptr;
  unsigned int* amax = nullptr;
  int* status = nullptr;
  void* x_stage = nullptr;
  void* out_stage = nullptr;
  // fused decode path (int4-g32 layers with an int4 shared expert; reads the grouped
  // GEMM's packed store)
  bool decode_ok = false;
  int decode_tmax = 0;          // largest T the decode scratch is sized for
  int n_sm = 0;
  uint32_t* dsync = nullptr;
  __half* dec_h16 = nullptr;
  float* dec_gu_part = nullptr;
  float* dec_y_part = nullptr;
  // grouped tcgen05 GEMM path
  bool gemm_ok = false;
  int gemm_rows = 0;            // rows of the expert-sorted activation matrices
  __half* x16s = nullptr;       // [gemm_rows, H] expert-sorted activations (fp16)
  __half* h16s = nullptr;       // [gemm_rows, I] expert-sorted h (fp16)
  float* ys = nullptr;          // [gemm_rows, H] expert-sorted down outputs (fp32)
  int32_t* inv = nullptr;       // [T*k] sorted row of each (token, slot)
  float* h32 = nullptr;         // [T*k, I] routed h before NVFP4 quantisation
  int4* gitems = nullptr;
  int32_t* g_nitems = nullptr;
  GemmMaps maps_up{}, maps_down{};
  uint8_t* gpack_up = nullptr;  // packed gate/up and down weights of the grouped GEMM
  uint8_t* gpack_down = nullptr;
  void* sh16_gu = nullptr;      // separately stored shared expert as fp16 [2I, H], [H, I]
  void* sh16_d = nullptr;
  GemmMaps maps_sh_up{}, maps_sh_down{};
  int gemm_chunk = 256;         // token rows per grouped-GEMM item
  // block-scaled FP4 path of NVFP4 layers (routed experts; the bf16 shared expert keeps the
  // fp16 kernel): weight stores in tile order with MMA-ordered scales, and the sorted
  // NVFP4 activations of the two GEMMs
  bool fp4_ok = false;
  uint8_t* f4_up_codes = nullptr;
  uint8_t* f4_up_sf = nullptr;
  uint8_t* f4_dn_codes = nullptr;
  uint8_t* f4_dn_sf = nullptr;
  uint8_t* xc = nullptr;        // [T*k, H/2] codes, [T*k, H/16] scales of the sorted x rows
  uint8_t* xsf = nullptr;
  uint8_t* hc = nullptr;        // [T*k, I/2] codes, [T*k, I/16] scales of the routed h rows
  uint8_t* hsf = nullptr;
  uint8_t* xtc = nullptr;       // [T, H/2] codes, [T, H/16] scales of each token's x
  uint8_t* xts = nullptr;
  Fp4Maps f4_up{}, f4_dn{};
  std::vector<void*> allocs;
  // HBM cache of host-resident experts (moe_layer_create_cached): the routed experts' packed
  // gate/up and down stores in pinned host memory, the HBM slots in gpack_up / gpack_down
  // (slot `slots` holds the shared expert), the device slot table, the read-back counts
  ExpertCache* cache = nullptr;
  std::vector<void*> host_allocs;
  uint8_t* host_up = nullptr;
  uint8_t* host_dn = nullptr;
  int32_t* d_slot = nullptr;
  int32_t* h_counts = nullptr;
  // routing workspace of moe_layer_prefetch (its own, so it may run beside a forward)
  float* logits_p = nullptr;
  int32_t* ids_p = nullptr;
  float* weights_p = nullptr;
  int32_t* counts_p = nullptr;
  int32_t* h_counts_p = nullptr;
  cudaEvent_t ev_x = nullptr;
  cudaStream_t route_stream = nullptr;   // prefetch routing (not behind the copies)
  // measurement
  std::vector<cudaEvent_t> events;   // kStageEvents per recorded forward
  int timing_cap = 0;
  int timing_used = 0;
  int64_t launches = 0;
  unsigned long long* trace = nullptr;   // decode-kernel phase timestamps (profiling)
  unsigned long long wait_ns = 2000000000ull;   // limit of the kernels' waits on other CTAs
  int identity_act = 0;                          // test-only: h = gate * up (no SiLU)
  int debug_checks = 0;                          // check each call's routing on the device
};

static constexpr int kStageEvents = 8;

namespace {

// Test hook: the n-th allocation from now fails (0 = off).
std::atomic<int> g_fail_alloc_at{0};
std::atomic<int> g_alloc_count{0};

bool forced_alloc_failure() {
  const int at = g_fail_alloc_at.load();
  return at > 0 && g_alloc_count.fetch_add(1) + 1 == at;
}

size_t act_bytes(int dt) { return dt == MOE_DT_F32 ? 4 : 2; }

int max_items_for(const moe_config& c, int T) {
  const long tk = (long)T * c.top_k;
  long n = tk / kTokChunk + (tk < c.n_experts ? tk : c.n_experts) + (T + kTokChunk - 1) / kTokChunk + 1;
  return (int)n;
}

struct DeviceGuard {
  int prev = -1;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    if (prev != dev) cudaSetDevice(dev);
  }
  ~DeviceGuard() {
    int cur = -1;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

moe_status validate_config(const moe_config* c) {
  if (c->hidden <= 0 || c->inter <= 0 || c->n_experts <= 0 || c->top_k <= 0 || c->n_group <= 0 ||
      c->topk_group <= 0 || c->max_tokens <= 0)
    return MOE_ERR_INVALID_ARG;
  if (!(c->routed_scaling_factor > 0.f)) return MOE_ERR_INVALID_ARG;
  if (c->expert_top_p != c->expert_top_p) return MOE_ERR_INVALID_ARG;   // NaN
  if (c->weight_format != MOE_W_INT4_G32 && c->weight_format != MOE_W_NVFP4 && !is_row_format(c->weight_format))
    return MOE_ERR_UNSUPPORTED;
  if (c->shared_format != c->weight_format && c->shared_format != MOE_W_BF16) return MOE_ERR_UNSUPPORTED;
  if (c->act_quant != MOE_ACT_NONE && c->act_quant != MOE_ACT_Q8_0) return MOE_ERR_UNSUPPORTED;
  if (c->act_quant == MOE_ACT_Q8_0 && (c->weight_format == MOE_W_NVFP4 || c->shared_format != c->weight_format))
    return MOE_ERR_UNSUPPORTED;
  if (c->act_dtype != MOE_DT_F32 && c->act_dtype != MOE_DT_BF16) return MOE_ERR_UNSUPPORTED;
  if (c->router_dtype != MOE_DT_F32 && c->router_dtype != MOE_DT_BF16) return MOE_ERR_UNSUPPORTED;
  if (c->hidden % 256 || c->inter % 64) return MOE_ERR_UNSUPPORTED;
  if ((size_t)kTokChunk * c->hidden * 4 > (size_t)kMaxDynSmem) return MOE_ERR_UNSUPPORTED;
  if (c->n_experts > 1024 || c->n_experts % c->n_group || c->n_group > 32) return MOE_ERR_UNSUPPORTED;
  const int G = c->n_experts / c->n_group;
  if (G < 2 || c->topk_group > c->n_group || c->top_k > c->topk_group * G || c->top_k > 32)
    return MOE_ERR_UNSUPPORTED;
  // work items index grid.y (<= 65535) and carry a 16-bit token-chunk field
  if (c->max_tokens > 16384 || max_items_for(*c, c->max_tokens) > 65535) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

moe_status dev_alloc(moe_layer* L, void** p, size_t bytes) {
  *p = nullptr;
  if (bytes == 0) return MOE_OK;
  if (forced_alloc_failure()) return MOE_ERR_OOM;
  if (cudaMalloc(p, bytes) != cudaSuccess) {
    cudaGetLastError();
    *p = nullptr;
    return MOE_ERR_OOM;
  }
  L->allocs.push_back(*p);
  return MOE_OK;
}

template <typename T>
moe_status dev_alloc_t(moe_layer* L, T** p, size_t bytes) {
  void* v = nullptr;
  moe_status s = dev_alloc(L, &v, bytes);
  *p = static_cast<T*>(v);
  return s;
}

void free_all(moe_layer* L) {
  delete L->cache;   // waits for its copies
  L->cache = nullptr;
  if (L->ev_x) cudaEventDestroy(L->ev_x);
  L->ev_x = nullptr;
  if (L->route_stream) {
    cudaStreamSynchronize(L->route_stream);
    cudaStreamDestroy(L->route_stream);
  }
  L->route_stream = nullptr;
  for (void* p : L->allocs) cudaFree(p);
  L->allocs.clear();
  for (void* p : L->host_allocs) cudaFreeHost(p);
  L->host_allocs.clear();
}

moe_status host_alloc(moe_layer* L, void** p, size_t bytes) {
  *p = nullptr;
  if (forced_alloc_failure()) return MOE_ERR_OOM;
  if (cudaHostAlloc(p, bytes, cudaHostAllocDefault) != cudaSuccess) {
    cudaGetLastError();
    *p = nullptr;
    return MOE_ERR_OOM;
  }
  L->host_allocs.push_back(*p);
  return MOE_OK;
}

// Upload one expert matrix family (codes, scales, tensor scales) of n experts into slots
// [first, first + n) of a store holding `cap` experts.
moe_status upload_family(const void* codes, const void* scales, const float* tscale, int fmt,
                         int rows, int K, int first, int n, uint8_t* dcodes, uint8_t* dscales,
                         float* dtscale, cudaStream_t s) {
  if (!codes) return MOE_ERR_INVALID_ARG;
  const size_t cb = (size_t)rows * row_code_bytes(fmt, K), sb = (size_t)rows * row_scale_bytes(fmt, K);
  if (cudaMemcpyAsync(dcodes + first * cb, codes, n * cb, cudaMemcpyDefault, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (sb) {
    if (!scales) return MOE_ERR_INVALID_ARG;
    if (cudaMemcpyAsync(dscales + first * sb, scales, n * sb, cudaMemcpyDefault, s) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  if (fmt == MOE_W_NVFP4) {
    if (!tscale) return MOE_ERR_INVALID_ARG;
    if (cudaMemcpyAsync(dtscale + first, tscale, n * sizeof(float), cudaMemcpyDefault, s) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

moe_status alloc_family(moe_layer* L, ExpertWeights& w, int fmt, int n, int H, int I) {
  moe_status st;
  const size_t gcb = (size_t)2 * I * row_code_bytes(fmt, H), gsb = (size_t)2 * I * row_scale_bytes(fmt, H);
  const size_t dcb = (size_t)H * row_code_bytes(fmt, I), dsb = (size_t)H * row_scale_bytes(fmt, I);
  uint8_t *gc, *gs, *dc, *ds;
  float *gt = nullptr, *dt = nullptr;
  if ((st = dev_alloc_t(L, &gc, n * gcb)) || (st = dev_alloc_t(L, &gs, n * gsb)) ||
      (st = dev_alloc_t(L, &dc, n * dcb)) || (st = dev_alloc_t(L, &ds, n * dsb)))
    return st;
  if (fmt == MOE_W_NVFP4 &&
      ((st = dev_alloc_t(L, &gt, n * sizeof(float))) || (st = dev_alloc_t(L, &dt, n * sizeof(float)))))
    return st;
  w = ExpertWeights{gc, gs, gt, dc, ds, dt};
  return MOE_OK;
}

// Store of a cached layer: each routed expert is uploaded row-major into a one-expert
// staging area, packed there into the grouped GEMM's layout and copied to pinned host
// memory; the shared expert is packed straight into its HBM slot (slot `slots`). Then the
// cache, the slot table, the read-back buffers and the prefetch workspace.
moe_status create_cache_store(moe_layer* L, const moe_config* c, const moe_weights* wt, int slots, cudaStream_t s) {
  moe_status st;
  const int H = c->hidden, I = c->inter, E = c->n_experts, k = c->top_k, Tm = c->max_tokens;
  const int fmt = c->weight_format;
  const size_t up_b = gemm_pack_bytes(2 * I, H, 1), dn_b = gemm_pack_bytes(H, I, 1);
  const size_t gcb = (size_t)2 * I * row_code_bytes(fmt, H), gsb = (size_t)2 * I * row_scale_bytes(fmt, H);
  const size_t dcb = (size_t)H * row_code_bytes(fmt, I), dsb = (size_t)H * row_scale_bytes(fmt, I);
  ExpertWeights stage{};
  uint8_t *pk_up, *pk_dn;
  void *hu, *hd;
  if ((st = alloc_family(L, stage, fmt, 1, H, I)) || (st = dev_alloc_t(L, &pk_up, up_b)) ||
      (st = dev_alloc_t(L, &pk_dn, dn_b)) || (st = dev_alloc_t(L, &L->gpack_up, (size_t)(slots + 1) * up_b)) ||
      (st = dev_alloc_t(L, &L->gpack_down, (size_t)(slots + 1) * dn_b)) ||
      (st = host_alloc(L, &hu, (size_t)E * up_b)) || (st = host_alloc(L, &hd, (size_t)E * dn_b)))
    return st;
  L->host_up = static_cast<uint8_t*>(hu);
  L->host_dn = static_cast<uint8_t*>(hd);
  uint8_t* sgc = const_cast<uint8_t*>(stage.gu_codes);
  uint8_t* sgs = const_cast<uint8_t*>(stage.gu_scales);
  uint8_t* sdc = const_cast<uint8_t*>(stage.d_codes);
  uint8_t* sds = const_cast<uint8_t*>(stage.d_scales);
  for (int e = 0; e <= E; ++e) {
    const bool sh = e == E;
    const uint8_t* gc = sh ? static_cast<const uint8_t*>(wt->sh_gu) : wt->gu_codes + (size_t)e * gcb;
    const uint8_t* gs = sh ? static_cast<const uint8_t*>(wt->sh_gu_scales)
                           : static_cast<const uint8_t*>(wt->gu_scales) + (size_t)e * gsb;
    const uint8_t* dc = sh ? static_cast<const uint8_t*>(wt->sh_d) : wt->d_codes + (size_t)e * dcb;
    const uint8_t* ds = sh ? static_cast<const uint8_t*>(wt->sh_d_scales)
                           : static_cast<const uint8_t*>(wt->d_scales) + (size_t)e * dsb;
    if ((st = upload_family(gc, gs, nullptr, fmt, 2 * I, H, 0, 1, sgc, sgs, nullptr, s)) ||
        (st = upload_family(dc, ds, nullptr, fmt, H, I, 0, 1, sdc, sds, nullptr, s)))
      return st;
    uint8_t* du = sh ? L->gpack_up + (size_t)slots * up_b : pk_up;
    uint8_t* dd = sh ? L->gpack_down + (size_t)slots * dn_b : pk_dn;
    if (launch_gemm_pack(sgc, sgs, H, 1, 2 * I, I, true, du, s) || launch_gemm_pack(sdc, sds, I, 1, H, I, false, dd, s))
      return MOE_ERR_CUDA;
    if (!sh && (cudaMemcpyAsync(L->host_up + (size_t)e * up_b, pk_up, up_b, cudaMemcpyDeviceToHost, s) ||
                cudaMemcpyAsync(L->host_dn + (size_t)e * dn_b, pk_dn, dn_b, cudaMemcpyDeviceToHost, s)))
      return MOE_ERR_CUDA;
  }
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  void *hc, *hcp;
  if ((st = dev_alloc_t(L, &L->d_slot, (size_t)(E + 1) * 4)) || (st = host_alloc(L, &hc, (size_t)(E + 1) * 4)) ||
      (st = host_alloc(L, &hcp, (size_t)(E + 1) * 4)) || (st = dev_alloc_t(L, &L->logits_p, (size_t)Tm * E * 4)) ||
      (st = dev_alloc_t(L, &L->ids_p, (size_t)Tm * k * 4)) || (st = dev_alloc_t(L, &L->weights_p, (size_t)Tm * k * 4)) ||
      (st = dev_alloc_t(L, &L->counts_p, (size_t)(E + 1) * 4)))
    return st;
  L->h_counts = static_cast<int32_t*>(hc);
  L->h_counts_p = static_cast<int32_t*>(hcp);
  if (cudaEventCreateWithFlags(&L->ev_x, cudaEventDisableTiming) != cudaSuccess ||
      cudaStreamCreateWithFlags(&L->route_stream, cudaStreamNonBlocking) != cudaSuccess)
    return MOE_ERR_CUDA;
  L->cache = new (std::nothrow) ExpertCache();
  if (!L->cache) return MOE_ERR_OOM;
  return L->cache->init(E, slots, up_b, dn_b, L->host_up, L->host_dn, L->gpack_up, L->gpack_down);
}

moe_status create_impl(moe_layer* L, const moe_config* c, const moe_weights* wt, cudaStream_t s,
                       int cache_slots = 0) {
  moe_status st;
  const int H = c->hidden, I = c->inter, E = c->n_experts, k = c->top_k, Tm = c->max_tokens;
  if (!wt->router_w || !wt->bias || !wt->gu_codes || !wt->d_codes || !wt->sh_gu || !wt->sh_d)
    return MOE_ERR_INVALID_ARG;
  if (expert_kernels_init() != cudaSuccess) return MOE_ERR_CUDA;
  L->shared_inline = c->shared_format == c->weight_format;
  const int n_store = E + (L->shared_inline ? 1 : 0);

  const size_t rw_bytes = (size_t)E * H * (c->router_dtype == MOE_DT_F32 ? 4 : 2);
  if ((st = dev_alloc(L, &L->router_w, rw_bytes)) || (st = dev_alloc_t(L, &L->bias, E * sizeof(float))))
    return st;
  if (cudaMemcpyAsync(L->router_w, wt->router_w, rw_bytes, cudaMemcpyDefault, s) ||
      cudaMemcpyAsync(L->bias, wt->bias, E * sizeof(float), cudaMemcpyDefault, s))
    return MOE_ERR_CUDA;

  if (cache_slots > 0) {
    if ((st = create_cache_store(L, c, wt, cache_slots, s))) return st;
  } else if ((st = alloc_family(L, L->w, c->weight_format, n_store, H, I))) {
    return st;
  }
  ExpertWeights& w = L->w;
  if (cache_slots > 0) {
    // routed and shared experts live in the cache store only
  } else if ((st = upload_family(wt->gu_codes, wt->gu_scales, wt->gu_tscale, c->weight_format, 2 * I, H, 0, E,
                          const_cast<uint8_t*>(w.gu_codes), const_cast<uint8_t*>(w.gu_scales),
                          const_cast<float*>(w.gu_tscale), s)) ||
      (st = upload_family(wt->d_codes, wt->d_scales, wt->d_tscale, c->weight_format, H, I, 0, E,
                          const_cast<uint8_t*>(w.d_codes), const_cast<uint8_t*>(w.d_scales),
                          const_cast<float*>(w.d_tscale), s)))
    return st;
  ExpertWeights* sw = &L->w;
  int slot = E;
  if (cache_slots > 0) {
    // shared expert packed into its HBM slot by create_cache_store
  } else if (!L->shared_inline) {
    if ((st = alloc_family(L, L->ws, c->shared_format, 1, H, I))) return st;
    sw = &L->ws;
    slot = 0;
  }
  if (cache_slots == 0 &&
      ((st = upload_family(wt->sh_gu, wt->sh_gu_scales, wt->sh_gu_tscale, c->shared_format, 2 * I, H, slot,
                           1, const_cast<uint8_t*>(sw->gu_codes), const_cast<uint8_t*>(sw->gu_scales),
                           const_cast<float*>(sw->gu_tscale), s)) ||
       (st = upload_family(wt->sh_d, wt->sh_d_scales, wt->sh_d_tscale, c->shared_format, H, I, slot, 1,
                           const_cast<uint8_t*>(sw->d_codes), const_cast<uint8_t*>(sw->d_scales),
                           const_cast<float*>(sw->d_tscale), s))))
    return st;

  const size_t ab = act_bytes(c->act_dtype);
  if ((st = dev_alloc_t(L, &L->logits, (size_t)Tm * E * 4)) ||
      (st = dev_alloc_t(L, &L->ids, (size_t)Tm * k * 4)) ||
      (st = dev_alloc_t(L, &L->weights, (size_t)Tm * k * 4)) ||
      (st = dev_alloc_t(L, &L->counts, (size_t)(E + 1) * 4)) ||
      (st = dev_alloc_t(L, &L->offsets, (size_t)(E + 2) * 4)) ||
      (st = dev_alloc_t(L, &L->entries, (size_t)Tm * k * 4)) ||
      (st = dev_alloc_t(L, &L->items, (size_t)max_items_for(*c, Tm) * 4)) ||
      (st = dev_alloc_t(L, &L->meta, 16 * 4)) ||
      (st = dev_alloc_t(L, &L->h, (size_t)Tm * (k + 1) * I * 4)) ||
      (st = dev_alloc_t(L, &L->out_acc, (size_t)Tm * H * 4)) ||
      (st = dev_alloc_t(L, &L->amax, 4 * sizeof(unsigned int))) ||
      (st = dev_alloc_t(L, &L->status, sizeof(int))) ||
      (st = dev_alloc(L, &L->x_stage, (size_t)Tm * H * ab)) ||
      (st = dev_alloc(L, &L->out_stage, (size_t)Tm * H * ab)))
    return st;
  if ((c->weight_format == MOE_W_NVFP4 || c->act_quant == MOE_ACT_Q8_0) &&
      (st = dev_alloc_t(L, &L->xq, (size_t)Tm * H * 4)))
    return st;

  int dev = 0;
  if (cudaGetDevice(&dev) || cudaDeviceGetAttribute(&L->n_sm, cudaDevAttrMultiProcessorCount, dev))
    return MOE_ERR_CUDA;
  // tensor-core router: an fp32 W_r is split into hi/mid/lo bf16 planes once; a bf16 W_r is
  // its own single plane
  if (router_mma_supported(c->act_dtype, H, E)) {
    if (router_mma_init() != cudaSuccess) return MOE_ERR_CUDA;
    if (c->router_dtype == MOE_DT_F32) {
      uint16_t* planes = nullptr;
      if ((st = dev_alloc_t(L, &planes, (size_t)3 * E * H * 2))) return st;
      if (launch_router_split(static_cast<const float*>(L->router_w), planes, (size_t)E * H, s) != cudaSuccess)
        return MOE_ERR_CUDA;
      L->router_planes = planes;
      L->router_nplanes = 3;
    } else {
      L->router_planes = static_cast<const uint16_t*>(L->router_w);
      L->router_nplanes = 1;
    }
    if ((st = dev_alloc_t(L, &L->router_part, router_mma_partial_floats(L->n_sm) * 4))) return st;
  }

  // grouped GEMM path: expert-sorted activation buffers and the TMA descriptors; a
  // separately stored (bf16) shared expert gets an fp16 copy for the same kernel
  // (per-row formats and Q8_0 activations run on the CUDA-core kernels only)
  L->gemm_ok = gemm_supported(H, I) && !is_row_format(c->weight_format) && c->act_quant == MOE_ACT_NONE &&
               gemm_kernels_init() == cudaSuccess && (L->shared_inline || c->shared_format == MOE_W_BF16);
  if (L->gemm_ok) {
    const int fmt = c->weight_format;
    L->gemm_rows = Tm * k + Tm;
    // NVFP4 routed experts with a separate shared expert run on the block-scaled FP4 kernel
    L->fp4_ok = fmt == MOE_W_NVFP4 && !L->shared_inline && fp4_gemm_supported(H, I) &&
                fp4_gemm_init() == cudaSuccess;
    L->gemm_chunk = L->fp4_ok ? kFp4MaxN : 256;
    if ((st = dev_alloc(L, reinterpret_cast<void**>(&L->x16s), (size_t)L->gemm_rows * H * 2)) ||
        (st = dev_alloc(L, reinterpret_cast<void**>(&L->h16s), (size_t)L->gemm_rows * I * 2)) ||
        (st = dev_alloc_t(L, &L->ys, (size_t)L->gemm_rows * H * 4)) ||
        (st = dev_alloc_t(L, &L->inv, (size_t)Tm * k * 4)) ||
        (st = dev_alloc_t(L, &L->gitems,
                          (size_t)gemm_max_items(Tm, k, E, true, true, L->gemm_chunk) * sizeof(int4))) ||
        (st = dev_alloc_t(L, &L->g_nitems, 4 * sizeof(int32_t))))
      return st;
    if (fmt == MOE_W_NVFP4 && (st = dev_alloc_t(L, &L->h32, (size_t)Tm * k * I * 4))) return st;
    if (L->fp4_ok) {
      const size_t rk = (size_t)Tm * k;
      if ((st = dev_alloc_t(L, &L->f4_up_codes, (size_t)E * 2 * I * (H / 2))) ||
          (st = dev_alloc_t(L, &L->f4_up_sf, fp4_scale_bytes(2 * I, H, E))) ||
          (st = dev_alloc_t(L, &L->f4_dn_codes, (size_t)E * H * (I / 2))) ||
          (st = dev_alloc_t(L, &L->f4_dn_sf, fp4_scale_bytes(H, I, E))) ||
          (st = dev_alloc_t(L, &L->xc, rk * (H / 2))) || (st = dev_alloc_t(L, &L->xsf, rk * (H / 16))) ||
          (st = dev_alloc_t(L, &L->hc, rk * (I / 2))) || (st = dev_alloc_t(L, &L->hsf, rk * (I / 16))) ||
          (st = dev_alloc_t(L, &L->xtc, (size_t)Tm * (H / 2))) || (st = dev_alloc_t(L, &L->xts, (size_t)Tm * (H / 16))))
        return st;
      if (launch_fp4_pack(L->w.gu_codes, L->w.gu_scales, H, E, 2 * I, I, true, L->f4_up_codes, L->f4_up_sf, s) ||
          launch_fp4_pack(L->w.d_codes, L->w.d_scales, I, E, H, I, false, L->f4_dn_codes, L->f4_dn_sf, s))
        return MOE_ERR_CUDA;
      bool ok = make_tmap_2d(&L->f4_up.w, L->f4_up_codes, 1, H / 2, (uint64_t)E * 2 * I, 128, 128, true) &&
                make_tmap_2d(&L->f4_dn.w, L->f4_dn_codes, 1, I / 2, (uint64_t)E * H, 128, 128, true);
      for (int b = 0; b < 4 && ok; ++b) {
        const uint32_t box = b < 3 ? 32u << b : (uint32_t)kFp4MaxN;
        ok = make_tmap_2d(&L->f4_up.act[b], L->xc, 1, H / 2, rk, 128, box, true) &&
             make_tmap_2d(&L->f4_dn.act[b], L->hc, 1, I / 2, rk, 128, box, true);
      }
      if (!ok) return MOE_ERR_CUDA;
    } else if (cache_slots == 0) {
      if ((st = dev_alloc_t(L, &L->gpack_up, gemm_pack_bytes(2 * I, H, n_store))) ||
          (st = dev_alloc_t(L, &L->gpack_down, gemm_pack_bytes(H, I, n_store))))
        return st;
      if (launch_gemm_pack(L->w.gu_codes, L->w.gu_scales, H, n_store, 2 * I, I, true, L->gpack_up, s) ||
          launch_gemm_pack(L->w.d_codes, L->w.d_scales, I, n_store, H, I, false, L->gpack_down, s))
        return MOE_ERR_CUDA;
    }
    for (int b = 0; b < 4 && L->gemm_ok; ++b)
      L->gemm_ok = make_tmap_2d(&L->maps_up.act[b], L->x16s, 2, H, L->gemm_rows, 64, 32u << b, true) &&
                   make_tmap_2d(&L->maps_down.act[b], L->h16s, 2, I, L->gemm_rows, 64, 32u << b, true);
    L->maps_up.codes = L->maps_up.act[0];       // unused by the packed-weight kernels
    L->maps_down.codes = L->maps_down.act[0];
    if (L->gemm_ok && !L->shared_inline) {
      if ((st = dev_alloc(L, &L->sh16_gu, (size_t)2 * I * H * 2)) || (st = dev_alloc(L, &L->sh16_d, (size_t)H * I * 2)))
        return st;
      if (launch_bf16_to_f16(L->ws.gu_codes, L->sh16_gu, (size_t)2 * I, H, true, I, s) ||
          launch_bf16_to_f16(L->ws.d_codes, L->sh16_d, (size_t)H, I, false, I, s))
        return MOE_ERR_CUDA;
      L->maps_sh_up = L->maps_up;
      L->maps_sh_down = L->maps_down;
      L->gemm_ok = make_tmap_2d(&L->maps_sh_up.codes, L->sh16_gu, 2, H, 2 * I, 64, 128, true) &&
                   make_tmap_2d(&L->maps_sh_down.codes, L->sh16_d, 2, I, H, 64, 128, true);
    }
  }
  // fused decode path: reads the grouped GEMM's packed store; scratch for min(max_tokens, 8)
  // tokens
  {
    const int Td = Tm < 8 ? Tm : 8;
    L->decode_ok = L->gemm_ok && !L->cache && c->weight_format == MOE_W_INT4_G32 && L->shared_inline &&
                   decode_supported(H, I, E, k, 1) && decode_kernels_init() == cudaSuccess;
    int occ = 0;
    if (L->decode_ok && (decode_occupancy(&occ) != cudaSuccess || occ < 1)) L->decode_ok = false;
    if (L->decode_ok) {
      int td = Td;
      while (td > 1 && !decode_supported(H, I, E, k, td)) --td;
      L->decode_tmax = td;
      const size_t nsync = decode_sync_words(I);
      if ((st = dev_alloc_t(L, &L->dsync, nsync * 4)) ||
          (st = dev_alloc_t(L, &L->dec_h16, decode_h16_elems(td, I, E, k) * 2)) ||
          (st = dev_alloc_t(L, &L->dec_gu_part, decode_gu_part_floats(td, H, I, E, k) * 4)) ||
          (st = dev_alloc_t(L, &L->dec_y_part, decode_y_part_floats(td, H, I, k) * 4)))
        return st;
      if (cudaMemsetAsync(L->dsync, 0, nsync * 4, s)) return MOE_ERR_CUDA;
    }
  }
  if (cudaMemsetAsync(L->status, 0, sizeof(int), s) || cudaMemsetAsync(L->meta, 0, 16 * 4, s))
    return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}

#define MOE_CK(call)                       \
  do {                                     \
    if ((call) != cudaSuccess) return MOE_ERR_CUDA; \
  } while (0)

// Kernel launch: counted, error-checked.
#define MOE_LAUNCH(call)   \
  do {                     \
    ++L->launches;         \
    MOE_CK(call);          \
  } while (0)

struct StageMarks {
  cudaEvent_t* ev = nullptr;
  cudaStream_t s;
  // External records become event nodes when the stream is being captured into a graph.
  cudaError_t mark(int i) {
    return ev ? cudaEventRecordWithFlags(ev[i], s, cudaEventRecordExternal) : cudaSuccess;
  }
};

void release_events(moe_layer* L) {
  for (cudaEvent_t e : L->events) cudaEventDestroy(e);
  L->events.clear();
  L->timing_cap = L->timing_used = 0;
}

// Grouped tcgen05 path after routing: expert-sorted activations, gate/up GEMM with the
// SwiGLU epilogue, down GEMM with the weighted-combine epilogue, output conversion.
moe_status forward_gemm(moe_layer* L, const void* x, int T, void* out, cudaStream_t s, StageMarks& m) {
  const moe_config& c = L->cfg;
  const int H = c.hidden, I = c.inter, E = c.n_experts, k = c.top_k;
  const bool nvfp4 = c.weight_format == MOE_W_NVFP4;
  const int Tk = T * k;
  const bool inl = L->shared_inline;
  // inline shared expert: one launch covers routed and shared items (n_items[2]);
  // otherwise the routed items (n_items[0]) and the fp16 shared expert (n_items[1], after
  // the routed ones) are separate launches
  const bool f4 = L->fp4_ok;
  const int chunk = L->gemm_chunk;
  const int routed_max = gemm_max_items(T, k, E, true, inl, chunk);
  const int shared_max = gemm_max_items(T, k, E, false, true, chunk);
  MOE_LAUNCH(launch_gemm_items(L->offsets, E, T, k, chunk, L->gitems, L->g_nitems, s));
  if (L->cache) {
    // host-resident experts: read the routed experts back, load the missing ones into HBM
    // slots (copy stream), then publish the slot table on this stream
    MOE_CK(cudaMemcpyAsync(L->h_counts, L->counts, (size_t)E * 4, cudaMemcpyDeviceToHost, s));
    MOE_CK(cudaStreamSynchronize(s));
    moe_status cs = L->cache->ensure(L->h_counts, false);
    if (cs || (cs = L->cache->wait_copies(s))) return cs;
    SlotTable t;
    for (int e = 0; e < E; ++e) t.slot[e] = L->cache->slot_of(e);
    t.slot[E] = L->cache->slots();
    MOE_LAUNCH(launch_set_slots(t, E + 1, L->d_slot, s));
  }
  if (nvfp4) MOE_LAUNCH(launch_amax(x, c.act_dtype, (size_t)T * H, L->amax, s));
  if (f4) {
    // routed rows as NVFP4 codes + scales; the bf16 shared expert reads fp16 x
    MOE_LAUNCH(launch_quant_gather_fp4(x, c.act_dtype, H, T, L->entries, k, L->amax, L->xtc, L->xts, L->xc, L->xsf,
                                       L->inv, L->offsets + E, s));
    MOE_LAUNCH(launch_gather_shared_rows(x, c.act_dtype, H, Tk, T, L->x16s, s));
  } else {
    MOE_LAUNCH(launch_gather_act(x, c.act_dtype, nvfp4, H, L->entries, Tk, k, Tk + T, L->x16s, L->amax,
                                 reinterpret_cast<__half*>(L->xq), L->inv, L->offsets + E, s));   // xq: NVFP4 scratch
  }
  MOE_CK(m.mark(2));
  GemmParams p{};
  p.items = L->gitems;
  p.n_items = L->g_nitems + (inl ? 2 : 0);
  p.H = H;
  p.I = I;
  p.T = T;
  p.top_k = k;
  p.h16 = L->h16s;
  p.h32 = L->h32;
  p.h_amax = L->amax + 1;
  p.y = L->ys;
  p.entries = L->entries;
  p.weights = L->weights;
  p.status = L->status;
  p.wait_ns = L->wait_ns;
  p.slot_of = L->cache ? L->d_slot : nullptr;
  p.identity_act = L->identity_act;
  p.trace = L->trace;
  p.trace_base = 16;
  GemmParams ps = p;   // separately stored fp16 shared expert
  ps.n_items = L->g_nitems + 1;
  ps.item_skip = L->g_nitems;
  ps.e_sub = E;
  ps.w_tscale = nullptr;
  ps.act_amax = nullptr;
  ps.trace_base = 48;

  p.K = ps.K = H;
  p.rows_per_expert = ps.rows_per_expert = 2 * I;
  p.mtiles = ps.mtiles = 2 * I / 128;
  p.wpack = L->gpack_up;
  p.w_tscale = L->w.gu_tscale;
  p.act_amax = L->amax;
  if (f4) {
    p.wsf = L->f4_up_sf;
    p.asf = L->xsf;
    MOE_LAUNCH(launch_gemm_fp4(0, L->f4_up, p, routed_max * p.mtiles, L->n_sm, s));
  } else {
    MOE_LAUNCH(launch_gemm(c.weight_format, 0, L->maps_up, p, routed_max * p.mtiles, L->n_sm, s));
  }
  MOE_CK(m.mark(3));
  if (!inl) MOE_LAUNCH(launch_gemm(kWF16, 0, L->maps_sh_up, ps, shared_max * ps.mtiles, L->n_sm, s));
  MOE_CK(m.mark(4));
  if (f4) MOE_LAUNCH(launch_quant_h_fp4(L->h32, (size_t)Tk * I, L->amax + 1, L->hc, L->hsf, s));
  else if (nvfp4) MOE_LAUNCH(launch_quant_h(L->h32, (size_t)Tk * I, L->amax + 1, L->h16s, s));
  MOE_CK(m.mark(5));
  p.K = ps.K = I;
  p.trace_base = 32;
  ps.trace = nullptr;   // the shared expert's down launch is not traced
  p.rows_per_expert = ps.rows_per_expert = H;
  p.mtiles = ps.mtiles = H / 128;
  p.wpack = L->gpack_down;
  p.w_tscale = L->w.d_tscale;
  p.act_amax = L->amax + 1;
  if (f4) {
    p.wsf = L->f4_dn_sf;
    p.asf = L->hsf;
    MOE_LAUNCH(launch_gemm_fp4(1, L->f4_dn, p, routed_max * p.mtiles, L->n_sm, s));
  } else {
    MOE_LAUNCH(launch_gemm(c.weight_format, 1, L->maps_down, p, routed_max * p.mtiles, L->n_sm, s));
  }
  if (!inl) MOE_LAUNCH(launch_gemm(kWF16, 1, L->maps_sh_down, ps, shared_max * ps.mtiles, L->n_sm, s));
  if (L->cache) {
    moe_status cs = L->cache->note_compute(s);   // the slots' last readers
    if (cs) return cs;
  }
  MOE_CK(m.mark(6));
  MOE_LAUNCH(launch_combine(L->ys, L->inv, L->ids, L->weights, T, k, H, out, c.act_dtype, s));
  MOE_CK(m.mark(7));
  return MOE_OK;
}

moe_status forward_impl(moe_layer* L, const void* x, int T, void* out, cudaStream_t s) {
  const moe_config& c = L->cfg;
  const int H = c.hidden, I = c.inter, E = c.n_experts, k = c.top_k;
  const bool nvfp4 = c.weight_format == MOE_W_NVFP4;
  StageMarks m;
  m.s = s;
  if (L->timing_used < L->timing_cap) m.ev = &L->events[(size_t)kStageEvents * L->timing_used++];
  if (L->cache && (L->path == MOE_PATH_GEMV || L->path == MOE_PATH_GENERIC)) return MOE_ERR_UNSUPPORTED;
  const bool decode = L->decode_ok && T <= L->decode_tmax && (long)T * k <= 64 &&
                     (L->path == MOE_PATH_AUTO || L->path == MOE_PATH_GEMV);
  if (L->path == MOE_PATH_GEMV && !decode) return MOE_ERR_UNSUPPORTED;
  if (L->path == MOE_PATH_GROUPED && !L->gemm_ok) return MOE_ERR_UNSUPPORTED;
  const bool gemm = !decode && L->gemm_ok && L->path != MOE_PATH_GENERIC;
  if (decode) {
    // one fused kernel: routing, gate/up, down + combine (recorded in the third stage slot)
    MOE_CK(m.mark(0));
    MOE_CK(m.mark(1));
    MOE_CK(m.mark(2));
    DecodeLaunch d{x, T, L->router_w, L->bias, H, I, E, k, c.n_group, c.topk_group,
                   c.routed_scaling_factor, c.expert_top_p, L->identity_act, L->gpack_up, L->gpack_down,
                   L->logits, L->ids,
                   L->weights, L->offsets, L->entries, L->dec_h16, L->dec_gu_part, L->dec_y_part,
                   out, L->dsync, L->status, L->wait_ns, L->trace};
    MOE_LAUNCH(launch_decode_fused(d, c.act_dtype, c.router_dtype, L->n_sm, s));
    if (L->debug_checks) MOE_LAUNCH(launch_check_routing(L->ids, L->offsets, L->entries, T, k, E, L->status, s));
    for (int i = 3; i < kStageEvents; ++i) MOE_CK(m.mark(i));
    return MOE_OK;
  }
  MOE_CK(m.mark(0));
  MOE_CK(cudaMemsetAsync(L->counts, 0, (E + 1) * sizeof(int32_t), s));
  MOE_CK(cudaMemsetAsync(L->amax, 0, 4 * sizeof(unsigned int), s));
  if (!gemm) MOE_CK(cudaMemsetAsync(L->out_acc, 0, (size_t)T * H * sizeof(float), s));
  if (L->router_planes)
    MOE_LAUNCH(launch_router_mma(x, L->router_planes, L->router_nplanes, L->logits, L->router_part, T, E, H,
                                 L->n_sm, s));
  else
    MOE_LAUNCH(launch_router_logits(x, c.act_dtype, L->router_w, c.router_dtype, L->logits, T, E, H, s));
  MOE_LAUNCH(launch_select(L->logits, L->bias, T, E, c.n_group, c.topk_group, k, c.routed_scaling_factor,
                           c.expert_top_p,
                           L->ids, L->weights, L->counts, L->status, s));
  MOE_LAUNCH(launch_group(L->ids, L->counts, T, k, E, L->shared_inline, L->offsets, L->entries,
                          gemm ? nullptr : L->items, L->meta, s));
  if (L->debug_checks) MOE_LAUNCH(launch_check_routing(L->ids, L->offsets, L->entries, T, k, E, L->status, s));
  MOE_CK(m.mark(1));
  if (gemm) return forward_gemm(L, x, T, out, s, m);
  const void* x_in = x;
  int x_dt = c.act_dtype;
  const bool q8 = c.act_quant == MOE_ACT_Q8_0;
  if (nvfp4) {
    MOE_LAUNCH(launch_amax(x, c.act_dtype, (size_t)T * H, L->amax, s));
    MOE_LAUNCH(launch_nvfp4_quant(x, c.act_dtype, L->xq, (size_t)T * H, L->amax, s));
    x_in = L->xq;
    x_dt = MOE_DT_F32;
  } else if (q8) {
    MOE_LAUNCH(launch_q8_0_quant(x, c.act_dtype, L->xq, (size_t)T * H, s));
    x_in = L->xq;
    x_dt = MOE_DT_F32;
  }
  MOE_CK(m.mark(2));
  ExpertGemvArgs a{};
  a.w = L->w;
  a.fmt = c.weight_format;
  a.H = H;
  a.I = I;
  a.E = E;
  a.top_k = k;
  a.T = T;
  a.x = x_in;
  a.x_dtype = x_dt;
  a.offsets = L->offsets;
  a.entries = L->entries;
  a.items = L->items;
  a.meta = L->meta;
  a.expert_base = E;
  a.h = L->h;
  a.h_amax = nvfp4 ? L->amax + 1 : nullptr;
  a.weights = L->weights;
  a.out_acc = L->out_acc;
  a.max_items = max_items_for(c, T);
  a.identity_act = L->identity_act;
  ExpertGemvArgs sh = a;
  if (!L->shared_inline) {
    sh.w = L->ws;
    sh.fmt = c.shared_format;
    sh.items = nullptr;
    sh.meta = nullptr;
    sh.expert_base = 0;
    sh.h_amax = nullptr;
    sh.max_items = (T + kTokChunk - 1) / kTokChunk;
    if (c.shared_format != MOE_W_NVFP4) {
      sh.x = x;
      sh.x_dtype = c.act_dtype;
    }
  }
  MOE_LAUNCH(launch_expert_up(a, s));
  MOE_CK(m.mark(3));
  if (!L->shared_inline) MOE_LAUNCH(launch_expert_up(sh, s));
  MOE_CK(m.mark(4));
  if (nvfp4) MOE_LAUNCH(launch_nvfp4_quant(L->h, MOE_DT_F32, L->h, (size_t)T * k * I, L->amax + 1, s));
  if (q8) MOE_LAUNCH(launch_q8_0_quant(L->h, MOE_DT_F32, L->h, (size_t)T * (k + 1) * I, s));   // routed + shared h
  MOE_CK(m.mark(5));
  MOE_LAUNCH(launch_expert_down(a, s));
  if (!L->shared_inline) MOE_LAUNCH(launch_expert_down(sh, s));
  MOE_CK(m.mark(6));
  MOE_LAUNCH(launch_finalize(L->out_acc, out, c.act_dtype, (size_t)T * H, s));
  MOE_CK(m.mark(7));
  return MOE_OK;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace

extern "C" {

moe_status moe_layer_create(const moe_config* cfg, const moe_weights* w, void* stream,
                            moe_layer** out) {
  if (!out) return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  if (!cfg || !w) return MOE_ERR_INVALID_ARG;
  moe_status st = validate_config(cfg);
  if (st) return st;
  moe_layer* L = new (std::nothrow) moe_layer();
  if (!L) return MOE_ERR_OOM;
  L->cfg = *cfg;
  if (cudaGetDevice(&L->device) != cudaSuccess) {
    delete L;
    return MOE_ERR_CUDA;
  }
  st = create_impl(L, cfg, w, static_cast<cudaStream_t>(stream));
  if (st) {
    cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    cudaGetLastError();
    free_all(L);
    delete L;
    return st;
  }
  *out = L;
  return MOE_OK;
}

moe_status moe_layer_forward(moe_layer* L, const void* x, int32_t T, void* out, void* stream) {
  if (!L) return MOE_ERR_INVALID_ARG;
  if (T < 0 || T > L->cfg.max_tokens) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !out || !aligned16(x) || !aligned16(out) || x == out) return MOE_ERR_INVALID_ARG;
  DeviceGuard g(L->device);
  return forward_impl(L, x, T, out, static_cast<cudaStream_t>(stream));
}

moe_status moe_layer_forward_host(moe_layer* L, const void* x_host, int32_t T, void* out_host,
                                  void* stream) {
  if (!L) return MOE_ERR_INVALID_ARG;
  if (T < 0 || T > L->cfg.max_tokens) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x_host || !out_host) return MOE_ERR_INVALID_ARG;
  DeviceGuard g(L->device);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t bytes = (size_t)T * L->cfg.hidden * act_bytes(L->cfg.act_dtype);
  if (cudaMemcpyAsync(L->x_stage, x_host, bytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  moe_status st = forward_impl(L, L->x_stage, T, L->out_stage, s);
  if (st) return st;
  if (cudaMemcpyAsync(out_host, L->out_stage, bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  return cudaStreamSynchronize(s) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status moe_layer_get_routing(moe_layer* L, int32_t T, int32_t* ids, float* weights,
                                 int32_t* offsets, int32_t* entries, void* stream) {
  if (!L || T < 0 || T > L->cfg.max_tokens) return MOE_ERR_INVALID_ARG;
  DeviceGuard g(L->device);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t tk = (size_t)T * L->cfg.top_k;
  if ((ids && cudaMemcpyAsync(ids, L->ids, tk * 4, cudaMemcpyDeviceToHost, s)) ||
      (weights && cudaMemcpyAsync(weights, L->weights, tk * 4, cudaMemcpyDeviceToHost, s)) ||
      (offsets && cudaMemcpyAsync(offsets, L->offsets, (L->cfg.n_experts + 1) * 4, cudaMemcpyDeviceToHost, s)) ||
      (entries && cudaMemcpyAsync(entries, L->entries, tk * 4, cudaMemcpyDeviceToHost, s)))
    return MOE_ERR_CUDA;
  return cudaStreamSynchronize(s) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status moe_layer_set_path(moe_layer* L, int32_t path) {
  if (!L || path < MOE_PATH_AUTO || path > MOE_PATH_GENERIC) return MOE_ERR_INVALID_ARG;
  L->path = path;
  return MOE_OK;
}

moe_status moe_layer_status(moe_layer* L) {
  if (!L) return MOE_ERR_INVALID_ARG;
  DeviceGuard g(L->device);
  if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  int code = 0;
  if (cudaMemcpy(&code, L->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  return static_cast<moe_status>(code);
}

moe_status moe_layer_enable_timing(moe_layer* L, int32_t enable) {
  if (!L || enable < 0) return MOE_ERR_INVALID_ARG;
  DeviceGuard g(L->device);
  release_events(L);
  for (long i = 0; i < (long)enable * kStageEvents; ++i) {
    cudaEvent_t e;
    if (cudaEventCreate(&e) != cudaSuccess) {
      release_events(L);
      return MOE_ERR_CUDA;
    }
    L->events.push_back(e);
  }
  L->timing_cap = enable;
  return MOE_OK;
}

moe_status moe_layer_stage_times(moe_layer* L, float* ms, int32_t* n_forwards) {
  if (!L || !ms) return MOE_ERR_INVALID_ARG;
  DeviceGuard g(L->device);
  if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;
  for (int j = 0; j < kStageEvents - 1; ++j) ms[j] = 0.f;
  for (int i = 0; i < L->timing_used; ++i) {
    cudaEvent_t* ev = &L->events[(size_t)kStageEvents * i];
    for (int j = 0; j < kStageEvents - 1; ++j) {
      float t = 0.f;
      if (cudaEventElapsedTime(&t, ev[j], ev[j + 1]) != cudaSuccess) return MOE_ERR_CUDA;
      ms[j] += t;
    }
  }
  if (n_forwards) *n_forwards = L->timing_used;
  L->timing_used = 0;
  return MOE_OK;
}

moe_status moe_layer_set_trace(moe_layer* L, void* buffer, int32_t n_ctas) {
  if (!L || n_ctas < 0 || (buffer && n_ctas < L->n_sm)) return MOE_ERR_INVALID_ARG;
  L->trace = buffer ? static_cast<unsigned long long*>(buffer) : nullptr;
  return MOE_OK;
}

moe_status moe_layer_launch_count(moe_layer* L, int64_t* count) {
  if (!L || !count) return MOE_ERR_INVALID_ARG;
  *count = L->launches;
  return MOE_OK;
}

moe_status moe_layer_set_wait_limit(moe_layer* L, int64_t ns) {
  if (!L || ns < 0) return MOE_ERR_INVALID_ARG;
  L->wait_ns = (unsigned long long)ns;
  return MOE_OK;
}

moe_status moe_layer_get_nvfp4_act(moe_layer* L, int32_t T, uint8_t* codes, uint8_t* scales, float* amax,
                                   void* stream) {
  if (!L || T < 0 || T > L->cfg.max_tokens || !codes || !scales || !amax) return MOE_ERR_INVALID_ARG;
  if (!L->fp4_ok) return MOE_ERR_UNSUPPORTED;
  DeviceGuard g(L->device);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t rows = (size_t)T * L->cfg.top_k, H = (size_t)L->cfg.hidden;
  if (cudaMemcpyAsync(codes, L->xc, rows * (H / 2), cudaMemcpyDeviceToHost, s) ||
      cudaMemcpyAsync(scales, L->xsf, rows * (H / 16), cudaMemcpyDeviceToHost, s) ||
      cudaMemcpyAsync(amax, L->amax, sizeof(float), cudaMemcpyDeviceToHost, s))
    return MOE_ERR_CUDA;
  return cudaStreamSynchronize(s) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// Layers with host-resident experts: int4-g32 routed and shared experts without Q8_0, on
// the grouped tensor-core path, with a slot table that holds every expert.
static moe_status cached_layer_support(const moe_config* c) {
  if (c->weight_format != MOE_W_INT4_G32 || c->shared_format != MOE_W_INT4_G32 || c->act_quant != MOE_ACT_NONE ||
      !gemm_supported(c->hidden, c->inter) || c->n_experts + 1 > kMaxSlotTable)
    return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

static int cached_min_slots(const moe_config* c) {
  return (long)c->max_tokens * c->top_k < c->n_experts ? c->max_tokens * c->top_k : c->n_experts;
}

moe_status moe_cache_slots_for_memory(const moe_config* cfg, uint64_t budget_bytes, int32_t* slots) {
  if (!slots) return MOE_ERR_INVALID_ARG;
  *slots = 0;
  if (!cfg) return MOE_ERR_INVALID_ARG;
  moe_status st = validate_config(cfg);
  if (st || (st = cached_layer_support(cfg))) return st;
  const uint64_t per = gemm_pack_bytes(2 * cfg->inter, cfg->hidden, 1) + gemm_pack_bytes(cfg->hidden, cfg->inter, 1);
  const uint64_t fit = budget_bytes / per;   // routed slots + the shared expert's slot
  if (fit < (uint64_t)cached_min_slots(cfg) + 1) return MOE_ERR_OOM;
  *slots = fit - 1 > (uint64_t)cfg->n_experts ? cfg->n_experts : (int32_t)(fit - 1);
  return MOE_OK;
}

moe_status moe_layer_create_cached(const moe_config* cfg, const moe_weights* w, int32_t slots, void* stream,
                                   moe_layer** out) {
  if (!out) return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  if (!cfg || !w) return MOE_ERR_INVALID_ARG;
  moe_status st = validate_config(cfg);
  if (st) return st;
  if (slots < cached_min_slots(cfg) || slots > cfg->n_experts) return MOE_ERR_INVALID_ARG;
  if ((st = cached_layer_support(cfg))) return st;
  moe_layer* L = new (std::nothrow) moe_layer();
  if (!L) return MOE_ERR_OOM;
  L->cfg = *cfg;
  if (cudaGetDevice(&L->device) != cudaSuccess) {
    delete L;
    return MOE_ERR_CUDA;
  }
  st = create_impl(L, cfg, w, static_cast<cudaStream_t>(stream), slots);
  if (!st && !L->gemm_ok) st = MOE_ERR_UNSUPPORTED;
  if (st) {
    cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    cudaGetLastError();
    free_all(L);
    delete L;
    return st;
  }
  L->path = MOE_PATH_GROUPED;
  *out = L;
  return MOE_OK;
}

moe_status moe_layer_prefetch(moe_layer* L, const void* x, int32_t T, void* stream) {
  if (!L || T < 0 || T > L->cfg.max_tokens || (T > 0 && !x)) return MOE_ERR_INVALID_ARG;
  if (!L->cache) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  DeviceGuard g(L->device);
  const moe_config& c = L->cfg;
  const int E = c.n_experts, H = c.hidden;
  cudaStream_t cs = L->route_stream;
  // predict on the layer's routing stream (not behind the copies in flight), after x is
  // ready on the caller's stream; the loads then go out on the copy stream
  if (cudaEventRecord(L->ev_x, static_cast<cudaStream_t>(stream)) || cudaStreamWaitEvent(cs, L->ev_x, 0) ||
      cudaMemsetAsync(L->counts_p, 0, (size_t)(E + 1) * 4, cs) ||
      launch_router_logits(x, c.act_dtype, L->router_w, c.router_dtype, L->logits_p, T, E, H, cs) ||
      launch_select(L->logits_p, L->bias, T, E, c.n_group, c.topk_group, c.top_k, c.routed_scaling_factor,
                    c.expert_top_p, L->ids_p, L->weights_p, L->counts_p, L->status, cs) ||
      cudaMemcpyAsync(L->h_counts_p, L->counts_p, (size_t)E * 4, cudaMemcpyDeviceToHost, cs) ||
      cudaStreamSynchronize(cs))
    return MOE_ERR_CUDA;
  L->launches += 2;
  return L->cache->ensure(L->h_counts_p, true);
}

moe_status moe_layer_cache_pin_hot(moe_layer* L, int32_t n) {
  if (!L) return MOE_ERR_INVALID_ARG;
  if (!L->cache) return MOE_ERR_UNSUPPORTED;
  DeviceGuard g(L->device);
  const moe_config& c = L->cfg;
  const int need = (long)c.max_tokens * c.top_k < c.n_experts ? c.max_tokens * c.top_k : c.n_experts;
  return L->cache->pin_hot(n, need);
}

moe_status moe_layer_cache_stats(moe_layer* L, int64_t* stats) {
  if (!L || !stats) return MOE_ERR_INVALID_ARG;
  if (!L->cache) return MOE_ERR_UNSUPPORTED;
  for (int i = 0; i < ExpertCache::kNumStats; ++i) stats[i] = L->cache->stats()[i];
  return MOE_OK;
}

moe_status moe_layer_cache_query(moe_layer* L, int32_t* slot_of, int32_t* pinned) {
  if (!L || !slot_of || !pinned) return MOE_ERR_INVALID_ARG;
  if (!L->cache) return MOE_ERR_UNSUPPORTED;
  for (int e = 0; e < L->cfg.n_experts; ++e) {
    slot_of[e] = L->cache->slot_of(e);
    pinned[e] = L->cache->pinned(e) ? 1 : 0;
  }
  return MOE_OK;
}

moe_status moe_layer_set_debug_checks(moe_layer* L, int32_t on) {
  if (!L || (on != 0 && on != 1)) return MOE_ERR_INVALID_ARG;
  L->debug_checks = on;
  return MOE_OK;
}

moe_status moe_check_routing(const int32_t* ids, const int32_t* offsets, const int32_t* entries, int32_t T,
                             int32_t top_k, int32_t n_experts, int32_t* status, void* stream) {
  if (!ids || !offsets || !entries || !status || T <= 0 || top_k <= 0 || n_experts <= 0)
    return MOE_ERR_INVALID_ARG;
  return launch_check_routing(ids, offsets, entries, T, top_k, n_experts, status,
                              static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}

moe_status moe_test_fail_allocation(int32_t nth) {
  if (nth < 0) return MOE_ERR_INVALID_ARG;
  g_alloc_count.store(0);
  g_fail_alloc_at.store(nth);
  return MOE_OK;
}

moe_status moe_layer_set_test_activation(moe_layer* L, int32_t identity) {
  if (!L || (identity != 0 && identity != 1)) return MOE_ERR_INVALID_ARG;
  L->identity_act = identity;
  return MOE_OK;
}

moe_status moe_layer_reset_status(moe_layer* L, void* stream) {
  if (!L) return MOE_ERR_INVALID_ARG;
  DeviceGuard g(L->device);
  return cudaMemsetAsync(L->status, 0, sizeof(int), static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}

void moe_layer_destroy(moe_layer* L) {
  if (!L) return;
  {
    DeviceGuard g(L->device);
    cudaDeviceSynchronize();
    release_events(L);
    free_all(L);
  }
  delete L;
}

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_OOM: return "MOE_ERR_OOM";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    case MOE_ERR_DEVICE_CHECK: return "MOE_ERR_DEVICE_CHECK";
  }
  return "MOE_ERR_UNKNOWN";
}

}  // extern "C"
