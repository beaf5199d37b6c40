/*
 * moe_layer.h - C ABI of the B300 quantised routed-MoE layer forward.
 *
 * The layer is the one the colibri engine runs for GLM-5.2 ("Show HN: Menjalankan GLM 5.2
 * di komputer lambat", section "Fitur utama yang diimplementasikan"): a DeepSeek-V3-style
 * sigmoid router with noaux_tc bias-corrected grouped top-k, routed_scaling_factor and an
 * always-on shared expert; batch-union grouping, so each selected expert's weights are
 * read once per call and applied to every token routed to it (same section, and
 * "16 Teknik Özellik ve Yazılım Çıkarımları" of "Show HN: GLM 5.2 Modelini Yavaş
 * Bilgisayarımda Çalıştırmak"); weight-only quantised SwiGLU experts in packed int4
 * (one fp16 scale per 32 input-dim elements) or NVFP4 (E2M1 codes, an E4M3 scale per
 * 16 elements and an fp32 tensor scale: "NVIDIA stellt neues GLM-5.2 NVFP4 Modell vor",
 * section "Technische Details und Quantisierungsansatz"); and the weighted combine.
 *
 * out[t] = sum_j w[t,j] * FFN_{ids[t,j]}(x[t]) + FFN_shared(x[t])
 *   FFN_e(v) = W_d^e (SiLU(W_g^e v) * (W_u^e v))
 *   s = sigmoid(x W_r^T);  b = s + bias (selection only)
 *   group score = sum of the two largest b per group of E/n_group experts
 *   keep the topk_group best groups; ids = top_k largest b among kept experts
 *   w[t,j] = s[ids[t,j]] / sum_j s[ids[t,j]] * routed_scaling_factor
 * For NVFP4 layers the activations feeding the routed experts (x, and h before the
 * down projection) are themselves quantised to NVFP4 with a per-call fp32 tensor scale
 * (amax / (6*448)); a bf16 shared expert and the router read the unquantised x.
 *
 * All entry points return a moe_status and never abort the process. Device pointers
 * are CUDA device (or managed) addresses on the device that was current at create time;
 * "host" pointers may be pageable or pinned host memory. Streams are cudaStream_t passed
 * as void* (NULL = the legacy default stream).
 */
#ifndef MOE_LAYER_H
#define MOE_LAYER_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,   /* a NULL/misaligned pointer, a size out of range */
  MOE_ERR_UNSUPPORTED = 2,   /* a shape or format combination this build does not run */
  MOE_ERR_OOM = 3,           /* device or pinned-host allocation failed */
  MOE_ERR_CUDA = 4,          /* a CUDA runtime call failed (launch, copy, sync) */
  MOE_ERR_TIMEOUT = 5,       /* a bounded device-side wait gave up */
  MOE_ERR_DEVICE_CHECK = 6   /* a device-side consistency check failed */
} moe_status;

/* storage formats */
enum { MOE_W_INT4_G32 = 0, MOE_W_NVFP4 = 1, MOE_W_BF16 = 2, MOE_W_INT8_ROW = 3, MOE_W_INT4_ROW = 4,
       MOE_W_INT2_ROW = 5 };
/* Activations into the expert matmuls: as given, or Q8_0-style int8 (per 32 elements of a
 * row, step d = fp16(amax / 127), code = clamp(rint(v / d), -127, 127); x before gate/up and
 * h before down, routed and shared experts). */
enum { MOE_ACT_NONE = 0, MOE_ACT_Q8_0 = 1 };
/* activation / router element types */
enum { MOE_DT_F32 = 0, MOE_DT_BF16 = 1 };
/*
 * forward-path selection (moe_layer_set_path):
 *   MOE_PATH_GEMV     fused decode kernel (int4 layers, T <= 8, T * top_k <= 64)
 *   MOE_PATH_GROUPED  grouped tcgen05 tensor-core GEMMs (H, I multiples of 256)
 *   MOE_PATH_GENERIC  CUDA-core batch-union kernels (any supported shape; slow, kept as a
 *                     cross-check of the fast paths)
 *   MOE_PATH_AUTO     GEMV when it applies, else GROUPED when it applies, else GENERIC
 */
enum { MOE_PATH_AUTO = 0, MOE_PATH_GEMV = 1, MOE_PATH_GROUPED = 2, MOE_PATH_GENERIC = 3 };

/*
 * Limits checked by moe_layer_create (outside them: MOE_ERR_UNSUPPORTED; a size <= 0 or an
 * rsf not > 0: MOE_ERR_INVALID_ARG):
 *   hidden      multiple of 256, at most 14336 (the CUDA-core kernels stage 4 tokens of x
 *               in fp32 in shared memory)
 *   inter       multiple of 64
 *   n_experts   at most 1024, a multiple of n_group; n_group at most 32, and at least 2
 *               experts per group
 *   topk_group  at most n_group
 *   top_k       at most 32 and at most topk_group * n_experts / n_group (the fused decode
 *               path takes top_k <= 16 with T * top_k <= 64; other layers skip it)
 *   max_tokens  at most 16384, and the work list of the CUDA-core kernels fits 16 bits:
 *               floor(max_tokens * top_k / 4) + min(max_tokens * top_k, n_experts)
 *               + ceil(max_tokens / 4) + 1 <= 65535
 */
typedef struct {
  int32_t hidden;              /* H */
  int32_t inter;               /* I: per-expert intermediate size */
  int32_t n_experts;           /* E routed experts (the shared expert is extra) */
  int32_t top_k;               /* experts per token */
  int32_t n_group;             /* groups of E/n_group experts */
  int32_t topk_group;          /* groups kept per token */
  int32_t max_tokens;          /* largest T forward will be called with */
  float routed_scaling_factor; /* rsf */
  int32_t weight_format;       /* routed experts: MOE_W_INT4_G32 | MOE_W_NVFP4 | MOE_W_INT*_ROW */
  int32_t shared_format;       /* shared expert: the routed format, or MOE_W_BF16 */
  int32_t act_dtype;           /* x and out: MOE_DT_F32 | MOE_DT_BF16 */
  int32_t router_dtype;        /* W_r: MOE_DT_F32 | MOE_DT_BF16 */
  float expert_top_p;          /* adaptive expert top-p; 0 (or >= 1) = off, see below */
  int32_t act_quant;           /* MOE_ACT_NONE | MOE_ACT_Q8_0 (per-row integer or int4_g32
                                  layers whose shared expert is in the routed format) */
} moe_config;

/*
 * Per-row integer formats ("Show HN: Menjalankan GLM 5.2 di komputer lambat", section "Fitur
 * utama yang diimplementasikan": int8, packed int4, packed int2, scale per-row): codes
 * [rows, K * bits / 8] two's complement (int8 one per byte; int4 element 2j in the low
 * nibble of byte j; int2 element 4j + i in bits 2i..2i+1 of byte j) and one fp32 scale per
 * row ([rows, 1]); w = code * scale. They and MOE_ACT_Q8_0 run on the CUDA-core batch-union
 * kernels (MOE_PATH_GENERIC; AUTO picks it, GEMV and GROUPED are MOE_ERR_UNSUPPORTED).
 */

/*
 * Adaptive expert top-p (the "--topp" option of "Show HN: Menjalankan GLM 5.2 di komputer
 * lambat", section "Mengunduh model dan menjalankannya": fewer experts per token, less
 * expert data read). With 0 < expert_top_p < 1, each token's top_k selected experts are
 * ordered by their unbiased score s (largest first, equal scores lower id first) and the
 * shortest prefix whose summed s reaches expert_top_p times the summed s of all top_k is
 * kept (an expert stays while the mass ranked before it is below that). The kept weights
 * are renormalised to routed_scaling_factor; a dropped slot reads id -1 and weight 0 in
 * moe_layer_get_routing and has no entry in the grouping (offsets[E] = the kept count).
 * Decisions within fp32 rounding of the threshold may differ from an fp64 evaluation.
 * A NaN value is MOE_ERR_INVALID_ARG.
 */

/*
 * Layer weights, read once by moe_layer_create (host or device memory, contiguous,
 * row-major). Routed arrays are stacked over the E experts:
 *   router_w  [E, H]           fp32 or bf16 (router_dtype)
 *   bias      [E]              fp32 e_score_correction_bias
 *   gu_codes  [E, 2I, H/2]     uint8; rows 0..I-1 gate, I..2I-1 up; element 2j in the
 *                              low nibble of byte j (int4: two's complement; NVFP4: E2M1)
 *   gu_scales [E, 2I, H/32]    fp16 (int4_g32)  |  [E, 2I, H/16] uint8 E4M3 (NVFP4)
 *   gu_tscale [E]              fp32 tensor scale (NVFP4 only, else NULL)
 *   d_codes   [E, H, I/2], d_scales [E, H, I/32 | I/16], d_tscale [E]  (down projection)
 * The shared expert uses the sh_* fields with the same layouts and no leading E
 * dimension; for MOE_W_BF16, sh_gu is [2I, H] bf16, sh_d is [H, I] bf16 and the scale
 * fields are NULL.
 */
typedef struct {
  const void* router_w;
  const float* bias;
  const uint8_t* gu_codes;
  const void* gu_scales;
  const float* gu_tscale;
  const uint8_t* d_codes;
  const void* d_scales;
  const float* d_tscale;
  const void* sh_gu;
  const void* sh_gu_scales;
  const float* sh_gu_tscale;
  const void* sh_d;
  const void* sh_d_scales;
  const float* sh_d_tscale;
} moe_weights;

typedef struct moe_layer moe_layer;

/*
 * Create a layer on the current CUDA device. Copies (and repacks) the weights into
 * library-owned device memory and allocates the workspace for cfg->max_tokens tokens;
 * the caller may free its weight buffers when this returns. Work is enqueued on
 * `stream` and completed before return.
 * Errors: MOE_ERR_INVALID_ARG (NULL pointer, bad sizes), MOE_ERR_UNSUPPORTED (shape or
 * format outside the limits documented in moe_config), MOE_ERR_OOM, MOE_ERR_CUDA.
 * On error *out is set to NULL and nothing is leaked.
 */
moe_status moe_layer_create(const moe_config* cfg, const moe_weights* w, void* stream,
                            moe_layer** out);

/*
 * out[T, H] = layer(x[T, H]); x and out are device pointers in act_dtype, row-major,
 * 16-byte aligned, not overlapping. 0 <= T <= max_tokens (T = 0 is a no-op).
 * Asynchronous on `stream`: no host synchronisation, no allocation, capturable in a
 * CUDA graph (a layer made by moe_layer_create_cached is the exception: see there). Not
 * thread-safe per layer (the workspace is shared by calls).
 * Routing results stay on the device; moe_layer_get_routing copies them out.
 * Errors, returned before or while enqueueing: MOE_ERR_INVALID_ARG (NULL layer, x or out,
 * a pointer not 16-byte aligned, x == out, T out of range); MOE_ERR_UNSUPPORTED when the
 * path forced by moe_layer_set_path does not apply to this layer or T; MOE_ERR_CUDA when a
 * launch or copy fails to enqueue; for a cached layer also the cache's errors. Device-side
 * failures (check violations, wait time-outs) are reported by moe_layer_status.
 */
moe_status moe_layer_forward(moe_layer* layer, const void* x, int32_t T, void* out, void* stream);

/*
 * Same computation with HOST buffers: copies x_host (T*H elements of act_dtype) to the
 * device, runs the forward and copies the result into out_host, then synchronises
 * `stream`. Uses the layer's own device staging buffers (allocated at create); the caller
 * keeps ownership of both host buffers, which may be pageable or pinned.
 * Errors: MOE_ERR_INVALID_ARG (NULL layer, T out of range, NULL x_host or out_host with
 * T > 0); the errors of moe_layer_forward; MOE_ERR_CUDA when a copy or the synchronisation
 * fails (a device-side failure of this forward surfaces here or in moe_layer_status).
 */
moe_status moe_layer_forward_host(moe_layer* layer, const void* x_host, int32_t T,
                                  void* out_host, void* stream);

/*
 * Copy the routing of the last forward (called with the same T) to host memory and
 * synchronise `stream`. Any output pointer may be NULL to skip it; the buffers are the
 * caller's. Errors: MOE_ERR_INVALID_ARG (NULL layer, T outside [0, max_tokens]),
 * MOE_ERR_CUDA (a copy or the synchronisation failed).
 *   ids     [T, top_k] int32 selected experts (slot order: descending biased score)
 *   weights [T, top_k] fp32 combine weights
 *   offsets [E + 1]    int32 exclusive scan of per-expert counts
 *   entries [T * top_k] int32 token*top_k + slot, grouped by expert, ascending token
 */
moe_status moe_layer_get_routing(moe_layer* layer, int32_t T, int32_t* ids, float* weights,
                                 int32_t* offsets, int32_t* entries, void* stream);

/* Force the expert path (MOE_PATH_*) for later forwards; AUTO picks by T and shape. A
 * forced path that does not apply to a forward makes it return MOE_ERR_UNSUPPORTED.
 * Errors: MOE_ERR_INVALID_ARG (NULL layer, a value outside MOE_PATH_*). */
moe_status moe_layer_set_path(moe_layer* layer, int32_t path);

/*
 * Synchronise the device and report the sticky device-side status word (MOE_OK,
 * MOE_ERR_TIMEOUT or MOE_ERR_DEVICE_CHECK) plus any pending CUDA error (MOE_ERR_CUDA).
 * MOE_ERR_INVALID_ARG for a NULL layer. The word stays set until moe_layer_reset_status.
 */
moe_status moe_layer_status(moe_layer* layer);

/*
 * Stage timing (for measurement): with enable = N > 0 the layer creates N x 8 CUDA
 * events and each of the next N forwards records 8 events on its stream at the stage
 * boundaries: start | routing (router logits, selection, grouping) | activation staging
 * (NVFP4 quantise, expert-sorted rows) | routed gate/up + SwiGLU (with a shared expert
 * stored in the routed format: it too; the fused decode kernel: the whole layer) |
 * separately stored shared expert's gate/up | h quantise (NVFP4) | down + combine |
 * output conversion |.
 * Events recorded while the stream is being captured become graph nodes and are timed
 * on replay. enable = 0 releases the events. Errors: MOE_ERR_INVALID_ARG (NULL layer,
 * enable < 0), MOE_ERR_CUDA (an event could not be created; none are kept then).
 */
moe_status moe_layer_enable_timing(moe_layer* layer, int32_t enable);

/*
 * Synchronise the device, then write into ms[0..6] the summed durations (milliseconds)
 * of the 7 stages over the forwards recorded since timing was enabled (or last read),
 * and their number into *n_forwards (which may be NULL); resets the record count. An empty
 * stage reads 0. ms is the caller's, 7 floats. Errors: MOE_ERR_INVALID_ARG (NULL layer or
 * ms), MOE_ERR_CUDA (the synchronisation or an event query failed).
 */
moe_status moe_layer_stage_times(moe_layer* layer, float* ms, int32_t* n_forwards);

/*
 * Profiling hook. With a device buffer of n_ctas x 64 uint64 (n_ctas >= the device's SM
 * count), later forwards write per-CTA records into buffer[cta * 64 + slot]:
 *  - fused decode kernel: %globaltimer stamps (ns) at its phase boundaries in slots 0 start,
 *    2 this CTA's router rows written, 3 every CTA's router rows seen, 7 selection done,
 *    15 routing published, 4 / 5 / 6 epilogue done with the shared gate/up / routed gate/up /
 *    shared down units, 12 all units done, 13 producer done issuing, 14 MMA warp done
 *    (tensor mode); clock-cycle counters in slots 16..28 (decoders: waiting for item data,
 *    for an accumulator or hand-off slot, busy, items; MMA warp (tensor mode): waiting for A,
 *    for an accumulator, h staging, units; epilogue: waiting, busy, last-arriver work;
 *    producer: waiting for a slot, items issued), 29 / 30 the epilogue thread's clock64 at
 *    slots 0 and 12 (their ratio to the ns stamps is the SM clock), 31 units, 32 h stager
 *    waiting, 33 / 34 MMA issue / loop cycles, 35 / 36 / 37 decoders waiting for the routing,
 *    for an expert's h, loop total;
 *  - grouped fp16/int4 GEMMs (the FP4 kernel writes none), slots 16..26 (gate/up), 32..42
 *    (down), 48..58 (separately stored
 *    shared expert, gate/up), clock cycles: +0 kernel, +1 MMA waiting for operands, +2 MMA
 *    waiting for an accumulator, +3 dequantiser waiting for weights, +4 dequantiser waiting
 *    for a free stage, +5 activation producer waiting, +6 weight producer waiting, +7
 *    epilogue waiting, +8 epilogue busy, +9 tiles, +10 dequantiser loop.
 * buffer = NULL switches it off (the default). The buffer stays the caller's and must stay
 * valid while traced forwards run. Errors: MOE_ERR_INVALID_ARG (NULL layer, n_ctas < 0, or
 * a buffer with n_ctas below the SM count).
 */
moe_status moe_layer_set_trace(moe_layer* layer, void* buffer, int32_t n_ctas);

/* Cumulative number of kernel launches this layer has issued (host-side count; a forward
 * captured into a CUDA graph counts once at capture). MOE_ERR_INVALID_ARG for a NULL layer
 * or count. */
moe_status moe_layer_launch_count(moe_layer* layer, int64_t* count);

/*
 * Failure-handling hook. Every device-side wait on work of other CTAs (the fused decode
 * kernel's router-row and gate/up completion counters; the grouped GEMM's pipeline waits)
 * gives up after `ns` nanoseconds (default 2e9), sets MOE_ERR_TIMEOUT in the layer's status
 * word, lets the copies and tensor-core operations it issued land, frees its tensor memory
 * and returns; the forward's output is then undefined. ns = 0 makes every such wait that is
 * not already satisfied give up at once, which exercises that path without a GPU fault.
 * ns < 0 is MOE_ERR_INVALID_ARG. Later forwards start from a clean state.
 */
moe_status moe_layer_set_wait_limit(moe_layer* layer, int64_t ns);

/*
 * Debug checks (a sanitizer substitute): with on = 1 every later forward checks its routing
 * on the device after the grouping: ids in [-1, E), offsets starting at 0, never decreasing
 * and ending at the number of routed slots (at most T * top_k), each entry of expert e's
 * range naming a slot whose id is e, tokens strictly ascending in each range. A violation
 * sets MOE_ERR_DEVICE_CHECK in the status word (moe_layer_status); nothing traps.
 * moe_check_routing runs the same checks on caller DEVICE arrays ids [T * top_k], offsets
 * [n_experts + 1], entries [T * top_k] and raises MOE_ERR_DEVICE_CHECK in the caller's
 * device int *status (enqueued on `stream`); the checks read only inside those arrays.
 */
moe_status moe_layer_set_debug_checks(moe_layer* layer, int32_t on);
moe_status moe_check_routing(const int32_t* ids, const int32_t* offsets, const int32_t* entries,
                             int32_t T, int32_t top_k, int32_t n_experts, int32_t* status,
                             void* stream);

/*
 * Test hook: after this call the nth device or host allocation made by the library fails
 * with MOE_ERR_OOM (nth = 0 switches it off; counting restarts at each call). Creation
 * then returns MOE_ERR_OOM and releases everything it had allocated.
 */
moe_status moe_test_fail_allocation(int32_t nth);

/*
 * Test-only: identity = 1 makes every path compute h = gate * up instead of SiLU(gate) * up
 * for later forwards (0 restores SiLU). It exists so that inputs chosen for exact
 * arithmetic (small integers, power-of-two scales) give outputs that an exact evaluation of
 * the same formula reproduces bit for bit. Anything but 0 or 1 is MOE_ERR_INVALID_ARG.
 */
moe_status moe_layer_set_test_activation(moe_layer* layer, int32_t identity);

/* Clear the sticky device status word (enqueued on `stream`). */
moe_status moe_layer_reset_status(moe_layer* layer, void* stream);

/*
 * Host-resident experts with an HBM cache ("Cara kerja eksekusi MoE berbasis streaming disk"
 * in "Show HN: Menjalankan GLM 5.2 di komputer lambat": a per-layer LRU cache of experts over
 * slower storage, an optional pinned hot store learned from usage counts; "Yönlendirici
 * İleriye Dönük Ön-Getirme" in "Show HN: GLM 5.2 Modelini Yavaş Bilgisayarımda
 * Çalıştırmak": the router predicts the next layer's experts so their loads start early).
 *
 * moe_layer_create_cached: like moe_layer_create, but the routed experts stay in pinned host
 * memory (the library's copy, in the tensor-core path's packed layout) and HBM holds `slots`
 * of them; the shared expert stays in HBM. Requires int4_g32 routed and shared experts, no
 * act_quant, H and I multiples of 256, and min(E, max_tokens * top_k) <= slots <= E
 * (MOE_ERR_INVALID_ARG otherwise for slots, MOE_ERR_UNSUPPORTED for the rest). Forwards on
 * the layer run the grouped tensor-core path (GEMV and GENERIC are MOE_ERR_UNSUPPORTED): the
 * routing runs on `stream`, the host reads the routed experts back (a synchronisation of
 * `stream`; such forwards cannot be captured into a CUDA graph), the missing ones are copied
 * into slots on the layer's copy stream (least recently used, unpinned experts that the call
 * does not need are evicted), and the expert kernels wait for those copies. Use one stream
 * for a cached layer's forwards and prefetches.
 *
 * moe_cache_slots_for_memory: the largest number of expert slots (at most n_experts) whose
 * HBM store, the shared expert's slot included, fits in budget_bytes for a layer that
 * moe_layer_create_cached accepts with this configuration: the sizing step of the expert
 * cache that "Fitur utama yang diimplementasikan" of "Show HN: Menjalankan GLM 5.2 di
 * komputer lambat" describes (the cache sized at start-up from the memory available). The
 * budget is the caller's share of free device memory for this layer's experts (for
 * instance cudaMemGetInfo's free bytes less the layers' workspaces, divided among the
 * layers of a stack). Host arithmetic only, no CUDA call. Errors: MOE_ERR_INVALID_ARG (a
 * NULL pointer, or a configuration moe_layer_create refuses as such), MOE_ERR_UNSUPPORTED
 * (a configuration moe_layer_create_cached does not take), MOE_ERR_OOM (the budget holds
 * fewer than min(n_experts, max_tokens * top_k) + 1 slots); *slots is 0 on any error.
 *
 * moe_layer_prefetch: predict the experts of x [T, H] (device, act_dtype) with this layer's
 * router on a routing stream of the layer's own (after the work already on `stream`; the
 * host waits for this routing only) and start loading the missing ones on the copy stream,
 * without waiting for the copies. For a stack of layers: prefetch layer l + 1 with layer l's
 * input before running layer l. Uses a routing workspace of its own.
 *
 * moe_layer_cache_pin_hot: pin the n experts most often routed so far (ties: lower id),
 * loading them if needed; pinned experts are never evicted; a new call replaces the pins.
 * MOE_ERR_INVALID_ARG if fewer than min(E, max_tokens * top_k) slots would stay unpinned.
 *
 * moe_layer_cache_stats: stats[0..5] = expert hits, misses, experts loaded by prefetch,
 * prefetched experts later used, bytes copied host -> device, evictions.
 * moe_layer_cache_query: slot_of[e] (-1 if not in HBM) and pinned[e] (0/1) for the E routed
 * experts, into host arrays.
 * All four return MOE_ERR_UNSUPPORTED on a layer created without a cache.
 */
moe_status moe_layer_create_cached(const moe_config* cfg, const moe_weights* w, int32_t slots,
                                   void* stream, moe_layer** out);
moe_status moe_cache_slots_for_memory(const moe_config* cfg, uint64_t budget_bytes, int32_t* slots);
moe_status moe_layer_prefetch(moe_layer* layer, const void* x, int32_t T, void* stream);
moe_status moe_layer_cache_pin_hot(moe_layer* layer, int32_t n);
moe_status moe_layer_cache_stats(moe_layer* layer, int64_t* stats);
moe_status moe_layer_cache_query(moe_layer* layer, int32_t* slot_of, int32_t* pinned);

/*
 * Inspection of the NVFP4 activation quantiser ("NVIDIA stellt neues GLM-5.2 NVFP4 Modell
 * vor", section "Technische Details und Quantisierungsansatz": E2M1 elements, one E4M3 scale
 * per 16 elements, an fp32 tensor scale). After a forward of T tokens that ran the grouped
 * path of an NVFP4 layer whose shared expert is stored separately (the layers that use the
 * block-scaled FP4 tensor cores), copies to HOST buffers, synchronously on `stream`:
 *   codes  [T * top_k, hidden / 2] uint8: the expert-sorted routed rows (row q is token
 *          entries[q] / top_k of moe_layer_get_routing), element 2j in the low nibble of
 *          byte j;
 *   scales [T * top_k, hidden / 16] uint8: the E4M3 scale of each 16-element block;
 *   amax   one float: the amax of |x| over the call; the tensor scale is amax / 2688.
 * The caller owns the buffers. Other layers return MOE_ERR_UNSUPPORTED; T outside
 * [0, max_tokens] or a NULL pointer is MOE_ERR_INVALID_ARG. T must be the last forward's T
 * (the contents are otherwise unspecified).
 */
moe_status moe_layer_get_nvfp4_act(moe_layer* layer, int32_t T, uint8_t* codes, uint8_t* scales,
                                   float* amax, void* stream);

/*
 * Routing without any allocation. The pages have no counterpart to this entry point: it
 * exists for callers that cannot call cudaMalloc when they need routing (code running
 * while a stream is captured into a CUDA graph, where allocation is not capturable; hosts
 * whose framework owns the device memory budget; runtimes that forbid allocation after
 * start-up). It computes the routing of moe_layer_forward + moe_layer_get_routing from
 * caller-owned DEVICE buffers, with the same selection and grouping kernels; the logits
 * come from the CUDA-core router kernels. Those add in another order than the tensor-core
 * router that a layer uses for bf16 activations. So the selections agree except where two
 * biased scores lie within fp32 rounding of each other. Inputs and outputs:
 *   x [T, H] (act_dtype), router_w [E, H] (router_dtype), bias [E] fp32
 *   -> ids [T, top_k] int32, weights [T, top_k] fp32, offsets [E + 1] int32,
 *      entries [T * top_k] int32 (layouts as in moe_layer_get_routing).
 * The kernels' scratch (logits, histogram, work list, status word) lives in one
 * file-scope __device__ array of about 1.04 MiB that every device loading the library
 * holds until the process exits. Checks, all made before any work is enqueued:
 *   MOE_ERR_INVALID_ARG: T < 0, H <= 0, E, n_group, topk_group or top_k <= 0, an unknown
 *     act_dtype or router_dtype, routed_scaling_factor not > 0, a NULL pointer (T > 0),
 *     x or router_w not 16-byte aligned, bias, ids, weights, offsets or entries not
 *     4-byte aligned;
 *   MOE_ERR_UNSUPPORTED: E > 1024, n_group > 32 or not dividing E, fewer than 2 experts
 *     per group, topk_group > n_group, top_k > topk_group * E / n_group or > 32, and the
 *     scratch limits T * E <= 262144 and T * top_k / 4 + min(T * top_k, E) + 1 <= 8192.
 * T = 0 returns MOE_OK and does nothing. Scores that are not finite (a NaN or infinite
 * logit) give an unspecified selection: the selection kernel's check word stays in the
 * scratch array and is not reported by this entry point.
 * The first call on a device looks up the array's device address (once per device, with
 * that device current) and caches it for the life of the process; make that first call
 * before any stream capture, and make no call after cudaDeviceReset on that device (the
 * cached address would be stale). Every call shares the one array: calls whose work
 * overlaps on the GPU (different streams, or concurrent host threads) race on it and must
 * be serialised by the caller. Asynchronous on `stream`; no host synchronisation.
 */
moe_status moe_route_noalloc(const void* x, int32_t act_dtype, int32_t T, int32_t H,
                             const void* router_w, int32_t router_dtype, const float* bias,
                             int32_t E, int32_t n_group, int32_t topk_group, int32_t top_k,
                             float routed_scaling_factor, int32_t* ids, float* weights,
                             int32_t* offsets, int32_t* entries, void* stream);

/* Free everything the layer owns. NULL is a no-op. */
void moe_layer_destroy(moe_layer* layer);

/* Static string naming a status code. */
const char* moe_status_string(moe_status status);

#ifdef __cplusplus
}
#endif

#endif /* MOE_LAYER_H */
