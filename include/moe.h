/*
 * moe.h -- C ABI of the GB300 routed Mixture-of-Experts FFN layer.
 *
 * What a layer computes (the hot path of the local-inference engines
 * described in "nano-cuda-moe-qwen38" -- memory-hierarchy and prefill
 * paragraphs --, "cyber-on-strata" -- two-tier memory section -- and the
 * Strata / Project Maya page -- "MoE architecture and hierarchical caching"
 * and "Strata tiers" sections): per token,
 *   z   = W_r x + b                       router logits (fp32 weights)
 *   S   = top-k of z (ties: lower id)     the experts that run
 *   w   = softmax of z over S             routing weights, sum to 1
 *   y   = sum_{e in S} w_e FFN_{slot(e)}(x) + FFN_shared(x)
 *   FFN(x) = W_d (silu(W_g x) * (W_u x))  SwiGLU expert
 * Routing variants (moe_layer_config.routing_flags, all off by default):
 *   MOE_ROUTING_NO_RENORM       w_e = softmax over all E logits, taken at
 *                               the selected experts (sums to less than 1)
 *   MOE_ROUTING_BIAS_SELECT_ONLY the bias b enters the selection only: S is
 *                               the top-k of W_r x + b, the weights use the
 *                               logits W_r x without b
 *   MOE_ROUTING_SHARED_GATE     the shared expert is scaled per token by
 *                               sigmoid(g . x), g = sh_gate_w [H] fp32
 * Every expert is reached through a slot table (the pages' VRAM expert
 * cache).  By default every expert has a slot in HBM (n_slots == n_experts);
 * with n_slots < n_experts only n_slots experts per layer stay in HBM, the
 * rest in a library-owned pinned host tier (the pages' RAM tier) read by
 * the GPU over the host link: see moe_layer_config.n_slots.  Expert weights are
 * symmetric 4-bit codes in blocks of 32 along the reduction dimension with
 * one binary16 scale per block (the block-scale idea of the pages' int8 KV
 * cache, one scale per 32 values): weight = (nibble - 8) * scale.
 *
 * Conventions for every entry point:
 *  - No C++ exceptions cross this boundary; errors are moe_status codes and
 *    a thread-local message from moe_last_error().
 *  - All work is asynchronous on the given CUDA stream (a cudaStream_t
 *    passed as void*, NULL = legacy default stream), except where stated.
 *  - Activation pointers (x, y, ids, weights) may be device pointers or host
 *    pointers (pinned or pageable).  Host inputs are copied into library
 *    buffers on the stream; when an output is a host pointer the call copies
 *    it back and synchronises the stream before returning.  Exception: in
 *    moe_forward and moe_stack_forward with at most 4 tokens, a pinned
 *    (page-locked, device-mapped) x with 16-byte alignment is read by the
 *    kernels in place and a pinned y is written in place, without staging
 *    copies; such an x, like the source of a stream-ordered copy, must stay
 *    unchanged until the stream reaches the call, and the call still
 *    synchronises before returning when y is a host pointer.
 *  - The library owns all device memory it uses (weights and workspaces are
 *    allocated in moe_layer_create); no other call allocates device memory.
 *  - Calls that use the same layer object must not run concurrently (they
 *    share its workspace); stack calls use the first layer's workspace.
 */
#ifndef MOE_GB300_MOE_H
#define MOE_GB300_MOE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct moe_layer moe_layer; /* opaque, owned by the library */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID = -1,  /* bad argument, config or weight table */
  MOE_ERR_CUDA = -2,     /* a CUDA runtime call failed */
  MOE_ERR_OOM = -3,      /* device allocation failed (create only) */
  MOE_ERR_CAPACITY = -4, /* n_tokens outside [1, max_tokens] */
  MOE_ERR_BOUNDS = -5,   /* a kernel met an out-of-range slot or non-finite logits */
  MOE_ERR_TIMEOUT = -6   /* a bounded device-side wait ran out */
} moe_status;

/* Routing variant bits for moe_layer_config.routing_flags; combinations are
 * allowed (MOE_ROUTING_SHARED_GATE needs shared_ffn > 0). */
enum {
  MOE_ROUTING_NO_RENORM = 1,
  MOE_ROUTING_BIAS_SELECT_ONLY = 2,
  MOE_ROUTING_SHARED_GATE = 4
};

/* Layer shape.  Limits: hidden % 128 == 0 and 128 <= hidden <= 8192;
 * 1 <= n_experts <= 1024; 1 <= top_k <= min(16, n_experts);
 * ffn % 128 == 0 and 128 <= ffn <= 4096; shared_ffn == 0 or a multiple of
 * 128 up to 4096; min(n_experts, 4 * top_k) <= n_slots <= n_experts;
 * 1 <= max_tokens <= 65536 (sizes the workspaces: above 4 tokens the
 * prefill workspace takes about 2 * max_tokens * ((top_k + 2) * hidden +
 * top_k * ffn + shared_ffn) bytes, 0.6 GB at 8192 tokens of a hidden 2048,
 * top-10, ffn 768 layer); routing_flags a
 * combination of the MOE_ROUTING_* bits (0: the default routing above).
 * moe_layer_create also refuses shapes whose single-token decode does not
 * fit the decode kernel's 227 KB of shared memory (one 16-row gate/up stage
 * is 18 * hidden bytes, so hidden = 8192 does not fit); a 2..4-token call
 * whose batch does not fit returns MOE_ERR_INVALID. */
typedef struct {
  int32_t hidden;     /* H */
  int32_t n_experts;  /* E */
  int32_t top_k;      /* k */
  int32_t ffn;        /* F: routed expert intermediate size */
  int32_t shared_ffn; /* Fs: shared expert intermediate size, 0 = none */
  int32_t n_slots;    /* S: expert-cache slots in HBM (see below) */
  int32_t max_tokens; /* largest n_tokens any call will pass */
  int32_t routing_flags; /* MOE_ROUTING_* bits */
} moe_layer_config;
/* Partial residency (n_slots < n_experts).  A copy of every expert stays in
 * pinned host memory owned by the library; n_slots experts also hold an HBM
 * slot, first the n_slots with the largest moe_layer_weights.expert_profile
 * values (ties: lower id; no profile: experts 0..n_slots-1).  Single-layer
 * and stack calls on 1..4 tokens look each selected expert up; a miss is
 * served in the same call: the layer's CTAs read the expert from the host
 * tier over the host link into the least recently used slot that this call
 * does not use (so the cache evolves with the traffic), then the layer
 * proceeds from HBM; results are the same as with every expert resident.
 * Larger batches (the prefill path) stream the experts their tokens select
 * from HBM slots or the host tier into a staging buffer shared by the
 * partially resident layers of the process (one layer's worth of experts),
 * then run as usual; calls on partially resident layers must not overlap on
 * the GPU.  moe_cache_stats reports hits and misses. */

/* Packed weights, all row-major with the reduction dimension contiguous.
 * A packed row of K weights is K/2 bytes of codes (byte i holds element 2i
 * in its low nibble and element 2i+1 in its high nibble) and K/32 binary16
 * scales (raw bits).  Routed tensors hold all E experts, expert e in row
 * slot_of_expert[e]:
 *   gate_q, up_q  [E][F][H/2]   gate_s, up_s  [E][F][H/32]
 *   down_q        [E][H][F/2]   down_s        [E][H][F/32]
 *   sh_gate_q, sh_up_q [Fs][H/2], sh_*_s [Fs][H/32]
 *   sh_down_q [H][Fs/2], sh_down_s [H][Fs/32]        (NULL when Fs == 0)
 *   router_w [E][H] fp32, router_bias [E] fp32 or NULL (zero bias)
 *   slot_of_expert [E]: a permutation of 0..E-1 (validated at create)
 *   sh_gate_w [H] fp32: shared-expert gate vector, read only with
 *   MOE_ROUTING_SHARED_GATE (NULL otherwise)
 *   expert_profile [E] fp32 or NULL: expected use of each expert, read only
 *   with n_slots < n_experts to choose the experts first placed in HBM. */
typedef struct {
  const float* router_w;
  const float* router_bias;
  const int32_t* slot_of_expert;
  const uint8_t* gate_q;
  const uint16_t* gate_s;
  const uint8_t* up_q;
  const uint16_t* up_s;
  const uint8_t* down_q;
  const uint16_t* down_s;
  const uint8_t* sh_gate_q;
  const uint16_t* sh_gate_s;
  const uint8_t* sh_up_q;
  const uint16_t* sh_up_s;
  const uint8_t* sh_down_q;
  const uint16_t* sh_down_s;
  const float* sh_gate_w;
  const float* expert_profile;
} moe_layer_weights;

/* Creates a layer: validates cfg and the slot table, allocates the layer's
 * HBM (weights + workspaces) and copies the weights in.  weights_on_device
 * = 1: every pointer in w is a device pointer, 0: host pointers.  The caller
 * keeps ownership of its buffers and may free them after the call returns
 * (the call synchronises the device).  On success *out owns everything and
 * must be released with moe_layer_destroy. */
moe_status moe_layer_create(const moe_layer_config* cfg, const moe_layer_weights* w,
                            int weights_on_device, moe_layer** out);

/* Frees a layer (NULL is a no-op).  Synchronises the device first. */
void moe_layer_destroy(moe_layer* layer);

/* Router + top-k only.  x_bf16 [T][H] (bf16 bits); outputs topk_ids [T][k]
 * (logical expert ids, descending selection logit, ties to the lower id) and
 * topk_w [T][k] (softmax over the selected logits, or as routing_flags
 * say). */
moe_status moe_route(moe_layer* layer, const void* x_bf16, int n_tokens, int32_t* topk_ids,
                     float* topk_w, void* stream);

/* One layer: y_bf16 [T][H] = layer(x_bf16 [T][H]).  x and y must not
 * overlap.  n_tokens <= 4 runs the decode path (fused dequant GEMVs);
 * larger batches run the prefill path (bucketed grouped GEMM on tcgen05),
 * whose results are bit-identical from call to call (each expert's
 * weighted rows are summed per token in one fixed order). */
moe_status moe_forward(moe_layer* layer, const void* x_bf16, int n_tokens, void* y_bf16,
                       void* stream);

/* Pre-norm residual stack: h_0 = x and, for l = 0..L-1,
 *   u_l     = bf16(h_l / sqrt(mean(h_l^2) + 1e-6))   (RMS norm, unit gain)
 *   h_{l+1} = bf16(h_l + bf16(layer_l(u_l)))
 * y = h_L.  The norm keeps the stack finite: without it the SwiGLU output,
 * which grows with the square of its input, makes a deep residual stack of
 * these layers diverge.  All layers must share one shape.  x == y is
 * allowed. */
moe_status moe_stack_forward(moe_layer* const* layers, int n_layers, const void* x_bf16,
                             int n_tokens, void* y_bf16, void* stream);

/* moe_stack_forward that also records, for every pointer that is not NULL
 * (device memory only): h_trace [L][T][H] = h_{l+1}, in_trace [L][T][H] =
 * u_l, y_trace [L][T][H] = bf16(layer_l(u_l)) (all bf16 bits), ids_trace
 * [L][T][k] = each layer's top-k ids. */
moe_status moe_stack_forward_traced(moe_layer* const* layers, int n_layers, const void* x_bf16,
                                    int n_tokens, void* y_bf16, void* h_trace_bf16,
                                    void* in_trace_bf16, void* y_trace_bf16, int32_t* ids_trace,
                                    void* stream);

/* Allocation-free decode of one layer (1..4 tokens), for callers that
 * cannot allocate device memory when they need a layer evaluated: code
 * that runs while a CUDA graph is being captured into a memory pool it does
 * not own, plug-ins hosted by a framework whose allocator is the only one
 * allowed to call cudaMalloc, and processes held to a fixed device-memory
 * budget after start-up.  The pages have no counterpart of this entry point.
 * Computes y = layer(x) like moe_forward, but from the caller's weights
 * (layout as in moe_layer_weights, n_slots == n_experts, router_bias
 * required).  Every pointer must be device memory of the current device
 * (or managed memory): the weights, router_w, slot_of_expert and
 * sh_gate_w 16-byte aligned, x [n_tokens][H] bf16 16-byte aligned,
 * router_bias and status_out 4-byte aligned; anything else returns
 * MOE_ERR_INVALID before any work is queued, as do shapes outside the
 * moe_layer_create limits.  All the scratch memory the kernel needs comes
 * from one static 128 KiB device array inside the library, present on every
 * GPU that loads it until the process exits; shapes whose scratch would not
 * fit (8 * hidden * 4 bytes of output accumulators plus 16 * n_experts
 * bytes of logits and about 1 KB more: hidden 2048 fits, hidden 4096 does
 * not) return MOE_ERR_CAPACITY.  No call allocates or frees device memory.
 * The first call on each device looks up the array's device address with
 * that device current: make it before any stream capture.  Every call
 * shares the array, so calls that overlap on the GPU (other streams, other
 * host threads) race on it.  status_out (optional, device int32) is zeroed,
 * then receives any error a kernel records (MOE_ERR_TIMEOUT, MOE_ERR_BOUNDS);
 * without it such an error goes to a scratch word that no call reads, so a
 * failed kernel leaves a wrong y unreported.  The slot table is only
 * bounds-checked by the kernel.  Asynchronous on `stream`; the bounded
 * waits use the MOE_WAIT_TIMEOUT_US limit of the other calls. */
moe_status moe_forward_noalloc(const moe_layer_config* cfg, const moe_layer_weights* w,
                               const void* x_bf16, int n_tokens, void* y_bf16,
                               int32_t* status_out, void* stream);

/* Introspection of the prefill path's token bucketing: after a moe_forward
 * or moe_route call with n_tokens > 4 on this layer, copies the bucket
 * offsets [E+1] (exclusive scan of the per-expert counts; offsets[E] = T*k)
 * and the token of every bucketed row [T*k] (rows sorted by expert, then by
 * token).  Host or device pointers; synchronises the stream.  n_tokens must
 * be the batch of that call. */
moe_status moe_last_buckets(moe_layer* layer, int n_tokens, int32_t* offsets, int32_t* perm_token,
                            void* stream);

/* Expert-cache statistics of a layer (synchronises `stream`): *hits and
 * *misses count the routed-expert lookups of the decode path (1..4-token
 * calls) since creation or the last reset (reset != 0 zeroes them after
 * reading); with every expert resident every lookup is a hit.
 * slot_of_expert (host pointer, [E], or NULL) receives the current slot of
 * every expert, -1 for those only in the host tier.  Any pointer may be
 * NULL. */
moe_status moe_cache_stats(moe_layer* layer, uint64_t* hits, uint64_t* misses,
                           int32_t* slot_of_expert, int reset, void* stream);

/* Synchronises `stream`, then returns and clears the layer's device error
 * word (MOE_ERR_BOUNDS or MOE_ERR_TIMEOUT if a kernel recorded one). */
moe_status moe_status_sync(moe_layer* layer, void* stream);

/* Per-kernel timing of the library's own launches, for measurement (off by
 * default; it adds two event records per launch).  While enabled, every
 * kernel launch is bracketed by CUDA events on its stream.
 * moe_profile_read synchronises on the recorded events, writes up to
 * max_entries rows -- kernel name (NUL-terminated, name_len bytes per row),
 * launch count, total milliseconds -- returns the number of rows and clears
 * the totals. */
moe_status moe_profile_enable(int enable);
int moe_profile_read(char* names, int name_len, int* counts, float* total_ms, int max_entries);

/* Message of the last failed call on this thread ("" if none). */
const char* moe_last_error(void);

/* ABI version (major * 100 + minor). */
int moe_version(void);

#ifdef __cplusplus
}
#endif

#endif
