/*
 * moe.h - C ABI of the tiered (HBM / host-UVA) sparse MoE layer for GB300.
 *
 * One forward pass of a sparse Mixture-of-Experts layer whose experts are
 * placed one by one either in GPU HBM or in pinned host memory, the per-expert
 * plan of "763B MoE in two 96 GB cards" (side-box on the per-expert plan in
 * section "Same idea, native vLLM fails": each expert's residence and read
 * path is decided on its own).  Host-resident experts are read in place by the
 * GPU through unified virtual addressing, with no copy into HBM ("763B ...",
 * section "Where the VRAM gap comes from", UVA side-box).  Optionally the HBM
 * holds an adaptive, frequency-admitted expert cache over a set of experts
 * that all live in pinned host memory ("Running a 24k-expert MoE on a single
 * 32 GB card", sections 2 and 3).
 *
 * The pass: router logits -> top-k with renormalised softmax weights ->
 * grouping of (token, expert) pairs by expert -> per-expert SwiGLU FFN over
 * symmetric int-b group-quantised weights -> weighted combine into token
 * order.  Every step runs in this library's CUDA kernels (sm_103a).
 *
 * Conventions for every call:
 *  - Return value: a moe_status.  No call aborts, throws or exits.  After an
 *    error, moe_last_error(plan) holds a one-line description.
 *  - "device" pointers are CUDA device (or managed) addresses on the plan's
 *    device; "host" pointers are ordinary CPU addresses.  Where a parameter
 *    accepts either, the library asks the CUDA runtime which one it is.
 *  - bf16 values are passed as their 16-bit patterns (uint16_t / void*).
 *  - Streams are cudaStream_t values passed as void* (NULL = legacy default).
 *  - A plan is used by one host thread at a time.  Calls that enqueue work
 *    are ordered on the stream given; a forward on a different stream than
 *    the previous one first waits for the previous one (the plan's scratch
 *    buffers are reused).  Forwards enqueued while their stream is being
 *    captured into a CUDA graph take no part in that ordering (the graph's
 *    own edges order its nodes): the caller orders a graph's launches
 *    against the plan's other work, as for any graph.  A call made while
 *    another call on the same plan is running on another thread returns
 *    MOE_ERR_STATE.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum moe_status {
  MOE_OK = 0,
  MOE_ERR_INVALID = 1,     /* bad argument, shape or index */
  MOE_ERR_OOM = 2,         /* HBM or pinned host memory not available for the request */
  MOE_ERR_CUDA = 3,        /* a CUDA call failed (text in moe_last_error) */
  MOE_ERR_TIMEOUT = 4,     /* a bounded device-side wait gave up (latched; see moe_layer_forward) */
  MOE_ERR_STATE = 5,       /* call not valid in the plan's current state */
  MOE_ERR_UNSUPPORTED = 6  /* well-formed request outside what the library implements */
} moe_status;

typedef enum moe_scale_dtype { MOE_SCALE_F32 = 0, MOE_SCALE_BF16 = 1, MOE_SCALE_F16 = 2 } moe_scale_dtype;

typedef enum moe_residence { MOE_RES_HBM = 0, MOE_RES_HOST = 1 } moe_residence;

typedef enum moe_cache_policy {
  /* Residence is exactly what moe_place_experts says, per expert. */
  MOE_POLICY_STATIC = 0,
  /* Every expert lives in pinned host memory; cache_slots HBM slots hold a
   * frequency-admitted subset ("Running a 24k-expert MoE ...", sections 2-3). */
  MOE_POLICY_LFU = 1
} moe_cache_policy;

typedef struct moe_plan moe_plan;

/* Shapes and budgets of a plan.  Fill every field; struct_size must be
 * sizeof(moe_plan_desc) (ABI versioning). */
typedef struct moe_plan_desc {
  uint32_t struct_size;
  int32_t num_layers;   /* L >= 1 */
  int32_t num_experts;  /* E, routed experts per layer, 1..4096 */
  int32_t hidden;       /* H: multiple of 256 */
  int32_t inter;        /* I: expert intermediate size, multiple of 128 */
  int32_t top_k;        /* k: 1..min(E, 8) */
  int32_t weight_bits;  /* b in {2, 3, 4} */
  int32_t group_size;   /* G: scale group along each matrix's reduction axis; 32, 64 or 128,
                           dividing H and I */
  int32_t scale_dtype;  /* moe_scale_dtype */
  int32_t max_tokens;   /* upper bound on T for every forward of this plan */
  int32_t cache_policy; /* moe_cache_policy */
  int32_t device;       /* CUDA device ordinal */
  int64_t hbm_experts;  /* STATIC: capacity of the HBM expert arena, in experts (the rest of
                           the L*E experts must be placed in host memory) */
  int64_t cache_slots;  /* LFU: number of HBM slots (0 = no cache: every read goes to host) */
  int32_t reserved0;    /* must be zero (host- and HBM-resident experts are always processed
                           by one grid, with a share of its CTAs given to the host experts) */
  int32_t aging_period; /* LFU: halve all access counts every aging_period steps (0 = never) */
  int64_t prefill_slots; /* HBM slots reserved for staging a long prompt's experts that are
                            not in HBM (moe_prefill_forward); 0 = none */
  int64_t reserved[3];   /* must be zero */
} moe_plan_desc;

/* One expert in the canonical interchange format.  Matrices: gate Wg [I][H],
 * up Wu [I][H], down Wd [H][I], row-major, quantised in groups of G along the
 * reduction axis (H for gate/up, I for down).  codes[m]: weight i (row-major
 * index) occupies bits [i*b, i*b + b) of a little-endian bit stream and holds
 * u = q + 2^(b-1), q in [-(2^(b-1) - 1), 2^(b-1) - 1].  scales[m]:
 * [rows][cols / G] in the plan's scale dtype; the dequantised weight is q * s.
 * Pointers may be host or device; they are read during the call only. */
typedef struct moe_expert_weights {
  const void* codes[3];
  const void* scales[3];
} moe_expert_weights;

/* Optional copies of the routing, for inspection (device pointers, each may
 * be NULL).  Written in stream order by moe_layer_forward. */
typedef struct moe_routing_out {
  float* logits;     /* [T][E] fp32 router logits */
  int32_t* topk_idx; /* [T][k] chosen experts, logit descending, ties to the lower index */
  float* topk_w;     /* [T][k] renormalised softmax weights */
  int32_t* counts;   /* [E] (token, expert) pairs per expert */
  int32_t* offsets;  /* [E + 1] exclusive prefix sums of counts */
  int32_t* perm;     /* [T*k] slot ids t*k + j ordered by (expert asc, token asc) */
  int32_t* inv;      /* [T*k] position of slot t*k + j in perm */
} moe_routing_out;

/* Counters since plan creation or the last reset.  An access is one distinct
 * expert routed in one layer forward (an expert chosen by several tokens of
 * the same forward is read once). */
typedef struct moe_cache_stats_t {
  uint64_t accesses;   /* distinct (layer, expert) reads */
  uint64_t hits;       /* ... served from HBM */
  uint64_t misses;     /* ... served from pinned host memory over the link */
  uint64_t admissions; /* LFU: experts admitted into a slot */
  uint64_t evictions;  /* LFU: experts evicted from a slot */
  uint64_t hbm_bytes;  /* expert weight bytes read from HBM (router weights included) */
  uint64_t host_bytes; /* expert weight bytes read from host memory */
  uint64_t fill_bytes; /* LFU: bytes written into HBM slots by admissions */
  uint64_t pairs;      /* (token, expert) pairs computed */
  uint64_t forwards;   /* layer forwards */
  uint64_t router_exact; /* prefill path: router logits computed in the library's fixed
                          * order -- T*E when the logits are requested, otherwise the
                          * candidates the bounded tensor-core pass leaves per token */
} moe_cache_stats_t;

/* Create a plan: validates the shapes, checks the memory it will need
 * against free HBM (minus a headroom of max(1 GiB, 2%)) and returns
 * MOE_ERR_OOM instead of failing later -- a plan that fits at load time and
 * dies under load is the failure "125B sparse model on one 32 GB consumer
 * card" describes in section "A compute buffer is what limits capacity";
 * allocates the HBM expert arena (STATIC) or slot arena (LFU), the pinned host
 * arena (every expert not in HBM; all experts under LFU; from the driver's
 * pinned allocator with the GPU's NUMA node preferred where the system reports
 * one, "763B MoE in two 96 GB cards", section "PCIe topology"), and all
 * scratch.  *out is set on success.  Test hook:
 * the environment variable MOE_FAULT containing "hbm_alloc" or
 * "pinned_alloc" makes that allocation fail (MOE_ERR_OOM, all released). */
moe_status moe_plan_create(const moe_plan_desc* desc, moe_plan** out);

/* Free everything the plan owns.  Waits for the plan's outstanding work. */
moe_status moe_plan_destroy(moe_plan* plan);

/* Router of `layer` (the gate that picks k of the E routed experts per token,
 * "763B MoE in two 96 GB cards", section "Where the VRAM gap comes from"):
 * wr [E][H] bf16 (host or device), bias [E] fp32 (host or device) or NULL for
 * none.  Copied; synchronous. */
moe_status moe_set_router(moe_plan* plan, int layer, const uint16_t* wr_bf16, const float* bias);

/* Replace the router bias of `layer` in stream order (bias [E] fp32, host or
 * device; host memory must stay valid until `stream` reaches the copy).  For
 * per-step bias updates without a synchronisation. */
moe_status moe_update_router_bias(moe_plan* plan, int layer, const float* bias, void* stream);

/* The same for layers first .. first+count-1 at once: bias [count][E] fp32,
 * row i for layer first+i, in one stream-ordered copy (the biases of all
 * layers sit contiguously in device memory).  MOE_ERR_INVALID for a layer
 * range outside [0, num_layers) or bias NULL; count == 0 does nothing. */
moe_status moe_update_router_biases(moe_plan* plan, int first, int count, const float* bias,
                                    void* stream);

/* Place experts first .. first+count-1 of `layer` -- the per-expert plan of
 * "763B MoE in two 96 GB cards" (side-box of section "Same idea, native vLLM
 * fails": each expert's residence and read path decided on its own): copy
 * each expert from the canonical format into its device layout at
 * residence[i] (MOE_RES_HBM or
 * MOE_RES_HOST; ignored under LFU, where every expert goes to host memory;
 * NULL = all HBM).  An expert may be placed again (its residence can change)
 * under STATIC; under LFU experts are placed once, before the first forward.
 * Synchronous: the caller may free its buffers on return.  MOE_ERR_OOM if an
 * arena is full. */
moe_status moe_place_experts(moe_plan* plan, int layer, int first, int count,
                             const uint8_t* residence, const moe_expert_weights* w);

/* Forward of `layer` on T tokens (route, group by expert, SwiGLU FFN of each
 * chosen expert read from HBM or in place from pinned host memory over UVA,
 * weighted combine: "763B MoE in two 96 GB cards", section "Where the VRAM gap
 * comes from" and its UVA side-box): x [T][H] bf16 device (16-byte aligned),
 * y [T][H] bf16 device (must not alias x).  0 <= T <= max_tokens; T = 0 is a
 * no-op.  Every expert of the layer must have been placed.  Stream-ordered,
 * no host synchronisation inside: y is valid when `stream` reaches the end
 * of the call.  If a previous forward's bounded device wait gave up, this
 * call returns MOE_ERR_TIMEOUT once (and resets the plan's scratch state).
 * dbg may be NULL. */
moe_status moe_layer_forward(moe_plan* plan, int layer, const void* x_bf16, int T, void* y_bf16,
                             void* stream, const moe_routing_out* dbg);

/* The same forward with the residual-stream update fused into its combine:
 * y as moe_layer_forward, and out[t][c] = bf16(float(y[t][c]) + residual[t][c])
 * (round to nearest even), so that a stack of layers -- consecutive MoE layers
 * of the pages' models, each fed the previous layer's output plus the residual
 * stream -- gets the next layer's input without a launch of its own.
 * residual [T][H] fp32 device, out [T][H] bf16 device, both 16-byte aligned;
 * out must not overlap x, y or residual, nor residual y (MOE_ERR_INVALID).
 * Otherwise as moe_layer_forward (dbg is NULL here). */
moe_status moe_layer_forward_residual(moe_plan* plan, int layer, const void* x_bf16, int T, void* y_bf16,
                                      const float* residual, void* out_bf16, void* stream);

/* Chunked prefill of a long prompt through `layer`: the prefill-aware cache of
 * "Running a 24k-expert MoE on a single 32 GB card", section 2 -- HBM slots
 * kept for the prompt's experts, and long inputs read in chunks of 8,192
 * tokens.  x [T][H] and y [T][H] bf16 device (16-byte aligned, not aliased),
 * any T >= 0; needs max_tokens > 8 (the chunks, min(8192, max_tokens) tokens
 * each, take the prefill path of moe_layer_forward).  When there is more than
 * one chunk, the layer's experts that are not in HBM (host-resident; under LFU
 * those the cache does not hold) are first copied into the plan's
 * prefill_slots, in ascending expert order as far as the slots go, and every
 * chunk reads the staged copies (the rest in place from pinned host memory):
 * each such expert crosses the host link once per prompt, not once per chunk.  These forwards leave the
 * LFU state untouched (no access counts, no misses queued), so a prompt that
 * routes to nearly every expert neither evicts nor retrains the decode cache;
 * moe_cache_stats counts their reads (staged experts as HBM hits) and the
 * staging copies (fill_bytes).  Stream-ordered like moe_layer_forward. */
moe_status moe_prefill_forward(moe_plan* plan, int layer, const void* x_bf16, int64_t T, void* y_bf16,
                               void* stream);

/* Same layer forward with HOST buffers: copies x (host [T][H] bf16) into the
 * plan's device staging buffer, runs the forward and copies y back into
 * y_host, all in stream order; the caller synchronises the stream before
 * reading y_host.  Pinned host buffers give asynchronous copies.  For a
 * decode-sized batch (T <= 8) in page-locked buffers (x_host 16-byte and
 * y_host 4-byte aligned) no copy engine is used: a copy kernel reads x_host
 * through its device mapping and the forward writes y_host through its own. */
moe_status moe_layer_forward_host(moe_plan* plan, int layer, const void* x_host, int T,
                                  void* y_host, void* stream);

/* End of one decode step (one token through all layers).  Under LFU, runs the
 * admission/eviction pass over the step's misses and fills the admitted
 * experts' slots, in stream order; the next step sees the new residence --
 * the cache that "adapts to the conversation" of "Running a 24k-expert MoE on
 * a single 32 GB card", section 2 (rules of the pass: moe_plan_desc's
 * cache_policy and aging_period).  Under STATIC it only advances the step
 * counter. */
moe_status moe_step_end(moe_plan* plan, void* stream);

/* Counters of `layer` (or of all layers for layer = -1); reset = 1 zeroes
 * them after reading.  Synchronises with the plan's device work.  The hit
 * rate these counters give is the measure of "Running a 24k-expert MoE on a
 * single 32 GB card", section 3 (a cache of ~70 % of the experts serving
 * 97.8-99.7 % of expert reads).  Under LFU each step queues its misses for
 * moe_step_end in a queue of num_layers * min(E, max_tokens * k) entries; a
 * forward that finds it full (a layer forwarded more than once between step
 * ends) latches the fact, and the next moe_layer_forward, moe_step_end or
 * moe_cache_stats that sees it returns MOE_ERR_STATE (this call, which
 * synchronises first, always sees it; *out is filled all the same). */
moe_status moe_cache_stats(moe_plan* plan, int layer, moe_cache_stats_t* out, int reset);

/* Residence of every expert of `layer` as seen by the next forward: out[e] =
 * slot index (>= 0, HBM) or -1 (host) -- the per-expert residence of the
 * per-expert plan ("763B MoE in two 96 GB cards", side-box of section "Same
 * idea, native vLLM fails") or of the cache ("Running a 24k-expert MoE on a
 * single 32 GB card", section 2).  Under STATIC, slot = position in the HBM
 * arena.  Synchronous. */
moe_status moe_residence_table(moe_plan* plan, int layer, int32_t* out_host);

/* Quantise w [rows][cols] fp32 (device) into the canonical format (the
 * low-bit expert weights of "763B MoE in two 96 GB cards", 3-bit, and of
 * "Running a 24k-expert MoE on a single 32 GB card", 2-bit, read here as
 * symmetric int-b group quantisation): codes
 * (device, rows*cols*bits/8 bytes) and scales (device, [rows][cols/group] in
 * scale_dtype), groups of `group` along cols.  Per group: s = amax / qmax
 * rounded to nearest-even in the scale dtype, q = clamp(rint(w / s), -qmax,
 * qmax) with qmax = 2^(bits-1) - 1, q = 0 when s = 0.  Stream-ordered. */
moe_status moe_quantize(const float* w, int rows, int cols, int bits, int group, int scale_dtype,
                        void* codes, void* scales, void* stream);

/* Measure the GPU's zero-copy read bandwidth from pinned host memory (the
 * link host experts are read over: "763B MoE in two 96 GB cards", UVA side-box
 * of section "Where the VRAM gap comes from") and its HBM read bandwidth, with a
 * streaming-read kernel over `bytes` bytes (>= 64 MiB recommended), best of
 * `iters` runs.  Synchronous; allocates and frees its own buffers. */
moe_status moe_probe_bandwidth(int device, size_t bytes, int iters, double* host_read_gbs,
                               double* hbm_read_gbs);

/* Routing that allocates nothing.  The source pages have no counterpart to
 * this call; it exists for callers that cannot allocate device memory at the
 * point where they route tokens -- for example a serving runtime that has
 * already reserved nearly all of HBM for its own pools (so a cudaMalloc would
 * fail or would have to come out of memory it manages), or code running where
 * an allocation call is not permitted.  It computes the router logits of x
 * [T][H] bf16 (device) against wr [E][H] bf16 (device), plus bias [E] fp32
 * (device) or NULL, in the same fixed fp32 summation order as
 * moe_layer_forward, and writes the top-k per token (logit descending, ties
 * to the lower expert index) to topk_idx [T][k] int32 and the renormalised
 * softmax weights to topk_w [T][k] fp32 (both device).  Work space for the
 * logits is a fixed device array of 262,144 floats (1 MiB) that every GPU
 * holds from the moment this library's device code is loaded into its
 * context until the process exits; T * E above that is rejected with
 * MOE_ERR_INVALID, as are H not a positive multiple of 256, k outside
 * [1, min(E, 8)], x or wr not 16-byte aligned, and a stream that belongs
 * to another device than the current one.  The first call on a device looks
 * up that array's device address (cudaGetSymbolAddress) with the device
 * current; under CUDA's lazy module loading this is also where the array's
 * memory is committed, so make that first call early (a call with T = 0 does
 * it and nothing else) and before any stream capture.  Selection follows the
 * same order as moe_layer_forward (an order-preserving integer key of each
 * logit, -0 equal to +0; ties to the lower expert index).
 * All calls share the one array, so calls whose work overlaps on the GPU
 * (different streams, or different host threads) race and give wrong
 * results; order them on one stream.  Stream-ordered; T = 0 does the
 * set-up only (its buffer pointers may be NULL).
 * Calls no allocator (no cudaMalloc, cudaFree or library allocation). */
moe_status moe_route_noalloc(const void* x_bf16, int T, int H, const void* wr_bf16,
                             const float* bias, int E, int k, int32_t* topk_idx, float* topk_w,
                             void* stream);

/* Test hook for the failure path.  The next decode forward (T <= 8) of `plan`
 * publishes none of its gate/up results, so every down-projection unit's
 * bounded wait for them runs out (about a second): the kernel latches a
 * timeout in the plan's error word and ends with wrong outputs; nothing
 * faults or hangs.  The call after that forward returns MOE_ERR_TIMEOUT (and
 * does nothing else); the plan is then usable again.  MOE_ERR_INVALID for
 * plan NULL. */
moe_status moe_debug_fail_next_forward(moe_plan* plan);

const char* moe_status_string(moe_status s);
/* Last error text of `plan` (or of the last call that had no plan, for NULL). */
const char* moe_last_error(const moe_plan* plan);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
