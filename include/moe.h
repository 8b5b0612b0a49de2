/*
 * moe.h -- C ABI of the routed mixture-of-experts FFN layer for one GB300 (sm_103a).
 *
 * The layer, per token t of a window of T tokens (Krasis white paper, sec. 5.3
 * "Per-token routed expert execution"; kairos-engine README, "The MoE forward"):
 *
 *   logits[t][e] = sum_h Wr[e][h] * x[t][h] (+ bias[e])           router GEMV
 *   ids[t][0..K), w[t][0..K) = top-K of logits[t], ties to the lower id;
 *       w = softmax over all E logits, renormalised over the K chosen
 *   buckets: the T*K (token, rank) pairs grouped by expert (expert-major)
 *   per chosen expert e: h = SwiGLU(Wg[e] x, Wu[e] x), y_e = Wd[e] h,
 *       with Wg, Wu, Wd block-quantised and dequantised on the fly
 *   y[t] = sum_{k=0}^{K-1} w[t][k] * y_{ids[t][k]}(x[t])   (fixed k order)
 *          + shared(x[t])                                 (optional shared expert)
 *
 * Weights live in a device arena. A flat slot table indexed by (layer, expert)
 * gives each expert's arena slot, or -1 when it is not resident; the kernels
 * read the table on the device, so a captured CUDA graph keeps working when
 * experts move (Krasis white paper, sec. 5.3).
 *
 * Conventions for every function:
 *   - Return MOE_OK (0) or a negative MOE_ERR_* code. Argument and shape errors
 *     are detected on the host, before anything is enqueued; the message is then
 *     available from moe_last_error() (thread-local).
 *   - Pointers to tensors are DEVICE pointers unless the name or comment says
 *     host. The caller owns every tensor; the library owns the opaque handles.
 *   - All GPU work is enqueued on the caller's stream (moe_stream_t is the CUDA
 *     runtime's cudaStream_t; 0 is the legacy default stream) with no host
 *     synchronisation, so the compute calls can be captured in a CUDA graph.
 *     Exceptions, stated per function: moe_slot_load with a pageable host blob,
 *     moe_status (synchronises the stream), and the create/destroy calls.
 *   - Conditions found on the device (absent expert, non-finite logit, bounds,
 *     timeout) never trap: the kernel records a MOE_STATUS_* bit in the
 *     context's status word, the affected contribution is zero, and the caller
 *     reads the bits with moe_status().
 *   - There is no CPU fallback. Every call runs on the GPU of its context.
 *   - Row-major everywhere. x [T][H], logits [T][E], ids/w [T][K], y [T][H].
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *moe_stream_t; /* same type as cudaStream_t */
typedef struct moe_ctx moe_ctx;
typedef struct moe_arena moe_arena;
typedef struct moe_slots moe_slots;

/* return codes */
#define MOE_OK 0
#define MOE_ERR_ARG (-1)          /* null pointer, bad enum, negative size */
#define MOE_ERR_SHAPE (-2)        /* dimensions the kernels do not support */
#define MOE_ERR_UNSUPPORTED (-3)  /* valid request with no implementation */
#define MOE_ERR_CUDA (-4)         /* a CUDA runtime call failed */
#define MOE_ERR_NOMEM (-5)        /* device allocation, arena or slot pool full */
#define MOE_ERR_EXPERT_ABSENT (-6)
#define MOE_ERR_NONFINITE (-7)
#define MOE_ERR_TIMEOUT (-8)
#define MOE_ERR_BOUNDS (-9)
#define MOE_ERR_WORKSPACE (-10)   /* ws_bytes below moe_layer_workspace() */

/* device status bits (moe_status) */
#define MOE_STATUS_EXPERT_ABSENT 1u /* a routed expert had no slot: it added 0 */
#define MOE_STATUS_NONFINITE 2u     /* a router logit was NaN or +-inf */
#define MOE_STATUS_TIMEOUT 4u       /* a bounded device wait gave up */
#define MOE_STATUS_BOUNDS 8u        /* an index failed a device range check */

typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype;

/* Block formats. Every block is 18 bytes in the canonical (caller-facing) form:
 * an fp16 scale d (2 bytes, little-endian) then 16 bytes of codes q.
 *   MOE_Q2_64: 64 weights of 2 bits; code n in bits 2(n%4)..2(n%4)+1 of code
 *              byte n/4 ("Strata in the source", sections "The byte budget, in
 *              code" and "The CPU kernels").
 *   MOE_Q4_32: 32 weights of 4 bits; code n in bits 4(n%2)..4(n%2)+3 of code
 *              byte n/2.
 * Weight value: d * (q - zero_point). The Strata article's Q2_0 reads codes
 * {0,1,2,3} as {-1,0,1,2} (zero_point 1); zero_point 2 gives {-2,-1,0,1}. Q4
 * uses zero_point 8. Allowed: 0..3 for Q2, 0..15 for Q4. */
typedef enum { MOE_Q4_32 = 0, MOE_Q2_64 = 1 } moe_quant;

typedef struct {
    int kind;       /* moe_quant */
    int zero_point; /* subtracted from every code */
} moe_format;

typedef enum { MOE_ACT_SWIGLU = 0, MOE_ACT_GEGLU_TANH = 1 } moe_act;

/* Route weights of the K chosen experts (the choice is the same for every kind:
 * the K largest logits, equal logits to the lower id; sigmoid is monotone, so
 * ranking sigmoid scores is ranking logits). Krasis white paper sec. 5.3 names
 * sigmoid top-k routers (Nemotron Nano) beside softmax ones.
 *   MOE_ROUTER_SOFTMAX       w_k = softmax over the K chosen logits (default)
 *   MOE_ROUTER_SIGMOID       w_k = 1 / (1 + exp(-logit_k))
 *   MOE_ROUTER_SIGMOID_NORM  the sigmoid scores divided by their sum over the K
 * All in fp32 (expf, IEEE division; sums in rank order). */
typedef enum { MOE_ROUTER_SOFTMAX = 0, MOE_ROUTER_SIGMOID = 1, MOE_ROUTER_SIGMOID_NORM = 2 } moe_router_kind;

/* ------------------------------------------------------------ context */

/* Create a context on CUDA device `device` (made current for the call). The
 * context owns the device status word. Not thread-safe to share between threads
 * that enqueue concurrently on different streams (the status word is shared). */
MOE_API int moe_ctx_create(int device, moe_ctx **out);
MOE_API int moe_ctx_destroy(moe_ctx *ctx);

/* Context options. MOE_OPT_PERSISTENT_DECODE (default 1): windows of up to 8
 * tokens (4 with fp32 x) run as one cooperative persistent kernel per call (a
 * whole moe_stack_forward chain per launch); 0 forces the multi-kernel path.
 * Both paths give the same bits. MOE_ERR_ARG for an unknown option. */
#define MOE_OPT_PERSISTENT_DECODE 1
MOE_API int moe_ctx_set_option(moe_ctx *ctx, int option, int value);

/* Read a context option into *value. Besides the settable options:
 * MOE_OPT_LAST_PATH (read only): which path the last moe_layer_forward*,
 * moe_layer_forward_static, moe_stack_forward* or moe_expert_ffn call on this
 * context ran for its experts: 1 the persistent decode kernel, 2 the tensor-core
 * (tcgen05) grouped GEMMs, 0 the multi-kernel mma.sync path (or no call yet).
 * MOE_ERR_ARG for an unknown option or a null pointer; setting
 * MOE_OPT_LAST_PATH is MOE_ERR_ARG too. */
#define MOE_OPT_LAST_PATH 2
MOE_API int moe_ctx_get_option(moe_ctx *ctx, int option, int *value);

/* MOE_OPT_PREFILL_MIN_T (default 64, settable, >= 1): windows of at least this
 * many tokens run their Q4 experts (routed and shared, H a multiple of 128) as
 * grouped GEMMs on the tensor cores (kairos-engine README, "Prefill and decode are
 * different machines"): weights dequantised to fp16 (w = fp16(d*(q-8)), one
 * rounding), x and h in fp16, fp32 accumulation. Those results differ from the
 * mma.sync path by that rounding (both stay within the oracle's tolerance).
 * Q2_0 experts and smaller windows keep the mma.sync path. The router of such a
 * window (bf16 x and Wr, any format) is a tensor-core GEMM too: its logits can
 * differ from the per-row CUDA-core order in the last bits, and moe_router_topk
 * follows the same rule, so a window routes identically through either entry. */
#define MOE_OPT_PREFILL_MIN_T 3

/* MOE_OPT_TEST_SKIP_ARRIVAL (default -1, settable, >= -1): a test hook for the
 * bounded waits. With value v >= 0, in every persistent decode launch CTA 0 leaves
 * out its router logits and its arrival flag of layer v of the launch (a signal
 * that never comes): every CTA's wait for the layer's logits gives up after about
 * a second, MOE_STATUS_TIMEOUT is set, the kernel stops and returns, and the context
 * stays usable (the call's outputs are then undefined). Nothing faults or traps. */
#define MOE_OPT_TEST_SKIP_ARRIVAL 4

/* Synchronise `stream`, then read and clear the device status bits into *bits.
 * Returns MOE_OK even when bits are set; the caller inspects them. */
MOE_API int moe_status(moe_ctx *ctx, moe_stream_t stream, uint32_t *bits);

/* Text of the last error raised on this thread ("" if none). */
MOE_API const char *moe_last_error(void);

/* Bytes of one expert blob (gate [F][H], up [F][H], down [H][F]; canonical and
 * device forms have the same size): 3*H*F / weights_per_block * 18.
 * ("Strata in the source", "The byte budget, in code": 1,382,400 bytes for
 * H=2560, F=640 in Q2_0.) H and F must be positive multiples of 64. */
MOE_API int moe_expert_bytes(moe_format fmt, int H, int F, size_t *out);

/* ------------------------------------------------------------ arena and slots */

/* One device allocation of `bytes` from which slot pools are carved. */
MOE_API int moe_arena_create(moe_ctx *ctx, size_t bytes, moe_arena **out);
MOE_API int moe_arena_destroy(moe_arena *arena);

/* A slot table for n_layers x n_experts experts of one shape (H, F) and format,
 * with `capacity` resident slots carved from `arena` (each slot holds one
 * expert in the device layout, rounded up to 256 bytes). Every table entry
 * starts at -1 (absent). Fails with MOE_ERR_NOMEM if the arena lacks room. */
MOE_API int moe_slots_create(moe_ctx *ctx, moe_arena *arena, int n_layers, int n_experts,
                     moe_format fmt, int H, int F, int capacity, moe_slots **out);
MOE_API int moe_slots_destroy(moe_slots *slots);

/* Make expert (layer, expert) resident. `blob` is the canonical blob of
 * moe_expert_bytes() bytes, host or device memory (nbytes must equal that
 * size). The blob is copied (host blobs through a device staging buffer owned
 * by `slots`), rewritten into the device layout in a free slot (or the slot the
 * expert already has), and only then is the table entry written, in stream
 * order, so no kernel can see the entry before the weights are in place. With a pageable host blob the
 * copy is synchronous with respect to the host; with a pinned or device blob
 * nothing blocks. The blob may be reused as soon as the call returns for
 * pageable memory, and after the stream reaches this point otherwise.
 * MOE_ERR_NOMEM if no slot is free. */
MOE_API int moe_slot_load(moe_slots *slots, int layer, int expert, const void *blob, size_t nbytes,
                  moe_stream_t stream);

/* Mark (layer, expert) absent (table entry -1, in stream order) and return its
 * slot to the free pool. A no-op for an absent expert. Work enqueued earlier on
 * `stream` still sees the old entry; work on other streams must be ordered by
 * the caller. */
MOE_API int moe_slot_evict(moe_slots *slots, int layer, int expert, moe_stream_t stream);

/* Host-side view of the table: the slot index of (layer, expert), or -1. */
MOE_API int moe_slot_lookup(const moe_slots *slots, int layer, int expert, int32_t *slot_out);

/* ------------------------------------------------------------ the steps */

/* Router GEMV and top-K (steps 1-2 above). x [T][H] (xt F32 or BF16); Wr [E][H]
 * (wt F32 or BF16); bias [E] f32 or NULL. Outputs ids [T][K] in rank order
 * (larger logit first, equal logits to the lower id; NaN ranks last and sets
 * MOE_STATUS_NONFINITE, as does +-inf) and w [T][K] f32 (softmax renormalised
 * over the K chosen; NaN for a token with a non-finite logit). logits_out
 * [T][E] f32 receives the logits and is required. Logits accumulate in fp32. 1 <= K <= min(E, 32),
 * E <= 4096, H % 8 == 0. */
MOE_API int moe_router_topk(moe_ctx *ctx, const void *x, moe_dtype xt, int T, int H, const void *Wr,
                    moe_dtype wt, const float *bias, int E, int K, float *logits_out,
                    int32_t *ids, float *w, moe_stream_t stream);

/* Stable counting sort of the T*K pairs p = t*K + k by expert ids[p] (kairos
 * README, "The MoE forward": the batch is bucketed by expert). counts [E];
 * offsets [E+1] (exclusive prefix sum, offsets[E] = T*K); perm [T*K] lists the
 * pairs of expert 0, then expert 1, ..., each in increasing p; active [E] lists
 * the experts with count > 0 in increasing order, *n_active (device int) their
 * number. Integer results are exact. ids outside [0, E) set MOE_STATUS_BOUNDS
 * and are left out of every bucket. */
MOE_API int moe_bucket(moe_ctx *ctx, const int32_t *ids, int T, int K, int E, int32_t *counts,
               int32_t *offsets, int32_t *perm, int32_t *active, int32_t *n_active,
               moe_stream_t stream);

/* Bytes of workspace moe_expert_ffn / moe_layer_forward / moe_stack_forward need
 * for up to T_max tokens with this layer description (below). */
typedef struct {
    const moe_slots *slots;  /* routed experts, table of n_layers x E */
    int layer;               /* which layer of `slots` */
    int H, E, K, F;          /* hidden, experts, top-K, expert FFN width */
    const void *Wr;          /* router weights [E][H] (device) */
    moe_dtype wr_dtype;
    const float *bias;       /* router bias [E] or NULL */
    const moe_slots *shared; /* shared expert (layer `layer`, expert 0) or NULL */
    int F_shared;            /* its FFN width */
    int act;                 /* moe_act */
    /* --- optional (zero / NULL = off) ---
     * router_scale [H] f32: per-input-dimension scale of the router input,
     *   logits = Wr (x * router_scale) (+ bias); the product x_h * s_h is rounded
     *   to fp32 and the dot product accumulates in fp32 (kairos README, "The MoE
     *   forward": the router scale is per input dimension).
     * down_scale [E] f32: per-expert scale of the down projection, folded into
     *   the route weight: the combine adds fp32(w_k * s_e) * y_k (kairos README:
     *   the down scale is per expert). A pair whose scaled weight is 0 does no
     *   expert work.
     * router_kind: moe_router_kind.
     * drop_eligible [E] u8, drop_protect_pct P, drop_mass_pct M: route-drop
     *   policy P/M (Krasis white paper sec. 7.2). Per token: the first
     *   ceil(K * P / 100) ranks are kept; among the later ranks whose expert is
     *   eligible (nonzero byte) and whose weight is positive, taken from the
     *   smallest weight up (equal weights: later rank first), routes are dropped
     *   while the dropped weight c (fp32, summed in that order) keeps
     *   c * 100 <= M * S, S = the sum of the K route weights in rank order
     *   (fp32); the first route that does not fit ends the scan. A dropped route
     *   keeps its place with weight 0 (no expert work, nothing added) and the
     *   survivors are not renormalised (sec. 7.3). The decision uses the route
     *   weights before down_scale. drop_eligible NULL = off.
     * omitted_out [T] f32 (device, NULL = not reported): the dropped share c / S
     *   of each token (0 when nothing is dropped). */
    const float *router_scale;
    const float *down_scale;
    int router_kind;
    const uint8_t *drop_eligible;
    int drop_protect_pct, drop_mass_pct;
    float *omitted_out;
} moe_layer_desc;

MOE_API int moe_layer_workspace(const moe_layer_desc *desc, int T_max, size_t *bytes);

/* Expert part of the layer (steps 4-6): with the routing (ids, w) and buckets
 * (offsets, perm from moe_bucket over the same ids) given, computes
 *   y[t] = sum_k w[t][k] * expert_{ids[t][k]}(x[t]) (+ shared(x[t]))
 * with the layer description's slots (desc->Wr, bias, router_scale and the
 * routing options are not read; desc->down_scale is: w becomes fp32(w *
 * down_scale[e])). Pairs with w == 0 do no expert work and add nothing. ws:
 * device workspace of at least moe_layer_workspace(desc, T) bytes, 256-byte
 * aligned. A router input other than the experts' input (a separately normed
 * tensor) is served by moe_router_topk on that input followed by this call. */
MOE_API int moe_expert_ffn(moe_ctx *ctx, const moe_layer_desc *desc, const void *x, moe_dtype xt, int T,
                   const int32_t *ids, const float *w, const int32_t *offsets,
                   const int32_t *perm, float *y, void *ws, size_t ws_bytes,
                   moe_stream_t stream);

/* The whole layer: router, top-K, buckets, experts, combine. y [T][H] f32.
 * logits_out [T][E] and ids_out [T][K] may be NULL. Deterministic: the same
 * inputs give the same bits, and token t's result does not depend on the other
 * tokens of the window or on T (Strata article, "Drafting and verifying": a
 * multi-token pass does per token what the single-token pass does). */
MOE_API int moe_layer_forward(moe_ctx *ctx, const moe_layer_desc *desc, const void *x, moe_dtype xt,
                      int T, float *y, float *logits_out, int32_t *ids_out, void *ws,
                      size_t ws_bytes, moe_stream_t stream);

/* Same, with x [T][H] and y [T][H] in HOST memory (pinned for asynchronous
 * copies): x is copied into the workspace, the layer runs, y is copied back, all
 * on `stream`. The host buffers must stay valid until the stream reaches the
 * end of the call. Needs moe_layer_workspace() + T*H*(4 + element size of xt)
 * bytes (rounded up to 256 each). */
MOE_API int moe_layer_forward_host(moe_ctx *ctx, const moe_layer_desc *desc, const void *x_host,
                           moe_dtype xt, int T, float *y_host, void *ws, size_t ws_bytes,
                           moe_stream_t stream);

/* A chain of n_layers MoE layers over a residual stream (one decode step of an
 * expert stack): for l in 0..n_layers-1:
 *   u = bf16(RMSNorm(resid))   (weightless, eps; kairos README "normalise")
 *   resid += layer_l(u)
 * resid [T][H] f32 is updated in place. trace_in [n_layers][T][H] bf16 and
 * trace_logits [n_layers][T][E] f32 may be NULL; when given they receive each
 * layer's input and router logits (for per-layer checks). All layers must share
 * H, E, K, F and the router dtype. */
MOE_API int moe_stack_forward(moe_ctx *ctx, const moe_layer_desc *layers, int n_layers, float *resid,
                      int T, float eps, void *trace_in, float *trace_logits, void *ws,
                      size_t ws_bytes, moe_stream_t stream);

/* Same chain with resid [T][H] f32 in HOST memory (pinned for asynchronous
 * copies): copied into the workspace, run through the n_layers layers, copied
 * back, all on `stream`. Needs moe_layer_workspace() + T*H*4 (rounded up to
 * 256) bytes. The host buffer must stay valid until the stream reaches the end
 * of the call. */
MOE_API int moe_stack_forward_host(moe_ctx *ctx, const moe_layer_desc *layers, int n_layers,
                                   float *resid_host, int T, float eps, void *ws, size_t ws_bytes,
                                   moe_stream_t stream);

/* Size of the library's fixed scratch area used by moe_layer_forward_static. */
#define MOE_STATIC_SCRATCH_BYTES (4 * 1024 * 1024)

/* moe_layer_forward without a workspace argument, for callers that cannot
 * allocate device memory: a host framework that owns the whole GPU through its
 * own memory pool and gives libraries no allocator, a latency-critical decode
 * loop that must not call cudaMalloc (it can synchronise the device), or a thin
 * binding with no way to size and keep a buffer. The paper has no counterpart:
 * it is a packaging choice of this library.
 *
 * The scratch is one file-scope device array of MOE_STATIC_SCRATCH_BYTES (4 MiB)
 * that every GPU loading the library holds until the process exits. This call
 * allocates nothing: no cudaMalloc, no cudaFree, no allocating library routine.
 * The first call on a device looks up the array's device address (with that
 * device current) and caches it; make that first call before any stream
 * capture. A window whose moe_layer_workspace() exceeds the array fails with
 * MOE_ERR_WORKSPACE (4 MiB covers decode and verify windows: about 150 KB at
 * T=1 and 600 KB at T=4 for the H=2560, E=512, top-10, F=640 layer; 1.5 MB at T=8
 * for the H=2816 layer with a 2112-wide shared expert). Every call on every
 * stream shares the array and leaves its contents behind; nothing in it needs
 * to start at zero (each call writes what it reads). Calls that overlap on the
 * GPU race on the array: serialise them (one stream, or events). Arguments and
 * results are those of moe_layer_forward. */
MOE_API int moe_layer_forward_static(moe_ctx *ctx, const moe_layer_desc *desc, const void *x,
                                     moe_dtype xt, int T, float *y, float *logits_out,
                                     int32_t *ids_out, moe_stream_t stream);

/* Weightless RMSNorm with bf16 output: out[t][h] = bf16(x[t][h] / sqrt(mean_h
 * x[t][h]^2 + eps)), x f32. H % 8 == 0. */
MOE_API int moe_rmsnorm_bf16(moe_ctx *ctx, const float *x, int T, int H, float eps, void *out,
                     moe_stream_t stream);

/* ------------------------------------------------------------ residency policies
 *
 * Host-side replacement policies that decide which (layer, expert) pairs stay
 * resident in a pool of `capacity` slots, fed with the routed ids of each layer
 * and token, and a driver that applies their decisions to a moe_slots pool
 * through moe_slot_load / moe_slot_evict (publish after the copy lands). Pure
 * host code: no GPU work except in moe_policy_apply.
 *
 *   MOE_POLICY_LRU (kairos README, "Decode, 2026-09-28/29"): on a routing event
 *     (the ids one token routes to in one layer) every resident id of the event
 *     becomes most recently used, in event order; then each missing id, in event
 *     order, is loaded, evicting the least recently used entry that is not in
 *     the event when the pool is full.
 *   MOE_POLICY_DECAYED_FREQ (kairos README, "2026-09-29: which experts to
 *     keep"): every entry has a score that halves every `half_life` tokens and
 *     gains 1 per access; misses load as for LRU, and the victim is the entry
 *     of lowest decayed score among those not in the event and not accessed in
 *     the last `recency_guard` tokens (all guarded: among those not in the
 *     event); equal scores go to the least recently used, then the lower
 *     (layer, expert).
 *   MOE_POLICY_LFU_SWAP (Strata article, "The cache's replacement rule"): misses
 *     do not load; every access adds 1 to a float counter of its pair; at the
 *     end of every `swap_every`-th token, per layer, the hottest missing experts
 *     (counter >= min_count) pair with the coldest resident ones (hottest first,
 *     coldest first; equal counters to the lower expert) and swap while the
 *     newcomer's counter is at least the resident's + margin; across layers only
 *     the max_swaps largest gains (newcomer - resident; equal gains to the lower
 *     layer, then the earlier pair) are kept. After every token every counter is
 *     multiplied by `decay`. Swapped-in experts count as resident from the next
 *     token (their copy lands first).
 *
 * The experts of the event being served are never evicted. Capacity counts
 * entries over all layers (one pool, like moe_slots). */
typedef enum { MOE_POLICY_LRU = 0, MOE_POLICY_DECAYED_FREQ = 1, MOE_POLICY_LFU_SWAP = 2 } moe_policy_kind;

typedef struct {
    int kind;           /* moe_policy_kind */
    int capacity;       /* resident entries, >= 1 */
    double half_life;   /* DECAYED_FREQ: tokens (32 in the README) */
    int recency_guard;  /* DECAYED_FREQ: tokens (2) */
    float decay;        /* LFU_SWAP: counter factor per token (0.7) */
    float margin;       /* LFU_SWAP: hysteresis (1.5) */
    float min_count;    /* LFU_SWAP: newcomer threshold (2.0) */
    int swap_every;     /* LFU_SWAP: tokens between swap rounds (4) */
    int max_swaps;      /* LFU_SWAP: swaps per round over all layers (96) */
} moe_policy_params;

typedef struct moe_policy moe_policy;

/* A policy over n_layers x n_experts pairs with an empty pool. */
MOE_API int moe_policy_create(const moe_policy_params *params, int n_layers, int n_experts,
                              moe_policy **out);
MOE_API int moe_policy_destroy(moe_policy *p);

/* Make the listed pairs resident without counting accesses (a shipped profile),
 * in list order, until the pool is full; returns how many were placed in *n_placed.
 * Every pair is checked first: one out of range gives MOE_ERR_ARG and places none. */
MOE_API int moe_policy_seed(moe_policy *p, const int32_t *layers, const int32_t *experts, int n,
                            int *n_placed);

/* One routing event: `ids` [n] (host) routed by the current token in `layer`.
 * hit [n] (host, may be NULL) gets 1 for ids resident before the event. Loads
 * decided now (LRU, DECAYED_FREQ) are appended to the plan: load_expert [n]
 * (experts of `layer` to load, event order) with the evicted pairs
 * evict_layer / evict_expert [n] (-1 where no eviction was needed); *n_loads
 * their number. Duplicate ids in one event count once. */
MOE_API int moe_policy_route(moe_policy *p, int layer, const int32_t *ids, int n, uint8_t *hit,
                             int32_t *load_expert, int32_t *evict_layer, int32_t *evict_expert,
                             int *n_loads);

/* A whole token's routing in one call, as a chained decode step reports it after
 * the step: ids [n_layers][K] (host), row l the event of layer l, routed for
 * layers 0 .. n_layers - 1 in that order. Exactly the decisions of n_layers calls
 * of moe_policy_route in layer order. hit [n_layers][K] (host, may be NULL). The
 * loads of all events are appended in event order to load_layer / load_expert
 * with evict_layer / evict_expert (cap entries each; cap must be at least
 * n_layers * K for LRU and DECAYED_FREQ, and the buffers may be NULL for
 * LFU_SWAP, which loads nothing here), their number in *n_loads. Every id is
 * checked before any state changes: MOE_ERR_ARG leaves the policy as it was. */
MOE_API int moe_policy_route_token(moe_policy *p, const int32_t *ids, int n_layers, int K, uint8_t *hit,
                                   int32_t *load_layer, int32_t *load_expert, int32_t *evict_layer,
                                   int32_t *evict_expert, int cap, int *n_loads);

/* End of the current token. LFU_SWAP makes its swap round's decisions and, with
 * plan buffers, returns them (at most cap swaps are made then): load_layer /
 * load_expert with evict_layer / evict_expert, *n_swaps (NULL buffers: a replay
 * that only updates residency). The other policies advance their clock and
 * return no swaps. */
MOE_API int moe_policy_end_token(moe_policy *p, int32_t *load_layer, int32_t *load_expert,
                                 int32_t *evict_layer, int32_t *evict_expert, int cap, int *n_swaps);

/* Residency of one pair (1 / 0) and the pool's occupancy. */
MOE_API int moe_policy_resident(const moe_policy *p, int layer, int expert, int *resident);
MOE_API int moe_policy_count(const moe_policy *p, int *n_resident);

/* Offline ceiling for a demand cache (Belady: evict the resident pair whose next
 * use is farthest away, never one of the event being served) over a recorded
 * trace: ids [T][n_layers][K] (host; token-major, then layer, events of K ids),
 * the pool of `capacity` first seeded with the listed pairs (as moe_policy_seed).
 * *hits gets the number of routed ids found resident (duplicates within an event
 * count once, as in moe_policy_route). */
MOE_API int moe_policy_belady(const int32_t *ids, int T, int n_layers, int K, int n_experts, int capacity,
                              const int32_t *seed_layers, const int32_t *seed_experts, int n_seed,
                              long long *hits);

/* Apply decisions to a slot pool on `stream`: for i in 0..n-1, evict
 * (evict_layer[i], evict_expert[i]) when evict_layer[i] >= 0, then load
 * (load_layer[i], load_expert[i]) from blobs[load_layer[i] * n_experts +
 * load_expert[i]] (host pointers to canonical blobs of nbytes; pinned memory
 * keeps the copies asynchronous). Each table entry is published only after its
 * copy lands (moe_slot_load); work enqueued earlier on `stream` still sees an
 * evicted expert, so a layer's own experts are never taken from under it. */
MOE_API int moe_policy_apply(moe_slots *slots, int n_experts, const void *const *blobs, size_t nbytes,
                             const int32_t *load_layer, const int32_t *load_expert,
                             const int32_t *evict_layer, const int32_t *evict_expert, int n,
                             moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H */
