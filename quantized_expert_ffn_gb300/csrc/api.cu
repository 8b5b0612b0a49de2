// api.cu -- the C ABI declared in include/moe.h: handles, validation, the slot
// table over the device arena, workspace carving and the order of launches.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "decode_persistent.cuh"
#include "prefill_gemm.cuh"
#include "moe_internal.cuh"

struct moe_ctx {
    int device;
    uint32_t *d_status;
    int persistent;   // MOE_OPT_PERSISTENT_DECODE
    int last_path;    // MOE_OPT_LAST_PATH
    int prefill_min;  // MOE_OPT_PREFILL_MIN_T
    int max_smem;    // opt-in shared memory per block
    int fault_layer;  // MOE_OPT_TEST_SKIP_ARRIVAL (-1: off)
};

struct moe_arena {
    moe_ctx *ctx;
    uint8_t *base;
    size_t bytes;
    size_t used;
};

struct moe_slots {
    moe_ctx *ctx;
    moe_arena *arena;
    int n_layers, n_experts;
    moe_format fmt;
    int H, F;
    int capacity;
    size_t stride;          // bytes per slot (expert bytes rounded up to 256)
    uint8_t *base;          // first slot
    int32_t *d_table;       // [n_layers * n_experts], -1 = absent
    std::vector<int32_t> h_table;
    std::vector<int32_t> free_slots;  // stack of free slot indices
    moe::QLayout layout;
    uint8_t *d_staging;     // canonical blob staging for host sources
};

namespace moe {

namespace {
thread_local std::string g_last_error;

struct DeviceGuard {
    int prev = -1;
    bool ok = true;
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
        if (prev != dev) ok = cudaSetDevice(dev) == cudaSuccess;
    }
    ~DeviceGuard() {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

__global__ void k_set_entry(int32_t *table, long long idx, int32_t value) { table[idx] = value; }
__global__ void k_fill_i32(int32_t *p, long long n, int32_t value) {
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
        p[i] = value;
}

int check_format(moe_format fmt) {
    if (fmt.kind == MOE_Q2_64) {
        if (fmt.zero_point < 0 || fmt.zero_point > 3) return set_error(MOE_ERR_ARG, "Q2 zero_point %d not in 0..3", fmt.zero_point);
    } else if (fmt.kind == MOE_Q4_32) {
        if (fmt.zero_point < 0 || fmt.zero_point > 15) return set_error(MOE_ERR_ARG, "Q4 zero_point %d not in 0..15", fmt.zero_point);
    } else {
        return set_error(MOE_ERR_ARG, "unknown block format %d", fmt.kind);
    }
    return MOE_OK;
}

int check_dims(int H, int F) {
    if (H <= 0 || F <= 0 || H % 64 || F % 64 || H > 8192 || F > 8192)
        return set_error(MOE_ERR_SHAPE, "H=%d, F=%d: need positive multiples of 64, at most 8192", H, F);
    return MOE_OK;
}

// Workspace carving for one layer call of up to T tokens.
struct WsLayout {
    size_t logits, ids, w, counts, offsets, perm, active, n_active, live, cols, groups_gu, groups_d, n_groups, h, yp,
        u, x16, bar, wide, total;
    size_t sync_bytes;  // persistent path: its synchronisation area (SyncLayout)
    int max_routed_gu, max_routed_d, max_shared, h_ld;
};

WsLayout ws_layout(const moe_layer_desc *d, int T, int nc_gu) {
    WsLayout W;
    const size_t P = (size_t)T * d->K;
    const int minEP = (int)((size_t)d->E < P ? d->E : P);
    W.max_routed_gu = (int)(P / nc_gu) + minEP;
    W.max_routed_d = (int)(P / 4) + minEP;
    W.max_shared = d->shared ? (T + 3) / 4 : 0;
    W.h_ld = d->F;
    if (d->shared && d->F_shared > W.h_ld) W.h_ld = d->F_shared;
    const int max_groups = (int)(P / 4) + minEP + W.max_shared;
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t at = o; o = align256(o + bytes); return at; };
    W.logits = take((size_t)T * d->E * 4);
    W.ids = take(P * 4);
    W.w = take(P * 4);
    W.counts = take((size_t)d->E * 4);
    W.offsets = take((size_t)(d->E + 1) * 4);
    W.perm = take(P * 4);
    W.active = take((size_t)d->E * 4);
    W.n_active = take(4);
    W.live = take(P * 4);
    W.cols = take((P + T) * 4);
    W.groups_gu = take((size_t)max_groups * sizeof(Group));
    W.groups_d = take((size_t)max_groups * sizeof(Group));
    W.n_groups = take(16);
    W.h = take((P + T) * (size_t)W.h_ld * 4);
    W.yp = take((P + T) * (size_t)d->H * 4);
    W.u = take((size_t)T * d->H * 2);
    W.x16 = take((P + T) * (size_t)d->H * 2);  // x in plan-column order (tensor-core path)
    W.sync_bytes = sync_layout(T, d->H, d->E, d->K, kMaxPersistLayers).bytes;
    W.bar = take(W.sync_bytes);
    W.wide = take(use_wide(T, d->K) ? wide_scratch_bytes(T, d->K, d->E) : 0);  // multi-CTA sort and plan
    W.total = o;
    return W;
}

int check_desc(const moe_layer_desc *d) {
    if (!d || !d->slots) return set_error(MOE_ERR_ARG, "null layer description or slots");
    const moe_slots *s = d->slots;
    if (d->H != s->H || d->F != s->F || d->E != s->n_experts)
        return set_error(MOE_ERR_SHAPE, "layer (H=%d, F=%d, E=%d) does not match its slots (H=%d, F=%d, E=%d)", d->H,
                         d->F, d->E, s->H, s->F, s->n_experts);
    if (d->layer < 0 || d->layer >= s->n_layers) return set_error(MOE_ERR_ARG, "layer %d out of range", d->layer);
    if (d->E < 1 || d->E > 1024) return set_error(MOE_ERR_SHAPE, "E=%d not in 1..1024", d->E);
    if (d->K < 1 || d->K > 32 || d->K > d->E) return set_error(MOE_ERR_SHAPE, "K=%d not in 1..min(E, 32)", d->K);
    if (d->act != MOE_ACT_SWIGLU && d->act != MOE_ACT_GEGLU_TANH) return set_error(MOE_ERR_ARG, "unknown activation %d", d->act);
    if (d->router_kind < MOE_ROUTER_SOFTMAX || d->router_kind > MOE_ROUTER_SIGMOID_NORM)
        return set_error(MOE_ERR_ARG, "unknown router kind %d", d->router_kind);
    if (d->drop_eligible && (d->drop_protect_pct < 0 || d->drop_protect_pct > 100 || d->drop_mass_pct < 0 ||
                             d->drop_mass_pct > 100))
        return set_error(MOE_ERR_ARG, "drop policy %d/%d not in 0..100", d->drop_protect_pct, d->drop_mass_pct);
    if (d->router_scale && (uintptr_t)d->router_scale % 16)
        return set_error(MOE_ERR_ARG, "router_scale not 16-byte aligned");
    if (d->shared) {
        const moe_slots *sh = d->shared;
        if (sh->H != d->H || sh->F != d->F_shared || sh->fmt.kind != s->fmt.kind)
            return set_error(MOE_ERR_SHAPE, "shared expert slots (H=%d, F=%d, kind %d) do not match H=%d F_shared=%d kind %d",
                             sh->H, sh->F, sh->fmt.kind, d->H, d->F_shared, s->fmt.kind);
        if (sh->h_table.empty() || sh->h_table[0] < 0)
            return set_error(MOE_ERR_EXPERT_ABSENT, "shared expert (layer 0, expert 0 of its slots) is not loaded");
    }
    if (s->ctx == nullptr) return set_error(MOE_ERR_ARG, "slots without context");
    return MOE_OK;
}

int check_ws(void *ws, size_t ws_bytes, size_t need) {
    if (!ws && need) return set_error(MOE_ERR_ARG, "null workspace");
    if ((uintptr_t)ws % 256) return set_error(MOE_ERR_ARG, "workspace not 256-byte aligned");
    if (ws_bytes < need) return set_error(MOE_ERR_WORKSPACE, "workspace %zu bytes < %zu needed", ws_bytes, need);
    return MOE_OK;
}

// Router logits: windows of at least MOE_OPT_PREFILL_MIN_T tokens with bf16 x and
// Wr run the GEMM on the tensor cores (fp32 accumulation in tensor memory); other
// windows use the CUDA-core kernel with the canonical per-row order, as does a
// router with a per-input-dimension scale (its input x * s is fp32).
int router_logits(moe_ctx *ctx, const void *x, moe_dtype xt, int T, int H, const void *Wr, moe_dtype wt,
                  const float *bias, const float *router_scale, int E, float *logits, cudaStream_t s) {
    if (!router_scale && T >= ctx->prefill_min && xt == MOE_BF16 && wt == MOE_BF16 && umma_router_supported(H) &&
        umma_fits(ctx->max_smem) && (uintptr_t)x % 16 == 0 && (uintptr_t)Wr % 16 == 0) {
        int sms = 0;
        MOE_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, ctx->device));
        UmmaArgs ua;
        memset(&ua, 0, sizeof ua);
        ua.mode = 2;
        ua.wr = (const __nv_bfloat16 *)Wr;
        ua.xb = (const __nv_bfloat16 *)x;
        ua.bias = bias;
        ua.logits = logits;
        ua.E = E;
        ua.H = H;
        ua.T = T;
        ua.n_mt = (E + 127) / 128;
        ua.status = ctx->d_status;
        // tiles of 64 tokens: a 4,096-token window keeps 64 SMs busy instead of 16
        int rc = make_tmap_2d(&ua.tmap_b, x, true, (unsigned long long)T, (unsigned long long)H,
                              (unsigned long long)H * 2, 64);
        if (!rc) rc = make_tmap_2d(&ua.tmap_a, Wr, true, (unsigned long long)E, (unsigned long long)H,
                                   (unsigned long long)H * 2, 128);
        if (rc) return rc;
        const int tiles = ua.n_mt * ((T + 63) / 64);
        return launch_umma(ua, tiles < sms ? tiles : sms, s);
    }
    return launch_router_logits(x, xt, T, H, Wr, wt, bias, router_scale, E, logits, s);
}

RouteOpts route_opts(const moe_layer_desc *d, int T) {
    RouteOpts o;
    o.kind = d->router_kind;
    o.down_scale = d->down_scale;
    o.drop_eligible = d->drop_eligible;
    o.drop_protect = d->drop_protect_pct;
    o.drop_mass = d->drop_mass_pct;
    o.omitted = T > 0 ? d->omitted_out : nullptr;
    return o;
}

// Steps 4-6 (plan, experts, combine) given ids, w, offsets, perm.
int run_experts(moe_ctx *ctx, const moe_layer_desc *d, const void *x, moe_dtype xt, int T, const int32_t *ids,
                const float *w, const int32_t *offsets, const int32_t *perm, float *y, int accumulate,
                uint8_t *ws, const WsLayout &W, cudaStream_t s) {
    const moe_slots *sl = d->slots;
    // prefill-sized windows of Q4 experts: tcgen05 grouped GEMMs on column groups of
    // up to 256 live pairs; otherwise the mma.sync kernels on groups of 8 (4) columns
    const bool umma = T >= ctx->prefill_min && umma_supported(sl->layout) &&
                      (!d->shared || umma_supported(d->shared->layout)) &&
                      umma_fits(ctx->max_smem);
    const int nc_gu = umma ? 256 : (xt == MOE_F32 ? 4 : 8);
    PlanArgs pa;
    pa.ids = ids;
    pa.w = w;
    pa.offsets = offsets;
    pa.perm = perm;
    pa.table = sl->d_table;
    pa.layer = d->layer;
    pa.capacity = sl->capacity;
    pa.T = T;
    pa.K = d->K;
    pa.E = d->E;
    pa.nc_gu = nc_gu;
    pa.nc_d = umma ? 256 : 4;
    pa.max_routed_gu = W.max_routed_gu;
    pa.max_routed_d = W.max_routed_d;
    pa.has_shared = d->shared != nullptr;
    pa.live = (int32_t *)(ws + W.live);
    pa.cols = (int32_t *)(ws + W.cols);
    pa.groups_gu = (Group *)(ws + W.groups_gu);
    pa.groups_d = (Group *)(ws + W.groups_d);
    pa.n_groups = (int32_t *)(ws + W.n_groups);
    pa.status = ctx->d_status;
    int rc = use_wide(T, d->K) ? launch_plan_wide(pa, (int32_t *)(ws + W.wide), s) : launch_plan(pa, s);
    if (rc) return rc;

    ExpertArgs ea;
    ea.src.arena_base = sl->base;
    ea.src.slot_stride = (long long)sl->stride;
    ea.src.capacity = sl->capacity;
    ea.src.L = sl->layout;
    ea.src.shared = nullptr;
    ea.src.LS = sl->layout;
    if (d->shared) {
        const moe_slots *sh = d->shared;
        ea.src.shared = sh->base + (size_t)sh->h_table[0] * sh->stride;
        ea.src.LS = sh->layout;
    }
    ea.cols = pa.cols;
    ea.T = T;
    ea.K = d->K;
    ea.x = x;
    ea.h = (float *)(ws + W.h);
    ea.h_ld = W.h_ld;
    ea.yp = (float *)(ws + W.yp);
    ea.act = d->act;
    ea.un = make_unpack(sl->fmt.zero_point);
    ea.un_s = d->shared ? make_unpack(d->shared->fmt.zero_point) : ea.un;
    ea.status = ctx->d_status;
    if (umma) {
        // x -> fp16 rows, then the gate/up GEMM (h as fp16 in plan-column rows) and
        // the down GEMM (y_pair), then the k-ordered combine
        const int maxc = (int)(T * d->K + T);
        __half *x16 = (__half *)(ws + W.x16);
        rc = launch_gather_f16(pa.cols, pa.n_groups + 2, x, xt == MOE_F32 ? 1 : 0, d->K, d->H, maxc, x16, s);
        if (rc) return rc;
        int sms = 0;
        MOE_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, ctx->device));
        const int box0 = 16, box_big = 256;
        UmmaArgs ua;
        memset(&ua, 0, sizeof ua);
        ua.mode = 0;
        ua.groups = pa.groups_gu;
        ua.n_groups = pa.n_groups;
        ua.max_routed = W.max_routed_gu;
        ua.n_shared = d->shared ? (T + nc_gu - 1) / nc_gu : 0;
        ua.n_mt = sl->layout.F / 64;
        ua.n_mt_s = d->shared ? d->shared->layout.F / 64 : 0;
        ua.cols = pa.cols;
        ua.T = T;
        ua.K = d->K;
        ua.act = d->act;
        ua.src = ea.src;
        ua.x16 = x16;
        ua.h16 = (__half *)(ws + W.h);
        ua.h16_ld = W.h_ld;
        ua.yp = ea.yp;
        ua.status = ctx->d_status;
        rc = make_tmap_2d(&ua.tmap_b, x16, false, (unsigned long long)maxc, (unsigned long long)d->H,
                          (unsigned long long)d->H * 2, box_big);
        for (int i = 0; i < 4 && !rc; ++i)
            rc = make_tmap_2d(&ua.tmap_bn[i], x16, false, (unsigned long long)maxc, (unsigned long long)d->H,
                              (unsigned long long)d->H * 2, box0 << i);
        if (!rc) rc = make_packed_maps(&ua.pk[0], 0, sl->layout, sl->base, (long long)sl->stride, sl->capacity);
        if (!rc && d->shared) rc = make_packed_maps(&ua.pk[2], 0, d->shared->layout, ea.src.shared, 0, 1);
        if (rc) return rc;
        rc = launch_umma(ua, sms, s);
        if (rc) return rc;
        rc = make_tmap_2d(&ua.tmap_b, ua.h16, false, (unsigned long long)maxc, (unsigned long long)W.h_ld,
                          (unsigned long long)W.h_ld * 2, box_big);
        for (int i = 0; i < 4 && !rc; ++i)
            rc = make_tmap_2d(&ua.tmap_bn[i], ua.h16, false, (unsigned long long)maxc, (unsigned long long)W.h_ld,
                              (unsigned long long)W.h_ld * 2, box0 << i);
        if (!rc) rc = make_packed_maps(&ua.pk[0], 1, sl->layout, sl->base, (long long)sl->stride, sl->capacity);
        if (!rc && d->shared) rc = make_packed_maps(&ua.pk[2], 1, d->shared->layout, ea.src.shared, 0, 1);
        if (rc) return rc;
        ua.mode = 1;
        ua.groups = pa.groups_d;
        ua.n_groups = pa.n_groups + 1;
        ua.max_routed = W.max_routed_d;
        ua.n_mt = sl->layout.H / 128;
        ua.n_mt_s = d->shared ? d->shared->layout.H / 128 : 0;
        rc = launch_umma(ua, sms, s);
        if (rc) return rc;
        ctx->last_path = 2;
        return launch_combine(ea.yp, w, pa.live, T, d->K, d->H, d->shared != nullptr, accumulate, y, s);
    }
    // gate/up
    ea.groups = pa.groups_gu;
    ea.n_groups = pa.n_groups;
    ea.max_routed = W.max_routed_gu;
    ea.n_shared = d->shared ? (T + nc_gu - 1) / nc_gu : 0;
    rc = launch_gateup(ea, xt, s);
    if (rc) return rc;
    // down
    ea.groups = pa.groups_d;
    ea.n_groups = pa.n_groups + 1;
    ea.max_routed = W.max_routed_d;
    ea.n_shared = d->shared ? (T + 3) / 4 : 0;
    rc = launch_down(ea, s);
    if (rc) return rc;
    return launch_combine(ea.yp, w, pa.live, T, d->K, d->H, d->shared != nullptr, accumulate, y, s);
}

// The persistent decode kernel runs a whole step (one layer, or a chain of
// layers) in one cooperative launch when the window is small and every layer
// has the same shapes and formats. Returns MOE_OK with *used = false when it
// does not apply (the multi-kernel path then runs).
int try_persistent(moe_ctx *ctx, const moe_layer_desc *layers, int n_layers, bool stack, const void *x,
                   moe_dtype xt, int T, float *out, float *logits_out, int32_t *ids_out, void *trace_in,
                   float *trace_logits, float eps, uint8_t *ws, const WsLayout &W, cudaStream_t s, bool *used) {
    *used = false;
    ctx->last_path = 0;
    if (!ctx->persistent || T < 1 || T > kMaxTok || (xt == MOE_F32 && T > 4)) return MOE_OK;
    const moe_layer_desc &d0 = layers[0];
    if (d0.K * T > 256) return MOE_OK;
    const moe_slots *s0 = d0.slots;
    for (int l = 0; l < n_layers; ++l) {
        const moe_layer_desc &d = layers[l];
        const moe_slots *sl = d.slots;
        if (d.H != d0.H || d.E != d0.E || d.K != d0.K || d.F != d0.F || d.act != d0.act || d.wr_dtype != d0.wr_dtype ||
            sl->fmt.kind != s0->fmt.kind || sl->fmt.zero_point != s0->fmt.zero_point ||
            (d.shared != nullptr) != (d0.shared != nullptr))
            return MOE_OK;
        if (d.shared && (d.F_shared != d0.F_shared || d.shared->fmt.zero_point != d0.shared->fmt.zero_point))
            return MOE_OK;
        if ((uintptr_t)d.Wr % 16) return MOE_OK;
    }
    if (xt == MOE_BF16 && (uintptr_t)x % 16) return MOE_OK;
    if (stack && (uintptr_t)out % 16) return MOE_OK;
    int G = 0;
    const int wr_bytes = d0.wr_dtype == MOE_BF16 ? 2 : 4;
    // the grid is one CTA per SM; the geometry depends on it through the router rows
    int sms = 0;
    MOE_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, ctx->device));
    if (d0.H > 3072 || d0.F > 3072 || (d0.shared && d0.F_shared > 4096)) return MOE_OK;
    PersistGeom geom = persist_geom(s0->fmt.kind, T, d0.H, d0.E, d0.K, d0.F, d0.shared ? d0.F_shared : 0, wr_bytes,
                                    xt == MOE_F32 ? 1 : 0, sms, (size_t)ctx->max_smem);
    if (geom.ring_bytes == 0 || geom.bytes > (size_t)ctx->max_smem) return MOE_OK;
    int rc = persist_max_ctas((int)geom.bytes, &G);
    if (rc) return rc;
    if (G != sms || G > kMaxGrid) return MOE_OK;
    if ((d0.E + G - 1) / G > 16) return MOE_OK;  // router rows per CTA

    PersistArgs a;
    memset(&a, 0, sizeof a);
    a.T = T;
    a.H = d0.H;
    a.E = d0.E;
    a.K = d0.K;
    a.act = d0.act;
    a.stack = stack ? 1 : 0;
    a.wr_bf16 = d0.wr_dtype == MOE_BF16;
    a.x_f32 = xt == MOE_F32;
    a.eps = eps;
    a.fault_layer = ctx->fault_layer;
    a.L = s0->layout;
    a.LS = d0.shared ? d0.shared->layout : s0->layout;
    a.un = make_unpack(s0->fmt.zero_point);
    a.un_s = d0.shared ? make_unpack(d0.shared->fmt.zero_point) : a.un;
    a.geom = geom;
    a.x = x;
    a.y = stack ? nullptr : out;
    a.resid = stack ? out : nullptr;
    a.logits = logits_out;
    a.ids_out = ids_out;
    a.h_ld = W.h_ld;
    const size_t hrows = (size_t)T * d0.K + T;
    a.h_hi = (__nv_bfloat16 *)(ws + W.h);
    a.h_lo = a.h_hi + hrows * W.h_ld;
    const SyncLayout SL = sync_layout(T, d0.H, d0.E, d0.K, kMaxPersistLayers);
    a.bar = (unsigned *)(ws + W.bar);
    a.gu_cnt = (int *)(ws + W.bar + SL.gu_cnt);
    a.lg_t = (unsigned long long *)(ws + W.bar + SL.lg_t);
    a.resid_t = (unsigned long long *)(ws + W.bar + SL.resid_t);
    a.yp_t = (unsigned long long *)(ws + W.bar + SL.yp_t);
    a.sync_bytes = SL.bytes;
    a.status = ctx->d_status;
    for (int l0 = 0; l0 < n_layers; l0 += kMaxPersistLayers) {
        const int n = n_layers - l0 < kMaxPersistLayers ? n_layers - l0 : kMaxPersistLayers;
        a.n_layers = n;
        a.trace_in = trace_in ? (__nv_bfloat16 *)trace_in + (size_t)l0 * T * d0.H : nullptr;
        a.trace_logits = trace_logits ? trace_logits + (size_t)l0 * T * d0.E : nullptr;
        for (int l = 0; l < n; ++l) {
            const moe_layer_desc &d = layers[l0 + l];
            PersistLayer &P = a.layers[l];
            P.Wr = d.Wr;
            P.bias = d.bias;
            P.table = d.slots->d_table;
            P.layer = d.layer;
            P.capacity = d.slots->capacity;
            P.arena = d.slots->base;
            P.stride = (long long)d.slots->stride;
            P.shared = d.shared ? d.shared->base + (size_t)d.shared->h_table[0] * d.shared->stride : nullptr;
            P.router_scale = d.router_scale;
            P.route = route_opts(&d, T);
        }
        rc = launch_decode_persistent(a, G, s);
        if (rc) return rc;
    }
    *used = true;
    ctx->last_path = 1;
    return MOE_OK;
}

// Router + top-K + bucket + experts for one layer; y written or accumulated.
int layer_core(moe_ctx *ctx, const moe_layer_desc *d, const void *x, moe_dtype xt, int T, float *y, int accumulate,
               float *logits_out, int32_t *ids_out, uint8_t *ws, const WsLayout &W, cudaStream_t s) {
    float *logits = logits_out ? logits_out : (float *)(ws + W.logits);
    int32_t *ids = ids_out ? ids_out : (int32_t *)(ws + W.ids);
    float *w = (float *)(ws + W.w);
    int rc = router_logits(ctx, x, xt, T, d->H, d->Wr, d->wr_dtype, d->bias, d->router_scale, d->E, logits, s);
    if (rc) return rc;
    rc = launch_topk(logits, T, d->E, d->K, ids, w, route_opts(d, T), ctx->d_status, s);
    if (rc) return rc;
    if (use_wide(T, d->K))
        rc = launch_bucket_wide(ids, T, d->K, d->E, (int32_t *)(ws + W.counts), (int32_t *)(ws + W.offsets),
                                (int32_t *)(ws + W.perm), (int32_t *)(ws + W.active), (int32_t *)(ws + W.n_active),
                                (int32_t *)(ws + W.wide), ctx->d_status, s);
    else
        rc = launch_bucket(ids, T, d->K, d->E, (int32_t *)(ws + W.counts), (int32_t *)(ws + W.offsets),
                           (int32_t *)(ws + W.perm), (int32_t *)(ws + W.active), (int32_t *)(ws + W.n_active),
                           ctx->d_status, s);
    if (rc) return rc;
    return run_experts(ctx, d, x, xt, T, ids, w, (int32_t *)(ws + W.offsets), (int32_t *)(ws + W.perm), y,
                       accumulate, ws, W, s);
}

}  // namespace

int set_error(int code, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return code;
}

int cuda_error(cudaError_t e, const char *what) {
    return set_error(MOE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

int ctx_device(const moe_ctx *ctx) { return ctx->device; }

int set_max_dynamic_smem(const void *kernel, int max_smem) {
    cudaFuncAttributes fa;
    MOE_CUDA_TRY(cudaFuncGetAttributes(&fa, kernel));
    MOE_CUDA_TRY(cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      max_smem - (int)fa.sharedSizeBytes));
    return MOE_OK;
}

}  // namespace moe

using namespace moe;

#define MOE_GUARD(ctx)                                                                  \
    DeviceGuard _guard((ctx)->device);                                                  \
    if (!_guard.ok) return set_error(MOE_ERR_CUDA, "cudaSetDevice(%d) failed", (ctx)->device)

extern "C" {

const char *moe_last_error(void) { return g_last_error.c_str(); }

int moe_expert_bytes(moe_format fmt, int H, int F, size_t *out) {
    if (!out) return set_error(MOE_ERR_ARG, "null output");
    int rc = check_format(fmt);
    if (rc) return rc;
    rc = check_dims(H, F);
    if (rc) return rc;
    const int bw = fmt.kind == MOE_Q2_64 ? 64 : 32;
    *out = (size_t)3 * H * F / bw * kBlockBytes;
    return MOE_OK;
}

int moe_ctx_create(int device, moe_ctx **out) {
    if (!out) return set_error(MOE_ERR_ARG, "null output");
    *out = nullptr;
    int n = 0;
    if (cudaGetDeviceCount(&n) != cudaSuccess || device < 0 || device >= n)
        return set_error(MOE_ERR_CUDA, "no CUDA device %d (%d visible)", device, n);
    DeviceGuard g(device);
    if (!g.ok) return set_error(MOE_ERR_CUDA, "cudaSetDevice(%d) failed", device);
    moe_ctx *c = new moe_ctx{device, nullptr, 1, 0, 64, 0, -1};
    cudaError_t e = cudaMalloc(&c->d_status, sizeof(uint32_t));
    if (e != cudaSuccess) {
        delete c;
        return cuda_error(e, "cudaMalloc(status)");
    }
    e = cudaMemset(c->d_status, 0, sizeof(uint32_t));
    if (e != cudaSuccess) {
        cudaFree(c->d_status);
        delete c;
        return cuda_error(e, "cudaMemset(status)");
    }
    // Kernel attributes are set here once, so no compute call (and no graph
    // capture) ever changes them.
    int max_smem = 0;
    int rc = MOE_OK;
    if (cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) != cudaSuccess)
        rc = set_error(MOE_ERR_CUDA, "cudaDeviceGetAttribute(max shared memory)");
    if (!rc) rc = init_router_attributes(max_smem);
    if (!rc) rc = init_bucket_attributes(max_smem);
    if (!rc) rc = init_expert_attributes(max_smem);
    if (!rc) rc = init_repack_attributes(max_smem);
    if (!rc) rc = init_persist_attributes(max_smem);
    if (!rc) rc = init_umma_attributes(max_smem);
    c->max_smem = max_smem;
    if (rc) {
        cudaFree(c->d_status);
        delete c;
        return rc;
    }
    *out = c;
    return MOE_OK;
}

int moe_ctx_destroy(moe_ctx *ctx) {
    if (!ctx) return MOE_OK;
    {
        DeviceGuard g(ctx->device);
        cudaFree(ctx->d_status);
    }
    delete ctx;
    return MOE_OK;
}

int moe_ctx_set_option(moe_ctx *ctx, int option, int value) {
    if (!ctx) return set_error(MOE_ERR_ARG, "null context");
    if (option == MOE_OPT_PERSISTENT_DECODE) {
        ctx->persistent = value != 0;
        return MOE_OK;
    }
    if (option == MOE_OPT_LAST_PATH) return set_error(MOE_ERR_ARG, "option %d is read only", option);
    if (option == MOE_OPT_PREFILL_MIN_T) {
        if (value < 1) return set_error(MOE_ERR_ARG, "MOE_OPT_PREFILL_MIN_T must be >= 1, got %d", value);
        ctx->prefill_min = value;
        return MOE_OK;
    }
    if (option == MOE_OPT_TEST_SKIP_ARRIVAL) {
        if (value < -1) return set_error(MOE_ERR_ARG, "MOE_OPT_TEST_SKIP_ARRIVAL must be >= -1, got %d", value);
        ctx->fault_layer = value;
        return MOE_OK;
    }
    return set_error(MOE_ERR_ARG, "unknown option %d", option);
}

int moe_ctx_get_option(moe_ctx *ctx, int option, int *value) {
    if (!ctx || !value) return set_error(MOE_ERR_ARG, "null argument");
    if (option == MOE_OPT_PERSISTENT_DECODE) {
        *value = ctx->persistent;
        return MOE_OK;
    }
    if (option == MOE_OPT_LAST_PATH) {
        *value = ctx->last_path;
        return MOE_OK;
    }
    if (option == MOE_OPT_PREFILL_MIN_T) {
        *value = ctx->prefill_min;
        return MOE_OK;
    }
    if (option == MOE_OPT_TEST_SKIP_ARRIVAL) {
        *value = ctx->fault_layer;
        return MOE_OK;
    }
    return set_error(MOE_ERR_ARG, "unknown option %d", option);
}

int moe_status(moe_ctx *ctx, moe_stream_t stream, uint32_t *bits) {
    if (!ctx || !bits) return set_error(MOE_ERR_ARG, "null argument");
    MOE_GUARD(ctx);
    MOE_CUDA_TRY(cudaStreamSynchronize((cudaStream_t)stream));
    uint32_t v = 0;
    MOE_CUDA_TRY(cudaMemcpy(&v, ctx->d_status, sizeof v, cudaMemcpyDeviceToHost));
    MOE_CUDA_TRY(cudaMemset(ctx->d_status, 0, sizeof v));
    *bits = v;
    return MOE_OK;
}

int moe_arena_create(moe_ctx *ctx, size_t bytes, moe_arena **out) {
    if (!ctx || !out || bytes == 0) return set_error(MOE_ERR_ARG, "bad arena arguments");
    *out = nullptr;
    MOE_GUARD(ctx);
    void *p = nullptr;
    cudaError_t e = cudaMalloc(&p, bytes);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return set_error(MOE_ERR_NOMEM, "arena of %zu bytes: %s", bytes, cudaGetErrorString(e));
    }
    *out = new moe_arena{ctx, (uint8_t *)p, bytes, 0};
    return MOE_OK;
}

int moe_arena_destroy(moe_arena *arena) {
    if (!arena) return MOE_OK;
    {
        DeviceGuard g(arena->ctx->device);
        cudaFree(arena->base);
    }
    delete arena;
    return MOE_OK;
}

int moe_slots_create(moe_ctx *ctx, moe_arena *arena, int n_layers, int n_experts, moe_format fmt, int H, int F,
                     int capacity, moe_slots **out) {
    if (!ctx || !arena || !out) return set_error(MOE_ERR_ARG, "null argument");
    *out = nullptr;
    if (arena->ctx != ctx) return set_error(MOE_ERR_ARG, "arena belongs to another context");
    int rc = check_format(fmt);
    if (rc) return rc;
    rc = check_dims(H, F);
    if (rc) return rc;
    if (n_layers < 1 || n_experts < 1 || capacity < 1 || (long long)n_layers * n_experts > (1LL << 30))
        return set_error(MOE_ERR_ARG, "bad table size %d x %d or capacity %d", n_layers, n_experts, capacity);
    MOE_GUARD(ctx);
    QLayout L = make_layout(fmt.kind, fmt.zero_point, H, F);
    const size_t stride = align256((size_t)L.expert_bytes);
    const size_t start = align256(arena->used);
    const size_t need = stride * (size_t)capacity;
    if (start + need > arena->bytes)
        return set_error(MOE_ERR_NOMEM, "arena: %zu bytes free, %d slots need %zu", arena->bytes - start, capacity, need);
    const size_t n = (size_t)n_layers * n_experts;
    int32_t *table = nullptr;
    MOE_CUDA_TRY(cudaMalloc(&table, n * sizeof(int32_t)));
    uint8_t *staging = nullptr;
    cudaError_t e = cudaMalloc(&staging, (size_t)L.expert_bytes);
    if (e != cudaSuccess) {
        cudaFree(table);
        return cuda_error(e, "cudaMalloc(staging)");
    }
    k_fill_i32<<<256, 256>>>(table, (long long)n, -1);
    e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        cudaFree(table);
        cudaFree(staging);
        return cuda_error(e, "slot table init");
    }
    moe_slots *s = new moe_slots;
    s->ctx = ctx;
    s->arena = arena;
    s->n_layers = n_layers;
    s->n_experts = n_experts;
    s->fmt = fmt;
    s->H = H;
    s->F = F;
    s->capacity = capacity;
    s->stride = stride;
    s->base = arena->base + start;
    s->d_table = table;
    s->h_table.assign(n, -1);
    s->free_slots.resize(capacity);
    for (int i = 0; i < capacity; ++i) s->free_slots[i] = capacity - 1 - i;  // pop gives 0, 1, 2, ...
    s->layout = L;
    s->d_staging = staging;
    arena->used = start + need;
    *out = s;
    return MOE_OK;
}

int moe_slots_destroy(moe_slots *s) {
    if (!s) return MOE_OK;
    {
        DeviceGuard g(s->ctx->device);
        cudaFree(s->d_table);
        cudaFree(s->d_staging);
    }
    delete s;
    return MOE_OK;
}

int moe_slot_load(moe_slots *s, int layer, int expert, const void *blob, size_t nbytes, moe_stream_t stream) {
    if (!s || !blob) return set_error(MOE_ERR_ARG, "null argument");
    if (layer < 0 || layer >= s->n_layers || expert < 0 || expert >= s->n_experts)
        return set_error(MOE_ERR_ARG, "expert (%d, %d) outside the %d x %d table", layer, expert, s->n_layers, s->n_experts);
    if (nbytes != (size_t)s->layout.expert_bytes)
        return set_error(MOE_ERR_SHAPE, "blob of %zu bytes, expected %lld", nbytes, s->layout.expert_bytes);
    MOE_GUARD(s->ctx);
    const size_t idx = (size_t)layer * s->n_experts + expert;
    int32_t slot = s->h_table[idx];
    const bool fresh = slot < 0;
    if (fresh) {
        if (s->free_slots.empty()) return set_error(MOE_ERR_NOMEM, "no free expert slot (capacity %d)", s->capacity);
        slot = s->free_slots.back();
    }
    cudaPointerAttributes attr;
    const uint8_t *src = (const uint8_t *)blob;
    if (cudaPointerGetAttributes(&attr, blob) != cudaSuccess) {
        cudaGetLastError();
        attr.type = cudaMemoryTypeUnregistered;
    }
    const cudaStream_t cs = (cudaStream_t)stream;
    if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged) {
        MOE_CUDA_TRY(cudaMemcpyAsync(s->d_staging, blob, nbytes, cudaMemcpyHostToDevice, cs));
        src = s->d_staging;
    }
    int rc = repack_expert(s->layout, src, s->base + (size_t)slot * s->stride, cs);
    if (rc) return rc;
    if (fresh) {
        k_set_entry<<<1, 1, 0, cs>>>(s->d_table, (long long)idx, slot);
        MOE_CUDA_TRY(cudaGetLastError());
        s->free_slots.pop_back();
        s->h_table[idx] = slot;
    }
    return MOE_OK;
}

int moe_slot_evict(moe_slots *s, int layer, int expert, moe_stream_t stream) {
    if (!s) return set_error(MOE_ERR_ARG, "null slots");
    if (layer < 0 || layer >= s->n_layers || expert < 0 || expert >= s->n_experts)
        return set_error(MOE_ERR_ARG, "expert (%d, %d) outside the table", layer, expert);
    const size_t idx = (size_t)layer * s->n_experts + expert;
    const int32_t slot = s->h_table[idx];
    if (slot < 0) return MOE_OK;
    MOE_GUARD(s->ctx);
    k_set_entry<<<1, 1, 0, (cudaStream_t)stream>>>(s->d_table, (long long)idx, -1);
    MOE_CUDA_TRY(cudaGetLastError());
    s->h_table[idx] = -1;
    s->free_slots.push_back(slot);
    return MOE_OK;
}

int moe_slot_lookup(const moe_slots *s, int layer, int expert, int32_t *slot_out) {
    if (!s || !slot_out) return set_error(MOE_ERR_ARG, "null argument");
    if (layer < 0 || layer >= s->n_layers || expert < 0 || expert >= s->n_experts)
        return set_error(MOE_ERR_ARG, "expert (%d, %d) outside the table", layer, expert);
    *slot_out = s->h_table[(size_t)layer * s->n_experts + expert];
    return MOE_OK;
}

int moe_router_topk(moe_ctx *ctx, const void *x, moe_dtype xt, int T, int H, const void *Wr, moe_dtype wt,
                    const float *bias, int E, int K, float *logits_out, int32_t *ids, float *w, moe_stream_t stream) {
    if (!ctx || !x || !Wr || !ids || !w) return set_error(MOE_ERR_ARG, "null argument");
    if ((xt != MOE_F32 && xt != MOE_BF16) || (wt != MOE_F32 && wt != MOE_BF16)) return set_error(MOE_ERR_ARG, "bad dtype");
    if (T < 0 || H <= 0 || H % 8 || H > 16384) return set_error(MOE_ERR_SHAPE, "T=%d, H=%d (H %% 8 == 0, <= 16384)", T, H);
    if (E < 1 || E > 1024 || K < 1 || K > 32 || K > E) return set_error(MOE_ERR_SHAPE, "E=%d, K=%d", E, K);
    if (T == 0) return MOE_OK;
    MOE_GUARD(ctx);
    const cudaStream_t s = (cudaStream_t)stream;
    float *logits = logits_out;
    if (!logits) return set_error(MOE_ERR_ARG, "logits_out is required by this implementation (pass a [T][E] buffer)");
    int rc = router_logits(ctx, x, xt, T, H, Wr, wt, bias, nullptr, E, logits, s);
    if (rc) return rc;
    return launch_topk(logits, T, E, K, ids, w, RouteOpts{}, ctx->d_status, s);
}

int moe_bucket(moe_ctx *ctx, const int32_t *ids, int T, int K, int E, int32_t *counts, int32_t *offsets,
               int32_t *perm, int32_t *active, int32_t *n_active, moe_stream_t stream) {
    if (!ctx || !counts || !offsets || !active || !n_active || (T * K > 0 && (!ids || !perm)))
        return set_error(MOE_ERR_ARG, "null argument");
    if (T < 0 || K < 1 || K > 32 || E < 1 || E > 1024 || (long long)T * K > (1LL << 26))
        return set_error(MOE_ERR_SHAPE, "T=%d, K=%d, E=%d", T, K, E);
    MOE_GUARD(ctx);
    return launch_bucket(ids, T, K, E, counts, offsets, perm, active, n_active, ctx->d_status, (cudaStream_t)stream);
}

int moe_layer_workspace(const moe_layer_desc *desc, int T_max, size_t *bytes) {
    if (!bytes) return set_error(MOE_ERR_ARG, "null output");
    int rc = check_desc(desc);
    if (rc) return rc;
    if (T_max < 0) return set_error(MOE_ERR_ARG, "T_max < 0");
    *bytes = ws_layout(desc, T_max, 4).total;
    return MOE_OK;
}

int moe_expert_ffn(moe_ctx *ctx, const moe_layer_desc *desc, const void *x, moe_dtype xt, int T, const int32_t *ids,
                   const float *w, const int32_t *offsets, const int32_t *perm, float *y, void *ws, size_t ws_bytes,
                   moe_stream_t stream) {
    if (!ctx || !x || !ids || !w || !offsets || !perm || !y) return set_error(MOE_ERR_ARG, "null argument");
    int rc = check_desc(desc);
    if (rc) return rc;
    if (xt != MOE_F32 && xt != MOE_BF16) return set_error(MOE_ERR_ARG, "bad dtype");
    if (T < 0) return set_error(MOE_ERR_ARG, "T < 0");
    if (T == 0) return MOE_OK;
    const WsLayout W = ws_layout(desc, T, xt == MOE_F32 ? 4 : 8);
    rc = check_ws(ws, ws_bytes, ws_layout(desc, T, 4).total);
    if (rc) return rc;
    MOE_GUARD(ctx);
    if (desc->down_scale) {
        // the given route weights with each expert's down scale folded in
        float *ws_w = (float *)((uint8_t *)ws + W.w);
        rc = launch_scale_weights(ids, w, desc->down_scale, T * desc->K, desc->E, ws_w, (cudaStream_t)stream);
        if (rc) return rc;
        w = ws_w;
    }
    return run_experts(ctx, desc, x, xt, T, ids, w, offsets, perm, y, 0, (uint8_t *)ws, W, (cudaStream_t)stream);
}

int moe_layer_forward(moe_ctx *ctx, const moe_layer_desc *desc, const void *x, moe_dtype xt, int T, float *y,
                      float *logits_out, int32_t *ids_out, void *ws, size_t ws_bytes, moe_stream_t stream) {
    if (!ctx || !x || !y) return set_error(MOE_ERR_ARG, "null argument");
    int rc = check_desc(desc);
    if (rc) return rc;
    if (!desc->Wr) return set_error(MOE_ERR_ARG, "null router weights");
    if (xt != MOE_F32 && xt != MOE_BF16) return set_error(MOE_ERR_ARG, "bad dtype");
    if (T < 0) return set_error(MOE_ERR_ARG, "T < 0");
    if (T == 0) return MOE_OK;
    const WsLayout W = ws_layout(desc, T, xt == MOE_F32 ? 4 : 8);
    rc = check_ws(ws, ws_bytes, ws_layout(desc, T, 4).total);
    if (rc) return rc;
    MOE_GUARD(ctx);
    bool used = false;
    rc = try_persistent(ctx, desc, 1, false, x, xt, T, y, logits_out, ids_out, nullptr, nullptr, 0.f, (uint8_t *)ws, W,
                        (cudaStream_t)stream, &used);
    if (rc || used) return rc;
    return layer_core(ctx, desc, x, xt, T, y, 0, logits_out, ids_out, (uint8_t *)ws, W, (cudaStream_t)stream);
}

int moe_layer_forward_host(moe_ctx *ctx, const moe_layer_desc *desc, const void *x_host, moe_dtype xt, int T,
                           float *y_host, void *ws, size_t ws_bytes, moe_stream_t stream) {
    if (!ctx || !x_host || !y_host) return set_error(MOE_ERR_ARG, "null argument");
    int rc = check_desc(desc);
    if (rc) return rc;
    if (!desc->Wr) return set_error(MOE_ERR_ARG, "null router weights");
    if (xt != MOE_F32 && xt != MOE_BF16) return set_error(MOE_ERR_ARG, "bad dtype");
    if (T < 0) return set_error(MOE_ERR_ARG, "T < 0");
    if (T == 0) return MOE_OK;
    const WsLayout W = ws_layout(desc, T, xt == MOE_F32 ? 4 : 8);
    const size_t base = ws_layout(desc, T, 4).total;
    const size_t xbytes = (size_t)T * desc->H * (xt == MOE_F32 ? 4 : 2), ybytes = (size_t)T * desc->H * 4;
    rc = check_ws(ws, ws_bytes, base + align256(xbytes) + align256(ybytes));
    if (rc) return rc;
    MOE_GUARD(ctx);
    uint8_t *w8 = (uint8_t *)ws;
    void *xd = w8 + base;
    float *yd = (float *)(w8 + base + align256(xbytes));
    const cudaStream_t s = (cudaStream_t)stream;
    MOE_CUDA_TRY(cudaMemcpyAsync(xd, x_host, xbytes, cudaMemcpyHostToDevice, s));
    bool used = false;
    rc = try_persistent(ctx, desc, 1, false, xd, xt, T, yd, nullptr, nullptr, nullptr, nullptr, 0.f, w8, W, s, &used);
    if (!rc && !used) rc = layer_core(ctx, desc, xd, xt, T, yd, 0, nullptr, nullptr, w8, W, s);
    if (rc) return rc;
    MOE_CUDA_TRY(cudaMemcpyAsync(y_host, yd, ybytes, cudaMemcpyDeviceToHost, s));
    return MOE_OK;
}

int moe_rmsnorm_bf16(moe_ctx *ctx, const float *x, int T, int H, float eps, void *out, moe_stream_t stream) {
    if (!ctx || !x || !out) return set_error(MOE_ERR_ARG, "null argument");
    if (T < 0 || H <= 0 || H % 8) return set_error(MOE_ERR_SHAPE, "T=%d, H=%d", T, H);
    if (!(eps >= 0.f)) return set_error(MOE_ERR_ARG, "eps must be >= 0");
    MOE_GUARD(ctx);
    return launch_rmsnorm_bf16(x, T, H, eps, (__nv_bfloat16 *)out, (cudaStream_t)stream);
}

int moe_stack_forward(moe_ctx *ctx, const moe_layer_desc *layers, int n_layers, float *resid, int T, float eps,
                      void *trace_in, float *trace_logits, void *ws, size_t ws_bytes, moe_stream_t stream) {
    if (!ctx || !layers || !resid || n_layers < 1) return set_error(MOE_ERR_ARG, "bad stack arguments");
    if (T < 0) return set_error(MOE_ERR_ARG, "T < 0");
    if (!(eps >= 0.f)) return set_error(MOE_ERR_ARG, "eps must be >= 0");
    for (int l = 0; l < n_layers; ++l) {
        int rc = check_desc(&layers[l]);
        if (rc) return rc;
        if (!layers[l].Wr) return set_error(MOE_ERR_ARG, "layer %d: null router weights", l);
        if (layers[l].H != layers[0].H || layers[l].E != layers[0].E || layers[l].K != layers[0].K ||
            layers[l].F != layers[0].F || layers[l].wr_dtype != layers[0].wr_dtype ||
            (layers[l].shared != nullptr) != (layers[0].shared != nullptr) || layers[l].F_shared != layers[0].F_shared)
            return set_error(MOE_ERR_SHAPE, "layer %d differs in shape from layer 0", l);
    }
    if (T == 0) return MOE_OK;
    const WsLayout W = ws_layout(&layers[0], T, 8);
    int rc = check_ws(ws, ws_bytes, ws_layout(&layers[0], T, 4).total);
    if (rc) return rc;
    MOE_GUARD(ctx);
    const cudaStream_t s = (cudaStream_t)stream;
    uint8_t *w8 = (uint8_t *)ws;
    const int H = layers[0].H, E = layers[0].E;
    bool used = false;
    rc = try_persistent(ctx, layers, n_layers, true, nullptr, MOE_BF16, T, resid, nullptr, nullptr, trace_in,
                        trace_logits, eps, w8, W, s, &used);
    if (rc || used) return rc;
    for (int l = 0; l < n_layers; ++l) {
        __nv_bfloat16 *u = trace_in ? (__nv_bfloat16 *)trace_in + (size_t)l * T * H : (__nv_bfloat16 *)(w8 + W.u);
        float *lg = trace_logits ? trace_logits + (size_t)l * T * E : nullptr;
        rc = launch_rmsnorm_bf16(resid, T, H, eps, u, s);
        if (rc) return rc;
        rc = layer_core(ctx, &layers[l], u, MOE_BF16, T, resid, 1, lg, nullptr, w8, W, s);
        if (rc) return rc;
    }
    return MOE_OK;
}

int moe_stack_forward_host(moe_ctx *ctx, const moe_layer_desc *layers, int n_layers, float *resid_host, int T,
                           float eps, void *ws, size_t ws_bytes, moe_stream_t stream) {
    if (!ctx || !layers || !resid_host || n_layers < 1) return set_error(MOE_ERR_ARG, "bad stack arguments");
    int rc = check_desc(&layers[0]);
    if (rc) return rc;
    if (T < 0) return set_error(MOE_ERR_ARG, "T < 0");
    if (T == 0) return MOE_OK;
    const size_t base = ws_layout(&layers[0], T, 4).total;
    const size_t rbytes = (size_t)T * layers[0].H * 4;
    rc = check_ws(ws, ws_bytes, base + align256(rbytes));
    if (rc) return rc;
    MOE_GUARD(ctx);
    float *rd = (float *)((uint8_t *)ws + base);
    const cudaStream_t s = (cudaStream_t)stream;
    MOE_CUDA_TRY(cudaMemcpyAsync(rd, resid_host, rbytes, cudaMemcpyHostToDevice, s));
    rc = moe_stack_forward(ctx, layers, n_layers, rd, T, eps, nullptr, nullptr, ws, base, stream);
    if (rc) return rc;
    MOE_CUDA_TRY(cudaMemcpyAsync(resid_host, rd, rbytes, cudaMemcpyDeviceToHost, s));
    return MOE_OK;
}

}  // extern "C"
