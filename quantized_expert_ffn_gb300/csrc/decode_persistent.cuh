// decode_persistent.cuh -- arguments of the persistent decode kernel.
#pragma once

#include "moe_internal.cuh"

namespace moe {

constexpr int kPersistThreads = 512;
constexpr int kMaxTok = 8;             // tokens per window on this path
constexpr int kMaxPersistLayers = 48;  // layers per launch (longer stacks: several launches)
constexpr size_t kRedBytes = (kPersistThreads / 32) * 32 * 8 * sizeof(float);
constexpr int kMaxRingBytes = 16384;   // weight ring per warp (bytes)
constexpr int kCandCap = 128;          // top-K candidates per token kept by the threshold pass
constexpr int kMaxSeg = 64;            // segment maxima per token in the threshold pass
constexpr int kMaxGrid = 512;          // CTAs of one launch (one per SM)
constexpr int kMaxUnits = kMaxTok * 32 + 1;  // distinct experts of a window + the shared expert

// Words of the launch's synchronisation area (zeroed before every launch), in order:
//   u32 [4]                         stop word at [1]
//   u32 [kMaxPersistLayers][kMaxUnits]  gate/up items done per expert of the plan
//   u64 [2][T*Ep + 4*kMaxGrid]      tagged logits (token rows padded to Ep, E rounded
//                                   up to 32) and the flags of the CTAs that own no
//                                   expert (one per 32 bytes), by layer parity
//   u64 [T*H]                       tagged residual (stack)
//   u64 [T*K + T][H]                tagged down outputs per pair (+ shared, per token)
// A tagged word holds a 32-bit value in its low half and the layer that wrote it
// (+1) in its high half; a reader waits until the tag it needs is there.
struct SyncLayout {
    size_t gu_cnt, lg_t, resid_t, yp_t, bytes;
};
inline SyncLayout sync_layout(int T, int H, int E, int K, int n_layers) {
    SyncLayout S;
    auto up16 = [](size_t v) { return (v + 15) & ~size_t(15); };
    S.gu_cnt = 16;
    S.lg_t = up16(S.gu_cnt + (size_t)n_layers * kMaxUnits * 4);
    S.resid_t = S.lg_t + (size_t)2 * ((size_t)T * ((E + 31) & ~31) + 4 * kMaxGrid) * 8;
    S.yp_t = S.resid_t + (size_t)T * H * 8;
    S.bytes = S.yp_t + (size_t)(T * K + T) * H * 8;
    return S;
}

// Dynamic shared memory:
//   [wr: router rows][tab: slot-table rows, 2 layers][xs, red | hst][rings | u]
// xs (layer input) serves the input, router and gate/up phases and red the
// gate/up reduction; hst (h limbs of the CTA's down experts) replaces both in the
// down phase. The per-warp weight rings carry gate/up and down chunks; u (RMSNorm
// staging, top-K candidates) uses the same bytes while the rings are empty.
struct PersistGeom {
    size_t off_wr, off_tab, off_xs, off_red, off_u, off_hst, off_ring;
    size_t hst_bytes;  // capacity of the h staging area
    int ring_bytes;    // per-warp ring of weight chunks
    int tab_ld;        // int32 entries per slot-table row copy
    size_t bytes;      // dynamic + static shared memory of the kernel
    size_t dyn_bytes;  // dynamic part
};

struct PersistLayer {
    const void *Wr;         // router rows [E][H] (16-byte aligned)
    const float *bias;      // [E] or null
    const int32_t *table;   // slot table of the layer's slots object
    int layer, capacity;    // row of the table; slots in the pool
    const uint8_t *arena;   // slot 0 of the pool
    long long stride;       // bytes per slot
    const uint8_t *shared;  // shared expert (device layout) or null
    const float *router_scale;  // [H] or null
    RouteOpts route;            // route-weight kind, drop policy, down scale
};

struct PersistArgs {
    int n_layers, T, H, E, K, act, stack, wr_bf16, x_f32;
    int fault_layer;  // test hook: CTA 0 publishes neither its logits nor its flag at layer fault_layer (-1: off)
    float eps;
    QLayout L, LS;
    Unpack un, un_s;
    PersistGeom geom;
    const void *x;        // single layer: input [T][H]
    float *y;             // single layer: output [T][H]
    float *resid;         // stack: residual [T][H], updated in place
    float *logits;        // [T][E] the caller's logits_out, or null
    float *trace_logits;  // stack: [n_layers][T][E] or null
    __nv_bfloat16 *trace_in;  // stack: [n_layers][T][H] or null
    int32_t *ids_out;     // single layer: [T][K] or null
    __nv_bfloat16 *h_hi, *h_lo;  // [T*K + T][h_ld]
    int h_ld;
    unsigned long long *yp_t;  // [T*K + T][H] tagged per-pair down outputs
    unsigned *bar;        // the synchronisation area (SyncLayout), zeroed before each launch
    int *gu_cnt;          // [n_layers][kMaxUnits] gate/up items done per plan expert
    unsigned long long *lg_t;     // [2][T*Ep + 4*kMaxGrid] tagged logits, flags
    unsigned long long *resid_t;  // [T*H] tagged residual between the layers of a stack
    size_t sync_bytes;    // bytes of the synchronisation area
    uint32_t *status;
    PersistLayer layers[kMaxPersistLayers];
};
static_assert(sizeof(PersistArgs) <= 32764, "kernel parameters must fit in 32,764 bytes");

PersistGeom persist_geom(int kind, int T, int H, int E, int K, int F, int F_shared, int wr_bytes, int x_f32, int G,
                         size_t max_smem);

int launch_decode_persistent(const PersistArgs &a, int G, cudaStream_t s);
int persist_max_ctas(int smem_bytes, int *G);
int init_persist_attributes(int max_smem);

}  // namespace moe
