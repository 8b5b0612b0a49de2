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
    int fault_layer;  // test hook: CTA 0 skips its arrival at layer fault_layer's first grid barrier (-1: off)
    float eps;
    QLayout L, LS;
    Unpack un, un_s;
    PersistGeom geom;
    const void *x;        // single layer: input [T][H]
    float *y;             // single layer: output [T][H]
    float *resid;         // stack: residual [T][H], updated in place
    float *logits;        // [T][E] (scratch, or the caller's logits_out)
    float *trace_logits;  // stack: [n_layers][T][E] or null
    __nv_bfloat16 *trace_in;  // stack: [n_layers][T][H] or null
    int32_t *ids_out;     // single layer: [T][K] or null
    __nv_bfloat16 *h_hi, *h_lo;  // [T*K + T][h_ld]
    int h_ld;
    float *yp;            // [T*K + T][H] per-pair down outputs
    int *d_cnt;           // [H/16] arrivals per output row tile
    unsigned *bar;        // [2]: arrivals, stop word; then the counters (all zeroed per launch)
    int sync_words;       // 32-bit words zeroed before each launch from bar on
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
