// prefill_gemm.cuh -- arguments of the tcgen05 grouped GEMMs for prefill windows.
#pragma once

#include <cuda.h>  // CUtensorMap (the encoder is reached through the runtime's driver entry point)
#include <cuda_fp16.h>

#include "moe_internal.cuh"

namespace moe {

// One launch runs the gate/up GEMM (mode 0: h = act(gate) * up, fp16, row = plan
// column) or the down GEMM (mode 1: y_pair rows, fp32) over every column group of
// the plan (groups of at most 256 live columns of one expert; the shared expert's
// groups start at max_routed) and every 128-row M-tile of the weights; or the
// router GEMM (mode 2: logits = Wr x + bias, bf16 operands) over 128-expert by
// 64-token tiles.
struct UmmaArgs {
    // 2-D tensor maps (128-byte swizzle): B rows (mode 0: x in plan
    // order, fp16; mode 1: h; mode 2: x, bf16) and, for mode 2, the router rows
    alignas(64) CUtensorMap tmap_b;
    alignas(64) CUtensorMap tmap_a;
    // modes 0 and 1: the B tensor again with boxes of 16, 32, 64 and 128 rows (CTA
    // pairs: 8 to 64, tmap_b 128), so a CTA moves the smallest box that holds its
    // rows of the group's round-up(n, 16) columns
    alignas(64) CUtensorMap tmap_bn[4];
    // packed weights as 3-D byte tensors [slot][row tile][bytes] (8-byte elements):
    // pk[0] / pk[1] routed experts, pk[2] / pk[3] the shared expert. Gate/up: [0|2]
    // boxes of the codes of a chunk (2,048 bytes x 4 row tiles), [1|3] its scales
    // (256 x 4); down: [0|2] a whole chunk (1,152 x 8), [1|3] a last half chunk (576 x 8).
    alignas(64) CUtensorMap pk[4];
    int mode;
    // mode 2
    const __nv_bfloat16 *wr;  // [E][H]
    const __nv_bfloat16 *xb;  // [T][H]
    const float *bias;        // [E] or null
    float *logits;            // [T][E]
    int E, H;
    const Group *groups;
    const int32_t *n_groups;  // routed group count (device)
    int max_routed, n_shared;
    int n_mt, n_mt_s;         // M-tiles per routed / shared group
    const int32_t *cols;      // plan columns: pair p >= 0, shared token -(t + 1)
    int T, K, act;
    ExpertSrc src;
    const __half *x16;        // gate/up B rows: x in plan-column order, [P + T][H] fp16
    __half *h16;              // [P + T][h16_ld] fp16, row = plan column
    int h16_ld;
    float *yp;                // [P + T][H] fp32: row p for pair p, P + t for the shared expert
    uint32_t *status;
};

// The GEMMs run for Q4 layouts whose H is a multiple of 128 and F of 64.
bool umma_supported(const QLayout &L);
// The router GEMM runs for bf16 x and Wr with H a multiple of 64.
bool umma_router_supported(int H);
// One CTA per SM; tiles round-robin over the CTAs.
int launch_umma(const UmmaArgs &a, int n_ctas, cudaStream_t s);
// out[i] = fp16(x[token of plan column i]) for the n_cols (device count) columns
int launch_gather_f16(const int32_t *cols, const int32_t *n_cols, const void *x, int xf32, int K, int H, int max_rows,
                      __half *out, cudaStream_t s);
// 2-D row-major tensor (rows x cols of 16-bit elements, row stride in bytes) as a
// tensor map with boxes of 64 elements x box_rows rows (<= 0: the B box) and the
// 128-byte swizzle; bf16 or fp16.
int make_tmap_2d(CUtensorMap *map, const void *base, bool bf16, unsigned long long rows, unsigned long long cols,
                 unsigned long long row_stride_bytes, int box_rows = 0);
// The packed-weight maps of one layout (routed arena or shared expert) for `mode`.
int make_packed_maps(CUtensorMap maps[2], int mode, const QLayout &L, const uint8_t *base, long long slot_stride,
                     int n_slots);
int init_umma_attributes(int max_smem);
// The kernel's shared memory (dynamic + static) fits in max_smem bytes per block.
bool umma_fits(int max_smem);

}  // namespace moe
