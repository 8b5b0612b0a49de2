// moe_internal.cuh -- shared definitions of the CUDA library (not part of the ABI).
//
// Device layout of one expert (written by repack.cu from the canonical blob,
// read by the expert kernels). The byte count equals the canonical blob's.
//
//   [gate/up section]  F/16 row tiles; tile r holds rows 16r..16r+15 of both the
//                      gate and the up matrix ([F][H]), as H/128 "chunks" of 128
//                      reduction indices (a last half chunk of 64 if H % 128 == 64).
//   [down section]     H/16 row tiles of the down matrix ([H][F]), chunks along F.
//
// One chunk of one matrix for a 16-row tile: the codes (CB bytes: 512 for Q2,
// 1024 for Q4) then the block scales (SB bytes: 64 for Q2, 128 for Q4); a half
// chunk holds half of each. A gate/up chunk is [gate codes][up codes][gate
// scales][up scales]; a down chunk is [codes][scales].
//
// Codes are arranged so that lane l of a warp reads its bytes with one 16-byte
// load per 512 bytes (offset 16*l, or 8*l in a Q2 half chunk) and each 32-bit
// word unpacks straight into A fragments of mma.sync.m16n8k16 (bf16, row-major
// A): fragment register a of lane (g = l/4, c = l%4) holds the weights of row
// g + 8*(a&1) at reduction indices 2c + 8*(a>>1) (+0 in the low half, +1 in the
// high half) of its 16-wide k-step.
//   Q2 word i: k-steps 2i (bit pairs p = 0..3) and 2i+1 (p = 4..7); the weight of
//              (p, half hb) sits at bits 16*hb + 2p, register a = p & 3.
//   Q4 word i: k-step i; nibble p (0..3) at bits 16*hb + 4p, register a = p.
// Scale words: word (b*8 + g) of a chunk's scale part holds the fp16 scales of
// rows g (low half) and g+8 (high half) for the chunk's block b.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

constexpr int kBlockBytes = 18;

struct QLayout {
    int kind, zp, H, F;
    int bw;              // weights per block (32 or 64)
    int cb, sb;          // code bytes / scale bytes per matrix per full chunk
    // gate/up section
    int gu_chunks;       // chunks along H (last one half if gu_half)
    int gu_half;
    int gu_chunk_bytes;  // bytes of a full gate/up chunk (2*cb + 2*sb)
    long long gu_tile_bytes;
    int gu_tiles;        // F / 16
    // down section
    int d_chunks, d_half;
    int d_chunk_bytes;   // cb + sb
    long long d_tile_bytes;
    int d_tiles;         // H / 16
    long long d_offset;  // byte offset of the down section
    long long expert_bytes;
};

inline QLayout make_layout(int kind, int zp, int H, int F) {
    QLayout L;
    L.kind = kind;
    L.zp = zp;
    L.H = H;
    L.F = F;
    L.bw = kind == MOE_Q2_64 ? 64 : 32;
    L.cb = kind == MOE_Q2_64 ? 512 : 1024;
    L.sb = kind == MOE_Q2_64 ? 64 : 128;
    L.gu_chunks = (H + 127) / 128;
    L.gu_half = (H % 128) != 0;
    L.gu_chunk_bytes = 2 * L.cb + 2 * L.sb;
    L.gu_tile_bytes = (long long)(H / 128) * L.gu_chunk_bytes + (L.gu_half ? L.gu_chunk_bytes / 2 : 0);
    L.gu_tiles = F / 16;
    L.d_chunks = (F + 127) / 128;
    L.d_half = (F % 128) != 0;
    L.d_chunk_bytes = L.cb + L.sb;
    L.d_tile_bytes = (long long)(F / 128) * L.d_chunk_bytes + (L.d_half ? L.d_chunk_bytes / 2 : 0);
    L.d_tiles = H / 16;
    L.d_offset = L.gu_tile_bytes * L.gu_tiles;
    L.expert_bytes = L.d_offset + L.d_tile_bytes * L.d_tiles;
    return L;
}

// One unit of expert work: up to `ncols` columns of one expert.
//   slot >= 0: routed expert in arena slot `slot`; columns are live pairs
//              cols[col0 .. col0+ncols) (pair p = t*K + k).
//   slot == -2: the shared expert; columns are tokens cols[col0 ..) encoded as
//              -(t+1).
struct Group {
    int slot, col0, ncols, pad;
};

// Everything the expert kernels need about one layer's weights.
struct ExpertSrc {
    const uint8_t *arena_base;  // slot s starts at arena_base + s * slot_stride
    long long slot_stride;
    int capacity;
    QLayout L;                  // routed experts
    const uint8_t *shared;      // shared expert (device layout) or null
    QLayout LS;                 // its layout (F = F_shared)
};

// ---------------------------------------------------------------- device helpers

__device__ __forceinline__ uint32_t lop_and_or(uint32_t a, uint32_t mask, uint32_t orv) {
    uint32_t d;
    // (a & mask) | orv
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(mask), "r"(orv));
    return d;
}

__device__ __forceinline__ uint32_t bf16x2_fma(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// bf16 bit patterns (exact values): 1, 1/4, 1/16.
constexpr uint32_t kBf16One = 0x3F80u, kBf16Quarter = 0x3E80u, kBf16Sixteenth = 0x3D80u;
constexpr uint32_t kMagic = 0x43004300u;  // bf16x2 {128, 128}

// bf16 bits of a small non-negative integer n (0 <= n < 256), exact.
__host__ __device__ inline uint32_t bf16_of_int(int n) {
    if (n == 0) return 0;
    int e = 0;
    while ((n >> (e + 1)) != 0) ++e;  // n in [2^e, 2^(e+1))
    uint32_t mant = ((uint32_t)n << (7 - e)) & 0x7F;  // 7 mantissa bits (exact for n < 256)
    return ((uint32_t)(127 + e) << 7) | mant;
}

// Per-format unpack constants: fma(code_bits | 128, scale_p, -(128*scale_p + zp)).
struct Unpack {
    uint32_t mul[3];  // bf16x2 {4^-p, 4^-p}
    uint32_t add[3];  // bf16x2 {-(128*4^-p + zp)}
};

__host__ __device__ inline Unpack make_unpack(int zp) {
    Unpack u;
    const uint32_t m[3] = {kBf16One, kBf16Quarter, kBf16Sixteenth};
    const int base[3] = {128, 32, 8};
    for (int p = 0; p < 3; ++p) {
        u.mul[p] = m[p] | (m[p] << 16);
        uint32_t a = bf16_of_int(base[p] + zp) | 0x8000u;  // negative
        u.add[p] = a | (a << 16);
    }
    return u;
}

// Q2 word -> 8 bf16x2 registers holding (q - zp) exactly; R[p] has the codes of
// bit pairs (2p, 16+2p).
__device__ __forceinline__ void unpack_q2(uint32_t w, const Unpack &u, uint32_t R[8]) {
    const uint32_t w6 = w >> 6, w12 = w >> 12;
    R[0] = bf16x2_fma(lop_and_or(w, 0x00030003u, kMagic), u.mul[0], u.add[0]);
    R[1] = bf16x2_fma(lop_and_or(w, 0x000C000Cu, kMagic), u.mul[1], u.add[1]);
    R[2] = bf16x2_fma(lop_and_or(w, 0x00300030u, kMagic), u.mul[2], u.add[2]);
    R[3] = bf16x2_fma(lop_and_or(w6, 0x00030003u, kMagic), u.mul[0], u.add[0]);
    R[4] = bf16x2_fma(lop_and_or(w6, 0x000C000Cu, kMagic), u.mul[1], u.add[1]);
    R[5] = bf16x2_fma(lop_and_or(w6, 0x00300030u, kMagic), u.mul[2], u.add[2]);
    R[6] = bf16x2_fma(lop_and_or(w12, 0x00030003u, kMagic), u.mul[0], u.add[0]);
    R[7] = bf16x2_fma(lop_and_or(w12, 0x000C000Cu, kMagic), u.mul[1], u.add[1]);
}

// Q4 word -> 4 bf16x2 registers holding (q - zp); R[p] has nibbles (4p, 16+4p).
__device__ __forceinline__ void unpack_q4(uint32_t w, const Unpack &u, uint32_t R[4]) {
    R[0] = bf16x2_fma(lop_and_or(w, 0x000F000Fu, kMagic), u.mul[0], u.add[0]);
    R[1] = bf16x2_fma(lop_and_or(w >> 4, 0x000F000Fu, kMagic), u.mul[0], u.add[0]);
    R[2] = bf16x2_fma(lop_and_or(w >> 8, 0x000F000Fu, kMagic), u.mul[0], u.add[0]);
    R[3] = bf16x2_fma(lop_and_or(w >> 12, 0x000F000Fu, kMagic), u.mul[0], u.add[0]);
}

// D = A(16x16 bf16) * B(16x8 bf16) + C, fp32 accumulate.
__device__ __forceinline__ void mma_bf16(float d[4], const uint32_t a[4], uint32_t b0, uint32_t b1,
                                         const float c[4]) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%10,%11,%12,%13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]),
          "f"(c[2]), "f"(c[3]));
}

__device__ __forceinline__ uint4 ldg_stream16(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint2 ldg_stream8(const void *p) {
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
                 : "=r"(v.x), "=r"(v.y)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t ldg_stream4(const void *p) {
    uint32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }

__device__ __forceinline__ float gelu_tanh_f(float g) {
    const float k0 = 0.7978845608028654f;  // sqrt(2/pi)
    return 0.5f * g * (1.0f + tanhf(k0 * (g + 0.044715f * g * g * g)));
}

__device__ __forceinline__ void set_status(uint32_t *status, uint32_t bit) {
    if (status) atomicOr(status, bit);
}

// split an fp32 value into two bf16 limbs hi + lo (|x - hi - lo| <= 2^-17 |x|)
__device__ __forceinline__ void split_bf16(float x, __nv_bfloat16 &hi, __nv_bfloat16 &lo) {
    hi = __float2bfloat16_rn(x);
    lo = __float2bfloat16_rn(x - __bfloat162float(hi));
}

}  // namespace moe

// ---------------------------------------------------------------- host helpers
namespace moe {
int set_error(int code, const char *fmt, ...);
int cuda_error(cudaError_t e, const char *what);
}  // namespace moe

#define MOE_CUDA_TRY(call)                                        \
    do {                                                          \
        cudaError_t _e = (call);                                  \
        if (_e != cudaSuccess) return ::moe::cuda_error(_e, #call); \
    } while (0)

namespace moe {

struct PlanArgs {
    const int32_t *ids;
    const float *w;
    const int32_t *offsets;
    const int32_t *perm;
    const int32_t *table;  // slot table of the routed experts, [n_layers][E]
    int layer, capacity;
    int T, K, E;
    int nc_gu, nc_d;                // columns per group
    int max_routed_gu, max_routed_d; // index of the first shared group
    int has_shared;
    int32_t *live;   // [T*K] 1 if the pair does expert work
    int32_t *cols;   // [T*K + T]
    Group *groups_gu, *groups_d;
    int32_t *n_groups;  // [3] routed group counts (gate/up, down), plan columns
    uint32_t *status;
};

// Route-weight options of one layer (moe_layer_desc's optional fields).
struct RouteOpts {
    int kind = MOE_ROUTER_SOFTMAX;            // moe_router_kind
    const float *down_scale = nullptr;        // [E] or null
    const uint8_t *drop_eligible = nullptr;   // [E] or null: no drops
    int drop_protect = 0, drop_mass = 0;      // P, M (percent)
    float *omitted = nullptr;                 // [T] or null
};

struct ExpertArgs {
    ExpertSrc src;
    const Group *groups;
    const int32_t *n_groups;  // routed group count (device)
    int max_routed;           // routed group slots (shared groups follow)
    int n_shared;             // shared groups (0 if none)
    const int32_t *cols;
    int T, K;
    const void *x;            // gate/up input [T][H] (bf16 or f32)
    float *h;                 // [T*K + T][h_ld]
    int h_ld;
    float *yp;                // [T*K + T][H]
    int act;
    Unpack un, un_s;          // unpack constants (routed, shared)
    uint32_t *status;
};

// Allow `kernel` the opt-in maximum of dynamic shared memory left beside its
// static shared memory.
int set_max_dynamic_smem(const void *kernel, int max_smem);
int init_router_attributes(int max_smem);
int init_bucket_attributes(int max_smem);
int init_expert_attributes(int max_smem);
int init_repack_attributes(int max_smem);
int repack_expert(const QLayout &L, const uint8_t *blob, uint8_t *dst, cudaStream_t stream);
int launch_router_logits(const void *x, moe_dtype xt, int T, int H, const void *Wr, moe_dtype wt,
                         const float *bias, const float *router_scale, int E, float *logits, cudaStream_t s);
int launch_topk(const float *logits, int T, int E, int K, int32_t *ids, float *w, const RouteOpts &ro,
                uint32_t *status, cudaStream_t s);
// w_out[p] = fp32(w[p] * down_scale[ids[p]]) (the route weight of pair p with its
// expert's down scale folded in; ids out of range give 0)
int launch_scale_weights(const int32_t *ids, const float *w, const float *down_scale, int P, int E, float *w_out,
                         cudaStream_t s);
int launch_bucket(const int32_t *ids, int T, int K, int E, int32_t *counts, int32_t *offsets, int32_t *perm,
                  int32_t *active, int32_t *n_active, uint32_t *status, cudaStream_t s);
int launch_plan(const PlanArgs &a, cudaStream_t s);
// Windows of more than 2,048 pairs (up to 1,024 x 1,024): the same sort and plan
// over one CTA per 1,024 pairs; `scratch` holds wide_scratch_bytes(T, K, E).
bool use_wide(int T, int K);
size_t wide_scratch_bytes(int T, int K, int E);
int launch_bucket_wide(const int32_t *ids, int T, int K, int E, int32_t *counts, int32_t *offsets, int32_t *perm,
                       int32_t *active, int32_t *n_active, int32_t *scratch, uint32_t *status, cudaStream_t s);
int launch_plan_wide(const PlanArgs &a, int32_t *scratch, cudaStream_t s);
int launch_gateup(const ExpertArgs &a, moe_dtype xt, cudaStream_t s);
int launch_down(const ExpertArgs &a, cudaStream_t s);
int launch_combine(const float *yp, const float *w, const int32_t *live, int T, int K, int H, int has_shared,
                   int accumulate, float *y, cudaStream_t s);
int launch_rmsnorm_bf16(const float *x, int T, int H, float eps, __nv_bfloat16 *out, cudaStream_t s);

}  // namespace moe
