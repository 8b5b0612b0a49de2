// decode_common.cuh -- device code shared by the multi-kernel path
// (expert_decode.cu, router.cu) and the persistent decode kernel
// (decode_persistent.cu). Both paths call these functions so that every output
// element is computed with the same operations in the same order: a token's
// result is the same bits whichever path runs it and however many tokens share
// the window.
#pragma once

#include "moe_internal.cuh"

namespace moe {

// ---------------------------------------------------------------- expert chunks

template <int KIND>
struct ChunkRegs;
template <>
struct ChunkRegs<MOE_Q2_64> {
    uint32_t w[4];
    uint32_t s[2];
};
template <>
struct ChunkRegs<MOE_Q4_32> {
    uint32_t w[8];
    uint32_t s[4];
};

// codes at `cp`, scales at `sp` (one matrix of one chunk), for lane `lane`
template <int KIND>
__device__ __forceinline__ void load_chunk(const uint8_t *cp, const uint8_t *sp, bool half, int lane,
                                           ChunkRegs<KIND> &r) {
    const int g = lane >> 2;
    if constexpr (KIND == MOE_Q2_64) {
        if (!half) {
            const uint4 v = ldg_stream16(cp + 16 * lane);
            r.w[0] = v.x; r.w[1] = v.y; r.w[2] = v.z; r.w[3] = v.w;
            r.s[0] = ldg_stream4(sp + 4 * g);
            r.s[1] = ldg_stream4(sp + 4 * (8 + g));
        } else {
            const uint2 v = ldg_stream8(cp + 8 * lane);
            r.w[0] = v.x; r.w[1] = v.y; r.w[2] = 0; r.w[3] = 0;
            r.s[0] = ldg_stream4(sp + 4 * g);
            r.s[1] = 0;
        }
    } else {
        const uint4 v = ldg_stream16(cp + 16 * lane);
        r.w[0] = v.x; r.w[1] = v.y; r.w[2] = v.z; r.w[3] = v.w;
        r.s[0] = ldg_stream4(sp + 4 * g);
        r.s[1] = ldg_stream4(sp + 4 * (8 + g));
        if (!half) {
            const uint4 u = ldg_stream16(cp + 512 + 16 * lane);
            r.w[4] = u.x; r.w[5] = u.y; r.w[6] = u.z; r.w[7] = u.w;
            r.s[2] = ldg_stream4(sp + 4 * (16 + g));
            r.s[3] = ldg_stream4(sp + 4 * (24 + g));
        } else {
            r.w[4] = r.w[5] = r.w[6] = r.w[7] = 0;
            r.s[2] = r.s[3] = 0;
        }
    }
}

__device__ __forceinline__ void apply_scale(uint32_t s, float blk[4], float acc[4]) {
    const float lo = __half2float(__ushort_as_half((unsigned short)(s & 0xFFFFu)));
    const float hi = __half2float(__ushort_as_half((unsigned short)(s >> 16)));
    acc[0] = fmaf(lo, blk[0], acc[0]);
    acc[1] = fmaf(lo, blk[1], acc[1]);
    acc[2] = fmaf(hi, blk[2], acc[2]);
    acc[3] = fmaf(hi, blk[3], acc[3]);
    blk[0] = blk[1] = blk[2] = blk[3] = 0.f;
}

// B operand of one n8 tile: lane (g, c) reads column g at brow + k (+8); a lane
// whose column is empty passes valid = false and multiplies zeros.
struct BTile {
    const __nv_bfloat16 *row;
    bool valid;
};

__device__ __forceinline__ uint32_t ld_b(const BTile &b, int k) {
    return b.valid ? *reinterpret_cast<const uint32_t *>(b.row + k) : 0u;
}

// NMAT matrices of one chunk (k0 = absolute reduction index of the chunk) times
// NB n8 tiles of B, accumulated into acc[m][nb].
template <int KIND, int NMAT, int NB>
__device__ __forceinline__ void mma_chunk(const ChunkRegs<KIND> (&r)[NMAT], bool half, const BTile (&bt)[NB],
                                          int k0, const Unpack &un, float (&acc)[NMAT][NB][4]) {
    float blk[NMAT][NB][4];
#pragma unroll
    for (int m = 0; m < NMAT; ++m)
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) blk[m][nb][0] = blk[m][nb][1] = blk[m][nb][2] = blk[m][nb][3] = 0.f;
    if constexpr (KIND == MOE_Q2_64) {
        const int nwords = half ? 2 : 4;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if (i >= nwords) break;
            uint32_t R[NMAT][8];
#pragma unroll
            for (int m = 0; m < NMAT; ++m) unpack_q2(r[m].w[i], un, R[m]);
#pragma unroll
            for (int hs = 0; hs < 2; ++hs) {
                const int k = k0 + 16 * (2 * i + hs);
#pragma unroll
                for (int nb = 0; nb < NB; ++nb) {
                    const uint32_t b0 = ld_b(bt[nb], k), b1 = ld_b(bt[nb], k + 8);
#pragma unroll
                    for (int m = 0; m < NMAT; ++m) mma_bf16(blk[m][nb], &R[m][4 * hs], b0, b1, blk[m][nb]);
                }
            }
            if (i & 1) {
#pragma unroll
                for (int m = 0; m < NMAT; ++m)
#pragma unroll
                    for (int nb = 0; nb < NB; ++nb) apply_scale(r[m].s[i >> 1], blk[m][nb], acc[m][nb]);
            }
        }
    } else {
        const int nwords = half ? 4 : 8;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (i >= nwords) break;
            uint32_t R[NMAT][4];
#pragma unroll
            for (int m = 0; m < NMAT; ++m) unpack_q4(r[m].w[i], un, R[m]);
            const int k = k0 + 16 * i;
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) {
                const uint32_t b0 = ld_b(bt[nb], k), b1 = ld_b(bt[nb], k + 8);
#pragma unroll
                for (int m = 0; m < NMAT; ++m) mma_bf16(blk[m][nb], R[m], b0, b1, blk[m][nb]);
            }
            if (i & 1) {
#pragma unroll
                for (int m = 0; m < NMAT; ++m)
#pragma unroll
                    for (int nb = 0; nb < NB; ++nb) apply_scale(r[m].s[i >> 1], blk[m][nb], acc[m][nb]);
            }
        }
    }
}

// The canonical split of a gate/up row tile's chunks into parts: part w sums
// chunks [w*n/S, (w+1)*n/S) and the S partial sums are added in part order
// (((p0 + p1) + p2) + ...). S = 4 for both formats: four groups of four warps per
// 16-warp CTA, 608 groups on 152 SMs, so every row tile of a one-token window has a
// group of its own (400 for the H=2560, E=512, top-10 layer; 484 for the
// Gemma-shaped layer with its shared expert) and the busy warps spread evenly over
// an SM's four sub-partitions. A part is five chunks at H = 2560 (Q2, 1,152 bytes
// each) and five or six at H = 2816 (Q4, 2,304 bytes each).
template <int KIND>
struct GuSplit {
    static constexpr int S = 4;
};
__host__ __device__ __forceinline__ int gu_split(int kind) {
    (void)kind;
    return 4;
}
__device__ __forceinline__ int gu_chunk_begin(int w, int n, int S) { return w * n / S; }

// bf16 hi/lo limbs of an fp32 value
__device__ __forceinline__ uint32_t pack_bf16x2(__nv_bfloat16 a, __nv_bfloat16 b) {
    return (uint32_t)__bfloat16_as_ushort(a) | ((uint32_t)__bfloat16_as_ushort(b) << 16);
}

__device__ __forceinline__ float act_f(int act, float g) {
    return act == MOE_ACT_GEGLU_TANH ? gelu_tanh_f(g) : silu_f(g);
}

// ---------------------------------------------------------------- router

// Router dot products with the canonical order: one expert row is shared by 4
// warps (128 lanes); lane L = 32q + lane accumulates h = 8L + 1024j .. +7 (j
// ascending, fmaf in h order), an xor butterfly sums each warp, and the four warp
// sums are added in warp order ((s0 + s1) + s2) + s3 by combine_router4. A
// token's logit does not depend on the other tokens. xf(t, h, v[8]) gives 8 fp32
// inputs of token t; tokens t >= nt are skipped.
constexpr int kRouterLanes = 128;

__device__ __forceinline__ void bf16x8_to_f32(uint4 a, float v[8]) {
    const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

template <typename WT>
__device__ __forceinline__ void load_w8(const WT *p, float v[8]);
template <>
__device__ __forceinline__ void load_w8<float>(const float *p, float v[8]) {
    const float4 a = *reinterpret_cast<const float4 *>(p);
    const float4 b = *reinterpret_cast<const float4 *>(p + 4);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
template <>
__device__ __forceinline__ void load_w8<__nv_bfloat16>(const __nv_bfloat16 *p, float v[8]) {
    bf16x8_to_f32(*reinterpret_cast<const uint4 *>(p), v);
}

// Partial logits of 128-lane slot L (0..127) for up to NT tokens; returns the
// warp-reduced partial (identical in every lane of the warp).
template <typename WT, int NT, typename XF>
__device__ __forceinline__ void router_partial(const WT *wrow, int H, int L, int nt, XF xf, float (&acc)[NT]) {
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[t] = 0.f;
    for (int h = L * 8; h < H; h += kRouterLanes * 8) {
        float wv[8];
        load_w8<WT>(wrow + h, wv);
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            if (t >= nt) break;
            float xv[8];
            xf(t, h, xv);
            float a = acc[t];
#pragma unroll
            for (int j = 0; j < 8; ++j) a = fmaf(wv[j], xv[j], a);
            acc[t] = a;
        }
    }
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        if (t >= nt) break;
        float a = acc[t];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
        acc[t] = a;
    }
}

// The four warp partials of one expert row, added in warp order.
__device__ __forceinline__ float combine_router4(const float *part /* [4] */) {
    return ((part[0] + part[1]) + part[2]) + part[3];
}

// ---------------------------------------------------------------- top-k

// a ranks before b: larger value first, equal values to the lower index, NaN
// below every number (NaNs among themselves by index). idx < 0 = no candidate.
__device__ __forceinline__ bool ranks_before(float va, int ia, float vb, int ib) {
    if (ib < 0) return ia >= 0;
    if (ia < 0) return false;
    const bool na = isnan(va), nb = isnan(vb);
    if (na != nb) return nb;
    if (!na && va != vb) return va > vb;
    return ia < ib;
}

// Top-K on 64-bit keys that order exactly like ranks_before: the high word maps
// the fp32 value monotonically to an unsigned integer (NaN lowest, -0 == +0), the
// low word is ~index (the lower index wins a tie). Key 0 means "no candidate".
__device__ __forceinline__ uint32_t topk_ord(float v) {
    if (isnan(v)) return 0u;
    uint32_t b = __float_as_uint(v);
    if (v == 0.f) b = 0;
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ unsigned long long topk_key_of(uint32_t ord, int idx) {
    return ((unsigned long long)ord << 32) | (uint32_t)(0xFFFFFFFFu - (uint32_t)idx);
}

__device__ __forceinline__ unsigned long long topk_key(float v, int idx) { return topk_key_of(topk_ord(v), idx); }

__device__ __forceinline__ int topk_key_index(unsigned long long k) {
    return k ? (int)(0xFFFFFFFFu - (uint32_t)k) : -1;
}

__device__ __forceinline__ float topk_key_value(unsigned long long k) {
    const uint32_t ord = (uint32_t)(k >> 32);
    const uint32_t b = (ord & 0x80000000u) ? (ord & 0x7FFFFFFFu) : ~ord;
    return __uint_as_float(b);
}

__device__ __forceinline__ unsigned long long shfl_xor64(unsigned long long v, int m) {
    const uint32_t lo = __shfl_xor_sync(0xffffffffu, (uint32_t)v, m);
    const uint32_t hi = __shfl_xor_sync(0xffffffffu, (uint32_t)(v >> 32), m);
    return ((unsigned long long)hi << 32) | lo;
}

__device__ __forceinline__ unsigned long long shfl64(unsigned long long v, int src) {
    const uint32_t lo = __shfl_sync(0xffffffffu, (uint32_t)v, src);
    const uint32_t hi = __shfl_sync(0xffffffffu, (uint32_t)(v >> 32), src);
    return ((unsigned long long)hi << 32) | lo;
}

// Warp bitonic sort of 32 keys (one per lane), largest first.
__device__ __forceinline__ unsigned long long warp_sort32(unsigned long long key, int lane) {
#pragma unroll
    for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
            const unsigned long long o = shfl_xor64(key, j);
            const bool lower = (lane & j) == 0, desc = (lane & k) == 0;
            const bool take = (lower == desc) ? (o > key) : (o < key);
            if (take) key = o;
        }
    }
    return key;
}

// Top 32 of two lists sorted largest first (one element per lane each): the
// element-wise max of A and reversed B is bitonic and holds the 32 largest; a
// bitonic merge sorts it.
__device__ __forceinline__ unsigned long long warp_merge32(unsigned long long a, unsigned long long b, int lane) {
    const unsigned long long br = shfl64(b, 31 - lane);
    unsigned long long c = a > br ? a : br;
#pragma unroll
    for (int j = 16; j > 0; j >>= 1) {
        const unsigned long long o = shfl_xor64(c, j);
        const bool lower = (lane & j) == 0;
        c = lower ? (o > c ? o : c) : (o < c ? o : c);
    }
    return c;
}

// Sorted keys of logits chunk `ch` (32 entries) of one token.
__device__ __forceinline__ unsigned long long topk_chunk_keys(const float *l, int E, int ch, int lane, bool &bad) {
    const int e = ch * 32 + lane;
    unsigned long long key = 0;
    if (e < E) {
        const float v = l[e];
        bad = !isfinite(v);
        key = topk_key(v, e);
    } else {
        bad = false;
    }
    return warp_sort32(key, lane);
}

// Rank of candidate key `k` among n candidate keys (number of larger keys).
__device__ __forceinline__ int topk_rank(unsigned long long k, const unsigned long long *cand, int n) {
    int r = 0;
    for (int i = 0; i < n; ++i) r += cand[i] > k;
    return r;
}

// Softmax of the K chosen logits (lane k holds the k-th; the first is the
// largest): w_k = exp(l_k - l_0) / sum_j exp(l_j - l_0), the sum in k order.
__device__ __forceinline__ float topk_weight(float sel_v, int K, int lane) {
    const float m = __shfl_sync(0xffffffffu, sel_v, 0);
    const float ex = lane < K ? expf(sel_v - m) : 0.f;
    float s = 0.f;
    for (int k = 0; k < K; ++k) s += __shfl_sync(0xffffffffu, ex, k);
    return ex / s;
}

// topk_weight with the same arithmetic (m = the first chosen logit, the sum in k
// order), the exponentials exchanged through this warp's 32-float shared-memory
// scratch instead of warp shuffles
__device__ __forceinline__ float topk_weight_smem(float sel_v, float m, int K, int lane, float *scratch) {
    const float ex = lane < K ? expf(sel_v - m) : 0.f;
    scratch[lane] = ex;
    __syncwarp();
    float s = 0.f;
    for (int k = 0; k < K; ++k) s += scratch[k];
    return ex / s;
}

// Route-drop policy P/M (Krasis white paper sec. 7.2) on the K route weights of
// one token (lane k < K holds choice k: weight w, expert si): the first
// ceil(K P / 100) ranks are kept; the later ranks with an eligible expert and a
// positive weight are taken from the smallest weight up (equal weights: later rank
// first) while the dropped sum c (fp32, in that order) keeps c * 100 <= M * S, S the
// fp32 sum of the K weights in rank order; the first that does not fit ends it.
// Dropped routes get weight 0 (sec. 7.3: no renormalisation). Scratch: this warp's
// 32 floats and 64 ints of shared memory. *share = c / S (0 if S = 0).
__device__ __forceinline__ float route_drop(const RouteOpts &o, float w, int si, int K, int lane, float *fs, int *is,
                                            float *share) {
    __syncwarp();
    const int protect = (K * o.drop_protect + 99) / 100;
    const bool cand = lane < K && lane >= protect && w > 0.f && o.drop_eligible[si] != 0;
    fs[lane] = lane < K ? w : 0.f;
    is[lane] = cand ? 1 : 0;
    __syncwarp();
    float S = 0.f;
    for (int k = 0; k < K; ++k) S += fs[k];
    int r = 0;
    if (cand)
        for (int j = protect; j < K; ++j) {
            const float wj = fs[j];
            r += is[j] && (wj < w || (wj == w && j > lane));
        }
    const int nc = __popc(__ballot_sync(0xffffffffu, cand));
    if (cand) is[32 + r] = lane;
    __syncwarp();
    // every lane walks the same list in the same order
    float c = 0.f;
    int nd = 0;
    const float lim = (float)o.drop_mass * S;
    for (int i = 0; i < nc; ++i) {
        const float c2 = c + fs[is[32 + i]];
        if (c2 * 100.f <= lim) {
            c = c2;
            ++nd;
        } else {
            break;
        }
    }
    *share = S > 0.f ? c / S : 0.f;
    __syncwarp();
    return (cand && r < nd) ? 0.f : w;
}

// Route weight of choice `lane` (< K) of one token: logit sv, expert si, m = the
// largest chosen logit. The kind's weight (softmax: topk_weight_smem's arithmetic;
// sigmoid: 1 / (1 + expf(-sv)); sigmoid_norm: that over the sum of the K in rank
// order), then the drop policy, then the expert's down scale. Lane 0 writes the
// dropped share to omitted[t] when omitted is not null. Every lane of the warp calls
// it; fs / is: this warp's 32 floats and 64 ints of shared memory.
__device__ __forceinline__ float route_weight(const RouteOpts &o, float sv, float m, int si, int K, int lane,
                                              float *fs, int *is, float *omitted, int t) {
    float w;
    if (o.kind == MOE_ROUTER_SOFTMAX) {
        w = topk_weight_smem(sv, m, K, lane, fs);
    } else {
        const float sg = lane < K ? 1.f / (1.f + expf(-sv)) : 0.f;
        if (o.kind == MOE_ROUTER_SIGMOID_NORM) {
            __syncwarp();
            fs[lane] = sg;
            __syncwarp();
            float sum = 0.f;
            for (int k = 0; k < K; ++k) sum += fs[k];
            w = sg / sum;
        } else {
            w = sg;
        }
    }
    if (o.drop_eligible) {
        float share;
        w = route_drop(o, w, si, K, lane, fs, is, &share);
        if (omitted && lane == 0) omitted[t] = share;
    } else if (omitted && lane == 0) {
        omitted[t] = 0.f;
    }
    if (o.down_scale && lane < K) w *= o.down_scale[si];
    return w;
}

// ---------------------------------------------------------------- rmsnorm

// RMSNorm with the canonical 512-lane order: thread i (0..511) accumulates x_h^2
// for h = i, i+512, ... with fmaf, an xor butterfly sums each warp, and the 16
// warp sums are added in warp order; r = 1 / sqrt(sum / H + eps) and the output
// is bf16(x_h * r).
constexpr int kNormThreads = 512;
constexpr int kNormWarps = kNormThreads / 32;

// Warp-reduced partial of thread `tid` (identical in every lane of its warp).
__device__ __forceinline__ float rms_partial(const float *xt, int H, int tid) {
    float acc = 0.f;
    for (int h = tid; h < H; h += kNormThreads) acc = fmaf(xt[h], xt[h], acc);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    return acc;
}

// Scale from the 16 warp partials.
__device__ __forceinline__ float rms_scale(const float *wsum, int H, float eps) {
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kNormWarps; ++w) tot += wsum[w];
    return 1.0f / sqrtf(tot / (float)H + eps);
}

}  // namespace moe
