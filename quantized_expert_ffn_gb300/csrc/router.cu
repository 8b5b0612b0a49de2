// router.cu -- router GEMV (logits = Wr x + bias) and softmax top-K.
//
// kairos-engine README, "The MoE forward": run the router GEMM to get the
// per-expert logits, take the top-k. Krasis white paper sec. 14.5: spreading the
// routing GEMV over many blocks beat one fused 512-thread block by 2.2x, so the
// GEMV here is a grid over experts and tokens, and top-K is a second kernel.
#include "moe_internal.cuh"

namespace moe {

namespace {

constexpr int kRouterTok = 8;   // tokens per CTA
constexpr int kRouterWarps = 8; // experts per CTA (one warp each)

template <typename T>
__device__ __forceinline__ void load8(const T *p, float v[8]);

template <>
__device__ __forceinline__ void load8<float>(const float *p, float v[8]) {
    const float4 a = *reinterpret_cast<const float4 *>(p);
    const float4 b = *reinterpret_cast<const float4 *>(p + 4);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

template <>
__device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16 *p, float v[8]) {
    const uint4 a = *reinterpret_cast<const uint4 *>(p);
    const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

// grid (ceil(E/8), ceil(T/8)), 256 threads. Each lane accumulates the products of
// its strided slice of h in a fixed order, then a fixed butterfly; a token's
// logit does not depend on which other tokens share the CTA.
template <typename XT, typename WT>
__global__ void __launch_bounds__(256) k_router_logits(const XT *__restrict__ x, const WT *__restrict__ Wr,
                                                       const float *__restrict__ bias, int T, int H, int E,
                                                       float *__restrict__ logits) {
    extern __shared__ __align__(16) float xs[];  // [8][H]
    const int t0 = blockIdx.y * kRouterTok;
    const int nt = min(kRouterTok, T - t0);
    for (int i = threadIdx.x; i < kRouterTok * H / 8; i += blockDim.x) {
        const int t = i / (H / 8), h = (i % (H / 8)) * 8;
        float v[8];
        if (t < nt) {
            load8<XT>(x + (size_t)(t0 + t) * H + h, v);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = 0.f;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) xs[t * H + h + j] = v[j];
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = blockIdx.x * kRouterWarps + warp;
    if (e >= E) return;
    float acc[kRouterTok];
#pragma unroll
    for (int t = 0; t < kRouterTok; ++t) acc[t] = 0.f;
    const WT *wrow = Wr + (size_t)e * H;
    for (int h = lane * 8; h < H; h += 256) {
        float wv[8];
        load8<WT>(wrow + h, wv);
#pragma unroll
        for (int t = 0; t < kRouterTok; ++t) {
            const float4 xa = *reinterpret_cast<const float4 *>(&xs[t * H + h]);
            const float4 xb = *reinterpret_cast<const float4 *>(&xs[t * H + h + 4]);
            float a = acc[t];
            a = fmaf(wv[0], xa.x, a); a = fmaf(wv[1], xa.y, a);
            a = fmaf(wv[2], xa.z, a); a = fmaf(wv[3], xa.w, a);
            a = fmaf(wv[4], xb.x, a); a = fmaf(wv[5], xb.y, a);
            a = fmaf(wv[6], xb.z, a); a = fmaf(wv[7], xb.w, a);
            acc[t] = a;
        }
    }
#pragma unroll
    for (int t = 0; t < kRouterTok; ++t) {
        float a = acc[t];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
        acc[t] = a;
    }
    if (lane == 0) {
        const float b = bias ? bias[e] : 0.f;
        for (int t = 0; t < nt; ++t) logits[(size_t)(t0 + t) * E + e] = acc[t] + b;
    }
}

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

constexpr int kTopkWarps = 8;

// One warp per token: K rounds of a warp arg-max over the not-yet-chosen logits
// (the order is total, so the winner does not depend on the reduction tree),
// then the softmax of the K chosen logits (= the full softmax renormalised).
__global__ void __launch_bounds__(256) k_topk(const float *__restrict__ logits, int T, int E, int K,
                                              int32_t *__restrict__ ids, float *__restrict__ w,
                                              uint32_t *status) {
    extern __shared__ float ls[];  // [8][E]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * kTopkWarps + warp;
    if (t >= T) return;
    float *l = ls + (size_t)warp * E;
    bool bad = false;
    for (int e = lane; e < E; e += 32) {
        const float v = logits[(size_t)t * E + e];
        l[e] = v;
        bad |= !isfinite(v);
    }
    bad = __any_sync(0xffffffffu, bad);
    __syncwarp();
    uint32_t taken = 0;  // bit i: element lane + 32 i chosen
    float sel_v = 0.f;   // lane k keeps the k-th chosen logit
    for (int k = 0; k < K; ++k) {
        float bv = 0.f;
        int bi = -1;
        for (int i = 0, e = lane; e < E; ++i, e += 32) {
            if (taken & (1u << i)) continue;
            const float v = l[e];
            if (ranks_before(v, e, bv, bi)) { bv = v; bi = e; }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ranks_before(ov, oi, bv, bi)) { bv = ov; bi = oi; }
        }
        if (bi >= 0 && (bi & 31) == lane) taken |= 1u << (bi >> 5);
        if (lane == k) sel_v = bv;
        if (lane == 0) ids[(size_t)t * K + k] = bi;
    }
    if (bad) {
        if (lane == 0) set_status(status, MOE_STATUS_NONFINITE);
        if (lane < K) w[(size_t)t * K + lane] = __int_as_float(0x7fc00000);
        return;
    }
    // softmax over the chosen logits; the first chosen is the maximum
    const float m = __shfl_sync(0xffffffffu, sel_v, 0);
    const float ex = lane < K ? expf(sel_v - m) : 0.f;
    float s = 0.f;
    for (int k = 0; k < K; ++k) s += __shfl_sync(0xffffffffu, ex, k);  // in k order
    if (lane < K) w[(size_t)t * K + lane] = ex / s;
}

}  // namespace

int launch_router_logits(const void *x, moe_dtype xt, int T, int H, const void *Wr, moe_dtype wt,
                         const float *bias, int E, float *logits, cudaStream_t s) {
    if (T == 0) return MOE_OK;
    const dim3 grid((E + kRouterWarps - 1) / kRouterWarps, (T + kRouterTok - 1) / kRouterTok);
    const size_t smem = (size_t)kRouterTok * H * sizeof(float);
    if (smem > 200 * 1024) return set_error(MOE_ERR_SHAPE, "router: H=%d too large", H);
#define MOE_ROUTER_CASE(XT, WT)                                                                     \
    {                                                                                               \
        k_router_logits<XT, WT><<<grid, 256, smem, s>>>((const XT *)x, (const WT *)Wr, bias, T, H, E, logits); \
    }
    if (xt == MOE_F32 && wt == MOE_F32) MOE_ROUTER_CASE(float, float)
    else if (xt == MOE_F32 && wt == MOE_BF16) MOE_ROUTER_CASE(float, __nv_bfloat16)
    else if (xt == MOE_BF16 && wt == MOE_F32) MOE_ROUTER_CASE(__nv_bfloat16, float)
    else MOE_ROUTER_CASE(__nv_bfloat16, __nv_bfloat16)
#undef MOE_ROUTER_CASE
    MOE_CUDA_TRY(cudaGetLastError());
    return MOE_OK;
}

int launch_topk(const float *logits, int T, int E, int K, int32_t *ids, float *w, uint32_t *status,
                cudaStream_t s) {
    if (T == 0) return MOE_OK;
    const size_t smem = (size_t)kTopkWarps * E * sizeof(float);
    k_topk<<<(T + kTopkWarps - 1) / kTopkWarps, 32 * kTopkWarps, smem, s>>>(logits, T, E, K, ids, w, status);
    MOE_CUDA_TRY(cudaGetLastError());
    return MOE_OK;
}

int init_router_attributes(int max_smem) {
    const void *ks[] = {(const void *)k_router_logits<float, float>, (const void *)k_router_logits<float, __nv_bfloat16>,
                        (const void *)k_router_logits<__nv_bfloat16, float>,
                        (const void *)k_router_logits<__nv_bfloat16, __nv_bfloat16>, (const void *)k_topk};
    for (const void *k : ks) MOE_CUDA_TRY(cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem));
    return MOE_OK;
}

}  // namespace moe
