// router.cu -- router GEMV (logits = Wr x + bias) and softmax top-K.
//
// kairos-engine README, "The MoE forward": run the router GEMM to get the
// per-expert logits, take the top-k. Krasis white paper sec. 14.5: spreading the
// routing GEMV over many blocks beat one fused 512-thread block by 2.2x, so the
// GEMV here is a grid over experts and tokens, and top-K is a second kernel.
#include "decode_common.cuh"

namespace moe {

namespace {

constexpr int kRouterTok = 8;   // tokens per CTA
constexpr int kRouterExp = 16;  // experts per CTA (one warp each)

// grid (ceil(E/16), ceil(T/8)), 512 threads: warp w owns expert row 16 bx + w and
// computes the four 128-lane slot partials of the canonical order (router_partial
// with L = 32q + lane, q = 0..3) one after another, then combine_router4. The
// x rows staged in shared memory serve 16 experts.
template <typename XT, typename WT>
__global__ void __launch_bounds__(32 * kRouterExp) k_router_logits(const XT *__restrict__ x, const WT *__restrict__ Wr,
                                                                   const float *__restrict__ bias,
                                                                   const float *__restrict__ rscale, int T, int H, int E,
                                                                   float *__restrict__ logits) {
    extern __shared__ __align__(16) float xs[];  // [8][H]
    const int t0 = blockIdx.y * kRouterTok;
    const int nt = min(kRouterTok, T - t0);
    for (int i = threadIdx.x; i < nt * H / 8; i += blockDim.x) {
        const int t = i / (H / 8), h = (i % (H / 8)) * 8;
        float v[8];
        load_w8<XT>(x + (size_t)(t0 + t) * H + h, v);
        if (rscale) {
            // the scaled router input x_h * s_h, rounded to fp32
            float sc[8];
            load_w8<float>(rscale + h, sc);
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] *= sc[j];
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) xs[t * H + h + j] = v[j];
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = blockIdx.x * kRouterExp + warp;
    if (e >= E) return;
    float part[4][kRouterTok];
#pragma unroll
    for (int q = 0; q < 4; ++q)
        router_partial<WT, kRouterTok>(Wr + (size_t)e * H, H, 32 * q + lane, nt,
                                       [&](int t, int h, float v[8]) {
                                           const float4 xa = *reinterpret_cast<const float4 *>(&xs[t * H + h]);
                                           const float4 xb = *reinterpret_cast<const float4 *>(&xs[t * H + h + 4]);
                                           v[0] = xa.x; v[1] = xa.y; v[2] = xa.z; v[3] = xa.w;
                                           v[4] = xb.x; v[5] = xb.y; v[6] = xb.z; v[7] = xb.w;
                                       },
                                       part[q]);
    // every lane holds the four warp-reduced slot sums; lane t writes token t
#pragma unroll
    for (int t = 0; t < kRouterTok; ++t) {
        if (t < nt && lane == t) {
            const float p4[4] = {part[0][t], part[1][t], part[2][t], part[3][t]};
            logits[(size_t)(t0 + t) * E + e] = combine_router4(p4) + (bias ? bias[e] : 0.f);
        }
    }
}

constexpr int kTopkWarps = 8;

// One warp per token: each 32-logit chunk is sorted (warp bitonic sort on keys
// that order like the ranking rule) and merged into a running top-32; lane k
// then holds the k-th choice. The top-K set and its order are unique, so this
// agrees with any other correct selection. Weights: softmax of the K chosen
// logits (= the full softmax renormalised over them).
__global__ void __launch_bounds__(256) k_topk(const float *__restrict__ logits, int T, int E, int K,
                                              int32_t *__restrict__ ids, float *__restrict__ w, const RouteOpts ro,
                                              uint32_t *status) {
    __shared__ float fs[kTopkWarps][32];
    __shared__ int is[kTopkWarps][64];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * kTopkWarps + warp;
    if (t >= T) return;
    const int nch = (E + 31) / 32;
    const float *l = logits + (size_t)t * E;
    bool bad = false;
    unsigned long long best = 0;
    for (int ch = 0; ch < nch; ++ch) {
        bool b;
        const unsigned long long keys = topk_chunk_keys(l, E, ch, lane, b);
        bad |= b;
        best = ch == 0 ? keys : warp_merge32(best, keys, lane);
    }
    bad = __any_sync(0xffffffffu, bad);
    const int si = topk_key_index(best);
    const float sv = topk_key_value(best);
    if (lane < K) ids[(size_t)t * K + lane] = si;
    if (bad) {
        if (lane == 0) {
            set_status(status, MOE_STATUS_NONFINITE);
            if (ro.omitted) ro.omitted[t] = 0.f;
        }
        if (lane < K) w[(size_t)t * K + lane] = __int_as_float(0x7fc00000);
        return;
    }
    const float m = __shfl_sync(0xffffffffu, sv, 0);
    const float wk = route_weight(ro, sv, m, si, K, lane, fs[warp], is[warp], ro.omitted, t);
    if (lane < K) w[(size_t)t * K + lane] = wk;
}

// w_out[p] = fp32(w[p] * down_scale[ids[p]]), as route_weight folds the scale
__global__ void k_scale_weights(const int32_t *__restrict__ ids, const float *__restrict__ w,
                                const float *__restrict__ down_scale, int P, int E, float *__restrict__ w_out) {
    const int p = blockIdx.x * blockDim.x + threadIdx.x;
    if (p >= P) return;
    const int e = ids[p];
    w_out[p] = (e >= 0 && e < E) ? w[p] * down_scale[e] : 0.f;
}

}  // namespace

int launch_router_logits(const void *x, moe_dtype xt, int T, int H, const void *Wr, moe_dtype wt,
                         const float *bias, const float *router_scale, int E, float *logits, cudaStream_t s) {
    if (T == 0) return MOE_OK;
    const dim3 grid((E + kRouterExp - 1) / kRouterExp, (T + kRouterTok - 1) / kRouterTok);
    const size_t smem = (size_t)kRouterTok * H * sizeof(float);
    if (smem > 200 * 1024) return set_error(MOE_ERR_SHAPE, "router: H=%d too large", H);
#define MOE_ROUTER_CASE(XT, WT)                                                                     \
    {                                                                                               \
        k_router_logits<XT, WT><<<grid, 32 * kRouterExp, smem, s>>>((const XT *)x, (const WT *)Wr, bias, router_scale, T, H, E, logits); \
    }
    if (xt == MOE_F32 && wt == MOE_F32) MOE_ROUTER_CASE(float, float)
    else if (xt == MOE_F32 && wt == MOE_BF16) MOE_ROUTER_CASE(float, __nv_bfloat16)
    else if (xt == MOE_BF16 && wt == MOE_F32) MOE_ROUTER_CASE(__nv_bfloat16, float)
    else MOE_ROUTER_CASE(__nv_bfloat16, __nv_bfloat16)
#undef MOE_ROUTER_CASE
    MOE_CUDA_TRY(cudaGetLastError());
    return MOE_OK;
}

int launch_topk(const float *logits, int T, int E, int K, int32_t *ids, float *w, const RouteOpts &ro,
                uint32_t *status, cudaStream_t s) {
    if (T == 0) return MOE_OK;
    k_topk<<<(T + kTopkWarps - 1) / kTopkWarps, 32 * kTopkWarps, 0, s>>>(logits, T, E, K, ids, w, ro, status);
    MOE_CUDA_TRY(cudaGetLastError());
    return MOE_OK;
}

int launch_scale_weights(const int32_t *ids, const float *w, const float *down_scale, int P, int E, float *w_out,
                         cudaStream_t s) {
    if (P == 0) return MOE_OK;
    k_scale_weights<<<(P + 255) / 256, 256, 0, s>>>(ids, w, down_scale, P, E, w_out);
    MOE_CUDA_TRY(cudaGetLastError());
    return MOE_OK;
}

int init_router_attributes(int max_smem) {
    const void *ks[] = {(const void *)k_router_logits<float, float>, (const void *)k_router_logits<float, __nv_bfloat16>,
                        (const void *)k_router_logits<__nv_bfloat16, float>,
                        (const void *)k_router_logits<__nv_bfloat16, __nv_bfloat16>, (const void *)k_topk};
    for (const void *k : ks) {
        int rc = set_max_dynamic_smem(k, max_smem);
        if (rc) return rc;
    }
    return MOE_OK;
}

}  // namespace moe
