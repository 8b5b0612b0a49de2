// expert_decode.cu -- the routed experts for decode and verify windows.
//
// Krasis white paper sec. 5.3: batched expert projections, activation/gating,
// weighted reduce; fusing the activation into the projection work cut a MoE
// layer from 30 launches to four. kairos-engine README, "Prefill and decode are
// different machines": the decode GEMV reads the quantised codes straight from
// memory with no dequantised scratch copy.
//
// Each expert's weights stream from HBM once per layer call. A warp unpacks
// 32-bit code words into bf16 A fragments holding (q - zero_point) exactly and
// multiplies them on the tensor cores (mma.sync m16n8k16, fp32 accumulate)
// against the bucket's tokens (B, one column per token). Each quantisation
// block accumulates from zero and is added to the running sum times its fp16
// scale, so the scale never touches a weight.
//
//   k_gateup:  CTA = (group, 16-row tile of gate and up), 4 warps splitting the
//              H chunks; fixed-order cross-warp sum; h = act(gate) * up.
//   k_down:    CTA = (group, 4 tiles of 16 output rows), one warp per tile;
//              y_pair = W_down h, unweighted, per (token, rank) pair.
//   k_combine: y[t] = sum_k w[t][k] y_pair[t*K+k] in k order (+ shared expert).
// fp32 inputs (x of fp32 layers, and h) enter as two bf16 limbs hi + lo in
// separate B columns, so a group holds at most 4 such columns.
#include "decode_common.cuh"

namespace moe {

namespace {

constexpr int kWarps = 4;  // down: one 16-row tile per warp

// Stream chunks [c_begin, c_end) of one tile through a window of W chunks held
// in registers (loads for the next W chunks are in flight while one computes).
template <int KIND, int NMAT, int NB, int W>
__device__ __forceinline__ void stream_chunks(const uint8_t *tile_ptr, int chunk_bytes, int cb, int sb,
                                              int c_begin, int c_end, int n_chunks, bool has_half,
                                              const BTile (&bt)[NB], const Unpack &un, int lane,
                                              float (&acc)[NMAT][NB][4]) {
    ChunkRegs<KIND> buf[W][NMAT];
    auto load = [&](int ch, ChunkRegs<KIND>(&r)[NMAT]) {
        const bool half = has_half && ch == n_chunks - 1;
        const int cbh = half ? cb / 2 : cb, sbh = half ? sb / 2 : sb;
        const uint8_t *cp = tile_ptr + (long long)ch * chunk_bytes;
#pragma unroll
        for (int m = 0; m < NMAT; ++m) load_chunk<KIND>(cp + m * cbh, cp + NMAT * cbh + m * sbh, half, lane, r[m]);
    };
#pragma unroll
    for (int j = 0; j < W; ++j)
        if (c_begin + j < c_end) load(c_begin + j, buf[j]);
    for (int base = c_begin; base < c_end; base += W) {
#pragma unroll
        for (int j = 0; j < W; ++j) {
            const int ch = base + j;
            if (ch < c_end) {
                mma_chunk<KIND, NMAT, NB>(buf[j], has_half && ch == n_chunks - 1, bt, ch * 128, un, acc);
                if (ch + W < c_end) load(ch + W, buf[j]);
            }
        }
    }
}

// token of a column value (pair p >= 0 or shared token -(t+1)) and its h / y_pair row
__device__ __forceinline__ int col_token(int cv, int K) { return cv >= 0 ? cv / K : -cv - 1; }
__device__ __forceinline__ int col_row(int cv, int T, int K) { return cv >= 0 ? cv : T * K + (-cv - 1); }

struct Task {
    Group grp;
    QLayout L;
    const uint8_t *wbase;
    int tile;  // gate/up: row tile; down: first of 4 row tiles
    bool shared;
};

// Resolve blockIdx.x into a task. Routed tasks first (max_routed groups x
// tiles_r), then shared (n_shared groups x tiles_s). Returns false if idle.
__device__ __forceinline__ bool resolve_task(const ExpertArgs &a, int tiles_r, int tiles_s, Task &t) {
    const int bid = blockIdx.x;
    const int routed_tasks = a.max_routed * tiles_r;
    if (bid < routed_tasks) {
        const int gi = bid / tiles_r;
        if (gi >= *a.n_groups) return false;
        t.grp = a.groups[gi];
        t.tile = bid % tiles_r;
        t.L = a.src.L;
        if (t.grp.slot < 0 || t.grp.slot >= a.src.capacity) {
            set_status(a.status, MOE_STATUS_BOUNDS);
            return false;
        }
        t.wbase = a.src.arena_base + (long long)t.grp.slot * a.src.slot_stride;
        t.shared = false;
    } else {
        const int b2 = bid - routed_tasks;
        const int gi = b2 / tiles_s;
        if (gi >= a.n_shared) return false;
        t.grp = a.groups[a.max_routed + gi];
        t.tile = b2 % tiles_s;
        t.L = a.src.LS;
        t.wbase = a.src.shared;
        t.shared = true;
    }
    return true;
}

template <int KIND, bool XF32>
__global__ void __launch_bounds__(32 * GuSplit<KIND>::S) k_gateup(ExpertArgs a) {
    constexpr int NW = GuSplit<KIND>::S;
    extern __shared__ __align__(16) uint8_t smem[];
    Task tk;
    if (!resolve_task(a, a.src.L.gu_tiles, a.src.shared ? a.src.LS.gu_tiles : 1, tk)) return;
    const QLayout &L = tk.L;
    const int H = L.H, ldx = H + 8;
    __nv_bfloat16 *xs = reinterpret_cast<__nv_bfloat16 *>(smem);
    float *red = reinterpret_cast<float *>(smem + (size_t)8 * ldx * sizeof(__nv_bfloat16));
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int ncols = tk.grp.ncols;
    // stage the group's tokens as bf16 B columns (fp32 x: hi in rows 0..3, lo in 4..7)
    for (int idx = tid; idx < 8 * (H / 8); idx += blockDim.x) {
        const int r = idx / (H / 8), h8 = (idx % (H / 8)) * 8;
        const int j = XF32 ? (r & 3) : r;
        uint4 out = make_uint4(0, 0, 0, 0);
        if (j < ncols) {
            const int t = col_token(a.cols[tk.grp.col0 + j], a.K);
            if constexpr (XF32) {
                const float *xp = reinterpret_cast<const float *>(a.x) + (size_t)t * H + h8;
                const float4 v0 = *reinterpret_cast<const float4 *>(xp);
                const float4 v1 = *reinterpret_cast<const float4 *>(xp + 4);
                const float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
                __nv_bfloat16 o[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    __nv_bfloat16 hi, lo;
                    split_bf16(v[q], hi, lo);
                    o[q] = r < 4 ? hi : lo;
                }
                out = *reinterpret_cast<const uint4 *>(o);
            } else {
                out = *reinterpret_cast<const uint4 *>(reinterpret_cast<const __nv_bfloat16 *>(a.x) +
                                                       (size_t)t * H + h8);
            }
        }
        *reinterpret_cast<uint4 *>(xs + (size_t)r * ldx + h8) = out;
    }
    __syncthreads();

    const Unpack un = tk.shared ? a.un_s : a.un;
    const int g = lane >> 2, c = lane & 3;
    const BTile bt[1] = {{xs + (size_t)g * ldx + 2 * c, true}};
    const int n_chunks = L.gu_chunks;
    const int c_begin = gu_chunk_begin(warp, n_chunks, NW), c_end = gu_chunk_begin(warp + 1, n_chunks, NW);
    const uint8_t *tile_ptr = tk.wbase + (long long)tk.tile * L.gu_tile_bytes;
    float acc3[2][1][4] = {};
    stream_chunks<KIND, 2, 1, 2>(tile_ptr, L.gu_chunk_bytes, L.cb, L.sb, c_begin, c_end, n_chunks, L.gu_half, bt,
                                 un, lane, acc3);
    float acc[2][4];
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[m][q] = acc3[m][0][q];
    // fixed-order sum over the NW warps
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int q = 0; q < 4; ++q) red[(warp * 32 + lane) * 8 + m * 4 + q] = acc[m][q];
    __syncthreads();
    if (warp != 0) return;
    float v[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        float s = red[lane * 8 + q];
#pragma unroll
        for (int w = 1; w < NW; ++w) s += red[(w * 32 + lane) * 8 + q];
        v[q] = s;
    }
    if constexpr (XF32) {
#pragma unroll
        for (int q = 0; q < 8; ++q) v[q] += __shfl_xor_sync(0xffffffffu, v[q], 2);
        if (c >= 2) return;
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int rr = g + 8 * (q >> 1), j = 2 * c + (q & 1);
        if (j >= ncols) continue;
        const float gv = v[q], uv = v[4 + q];
        const float act = act_f(a.act, gv);
        const int row = col_row(a.cols[tk.grp.col0 + j], a.T, a.K);
        a.h[(size_t)row * a.h_ld + tk.tile * 16 + rr] = act * uv;
    }
}

template <int KIND>
__global__ void __launch_bounds__(32 * kWarps) k_down(ExpertArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    Task tk;
    const int tiles_r = (a.src.L.d_tiles + kWarps - 1) / kWarps;
    const int tiles_s = a.src.shared ? (a.src.LS.d_tiles + kWarps - 1) / kWarps : 1;
    if (!resolve_task(a, tiles_r, tiles_s, tk)) return;
    const QLayout &L = tk.L;
    const int F = L.F, ldx = F + 8;
    __nv_bfloat16 *xs = reinterpret_cast<__nv_bfloat16 *>(smem);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int ncols = tk.grp.ncols;
    // h of the group's columns as hi (rows 0..3) and lo (rows 4..7) limbs
    for (int idx = tid; idx < 8 * (F / 8); idx += blockDim.x) {
        const int r = idx / (F / 8), f8 = (idx % (F / 8)) * 8;
        const int j = r & 3;
        uint4 out = make_uint4(0, 0, 0, 0);
        if (j < ncols) {
            const int row = col_row(a.cols[tk.grp.col0 + j], a.T, a.K);
            const float *hp = a.h + (size_t)row * a.h_ld + f8;
            const float4 v0 = *reinterpret_cast<const float4 *>(hp);
            const float4 v1 = *reinterpret_cast<const float4 *>(hp + 4);
            const float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
            __nv_bfloat16 o[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                __nv_bfloat16 hi, lo;
                split_bf16(v[q], hi, lo);
                o[q] = r < 4 ? hi : lo;
            }
            out = *reinterpret_cast<const uint4 *>(o);
        }
        *reinterpret_cast<uint4 *>(xs + (size_t)r * ldx + f8) = out;
    }
    __syncthreads();
    const int tile = tk.tile * kWarps + warp;
    if (tile >= L.d_tiles) return;
    const Unpack un = tk.shared ? a.un_s : a.un;
    const int g = lane >> 2, c = lane & 3;
    const BTile bt[1] = {{xs + (size_t)g * ldx + 2 * c, true}};
    const uint8_t *tile_ptr = tk.wbase + L.d_offset + (long long)tile * L.d_tile_bytes;
    float acc3[1][1][4] = {};
    stream_chunks<KIND, 1, 1, 2>(tile_ptr, L.d_chunk_bytes, L.cb, L.sb, 0, L.d_chunks, L.d_chunks, L.d_half, bt, un,
                                 lane, acc3);
    float acc[1][4];
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[0][q] = acc3[0][0][q];
    float v[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) v[q] = acc[0][q] + __shfl_xor_sync(0xffffffffu, acc[0][q], 2);
    if (c >= 2) return;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int rr = g + 8 * (q >> 1), j = 2 * c + (q & 1);
        if (j >= ncols) continue;
        const int row = col_row(a.cols[tk.grp.col0 + j], a.T, a.K);
        a.yp[(size_t)row * L.H + tile * 16 + rr] = v[q];
    }
}

__global__ void __launch_bounds__(256) k_combine(const float *__restrict__ yp, const float *__restrict__ w,
                                                 const int32_t *__restrict__ live, int T, int K, int H,
                                                 int has_shared, int accumulate, float *y) {
    const int j = blockIdx.x * 256 + threadIdx.x, t = blockIdx.y;
    if (j >= H) return;
    float acc = 0.f;
    for (int k = 0; k < K; ++k) {
        const int p = t * K + k;
        if (live[p]) acc = fmaf(w[p], yp[(size_t)p * H + j], acc);
    }
    if (has_shared) acc += yp[(size_t)(T * K + t) * H + j];
    float *yt = y + (size_t)t * H + j;
    *yt = accumulate ? *yt + acc : acc;
}

// k_combine on 4 consecutive outputs per thread (H % 4 == 0, 16-byte aligned
// rows): each batch of 8 pairs' loads is in flight together; the same sum in k
// order as k_combine.
__global__ void __launch_bounds__(256) k_combine4(const float *__restrict__ yp, const float *__restrict__ w,
                                                  const int32_t *__restrict__ live, int T, int K, int H,
                                                  int has_shared, int accumulate, float *y) {
    const int j = (blockIdx.x * 256 + threadIdx.x) * 4, t = blockIdx.y;
    if (j >= H) return;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k0 = 0; k0 < K; k0 += 8) {
        float4 v[8];
        float wk[8];
        bool on[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int k = k0 + u, p = t * K + k;
            on[u] = k < K && live[p] != 0;
            wk[u] = on[u] ? w[p] : 0.f;
            v[u] = on[u] ? __ldcs(reinterpret_cast<const float4 *>(yp + (size_t)p * H + j)) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            if (on[u]) {
                acc.x = fmaf(wk[u], v[u].x, acc.x);
                acc.y = fmaf(wk[u], v[u].y, acc.y);
                acc.z = fmaf(wk[u], v[u].z, acc.z);
                acc.w = fmaf(wk[u], v[u].w, acc.w);
            }
        }
    }
    if (has_shared) {
        const float4 sh = __ldcs(reinterpret_cast<const float4 *>(yp + (size_t)(T * K + t) * H + j));
        acc.x += sh.x;
        acc.y += sh.y;
        acc.z += sh.z;
        acc.w += sh.w;
    }
    float4 *yt = reinterpret_cast<float4 *>(y + (size_t)t * H + j);
    if (accumulate) {
        const float4 o = *yt;
        acc.x = o.x + acc.x;
        acc.y = o.y + acc.y;
        acc.z = o.z + acc.z;
        acc.w = o.w + acc.w;
    }
    *yt = acc;
}

__global__ void __launch_bounds__(kNormThreads) k_rmsnorm_bf16(const float *__restrict__ x, int H, float eps,
                                                               __nv_bfloat16 *__restrict__ out) {
    __shared__ float ws[kNormWarps];
    const int t = blockIdx.x, tid = threadIdx.x;
    const float *xt = x + (size_t)t * H;
    const float s = rms_partial(xt, H, tid);
    if ((tid & 31) == 0) ws[tid >> 5] = s;
    __syncthreads();
    const float r = rms_scale(ws, H, eps);
    for (int h = tid; h < H; h += kNormThreads) out[(size_t)t * H + h] = __float2bfloat16_rn(xt[h] * r);
}

}  // namespace

int launch_gateup(const ExpertArgs &a, moe_dtype xt, cudaStream_t s) {
    const int tasks = a.max_routed * a.src.L.gu_tiles + (a.src.shared ? a.n_shared * a.src.LS.gu_tiles : 0);
    if (tasks == 0) return MOE_OK;
    const int H = a.src.L.H;
    const int NW = gu_split(a.src.L.kind);
    const size_t smem = (size_t)8 * (H + 8) * 2 + (size_t)NW * 32 * 8 * 4;
#define MOE_GU_CASE(KIND, XF)                                                                          \
    {                                                                                                  \
        k_gateup<KIND, XF><<<tasks, 32 * GuSplit<KIND>::S, smem, s>>>(a);                              \
    }
    const bool f32 = xt == MOE_F32;
    if (a.src.L.kind == MOE_Q2_64) {
        if (f32) MOE_GU_CASE(MOE_Q2_64, true) else MOE_GU_CASE(MOE_Q2_64, false)
    } else {
        if (f32) MOE_GU_CASE(MOE_Q4_32, true) else MOE_GU_CASE(MOE_Q4_32, false)
    }
#undef MOE_GU_CASE
    MOE_CUDA_TRY(cudaGetLastError());
    return MOE_OK;
}

int launch_down(const ExpertArgs &a, cudaStream_t s) {
    const int tiles_r = (a.src.L.d_tiles + kWarps - 1) / kWarps;
    const int tiles_s = a.src.shared ? (a.src.LS.d_tiles + kWarps - 1) / kWarps : 0;
    const int tasks = a.max_routed * tiles_r + (a.src.shared ? a.n_shared * tiles_s : 0);
    if (tasks == 0) return MOE_OK;
    int Fmax = a.src.L.F;
    if (a.src.shared && a.src.LS.F > Fmax) Fmax = a.src.LS.F;
    const size_t smem = (size_t)8 * (Fmax + 8) * 2;
    if (a.src.L.kind == MOE_Q2_64) {
        k_down<MOE_Q2_64><<<tasks, 32 * kWarps, smem, s>>>(a);
    } else {
        k_down<MOE_Q4_32><<<tasks, 32 * kWarps, smem, s>>>(a);
    }
    MOE_CUDA_TRY(cudaGetLastError());
    return MOE_OK;
}

int init_expert_attributes(int max_smem) {
    const void *ks[] = {(const void *)k_gateup<MOE_Q2_64, true>, (const void *)k_gateup<MOE_Q2_64, false>,
                        (const void *)k_gateup<MOE_Q4_32, true>, (const void *)k_gateup<MOE_Q4_32, false>,
                        (const void *)k_down<MOE_Q2_64>, (const void *)k_down<MOE_Q4_32>};
    for (const void *k : ks) {
        int rc = set_max_dynamic_smem(k, max_smem);
        if (rc) return rc;
    }
    return MOE_OK;
}

int launch_combine(const float *yp, const float *w, const int32_t *live, int T, int K, int H, int has_shared,
                   int accumulate, float *y, cudaStream_t s) {
    if (T == 0) return MOE_OK;
    if (H % 4 == 0 && ((uintptr_t)yp & 15) == 0 && ((uintptr_t)y & 15) == 0)
        k_combine4<<<dim3((H / 4 + 255) / 256, T), 256, 0, s>>>(yp, w, live, T, K, H, has_shared, accumulate, y);
    else
        k_combine<<<dim3((H + 255) / 256, T), 256, 0, s>>>(yp, w, live, T, K, H, has_shared, accumulate, y);
    MOE_CUDA_TRY(cudaGetLastError());
    return MOE_OK;
}

int launch_rmsnorm_bf16(const float *x, int T, int H, float eps, __nv_bfloat16 *out, cudaStream_t s) {
    if (T == 0) return MOE_OK;
    k_rmsnorm_bf16<<<T, kNormThreads, 0, s>>>(x, H, eps, out);
    MOE_CUDA_TRY(cudaGetLastError());
    return MOE_OK;
}

}  // namespace moe
