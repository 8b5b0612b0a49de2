// decode_persistent.cu -- one cooperative launch per decode step: every SM runs
// one CTA that walks through all the layers of the step, phase by phase, with a
// grid barrier between phases that depend on each other.
//
// Per layer (Krasis white paper sec. 5.3; kairos-engine README "The MoE forward"):
//   N  layer input: x (single layer) or u = bf16(RMSNorm(resid)) (stack), every
//      CTA for itself (no barrier needed: all read the same resid);
//   R  router logits: CTA c owns experts c, c+G, ...; their router rows were
//      prefetched into shared memory while the previous layer ran;
//   -- barrier --
//   T  top-K, weights and the plan (distinct experts, their live columns): every
//      CTA computes the same result from the logits, so no further barrier;
//   GU gate/up items (16 rows of one expert, all H) are dealt round-robin over
//      CTAs and over the 4 quads of 4 warps in a CTA; each warp streams a quarter
//      of the item's chunks through registers; h = act(gate) * up;
//   -- barrier --
//   D  output row tiles (16 rows x all chosen experts) are dealt over CTAs; the
//      warps of a CTA share the experts; the combine adds the experts in k order
//      (+ the shared expert) and writes y, or adds into resid;
//   -- barrier (stack only) --
//
// Arithmetic per output element is exactly that of the multi-kernel path
// (same device functions, same split of the reduction, same orders), so results
// match it bit for bit. Waits are bounded: a barrier that does not complete
// within about a second sets MOE_STATUS_TIMEOUT and every CTA leaves.
#include "decode_common.cuh"
#include "decode_persistent.cuh"

namespace moe {

namespace {

constexpr int kPWarps = kPersistThreads / 32;
constexpr long long kSpinCycles = 2000000000LL;  // about 1 s at GB300 clocks

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ unsigned ld_relaxed_u32(const unsigned *p) {
    unsigned v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async4(void *smem, const void *gmem) {
    const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Ask L2 to fetch [p, p + bytes) from HBM (bytes a multiple of 16, p 16-aligned).
__device__ __forceinline__ void prefetch_l2(const void *p, unsigned bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ void quad_sync(int quad) {
    asm volatile("bar.sync %0, 128;" ::"r"(quad + 1) : "memory");
}

// Barrier over all CTAs of the (co-resident) grid. bar[0] counts arrivals
// monotonically within the launch; bar[1] is the abort word. Returns false when
// the kernel must stop (this or another CTA gave up waiting).
__device__ bool grid_sync(unsigned *bar, unsigned &target, uint32_t *status, int *s_flag) {
    target += gridDim.x;
    __syncthreads();
    if (threadIdx.x == 0) {
        // release: every write of this CTA (ordered before by the bar.sync above)
        // is visible before the arrival is
        asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(bar) : "memory");
        const long long t0 = clock64();
        int stop = 0;
        while ((int)(ld_acquire_u32(bar) - target) < 0) {
            if (ld_relaxed_u32(bar + 1)) {
                stop = 1;
                break;
            }
            if (clock64() - t0 > kSpinCycles) {
                atomicExch(bar + 1, 1u);
                set_status(status, MOE_STATUS_TIMEOUT);
                stop = 1;
                break;
            }
        }
        *s_flag = stop;
    }
    __syncthreads();
    return *s_flag == 0;
}

// Dynamic shared memory: [xs: 8 rows x (H+8) bf16][wr: router rows of this
// CTA][u: top-k candidates | (gate/up reduction + down partial sums)]; offsets in
// PersistGeom (identical on host and device). The plan lives in static arrays.
struct Plan {
    int ids[256], live[256], sorted[256], cols[256], cexp[256], cslot[256];
    float w[256];
    int ustart[264], uexp[264], uslot[264];
    int misc[16];
    alignas(16) int32_t table[1024];  // slot-table row of the current layer
    float bias[16];                   // router bias of this CTA's experts
    float rpart[16][kMaxTok][4];      // router partial sums [row][token][warp]
    unsigned long long sel[kMaxTok][32];  // chosen keys per token, rank order  // 0: distinct live experts, 1: live pairs, 2: stop flag, 4..11: bad token
};

// Prefetch the router rows this CTA owns for layer l into shared memory.
__device__ void prefetch_router(const PersistArgs &a, int l, uint8_t *wr_s, int32_t *tab_s, float *bias_s) {
    const int G = gridDim.x, c = blockIdx.x;
    const int wsz = a.wr_bf16 ? 2 : 4;
    const int row_bytes = a.H * wsz;
    const uint8_t *Wr = reinterpret_cast<const uint8_t *>(a.layers[l].Wr);
    int nr = 0;
    for (int e = c; e < a.E; e += G) ++nr;
    const int per_row = row_bytes / 16;
    for (int i = threadIdx.x; i < nr * per_row; i += blockDim.x) {
        const int r = i / per_row, o = (i % per_row) * 16;
        const int e = c + r * G;
        cp_async16(wr_s + (size_t)r * row_bytes + o, Wr + (size_t)e * row_bytes + o);
    }
    if (a.layers[l].bias)
        for (int r = threadIdx.x; r < nr; r += blockDim.x) cp_async4(bias_s + r, a.layers[l].bias + c + r * G);
    // the slot-table row of this layer (E int32, E a multiple of 4 or copied by 4s)
    const int32_t *tab = a.layers[l].table + (size_t)a.layers[l].layer * a.E;
    if (((uintptr_t)tab & 15) == 0 && (a.E & 3) == 0) {
        for (int i = threadIdx.x; i < a.E / 4; i += blockDim.x) cp_async16(tab_s + 4 * i, tab + 4 * i);
    } else {
        for (int i = threadIdx.x; i < a.E; i += blockDim.x) tab_s[i] = tab[i];
    }
    cp_async_commit();
}

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

// Register window per format: Q2 chunks are half the bytes of Q4 chunks.
template <int KIND>
struct Win {
    static constexpr int GU = KIND == MOE_Q2_64 ? 2 : 1;
    static constexpr int D = KIND == MOE_Q2_64 ? 2 : 1;
};

template <int KIND, bool XF32>
__global__ void __launch_bounds__(kPersistThreads, 1) k_decode(const __grid_constant__ PersistArgs a) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    __shared__ Plan s;
    __nv_bfloat16 *const xs = reinterpret_cast<__nv_bfloat16 *>(smem_raw + a.geom.off_xs);
    uint8_t *const wr_s = smem_raw + a.geom.off_wr;
    float *const u_region = reinterpret_cast<float *>(smem_raw + a.geom.off_u);
    float *const ypart = reinterpret_cast<float *>(smem_raw + a.geom.off_yp);
    __nv_bfloat16 *const hst = reinterpret_cast<__nv_bfloat16 *>(smem_raw + a.geom.off_hst);
    const int G = gridDim.x, cta = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int T = a.T, H = a.H, E = a.E, K = a.K, P = T * K;
    const int ldx = H + 8;
    const int g = lane >> 2, c = lane & 3;
    unsigned target = 0;
    int *s_flag = &s.misc[2];

    prefetch_router(a, 0, wr_s, s.table, s.bias);
    for (int l = 0; l < a.n_layers; ++l) {
        const PersistLayer &Ly = a.layers[l];
        // ------------------------------------------------ N: layer input
        if (a.stack) {
            // rmsnorm of resid with the canonical 256-thread order, two tokens at a time;
            // resid is staged once in shared memory (one global round trip)
            float *rs = u_region;  // [T][H]
            const float4 *r4 = reinterpret_cast<const float4 *>(a.resid);
            for (int idx = tid; idx < T * H / 4; idx += blockDim.x) reinterpret_cast<float4 *>(rs)[idx] = r4[idx];
            __syncthreads();
            const int half = tid >> 8, i = tid & 255;
            float r_t[kMaxTok / 2];
            float ss[kMaxTok / 2];
#pragma unroll
            for (int j = 0; j < kMaxTok / 2; ++j) {
                const int t = half + 2 * j;
                float acc = 0.f;
                if (t < T) {
                    const float *xt = rs + (size_t)t * H;
                    for (int h = i; h < H; h += kNormThreads) acc = fmaf(xt[h], xt[h], acc);
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
                ss[j] = acc;
            }
            __shared__ float wsum[kMaxTok * 8];
            if (lane == 0) {
#pragma unroll
                for (int j = 0; j < kMaxTok / 2; ++j) {
                    const int t = half + 2 * j;
                    if (t < T) wsum[t * 8 + (i >> 5)] = ss[j];
                }
            }
            __syncthreads();
#pragma unroll
            for (int j = 0; j < kMaxTok / 2; ++j) {
                const int t = half + 2 * j;
                float tot = 0.f;
                if (t < T) {
#pragma unroll
                    for (int w = 0; w < 8; ++w) tot += wsum[t * 8 + w];
                }
                r_t[j] = 1.0f / sqrtf(tot / (float)H + a.eps);
            }
#pragma unroll
            for (int j = 0; j < kMaxTok / 2; ++j) {
                const int t = half + 2 * j;
                if (t < T) {
                    const float *xt = rs + (size_t)t * H;
                    for (int h = i; h < H; h += kNormThreads) {
                        const __nv_bfloat16 u = __float2bfloat16_rn(xt[h] * r_t[j]);
                        xs[(size_t)t * ldx + h] = u;
                        if (a.trace_in && cta == 0) a.trace_in[((size_t)l * T + t) * H + h] = u;
                    }
                }
            }
        } else if (XF32) {
            // hi limbs in rows 0..3, lo limbs in rows 4..7
            const float *x = reinterpret_cast<const float *>(a.x);
            for (int idx = tid; idx < T * H; idx += blockDim.x) {
                const int t = idx / H, h = idx % H;
                __nv_bfloat16 hi, lo;
                split_bf16(x[idx], hi, lo);
                xs[(size_t)t * ldx + h] = hi;
                xs[(size_t)(4 + t) * ldx + h] = lo;
            }
        } else {
            const uint4 *x = reinterpret_cast<const uint4 *>(a.x);
            for (int idx = tid; idx < T * H / 8; idx += blockDim.x) {
                const int t = idx / (H / 8), h8 = (idx % (H / 8)) * 8;
                *reinterpret_cast<uint4 *>(xs + (size_t)t * ldx + h8) = x[idx];
            }
        }
        cp_async_wait_all();
        __syncthreads();
        // ------------------------------------------------ R: router logits of my experts
        {
            const int wsz = a.wr_bf16 ? 2 : 4;
            const int q = warp & 3;
            const int nr = (E - cta + G - 1) / G;  // experts cta, cta + G, ...
            auto xf = [&](int t, int h, float v[8]) {
                if (XF32 && !a.stack)
                    load_w8<float>(reinterpret_cast<const float *>(a.x) + (size_t)t * H + h, v);
                else
                    bf16x8_to_f32(*reinterpret_cast<const uint4 *>(xs + (size_t)t * ldx + h), v);
            };
            for (int r = warp >> 2; r < nr; r += kPWarps / 4) {
                float acc[kMaxTok];
                const uint8_t *wrow = wr_s + (size_t)r * H * wsz;
                if (a.wr_bf16)
                    router_partial<__nv_bfloat16, kMaxTok>(reinterpret_cast<const __nv_bfloat16 *>(wrow), H,
                                                           32 * q + lane, T, xf, acc);
                else
                    router_partial<float, kMaxTok>(reinterpret_cast<const float *>(wrow), H, 32 * q + lane, T, xf,
                                                   acc);
                if (lane == 0)
                    for (int t = 0; t < T; ++t) s.rpart[r][t][q] = acc[t];
            }
            __syncthreads();
            if (tid < nr * T) {
                const int r = tid / T, t = tid % T;
                const int e = cta + r * G;
                const float v = combine_router4(&s.rpart[r][t][0]) + (Ly.bias ? s.bias[r] : 0.f);
                a.logits[(size_t)t * E + e] = v;
                if (a.trace_logits) a.trace_logits[((size_t)l * T + t) * E + e] = v;
            }
        }
        __syncthreads();
        
        if (!grid_sync(a.bar, target, a.status, s_flag)) break;
        // ------------------------------------------------ T: top-K and the plan (every CTA)
        {
            const int nch = (E + 31) / 32;
            unsigned long long *lists = reinterpret_cast<unsigned long long *>(u_region);  // [T][nch][32]
            if (tid < kMaxTok) s.misc[4 + tid] = 0;
            __syncthreads();
            for (int task = warp; task < T * nch; task += kPWarps) {
                const int t = task / nch, ch = task % nch;
                bool bad;
                const unsigned long long key = topk_chunk_keys(a.logits + (size_t)t * E, E, ch, lane, bad);
                if (__any_sync(0xffffffffu, bad) && lane == 0) s.misc[4 + t] = 1;
                lists[((size_t)t * nch + ch) * 32 + lane] = key;
            }
            __syncthreads();
            const int kc = K < 32 ? K : 32;
            const int C = nch * kc;  // candidates per token: the best kc of each chunk
            if (C <= 256) {
                // rank of each candidate among its token's candidates = its place in the top-K
                for (int idx = tid; idx < T * C; idx += blockDim.x) {
                    const int t = idx / C, c = idx % C;
                    const unsigned long long *lt = lists + (size_t)t * nch * 32;
                    const unsigned long long key = lt[(c / kc) * 32 + c % kc];
                    int r = 0;
                    for (int ch = 0; ch < nch; ++ch)
                        for (int i2 = 0; i2 < kc; ++i2) r += lt[ch * 32 + i2] > key;
                    if (r < K) s.sel[t][r] = key;
                }
                __syncthreads();
            } else {
            // merge tree: list i absorbs list i + stride (the top 32 of the union, sorted)
            for (int stride = 1; stride < nch; stride *= 2) {
                const int groups = (nch + 2 * stride - 1) / (2 * stride);
                for (int task = warp; task < T * groups; task += kPWarps) {
                    const int t = task / groups, i0 = (task % groups) * 2 * stride;
                    if (i0 + stride < nch) {
                        unsigned long long *la = lists + ((size_t)t * nch + i0) * 32;
                        const unsigned long long m = warp_merge32(la[lane], la[stride * 32 + lane], lane);
                        __syncwarp();
                        la[lane] = m;
                    }
                }
                __syncthreads();
            }
            if (tid < T * 32) s.sel[tid >> 5][tid & 31] = lists[(size_t)(tid >> 5) * nch * 32 + (tid & 31)];
            __syncthreads();
            }
            if (warp < T) {
                const int t = warp;
                const unsigned long long key = s.sel[t][lane];
                const int si = topk_key_index(key);
                const float sv = topk_key_value(key);
                const bool bad = s.misc[4 + t] != 0;
                const float wk = bad ? __int_as_float(0x7fc00000) : topk_weight(sv, K, lane);
                if (lane < K) {
                    s.ids[t * K + lane] = si;
                    s.w[t * K + lane] = wk;
                    if (a.ids_out && cta == 0) a.ids_out[(size_t)t * K + lane] = si;
                }
                if (bad && lane == 0 && cta == 0) set_status(a.status, MOE_STATUS_NONFINITE);
            }
            __syncthreads();
            // stable order of pairs by expert: rank = #{q : (id_q, q) < (id_p, p)}
            if (tid < P) {
                const int ep = s.ids[tid];
                int rank = 0;
                for (int q = 0; q < P; ++q) {
                    const int eq = s.ids[q];
                    rank += (eq < ep) || (eq == ep && q < tid);
                }
                s.sorted[rank] = tid;
            }
            __syncthreads();
            if (warp == 0) {
                int running = 0;
                bool absent = false, oob = false;
                for (int base = 0; base < P; base += 32) {
                    const int r = base + lane;
                    int p = -1, e = -1, slot = -1, live = 0;
                    if (r < P) {
                        p = s.sorted[r];
                        e = s.ids[p];
                        slot = s.table[e];
                        if (slot < 0) absent = true;
                        else if (slot >= Ly.capacity) oob = true;
                        else live = s.w[p] != 0.f;
                        s.live[p] = live;
                    }
                    const unsigned m = __ballot_sync(0xffffffffu, live);
                    if (live) {
                        const int pos = running + __popc(m & ((1u << lane) - 1));
                        s.cols[pos] = p;
                        s.cexp[pos] = e;
                        s.cslot[pos] = slot;
                    }
                    running += __popc(m);
                }
                absent = __any_sync(0xffffffffu, absent);
                oob = __any_sync(0xffffffffu, oob);
                if (cta == 0 && lane == 0) {
                    if (absent) set_status(a.status, MOE_STATUS_EXPERT_ABSENT);
                    if (oob) set_status(a.status, MOE_STATUS_BOUNDS);
                }
                __syncwarp();
                const int nlive = running;
                int nu = 0;
                for (int base = 0; base < nlive; base += 32) {
                    const int i = base + lane;
                    const bool first = i < nlive && (i == 0 || s.cexp[i - 1] != s.cexp[i]);
                    const unsigned m = __ballot_sync(0xffffffffu, first);
                    if (first) {
                        const int u = nu + __popc(m & ((1u << lane) - 1));
                        s.ustart[u] = i;
                        s.uexp[u] = s.cexp[i];
                        s.uslot[u] = s.cslot[i];
                    }
                    nu += __popc(m);
                }
                if (lane == 0) {
                    s.ustart[nu] = nlive;
                    s.misc[0] = nu;
                    s.misc[1] = nlive;
                }
            }
            __syncthreads();
        }
        const int nU = s.misc[0];
        const bool has_shared = Ly.shared != nullptr;
        // the table row and router rows of the next layer (the buffers are free now)
        if (l + 1 < a.n_layers) prefetch_router(a, l + 1, wr_s, s.table, s.bias);
        // every weight byte this CTA will read in this layer, requested from HBM now:
        // gate/up items (one request per item), then down tiles (one per expert and tile)
        {
            const int tilesF = a.L.gu_tiles;
            const int n_items = nU * tilesF + (has_shared ? a.LS.gu_tiles : 0);
            for (int j = cta + G * warp; j < n_items && warp < 4; j += G * 4) {
                if (lane == 0) {
                    const bool sh = j >= nU * tilesF;
                    const QLayout &LL = sh ? a.LS : a.L;
                    const uint8_t *wb = sh ? Ly.shared : Ly.arena + (long long)s.uslot[j / tilesF] * Ly.stride;
                    const int rt = sh ? j - nU * tilesF : j % tilesF;
                    prefetch_l2(wb + (long long)rt * LL.gu_tile_bytes, (unsigned)LL.gu_tile_bytes);
                }
            }
            const int n_tasks = nU + (has_shared ? 1 : 0);
            int k = 0;
            for (int r = cta; r < a.L.d_tiles; r += G)
                for (int ti = 0; ti < n_tasks; ++ti, ++k) {
                    if ((k % kPWarps) != warp || lane != 0) continue;
                    const bool sh = ti >= nU;
                    const QLayout &LL = sh ? a.LS : a.L;
                    const uint8_t *wb = sh ? Ly.shared : Ly.arena + (long long)s.uslot[ti] * Ly.stride;
                    prefetch_l2(wb + LL.d_offset + (long long)r * LL.d_tile_bytes, (unsigned)LL.d_tile_bytes);
                }
        }
        // ------------------------------------------------ GU: gate/up + activation
        {
            const QLayout &L = a.L;
            const int tilesF = L.gu_tiles;
            const int tilesS = has_shared ? a.LS.gu_tiles : 0;
            const int n_items = nU * tilesF + tilesS;
            const int quad = warp >> 2, q = warp & 3;
            for (int j = cta + G * quad; j < n_items; j += G * 4) {
                const bool shared = j >= nU * tilesF;
                int rt, ncols, col0 = 0;
                const uint8_t *wbase;
                const QLayout &LL = shared ? a.LS : a.L;
                if (!shared) {
                    const int u = j / tilesF;
                    rt = j % tilesF;
                    col0 = s.ustart[u];
                    ncols = s.ustart[u + 1] - col0;
                    wbase = Ly.arena + (long long)s.uslot[u] * Ly.stride;
                } else {
                    rt = j - nU * tilesF;
                    ncols = T;
                    wbase = Ly.shared;
                }
                // B column g: token of column g (x bf16), or hi/lo limb rows (x fp32)
                const int jc = XF32 ? (g & 3) : g;
                const bool valid = jc < ncols;
                int trow = 0;
                if (valid) {
                    const int t = shared ? jc : s.cols[col0 + jc] / K;
                    trow = XF32 ? ((g < 4) ? t : 4 + t) : t;
                }
                const BTile bt[1] = {{xs + (size_t)trow * ldx + 2 * c, valid}};
                const int n_chunks = LL.gu_chunks;
                const int cb0 = gu_chunk_begin(q, n_chunks), cb1 = gu_chunk_begin(q + 1, n_chunks);
                const uint8_t *tile_ptr = wbase + (long long)rt * LL.gu_tile_bytes;
                float acc[2][1][4] = {};
                stream_chunks<KIND, 2, 1, Win<KIND>::GU>(tile_ptr, LL.gu_chunk_bytes, LL.cb, LL.sb, cb0, cb1,
                                                         n_chunks, LL.gu_half, bt, shared ? a.un_s : a.un, lane,
                                                         acc);
                float *red = u_region + (size_t)quad * (4 * 32 * 8);
#pragma unroll
                for (int m = 0; m < 2; ++m)
#pragma unroll
                    for (int e4 = 0; e4 < 4; ++e4) red[(q * 32 + lane) * 8 + m * 4 + e4] = acc[m][0][e4];
                quad_sync(quad);
                if (q == 0) {
                    float v[8];
#pragma unroll
                    for (int e8 = 0; e8 < 8; ++e8) {
                        float sum = red[lane * 8 + e8];
#pragma unroll
                        for (int w = 1; w < 4; ++w) sum += red[(w * 32 + lane) * 8 + e8];
                        v[e8] = sum;
                    }
                    if (XF32) {
#pragma unroll
                        for (int e8 = 0; e8 < 8; ++e8) v[e8] += __shfl_xor_sync(0xffffffffu, v[e8], 2);
                    }
                    if (!XF32 || c < 2) {
#pragma unroll
                        for (int e4 = 0; e4 < 4; ++e4) {
                            const int rr = g + 8 * (e4 >> 1), jj = 2 * c + (e4 & 1);
                            if (jj < ncols) {
                                const float hv = act_f(a.act, v[e4]) * v[4 + e4];
                                const int row = shared ? P + jj : s.cols[col0 + jj];
                                __nv_bfloat16 hi, lo;
                                split_bf16(hv, hi, lo);
                                const size_t o = (size_t)row * a.h_ld + rt * 16 + rr;
                                a.h_hi[o] = hi;
                                a.h_lo[o] = lo;
                            }
                        }
                    }
                }
                quad_sync(quad);
            }
        }
        if (!grid_sync(a.bar, target, a.status, s_flag)) break;
        // ------------------------------------------------ D: down projection + combine
        {
            const QLayout &L = a.L;
            const int n_tasks = nU + (has_shared ? 1 : 0);
            // h limbs of the live columns (plan order) and of the shared tokens, staged
            // once: row i of the routed part at hst + i*ldh (hi) and hst + lo_off + i*ldh
            // (lo); lo_off makes hi and lo rows fall on different banks
            const int nlive = s.misc[1];
            const bool staged = a.geom.hst_bytes != 0;
            const int ldh = L.F + 8, ldhs = a.LS.F + 8;
            const int lo_off = ((nlive * ldh + 63) & ~63) + 32;
            __nv_bfloat16 *const hss = hst + (((lo_off + nlive * ldh) + 63) & ~63);
            const int lo_off_s = ((T * ldhs + 63) & ~63) + 32;
            if (staged) {
                const int vpr = L.F / 8;  // 16-byte vectors per routed row
                for (int idx = tid; idx < nlive * 2 * vpr; idx += blockDim.x) {
                    const int i = idx / (2 * vpr), rem = idx % (2 * vpr), limb = rem / vpr, v = rem % vpr;
                    const __nv_bfloat16 *src = (limb ? a.h_lo : a.h_hi) + (size_t)s.cols[i] * a.h_ld + v * 8;
                    *reinterpret_cast<uint4 *>(hst + (limb ? lo_off : 0) + i * ldh + v * 8) =
                        *reinterpret_cast<const uint4 *>(src);
                }
                if (has_shared) {
                    const int vps = a.LS.F / 8;
                    for (int idx = tid; idx < T * 2 * vps; idx += blockDim.x) {
                        const int t = idx / (2 * vps), rem = idx % (2 * vps), limb = rem / vps, v = rem % vps;
                        const __nv_bfloat16 *src = (limb ? a.h_lo : a.h_hi) + (size_t)(P + t) * a.h_ld + v * 8;
                        *reinterpret_cast<uint4 *>(hss + (limb ? lo_off_s : 0) + t * ldhs + v * 8) =
                            *reinterpret_cast<const uint4 *>(src);
                    }
                }
                __syncthreads();
            }
            for (int r = cta; r < L.d_tiles; r += G) {
                for (int ti = warp; ti < n_tasks; ti += kPWarps) {
                    const bool shared = ti >= nU;
                    const QLayout &LL = shared ? a.LS : a.L;
                    int ncols, col0 = 0;
                    const uint8_t *wbase;
                    if (!shared) {
                        col0 = s.ustart[ti];
                        ncols = s.ustart[ti + 1] - col0;
                        wbase = Ly.arena + (long long)s.uslot[ti] * Ly.stride;
                    } else {
                        ncols = T;
                        wbase = Ly.shared;
                    }
                    const uint8_t *tile_ptr = wbase + LL.d_offset + (long long)r * LL.d_tile_bytes;
                    const Unpack &un = shared ? a.un_s : a.un;
                    // B tiles: columns nb*4 + (g & 3); lanes g < 4 read hi limbs, g >= 4 lo limbs
                    auto make_bt = [&](int nb) {
                        const int jc = nb * 4 + (g & 3);
                        BTile b{a.h_hi, false};
                        if (jc < ncols) {
                            if (staged) {
                                b.row = shared ? hss + (g < 4 ? 0 : lo_off_s) + jc * ldhs + 2 * c
                                               : hst + (g < 4 ? 0 : lo_off) + (col0 + jc) * ldh + 2 * c;
                            } else {
                                const int row = shared ? P + jc : s.cols[col0 + jc];
                                b.row = (g < 4 ? a.h_hi : a.h_lo) + (size_t)row * a.h_ld + 2 * c;
                            }
                            b.valid = true;
                        }
                        return b;
                    };
                    auto emit = [&](int nb, float (&acc)[4]) {
                        float v[4];
#pragma unroll
                        for (int e4 = 0; e4 < 4; ++e4) v[e4] = acc[e4] + __shfl_xor_sync(0xffffffffu, acc[e4], 2);
                        if (c < 2) {
#pragma unroll
                            for (int e4 = 0; e4 < 4; ++e4) {
                                const int rr = g + 8 * (e4 >> 1), jj = nb * 4 + 2 * c + (e4 & 1);
                                if (jj < ncols) {
                                    const int row = shared ? P + jj : s.cols[col0 + jj];
                                    ypart[row * 16 + rr] = v[e4];
                                }
                            }
                        }
                    };
                    if (ncols > 4) {
                        const BTile bt[2] = {make_bt(0), make_bt(1)};
                        float acc[1][2][4] = {};
                        stream_chunks<KIND, 1, 2, Win<KIND>::D>(tile_ptr, LL.d_chunk_bytes, LL.cb, LL.sb, 0,
                                                                LL.d_chunks, LL.d_chunks, LL.d_half, bt, un, lane, acc);
                        emit(0, acc[0][0]);
                        emit(1, acc[0][1]);
                    } else {
                        const BTile bt[1] = {make_bt(0)};
                        float acc[1][1][4] = {};
                        stream_chunks<KIND, 1, 1, Win<KIND>::D>(tile_ptr, LL.d_chunk_bytes, LL.cb, LL.sb, 0,
                                                                LL.d_chunks, LL.d_chunks, LL.d_half, bt, un, lane, acc);
                        emit(0, acc[0][0]);
                    }
                }
                __syncthreads();
                if (tid < T * 16) {
                    const int t = tid >> 4, rr = tid & 15;
                    float acc = 0.f;
                    for (int k = 0; k < K; ++k) {
                        const int p = t * K + k;
                        if (s.live[p]) acc = fmaf(s.w[p], ypart[p * 16 + rr], acc);
                    }
                    if (has_shared) acc += ypart[(P + t) * 16 + rr];
                    const size_t o = (size_t)t * H + r * 16 + rr;
                    if (a.stack)
                        a.resid[o] = a.resid[o] + acc;
                    else
                        a.y[o] = acc;
                }
                __syncthreads();
            }
        }
        if (a.stack && l + 1 < a.n_layers) {
            if (!grid_sync(a.bar, target, a.status, s_flag)) break;
        }
    }
    cp_async_wait_all();
}

}  // namespace

PersistGeom persist_geom(int T, int H, int E, int K, int F, int F_shared, int wr_bytes, int G, size_t max_smem) {
    PersistGeom g;
    auto al = [](size_t v) { return (v + 127) & ~size_t(127); };
    const int nr = (E + G - 1) / G;
    const int P = T * K;
    g.off_wr = 0;
    g.off_xs = al((size_t)nr * H * wr_bytes);
    const size_t xs_bytes = (size_t)kMaxTok * (H + 8) * 2;
    g.off_u = g.off_xs + al(xs_bytes);
    const size_t topk_part = (size_t)T * ((E + 31) / 32) * 32 * 8;
    const size_t norm_part = (size_t)T * H * 4;
    size_t u = kRedBytes;
    if (topk_part > u) u = topk_part;
    if (norm_part > u) u = norm_part;
    const size_t yp_bytes = (size_t)(P + T) * 16 * 4;
    const size_t stat = sizeof(Plan);
    // h staging: hi and lo rows of up to P routed columns (F + 8 wide) and T shared rows
    size_t hst = ((size_t)2 * P * (F + 8) + (F_shared ? (size_t)2 * T * (F_shared + 8) : 0) + 256) * 2;
    g.off_hst = g.off_xs;
    g.hst_bytes = hst;
    g.off_yp = al(g.off_hst + hst);
    size_t dyn = g.off_u + al(u);
    if (g.off_yp + yp_bytes > dyn) dyn = g.off_yp + yp_bytes;
    if (dyn + stat > max_smem) {  // no room: the down phase reads h from global memory
        g.hst_bytes = 0;
        g.off_yp = g.off_xs;
        dyn = g.off_u + al(u);
        if (g.off_yp + yp_bytes > dyn) dyn = g.off_yp + yp_bytes;
    }
    g.dyn_bytes = dyn;
    g.bytes = dyn + stat;
    return g;
}

int launch_decode_persistent(const PersistArgs &a, int G, cudaStream_t s) {
    const void *kern;
    if (a.L.kind == MOE_Q2_64)
        kern = a.x_f32 ? (const void *)k_decode<MOE_Q2_64, true> : (const void *)k_decode<MOE_Q2_64, false>;
    else
        kern = a.x_f32 ? (const void *)k_decode<MOE_Q4_32, true> : (const void *)k_decode<MOE_Q4_32, false>;
    MOE_CUDA_TRY(cudaMemsetAsync(a.bar, 0, 2 * sizeof(unsigned), s));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(G);
    cfg.blockDim = dim3(kPersistThreads);
    cfg.dynamicSmemBytes = a.geom.dyn_bytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void *args[] = {const_cast<PersistArgs *>(&a)};
    MOE_CUDA_TRY(cudaLaunchKernelExC(&cfg, kern, args));
    return MOE_OK;
}

int persist_max_ctas(int smem_bytes, int *G) {
    int dev = 0, sms = 0, coop = 0;
    MOE_CUDA_TRY(cudaGetDevice(&dev));
    MOE_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    MOE_CUDA_TRY(cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev));
    if (!coop) {
        *G = 0;
        return MOE_OK;
    }
    int per_sm = 0;
    MOE_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_decode<MOE_Q2_64, false>, kPersistThreads,
                                                               smem_bytes - (int)sizeof(Plan)));
    int per_sm2 = 0;
    MOE_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm2, k_decode<MOE_Q4_32, false>, kPersistThreads,
                                                               smem_bytes - (int)sizeof(Plan)));
    if (per_sm2 < per_sm) per_sm = per_sm2;
    *G = per_sm >= 1 ? sms : 0;
    return MOE_OK;
}

int init_persist_attributes(int max_smem) {
    const void *ks[] = {(const void *)k_decode<MOE_Q2_64, true>, (const void *)k_decode<MOE_Q2_64, false>,
                        (const void *)k_decode<MOE_Q4_32, true>, (const void *)k_decode<MOE_Q4_32, false>};
    for (const void *k : ks) {
        int rc = set_max_dynamic_smem(k, max_smem);
        if (rc) return rc;
    }
    return MOE_OK;
}

}  // namespace moe
