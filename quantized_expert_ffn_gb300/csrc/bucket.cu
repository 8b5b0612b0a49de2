// bucket.cu -- expert-major bucketing of the (token, rank) pairs and the plan of
// expert work groups built from the buckets.
//
// kairos-engine README, "The MoE forward": the expert loop buckets the whole
// batch by expert, then runs each expert once over every token that chose it.
// Strata article, "The plan: three destinations per expert": a verify window's
// routed ids are deduplicated, so an expert chosen by two tokens is computed once
// for both. Both follow from one stable counting sort.
#include "moe_internal.cuh"

namespace moe {

namespace {

constexpr int kBucketThreads = 1024;

// Block-wide exclusive scan of one int per thread; returns the prefix and writes
// the block total to *total. All threads of the block must call it.
__device__ int block_exclusive_scan(int v, int *total, int *scratch /* >= 33 ints */) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += n;
    }
    if (lane == 31) scratch[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        int s = lane < nw ? scratch[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += n;
        }
        if (lane < nw) scratch[lane] = s;  // inclusive per-warp totals
        if (lane == 31) scratch[32] = s;
    }
    __syncthreads();
    const int warp_base = warp > 0 ? scratch[warp - 1] : 0;
    *total = scratch[32];
    __syncthreads();
    return warp_base + inc - v;
}

// The groups of one expert's my_lc live pairs (plan columns my_cs ..), at most nc
// columns each; every thread of the CTA calls it (tid < E: expert tid). With
// nc = 256 (the tensor-core GEMMs, whose CTAs take tiles round-robin in list
// order) the list is ordered for the schedule: every full group first, in expert
// order, then the partial groups from the largest down, so that the longest tiles
// start first. A group's tiles compute their outputs alone, so the order changes
// no result. Other widths keep expert order. *total = number of groups.
__device__ void emit_groups(int E, int my_lc, int my_cs, int slot, int nc, Group *groups, int *total, int *scr) {
    __shared__ int hist[256];
    const int tid = threadIdx.x;
    if (nc != 256) {
        const int ng = tid < E ? (my_lc + nc - 1) / nc : 0;
        const int gb = block_exclusive_scan(ng, total, scr);
        if (tid < E)
            for (int j = 0; j < ng; ++j) groups[gb + j] = Group{slot, my_cs + j * nc, min(nc, my_lc - j * nc), 0};
        return;
    }
    const int nfull = tid < E ? my_lc / 256 : 0, part = tid < E ? my_lc % 256 : 0;
    int tot_full, tot_part;
    const int fb = block_exclusive_scan(nfull, &tot_full, scr);
    for (int i = tid; i < 256; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    const int rank = part > 0 ? atomicAdd(&hist[part], 1) : 0;  // place among groups of its size
    __syncthreads();
    // start of each size's run: the full groups, then sizes 255, 254, ..., 1
    const int v = tid < 255 ? hist[255 - tid] : 0;
    const int start = block_exclusive_scan(v, &tot_part, scr);
    if (tid < 255) hist[255 - tid] = start;
    __syncthreads();
    if (tid < E) {
        for (int j = 0; j < nfull; ++j) groups[fb + j] = Group{slot, my_cs + j * 256, 256, 0};
        if (part > 0) groups[tot_full + hist[part] + rank] = Group{slot, my_cs + nfull * 256, part, 0};
    }
    *total = tot_full + tot_part;
    __syncthreads();
}

// One CTA of 1024 threads. Counting pass (order-free), exclusive scan, then the
// stable placement: pairs are placed in chunks of 1024 in pair order; inside a
// chunk a pair's rank among equal experts = (count in earlier warps) + (count in
// earlier lanes of its warp), so perm lists each expert's pairs in increasing p.
__global__ void __launch_bounds__(kBucketThreads) k_bucket(const int32_t *__restrict__ ids, int P, int E,
                                                           int32_t *counts, int32_t *offsets, int32_t *perm,
                                                           int32_t *active, int32_t *n_active,
                                                           uint32_t *status) {
    extern __shared__ int sm[];
    int *cnt = sm;              // [E]
    int *base = cnt + E;        // [E] running placement base
    int *wt = base + E;         // [32][E] per-warp counts of the current chunk
    int *scr = wt + 32 * E;     // [64] scan scratch
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int e = tid; e < E; e += blockDim.x) cnt[e] = 0;
    __syncthreads();
    bool oob = false;
    for (int p = tid; p < P; p += blockDim.x) {
        const int e = ids[p];
        if (e >= 0 && e < E) atomicAdd(&cnt[e], 1);
        else oob = true;
    }
    if (__syncthreads_or(oob) && tid == 0) set_status(status, MOE_STATUS_BOUNDS);
    // exclusive scan of counts over E (E <= 1024 = one element per thread)
    {
        const int c = tid < E ? cnt[tid] : 0;
        int total;
        const int pre = block_exclusive_scan(c, &total, scr);
        if (tid < E) {
            counts[tid] = c;
            offsets[tid] = pre;
            base[tid] = pre;
        }
        if (tid == 0) offsets[E] = total;
        const int act = (tid < E && c > 0) ? 1 : 0;
        int nact;
        const int apos = block_exclusive_scan(act, &nact, scr);
        if (act) active[apos] = tid;
        if (tid == 0) *n_active = nact;
    }
    __syncthreads();
    for (int c0 = 0; c0 < P; c0 += blockDim.x) {
        for (int i = tid; i < 32 * E; i += blockDim.x) wt[i] = 0;
        __syncthreads();
        const int p = c0 + tid;
        int e = p < P ? ids[p] : -1;
        if (e >= E) e = -1;
        const unsigned same = __match_any_sync(0xffffffffu, e);
        const int rank = __popc(same & ((1u << lane) - 1));
        if (e >= 0 && rank == 0) wt[warp * E + e] = __popc(same);
        __syncthreads();
        for (int ee = tid; ee < E; ee += blockDim.x) {
            int run = base[ee];
            for (int w = 0; w < 32; ++w) {
                const int c = wt[w * E + ee];
                wt[w * E + ee] = run;
                run += c;
            }
            base[ee] = run;
        }
        __syncthreads();
        if (e >= 0) perm[wt[warp * E + e] + rank] = p;
        __syncthreads();
    }
}

// Plan: live pairs (weight != 0 and the expert resident) in bucket order form
// the column list; each expert's live pairs are cut into groups of at most
// nc_gu (gate/up) and nc_d (down) columns. Shared-expert groups cover all T
// tokens and sit after the routed groups' maximum count.
__global__ void __launch_bounds__(kBucketThreads) k_plan(PlanArgs a) {
    extern __shared__ int sm[];
    const int tid = threadIdx.x;
    const int P = a.T * a.K, E = a.E;
    int *lc = sm;          // [E] live count per expert
    int *cstart = lc + E;  // [E]
    int *scr = cstart + E; // [64]
    bool absent = false, oob = false;
    for (int p = tid; p < P; p += blockDim.x) a.live[p] = 0;
    if (tid < E) lc[tid] = 0;
    __syncthreads();
    const int nb = a.offsets[E];  // pairs with an id in range (the rest were left out)
    // thread `tid` owns bucket positions [i0, i1): one pass counts its live pairs (and
    // each expert's, flushed per run of equal experts), one scan places them
    const int per = (nb + (int)blockDim.x - 1) / (int)blockDim.x;
    const int i0 = min(nb, tid * per), i1 = min(nb, i0 + per);
    int my_live = 0, run_e = -1, run_n = 0;
    // batches of 8 positions: each level of the lookups (pair, expert, slot and
    // weight) is issued for the whole batch before the next
    constexpr int kB = 8;
    for (int ib = i0; ib < i1; ib += kB) {
        int pp[kB], ee[kB], sl[kB];
        float ww[kB];
#pragma unroll
        for (int j = 0; j < kB; ++j) pp[j] = ib + j < i1 ? a.perm[ib + j] : -1;
#pragma unroll
        for (int j = 0; j < kB; ++j) ee[j] = pp[j] >= 0 ? a.ids[pp[j]] : -1;
#pragma unroll
        for (int j = 0; j < kB; ++j) {
            const bool in = pp[j] >= 0 && ee[j] >= 0 && ee[j] < E;
            sl[j] = in ? a.table[(size_t)a.layer * E + ee[j]] : -1;
            ww[j] = in ? a.w[pp[j]] : 0.f;
        }
#pragma unroll
        for (int j = 0; j < kB; ++j) {
            if (pp[j] < 0) break;
            const int p = pp[j], e = ee[j];
            int live = 0;
            if (e >= 0 && e < E) {
                if (sl[j] < 0) absent = true;
                else if (sl[j] >= a.capacity) oob = true;
                else live = ww[j] != 0.f;
            } else {
                oob = true;
            }
            a.live[p] = live;
            my_live += live;
            if (e != run_e) {
                if (run_n && run_e >= 0 && run_e < E) atomicAdd(&lc[run_e], run_n);
                run_e = e;
                run_n = 0;
            }
            run_n += live;
        }
    }
    if (run_n && run_e >= 0 && run_e < E) atomicAdd(&lc[run_e], run_n);
    int nlive;
    int pos = block_exclusive_scan(my_live, &nlive, scr);
    for (int ib = i0; ib < i1; ib += kB) {
        int pp[kB], lv[kB];
#pragma unroll
        for (int j = 0; j < kB; ++j) pp[j] = ib + j < i1 ? a.perm[ib + j] : -1;
#pragma unroll
        for (int j = 0; j < kB; ++j) lv[j] = pp[j] >= 0 ? a.live[pp[j]] : 0;
#pragma unroll
        for (int j = 0; j < kB; ++j)
            if (lv[j]) a.cols[pos++] = pp[j];
    }
    if (__syncthreads_or(absent) && tid == 0) set_status(a.status, MOE_STATUS_EXPERT_ABSENT);
    if (__syncthreads_or(oob) && tid == 0) set_status(a.status, MOE_STATUS_BOUNDS);
    // live count per expert (its pairs are offsets[e]..offsets[e+1] of perm)
    const int my_lc = tid < E ? lc[tid] : 0;
    int dummy;
    const int my_cs = block_exclusive_scan(tid < E ? my_lc : 0, &dummy, scr);
    if (tid < E) cstart[tid] = my_cs;
    __syncthreads();
    // groups
    int tot_gu, tot_d;
    const int slot = (tid < E && my_lc > 0) ? a.table[(size_t)a.layer * E + tid] : -1;
    emit_groups(E, tid < E ? my_lc : 0, my_cs, slot, a.nc_gu, a.groups_gu, &tot_gu, scr);
    emit_groups(E, tid < E ? my_lc : 0, my_cs, slot, a.nc_d, a.groups_d, &tot_d, scr);
    if (tid == 0) {
        a.n_groups[0] = tot_gu;
        a.n_groups[1] = tot_d;
        a.n_groups[2] = nlive + (a.has_shared ? a.T : 0);  // plan columns
    }
    if (a.has_shared) {
        for (int t = tid; t < a.T; t += blockDim.x) a.cols[nlive + t] = -(t + 1);
        const int sg_gu = (a.T + a.nc_gu - 1) / a.nc_gu, sg_d = (a.T + a.nc_d - 1) / a.nc_d;
        for (int j = tid; j < sg_gu; j += blockDim.x)
            a.groups_gu[a.max_routed_gu + j] = Group{-2, nlive + j * a.nc_gu, min(a.nc_gu, a.T - j * a.nc_gu), 0};
        for (int j = tid; j < sg_d; j += blockDim.x)
            a.groups_d[a.max_routed_d + j] = Group{-2, nlive + j * a.nc_d, min(a.nc_d, a.T - j * a.nc_d), 0};
    }
}

// ---------------------------------------------------------------- wide windows
// The same stable counting sort and plan spread over one CTA per 1,024 pairs (or
// bucket positions): a single CTA is bound by its own share of the L2 bandwidth
// once the window holds tens of thousands of pairs. Outputs are identical to
// k_bucket / k_plan.

// Per-chunk expert histogram: cc[c][e] = pairs of chunk c with id e.
__global__ void __launch_bounds__(kBucketThreads) k_bucket_count(const int32_t *__restrict__ ids, int P, int E,
                                                                 int32_t *cc, uint32_t *status) {
    extern __shared__ int sm[];
    const int tid = threadIdx.x, c = blockIdx.x;
    for (int e = tid; e < E; e += blockDim.x) sm[e] = 0;
    __syncthreads();
    const int p = c * kBucketThreads + tid;
    bool oob = false;
    if (p < P) {
        const int e = ids[p];
        if (e >= 0 && e < E) atomicAdd(&sm[e], 1);
        else oob = true;
    }
    if (__syncthreads_or(oob) && tid == 0) set_status(status, MOE_STATUS_BOUNDS);
    for (int e = tid; e < E; e += blockDim.x) cc[(size_t)c * E + e] = sm[e];
}

// Stable placement of chunk c (the in-chunk rank as in k_bucket). The scan is
// folded in: expert e's base in chunk c is its offset (exclusive scan of the
// totals) plus its pairs in the chunks before c, which every CTA sums from the
// per-chunk histograms; CTA 0 also writes the totals, offsets and active experts.
__global__ void __launch_bounds__(kBucketThreads) k_bucket_place(const int32_t *__restrict__ ids, int P, int E, int C,
                                                                 const int32_t *__restrict__ cc, int32_t *counts,
                                                                 int32_t *offsets, int32_t *active, int32_t *n_active,
                                                                 int32_t *perm) {
    extern __shared__ int sm[];
    __shared__ int scr[64];
    int *base = sm;       // [E]
    int *wt = base + E;   // [32][E]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, c = blockIdx.x;
    int before = 0, run = 0;  // expert tid: pairs in the chunks before c, in all chunks
    if (tid < E) {
        // batches of 8 chunks: the loads of a batch are in flight together
        for (int c0 = 0; c0 < C; c0 += 8) {
            int v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = c0 + j < C ? cc[(size_t)(c0 + j) * E + tid] : 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (c0 + j == c) before = run;
                run += v[j];
            }
        }
    }
    int total;
    const int pre = block_exclusive_scan(tid < E ? run : 0, &total, scr);
    if (tid < E) base[tid] = pre + before;
    if (c == 0) {
        if (tid < E) {
            counts[tid] = run;
            offsets[tid] = pre;
        }
        if (tid == 0) offsets[E] = total;
        const int act = (tid < E && run > 0) ? 1 : 0;
        int nact;
        const int apos = block_exclusive_scan(act, &nact, scr);
        if (act) active[apos] = tid;
        if (tid == 0) *n_active = nact;
    }
    for (int i = tid; i < 32 * E; i += blockDim.x) wt[i] = 0;
    __syncthreads();
    const int p = c * kBucketThreads + tid;
    int e = p < P ? ids[p] : -1;
    if (e >= E) e = -1;
    const unsigned same = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(same & ((1u << lane) - 1));
    if (e >= 0 && rank == 0) wt[warp * E + e] = __popc(same);
    __syncthreads();
    for (int ee = tid; ee < E; ee += blockDim.x) {
        int r = base[ee];
        for (int w = 0; w < 32; ++w) {
            const int n = wt[w * E + ee];
            wt[w * E + ee] = r;
            r += n;
        }
    }
    __syncthreads();
    if (e >= 0) perm[wt[warp * E + e] + rank] = p;
}

// Plan, pass 1 (one CTA per 1,024 bucket positions): liveness of the pair at
// each position, the CTA's live pairs per expert (lcb[c][e]) and in all (blk[c]);
// pairs whose id is out of range (not in the buckets) are marked dead by their
// own index.
__global__ void __launch_bounds__(kBucketThreads) k_plan_live(PlanArgs a, int32_t *lcb, int32_t *blk) {
    extern __shared__ int hl[];  // [E]
    const int tid = threadIdx.x, i = blockIdx.x * kBucketThreads + tid;
    const int P = a.T * a.K, E = a.E;
    for (int e = tid; e < E; e += blockDim.x) hl[e] = 0;
    __syncthreads();
    const int nb = a.offsets[E];
    bool absent = false, oob = false;
    int live = 0, e = -1;
    if (i < nb) {
        const int p = a.perm[i];
        e = a.ids[p];
        const int slot = a.table[(size_t)a.layer * E + e];
        if (slot < 0) absent = true;
        else if (slot >= a.capacity) oob = true;
        else live = a.w[p] != 0.f;
        a.live[p] = live;
    }
    if (i < P) {
        const int ei = a.ids[i];
        if (ei < 0 || ei >= E) {
            a.live[i] = 0;
            oob = true;
        }
    }
    const unsigned same = __match_any_sync(0xffffffffu, live ? e : -1);
    if (live && (same & ((1u << (tid & 31)) - 1)) == 0) atomicAdd(&hl[e], __popc(same));
    const int n = __syncthreads_count(live);
    for (int ee = tid; ee < E; ee += blockDim.x) lcb[(size_t)blockIdx.x * E + ee] = hl[ee];
    if (tid == 0) blk[blockIdx.x] = n;
    if (__syncthreads_or(absent) && tid == 0) set_status(a.status, MOE_STATUS_EXPERT_ABSENT);
    if (__syncthreads_or(oob) && tid == 0) set_status(a.status, MOE_STATUS_BOUNDS);
}

// Plan, pass 2 (one CTA per 1,024 bucket positions): the live pairs in bucket
// order are the routed plan columns, after the live pairs of the CTAs before.
// CTA 0 also sums the live pairs per expert, builds the groups and the group
// counts, and writes the shared expert's columns and groups.
__global__ void __launch_bounds__(kBucketThreads) k_plan_cols(PlanArgs a, int nblk, const int32_t *lcb,
                                                              const int32_t *blk) {
    __shared__ int scr[64];
    __shared__ int cta_base;
    const int tid = threadIdx.x, i = blockIdx.x * kBucketThreads + tid, E = a.E;
    int nlive;
    const int bb = block_exclusive_scan(tid < nblk ? blk[tid] : 0, &nlive, scr);
    if (tid == (int)blockIdx.x) cta_base = bb;  // blockIdx.x < nblk <= blockDim.x
    __syncthreads();
    const int nb = a.offsets[E];
    int p = -1, live = 0;
    if (i < nb) {
        p = a.perm[i];
        live = a.live[p];
    }
    int dummy;
    const int pre = block_exclusive_scan(live, &dummy, scr);
    if (live) a.cols[cta_base + pre] = p;
    if (blockIdx.x != 0) return;
    int my_lc = 0;
    if (tid < E) {
        for (int c0 = 0; c0 < nblk; c0 += 8) {
            int v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = c0 + j < nblk ? lcb[(size_t)(c0 + j) * E + tid] : 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) my_lc += v[j];
        }
    }
    const int my_cs = block_exclusive_scan(my_lc, &dummy, scr);
    int tot_gu, tot_d;
    const int slot = (tid < E && my_lc > 0) ? a.table[(size_t)a.layer * E + tid] : -1;
    emit_groups(E, my_lc, my_cs, slot, a.nc_gu, a.groups_gu, &tot_gu, scr);
    emit_groups(E, my_lc, my_cs, slot, a.nc_d, a.groups_d, &tot_d, scr);
    if (tid == 0) {
        a.n_groups[0] = tot_gu;
        a.n_groups[1] = tot_d;
        a.n_groups[2] = nlive + (a.has_shared ? a.T : 0);
    }
    if (a.has_shared) {
        for (int t = tid; t < a.T; t += blockDim.x) a.cols[nlive + t] = -(t + 1);
        const int sg_gu = (a.T + a.nc_gu - 1) / a.nc_gu, sg_d = (a.T + a.nc_d - 1) / a.nc_d;
        for (int j = tid; j < sg_gu; j += blockDim.x)
            a.groups_gu[a.max_routed_gu + j] = Group{-2, nlive + j * a.nc_gu, min(a.nc_gu, a.T - j * a.nc_gu), 0};
        for (int j = tid; j < sg_d; j += blockDim.x)
            a.groups_d[a.max_routed_d + j] = Group{-2, nlive + j * a.nc_d, min(a.nc_d, a.T - j * a.nc_d), 0};
    }
}

}  // namespace

int launch_bucket(const int32_t *ids, int T, int K, int E, int32_t *counts, int32_t *offsets, int32_t *perm,
                  int32_t *active, int32_t *n_active, uint32_t *status, cudaStream_t s) {
    const size_t smem = ((size_t)2 * E + 32 * (size_t)E + 64) * sizeof(int);
    k_bucket<<<1, kBucketThreads, smem, s>>>(ids, T * K, E, counts, offsets, perm, active, n_active, status);
    MOE_CUDA_TRY(cudaGetLastError());
    return MOE_OK;
}

int init_bucket_attributes(int max_smem) {
    int rc = set_max_dynamic_smem((const void *)k_bucket, max_smem);
    if (!rc) rc = set_max_dynamic_smem((const void *)k_plan, max_smem);
    if (!rc) rc = set_max_dynamic_smem((const void *)k_bucket_place, max_smem);
    return rc;
}

// The bucket's per-chunk histograms, then (reusing the same ints) the plan's
// per-CTA live counts per expert and per CTA.
size_t wide_scratch_bytes(int T, int K, int E) {
    const size_t C = ((size_t)T * K + kBucketThreads - 1) / kBucketThreads;
    return (C * (size_t)E + C) * sizeof(int32_t);
}

bool use_wide(int T, int K) {
    const long long P = (long long)T * K;
    return P > 2 * kBucketThreads && P <= (long long)kBucketThreads * kBucketThreads;
}

int launch_bucket_wide(const int32_t *ids, int T, int K, int E, int32_t *counts, int32_t *offsets, int32_t *perm,
                       int32_t *active, int32_t *n_active, int32_t *scratch, uint32_t *status, cudaStream_t s) {
    const int P = T * K, C = (P + kBucketThreads - 1) / kBucketThreads;
    k_bucket_count<<<C, kBucketThreads, (size_t)E * sizeof(int), s>>>(ids, P, E, scratch, status);
    MOE_CUDA_TRY(cudaGetLastError());
    k_bucket_place<<<C, kBucketThreads, (size_t)33 * E * sizeof(int), s>>>(ids, P, E, C, scratch, counts, offsets,
                                                                           active, n_active, perm);
    MOE_CUDA_TRY(cudaGetLastError());
    return MOE_OK;
}

int launch_plan_wide(const PlanArgs &a, int32_t *scratch, cudaStream_t s) {
    const int P = a.T * a.K, C = (P + kBucketThreads - 1) / kBucketThreads;
    int32_t *lcb = scratch, *blk = scratch + (size_t)C * a.E;
    k_plan_live<<<C, kBucketThreads, (size_t)a.E * sizeof(int32_t), s>>>(a, lcb, blk);
    MOE_CUDA_TRY(cudaGetLastError());
    k_plan_cols<<<C, kBucketThreads, 0, s>>>(a, C, lcb, blk);
    MOE_CUDA_TRY(cudaGetLastError());
    return MOE_OK;
}

int launch_plan(const PlanArgs &a, cudaStream_t s) {
    const size_t smem = ((size_t)2 * a.E + 64) * sizeof(int);
    k_plan<<<1, kBucketThreads, smem, s>>>(a);
    MOE_CUDA_TRY(cudaGetLastError());
    return MOE_OK;
}

}  // namespace moe
