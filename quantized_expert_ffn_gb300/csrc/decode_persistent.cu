// decode_persistent.cu -- one cooperative launch per decode step: every SM runs
// one CTA that walks through all the layers of the step, phase by phase.
//
// Per layer (Krasis white paper sec. 5.3; kairos-engine README "The MoE forward"):
//   N  layer input: x (single layer) or u = bf16(RMSNorm(resid)) (stack), every
//      CTA for itself from the same resid;
//   R  router logits: CTA c owns experts c, c+G, ...; four warps share a row; the
//      rows, bias and slot-table row were prefetched into shared memory during the
//      previous layer, and the next layer's are requested during the down phase;
//      the logits are published as tagged words, with a flag per CTA;
//   T  top-K, weights and the plan, every CTA the same result from the logits (read
//      as soon as every CTA's tagged words are there): the K-th largest of a few
//      segment maxima is a threshold, the experts at or above it are ranked exactly;
//      the distinct live experts and their columns; the split of the down work;
//   GU gate/up items (16 rows of one expert, all of H) are dealt round-robin over
//      CTAs and over the groups of S = 4 warps of a CTA; warp q of a group sums
//      part q of H; the group adds the parts in order, applies the activation,
//      writes h and counts the item for its expert;
//   D  down units (one expert x 16 output rows) in expert order, split over the
//      CTAs so that gate/up plus down bytes are even, then over the CTA's warps; a
//      CTA waits only until the gate/up items of its own units' experts are
//      counted, then stages their h in shared memory; a unit's outputs are tagged
//      words; the warp that ran the last task's unit of a row tile combines the
//      tile in k order (+ the shared expert) once every pair's words are there, and
//      writes y, or the next layer's residual as tagged words.
//
// No grid-wide barrier: every exchange between CTAs is either data that carries
// its own readiness (a 64-bit word = 32-bit value + the layer that wrote it, read
// with one round trip as soon as it is there) or a per-expert counter
// (release/acquire). The order of the phases makes reuse safe: a CTA publishes its
// layer-l logits only after reading layer l's input, and layer l's residual output
// is written only after every CTA's layer-l logits are seen, so no word is
// overwritten before everyone has read it (logits alternate between two buffers).
//
// Weights move through one ring per warp in shared memory, filled by bulk copies
// (TMA, cp.async.bulk, completion counted on an mbarrier) of a few chunks each, in
// the order the warp consumes them: its gate/up chunks, then its down chunks. One
// lane issues a copy and nobody waits for the issue; a down chunk does not depend
// on h, so a warp requests its down weights as soon as ring space frees up during
// gate/up, and the whole layer's expert bytes are in flight from the moment the
// plan is known.
//
// Arithmetic per output element is that of the multi-kernel path (same device
// functions, same splits of the reductions, same orders), so results match it bit
// for bit. Every wait is bounded: a wait or a copy that does not complete in about
// a second sets MOE_STATUS_TIMEOUT and the stop word, every CTA leaves at its next
// wait; before a warp leaves it waits (bounded) for every copy it issued.
#include <type_traits>

#include "decode_common.cuh"
#include "decode_persistent.cuh"

namespace moe {

namespace {

constexpr int kPWarps = kPersistThreads / 32;
constexpr long long kSpinCycles = 2000000000LL;  // about 1 s at GB300 clocks

// Static shared memory: the plan of the current layer and small per-CTA state.
struct alignas(16) Plan {
    int ids[256], live[256], sorted[256], cols[256], cexp[256], cslot[256];
    float w[256];
    int ustart[264], uexp[264], uslot[264];
    // 0: distinct live experts, 1: live pairs, 2: stop flag, 4..11: token t has a
    // non-finite logit, 12 / 13: first / end down unit of this CTA
    int misc[16];
    int ncand[kMaxTok];
    uint32_t theta[kMaxTok];
    float bias[2][16];                    // router bias of this CTA's experts, by layer parity
    float rpart[16][kMaxTok][4];          // router partial sums [row][token][warp]
    float wsum[kMaxTok][kNormWarps];      // RMSNorm warp sums
    unsigned long long sel[kMaxTok][32];  // chosen keys per token, rank order
    float wex[kMaxTok][32];               // route-weight scratch per token
    uint64_t ring_bar[kPersistThreads / 32][8];  // weight-ring mbarriers per warp
    uint64_t rbar;                               // router-row copies
};

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

__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_relaxed_u64(unsigned long long *p, unsigned long long v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long tagged(unsigned tag, uint32_t v) {
    return ((unsigned long long)tag << 32) | v;
}

// One wait of one thread (a fresh Waiter per wait). It gives up after about a
// second: it sets MOE_STATUS_TIMEOUT and the stop word, and returns false; it also
// returns false as soon as another thread has set the stop word.
struct Waiter {
    unsigned *stop;
    uint32_t *status;
    long long t0 = 0;
    unsigned it = 0;
    // false: stop waiting. Polls follow each other without a pause (sleeping between
    // them, even for tens of nanoseconds, delayed the chain more than the polling
    // traffic it saved).
    __device__ __forceinline__ bool keep_going() {
        if (it == 0) t0 = clock64();
        ++it;
        if ((it & 15) == 0) {
            if (ld_relaxed_u32(stop)) return false;
            if (clock64() - t0 > kSpinCycles) {
                atomicExch(stop, 1u);
                set_status(status, MOE_STATUS_TIMEOUT);
                return false;
            }
        }
        return true;
    }
};

// Load the tagged words addr(i) for the bits i of `mask` (i < N) with all loads in
// flight, again for the ones not yet written with `tag`, until every one is; their
// values in v. False if the wait gave up.
template <int N, typename Addr>
__device__ __forceinline__ bool wait_tagged(Addr addr, unsigned mask, unsigned tag, uint32_t (&v)[N], Waiter w) {
    unsigned long long x[N];
#pragma unroll
    for (int i = 0; i < N; ++i)
        if (mask >> i & 1u) x[i] = ld_relaxed_u64(addr(i));
    for (;;) {
        bool all = true;
#pragma unroll
        for (int i = 0; i < N; ++i)
            if ((mask >> i & 1u) && (unsigned)(x[i] >> 32) != tag) all = false;
        if (all) break;
        if (!w.keep_going()) return false;
#pragma unroll
        for (int i = 0; i < N; ++i)
            if ((mask >> i & 1u) && (unsigned)(x[i] >> 32) != tag) x[i] = ld_relaxed_u64(addr(i));
    }
#pragma unroll
    for (int i = 0; i < N; ++i) v[i] = (mask >> i & 1u) ? (uint32_t)x[i] : 0u;
    return true;
}

// Wait until counter *p reaches `target` (relaxed polling, then an acquire fence:
// what was written before the releasing increments is visible to this thread).
__device__ __forceinline__ bool wait_count(const int *p, int target, Waiter w) {
    while ((int)ld_relaxed_u32(reinterpret_cast<const unsigned *>(p)) < target)
        if (!w.keep_going()) return false;
    asm volatile("fence.acq_rel.gpu;" ::: "memory");
    return true;
}

// ------------------------------------------------------------------ weight ring
// One ring of R bytes per warp. A piece (a few consecutive chunks of one tile, a
// contiguous chunk image in global memory) is copied by one bulk copy that
// completes on one of the warp's kRingBars mbarriers; pieces are consumed in
// issue order. A piece that would cross the end of the ring starts at the next
// lap; producer and consumer apply the same rule to the same piece sizes, so they
// agree on every placement.
constexpr int kRingBars = 8;  // pieces in flight per warp

__device__ __forceinline__ unsigned smem_u32(const void *p) { return (unsigned)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t *m, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(m)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *m, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(m)), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *m, unsigned parity) {
    unsigned ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(smem_u32(m)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase of parity `parity` to complete; false after about a second.
__device__ __forceinline__ bool mbar_wait(uint64_t *m, unsigned parity) {
    if (mbar_try_wait(m, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(m, parity))
        if (clock64() - t0 > kSpinCycles) return false;
    return true;
}

__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, unsigned bytes, uint64_t *m) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(m))
                 : "memory");
}

struct Ring {
    uint8_t *base;
    uint64_t *bar;         // kRingBars mbarriers
    int R;                 // bytes
    int head, tail;        // bytes taken / released (monotonic, lap padding included)
    int issued, consumed;  // pieces
    int front;             // counter value of the piece being consumed
};

__device__ __forceinline__ int ring_place(int at, int bytes, int R) {
    const int pos = at % R;
    return pos + bytes > R ? at + (R - pos) : at;
}

// Request `bytes` from src as the next piece; false (nothing issued) if the ring
// has no room. Every lane of the warp calls it with the same arguments.
__device__ __forceinline__ bool ring_push(Ring &r, const uint8_t *src, int bytes, int lane) {
    if (r.issued - r.consumed >= kRingBars) return false;
    if (r.issued == r.consumed) r.head = r.tail = 0;  // empty: start at offset 0 (a piece <= R always fits)
    const int at = ring_place(r.head, bytes, r.R);
    if (at + bytes - r.tail > r.R) return false;
    if (lane == 0) {
        uint64_t *m = r.bar + r.issued % kRingBars;
        // the warp's earlier reads of these bytes (ordered by the __syncwarp of
        // ring_pop) come before the copy's writes
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_expect_tx(m, (unsigned)bytes);
        bulk_g2s(r.base + at % r.R, src, (unsigned)bytes, m);
    }
    r.head = at + bytes;
    ++r.issued;
    return true;
}

// Wait until the oldest piece (`bytes` long) has landed; its address. A copy that
// does not land in about a second sets MOE_STATUS_TIMEOUT and the stop word.
__device__ __forceinline__ const uint8_t *ring_front(Ring &r, int bytes, uint32_t *status, unsigned *bar) {
    r.front = ring_place(r.tail, bytes, r.R);
    if (!mbar_wait(r.bar + r.consumed % kRingBars, (unsigned)(r.consumed / kRingBars) & 1u)) {
        if ((threadIdx.x & 31) == 0) {
            set_status(status, MOE_STATUS_TIMEOUT);
            atomicExch(bar + 1, 1u);
        }
    }
    return r.base + r.front % r.R;
}

// Release the oldest piece (every lane has read what it needs from it).
__device__ __forceinline__ void ring_pop(Ring &r, int bytes) {
    __syncwarp();
    r.tail = r.front + bytes;
    ++r.consumed;
}

// Wait (bounded) for every piece still in flight.
__device__ __forceinline__ void ring_drain(Ring &r) {
    for (; r.consumed < r.issued; ++r.consumed)
        mbar_wait(r.bar + r.consumed % kRingBars, (unsigned)(r.consumed / kRingBars) & 1u);
}

// Bytes of the piece of chunks [c0, c0 + nc) of a tile of n chunks (the last
// chunk is half when has_half).
__device__ __forceinline__ int piece_bytes(int cbytes, int has_half, int n, int c0, int nc) {
    return nc * cbytes - ((has_half && c0 + nc == n) ? cbytes / 2 : 0);
}

// Chunk registers from shared memory (same offsets as the global layout).
template <int KIND>
__device__ __forceinline__ void load_chunk_s(const uint8_t *cp, const uint8_t *sp, bool half, int lane,
                                             ChunkRegs<KIND> &r) {
    const int g = lane >> 2;
    if constexpr (KIND == MOE_Q2_64) {
        if (!half) {
            const uint4 v = *reinterpret_cast<const uint4 *>(cp + 16 * lane);
            r.w[0] = v.x; r.w[1] = v.y; r.w[2] = v.z; r.w[3] = v.w;
            r.s[0] = *reinterpret_cast<const uint32_t *>(sp + 4 * g);
            r.s[1] = *reinterpret_cast<const uint32_t *>(sp + 4 * (8 + g));
        } else {
            const uint2 v = *reinterpret_cast<const uint2 *>(cp + 8 * lane);
            r.w[0] = v.x; r.w[1] = v.y; r.w[2] = 0; r.w[3] = 0;
            r.s[0] = *reinterpret_cast<const uint32_t *>(sp + 4 * g);
            r.s[1] = 0;
        }
    } else {
        const uint4 v = *reinterpret_cast<const uint4 *>(cp + 16 * lane);
        r.w[0] = v.x; r.w[1] = v.y; r.w[2] = v.z; r.w[3] = v.w;
        r.s[0] = *reinterpret_cast<const uint32_t *>(sp + 4 * g);
        r.s[1] = *reinterpret_cast<const uint32_t *>(sp + 4 * (8 + g));
        if (!half) {
            const uint4 u = *reinterpret_cast<const uint4 *>(cp + 512 + 16 * lane);
            r.w[4] = u.x; r.w[5] = u.y; r.w[6] = u.z; r.w[7] = u.w;
            r.s[2] = *reinterpret_cast<const uint32_t *>(sp + 4 * (16 + g));
            r.s[3] = *reinterpret_cast<const uint32_t *>(sp + 4 * (24 + g));
        } else {
            r.w[4] = r.w[5] = r.w[6] = r.w[7] = 0;
            r.s[2] = r.s[3] = 0;
        }
    }
}

// Request the router rows this CTA owns for layer l, their bias and the layer's
// slot-table row into shared memory; called by one warp. The rows (H * wsz bytes
// each, contiguous in global memory) and the table row go by bulk copies that
// complete on `m` (one phase per call), the few bias words by cp.async (one
// commit group per lane).
__device__ void prefetch_router(const PersistArgs &a, int l, uint8_t *wr_s, int32_t *tab_s, float *bias_s,
                                uint64_t *m) {
    const int G = gridDim.x, c = blockIdx.x, lane = threadIdx.x & 31;
    const int wsz = a.wr_bf16 ? 2 : 4;
    const int row_bytes = a.H * wsz;
    const uint8_t *Wr = reinterpret_cast<const uint8_t *>(a.layers[l].Wr);
    const int nrb = (a.E + G - 1) / G, e0 = c * nrb;  // my experts: e0 .. e0 + nr - 1
    const int nr = a.E - e0 < nrb ? (a.E - e0 > 0 ? a.E - e0 : 0) : nrb;
    const int32_t *tab = a.layers[l].table + (size_t)a.layers[l].layer * a.E;
    const bool tab_bulk = ((uintptr_t)tab & 15) == 0 && (a.E & 3) == 0;
    if (lane == 0) {
        // the CTA's earlier reads of these bytes (ordered before by a CTA barrier)
        // come before the copies' writes
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_expect_tx(m, (unsigned)(nr * row_bytes + (tab_bulk ? a.E * 4 : 0)));
        if (nr > 0) bulk_g2s(wr_s, Wr + (size_t)e0 * row_bytes, (unsigned)(nr * row_bytes), m);
        if (tab_bulk) bulk_g2s(tab_s, tab, (unsigned)(a.E * 4), m);
    }
    if (!tab_bulk)
        for (int i = lane; i < a.E; i += 32) cp_async4(tab_s + i, tab + i);
    if (a.layers[l].bias)
        for (int r = lane; r < nr; r += 32) cp_async4(bias_s + r, a.layers[l].bias + e0 + r);
    cp_async_commit();
}

// Top-K keys of every token by sorting 32-logit chunks and merging them pairwise
// (used when the threshold pass keeps too many candidates, e.g. many equal
// logits); lg: the layer's tagged logits ([T][ceil(E/32) * 32]), all written.
// lists: T * ceil(E/32) * 32 keys of scratch.
__device__ void topk_sort_merge(const unsigned long long *lg, int T, int E, unsigned long long *lists,
                                unsigned long long (*sel)[32]) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nch = (E + 31) / 32;
    for (int task = warp; task < T * nch; task += kPWarps) {
        const int t = task / nch, ch = task % nch;
        const int e = ch * 32 + lane;
        const unsigned long long key =
            e < E ? topk_key(__uint_as_float((uint32_t)__ldcg(lg + (size_t)t * nch * 32 + e)), e) : 0ull;
        lists[((size_t)t * nch + ch) * 32 + lane] = warp_sort32(key, lane);
    }
    __syncthreads();
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
    if (tid < T * 32) sel[tid >> 5][tid & 31] = lists[(size_t)(tid >> 5) * nch * 32 + (tid & 31)];
}

// The combine of row tile r of layer l by one warp (a separate function: its
// registers do not weigh on the rest of the kernel). The tile's words, one token
// at a time: lane (h, rr) = (lane / 16, lane % 16) reads output rr of pairs
// k = k0 + 2u + h (u < kCw; k < K routed, k = K the shared expert), so a warp load
// covers two pairs' lines; they land in cs (the warp's ring memory, empty once the
// warp's units are done) and lanes 0..15 add them in k order.
__device__ __noinline__ void combine_tile(const PersistArgs &a, const int *live, const float *w, float *cs, int r,
                                          int l, bool has_shared, int lane) {
    constexpr int kCw = 6;
    const int T = a.T, K = a.K, H = a.H, P = T * K, KK = K + 1;
    const int rr = lane & 15, hh = lane >> 4;
    for (int t = 0; t < T; ++t) {
        bool ok = true;
        for (int k0 = 0; k0 < KK && ok; k0 += 2 * kCw) {
            uint32_t v[kCw];
            unsigned m = 0;
#pragma unroll
            for (int u = 0; u < kCw; ++u) {
                const int k = k0 + 2 * u + hh;
                if (k < K ? live[t * K + k] != 0 : (k == K && has_shared)) m |= 1u << u;
            }
            const unsigned long long *base = a.yp_t + (size_t)r * 16 + rr;
            ok = wait_tagged<kCw>(
                [&](int u) {
                    const int k = k0 + 2 * u + hh;
                    return base + (size_t)(k < K ? t * K + k : P + t) * H;
                },
                m, (unsigned)(l + 1), v, Waiter{a.bar + 1, a.status});
#pragma unroll
            for (int u = 0; u < kCw; ++u)
                if (m >> u & 1u) cs[(k0 + 2 * u + hh) * 16 + rr] = __uint_as_float(v[u]);
        }
        if (!__all_sync(0xffffffffu, ok)) return;
        __syncwarp();
        if (lane < 16) {
            const size_t oo = (size_t)t * H + (size_t)r * 16 + rr;
            // the layer's input residual: the caller's at layer 0, else the tagged
            // words of the previous layer (already there: read in N)
            const float rv = !a.stack ? 0.f
                             : l == 0 ? __ldcg(a.resid + oo)
                                      : __uint_as_float((uint32_t)ld_relaxed_u64(a.resid_t + oo));
            float acc = 0.f;
            for (int k = 0; k < K; ++k)
                if (live[t * K + k]) acc = fmaf(w[t * K + k], cs[k * 16 + rr], acc);
            if (has_shared) acc += cs[K * 16 + rr];
            // the stack's output: tagged words for the next layer of the launch (a
            // token's 16 words of a tile fill one 128-byte line, written by this
            // warp alone), the caller's resid after the last
            if (!a.stack)
                a.y[oo] = acc;
            else if (l + 1 == a.n_layers)
                a.resid[oo] = rv + acc;
            else
                st_relaxed_u64(a.resid_t + oo, tagged(l + 1, __float_as_uint(rv + acc)));
        }
        __syncwarp();
    }
}

// OPTS: some layer of the launch has a router scale or non-default route options;
// without them the kernel carries none of that code (it costs the serial steps
// measurable time even when skipped)
template <int KIND, bool XF32, bool OPTS>
__global__ void __launch_bounds__(kPersistThreads, 1) k_decode(const __grid_constant__ PersistArgs a) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    __shared__ Plan s;
    __nv_bfloat16 *const xs = reinterpret_cast<__nv_bfloat16 *>(smem_raw + a.geom.off_xs);
    uint8_t *const wr_s = smem_raw + a.geom.off_wr;
    int32_t *const tab_s = reinterpret_cast<int32_t *>(smem_raw + a.geom.off_tab);
    uint8_t *const u_region = smem_raw + a.geom.off_u;
    __nv_bfloat16 *const hst = reinterpret_cast<__nv_bfloat16 *>(smem_raw + a.geom.off_hst);
    float *const red = reinterpret_cast<float *>(smem_raw + a.geom.off_red);
    const int G = gridDim.x, cta = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int T = a.T, H = a.H, E = a.E, K = a.K, P = T * K;
    const int ldx = H + 8;
    const int g = lane >> 2, c = lane & 3;
    const int tab_ld = a.geom.tab_ld;
    constexpr int S_GU = GuSplit<KIND>::S;
    constexpr int NG = kPWarps / S_GU;  // gate/up warp groups per CTA
    static_assert((size_t)NG * S_GU * 32 * 8 * sizeof(float) <= kRedBytes, "gate/up reduction scratch");
    const QLayout &L = a.L;
    const int dt = L.d_tiles;  // output row tiles (the shared expert has the same)

    static_assert(kRingBars == 8, "Plan::ring_bar holds 8 mbarriers per warp");
    Ring ring;
    ring.base = smem_raw + a.geom.off_ring + (size_t)warp * a.geom.ring_bytes;
    ring.bar = s.ring_bar[warp];
    ring.R = a.geom.ring_bytes;
    ring.head = ring.tail = ring.issued = ring.consumed = ring.front = 0;
    if (lane < kRingBars) mbar_init(&s.ring_bar[warp][lane], 1);
    if (tid == 0) mbar_init(&s.rbar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    __syncthreads();
    // chunks per piece: two pieces of each kind fit in the ring at once; larger pieces
    // mean fewer bulk copies (the copy engine takes them one at a time)
    const int pcg_fit = a.geom.ring_bytes / (2 * L.gu_chunk_bytes);
    const int pcg2 = pcg_fit < 1 ? 1 : (pcg_fit > 8 ? 8 : pcg_fit);
    const int pcd_fit = a.geom.ring_bytes / (2 * L.d_chunk_bytes);
    const int pcd = pcd_fit < 1 ? 1 : (pcd_fit > 8 ? 8 : pcd_fit);

    if (warp == 0) prefetch_router(a, 0, wr_s, tab_s, s.bias[0], &s.rbar);
    int r_issued = 1, r_done = 0;  // router prefetches issued / waited for
    for (int l = 0; l < a.n_layers; ++l) {
        const PersistLayer &Ly = a.layers[l];
        const int32_t *const tab = tab_s + (l & 1) * tab_ld;
        if (tid < kMaxTok) {
            s.misc[4 + tid] = 0;
            s.ncand[tid] = 0;
            s.theta[tid] = 0xFFFFFFFFu;
        }
        // ------------------------------------------------ N: layer input
        if (a.stack) {
            // RMSNorm of resid in the canonical order of rms_partial / rms_scale;
            // resid is staged once in shared memory. Layer 0 of a launch reads the
            // caller's resid; a later layer waits for the words the previous layer's
            // combine wrote (tagged l), every thread for its own words.
            float *rs = reinterpret_cast<float *>(u_region);  // [T][H]
            bool fail = false;
            if (l == 0) {
                const float4 *r4 = reinterpret_cast<const float4 *>(a.resid);
                for (int idx = tid; idx < T * H / 4; idx += kPersistThreads)
                    reinterpret_cast<float4 *>(rs)[idx] = __ldcg(r4 + idx);
            } else {
                for (int b0 = 0; b0 < T * H && !fail; b0 += 8 * kPersistThreads) {
                    const unsigned long long *base = a.resid_t + b0 + tid;
                    uint32_t v[8];
                    unsigned m = 0;
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        if (b0 + u * kPersistThreads + tid < T * H) m |= 1u << u;
                    fail = !wait_tagged<8>([&](int u) { return base + u * kPersistThreads; }, m, (unsigned)l, v,
                                           Waiter{a.bar + 1, a.status});
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        if (m >> u & 1u) rs[b0 + u * kPersistThreads + tid] = __uint_as_float(v[u]);
                }
            }
            if (__syncthreads_or(fail)) break;
            for (int t = 0; t < T; ++t) {
                const float p = rms_partial(rs + (size_t)t * H, H, tid);
                if (lane == 0) s.wsum[t][warp] = p;
            }
            __syncthreads();
            for (int t = 0; t < T; ++t) {
                const float r = rms_scale(s.wsum[t], H, a.eps);
                const float *xt = rs + (size_t)t * H;
                for (int h = tid; h < H; h += kPersistThreads) {
                    const __nv_bfloat16 u = __float2bfloat16_rn(xt[h] * r);
                    xs[(size_t)t * ldx + h] = u;
                    if (a.trace_in && cta == 0) a.trace_in[((size_t)l * T + t) * H + h] = u;
                }
            }
        } else if (XF32) {
            // hi limbs in rows 0..3, lo limbs in rows 4..7
            const float *x = reinterpret_cast<const float *>(a.x);
            for (int idx = tid; idx < T * H; idx += kPersistThreads) {
                const int t = idx / H, h = idx % H;
                __nv_bfloat16 hi, lo;
                split_bf16(x[idx], hi, lo);
                xs[(size_t)t * ldx + h] = hi;
                xs[(size_t)(4 + t) * ldx + h] = lo;
            }
        } else {
            const uint4 *x = reinterpret_cast<const uint4 *>(a.x);
            for (int idx = tid; idx < T * H / 8; idx += kPersistThreads) {
                const int t = idx / (H / 8), h8 = (idx % (H / 8)) * 8;
                *reinterpret_cast<uint4 *>(xs + (size_t)t * ldx + h8) = x[idx];
            }
        }
        // this layer's router rows, bias and table row
        cp_async_wait_all();
        if (!mbar_wait(&s.rbar, (unsigned)l & 1u) && tid == 0) {
            set_status(a.status, MOE_STATUS_TIMEOUT);
            atomicExch(a.bar + 1, 1u);
        }
        r_done = l + 1;
        __syncthreads();
        // ------------------------------------------------ R: router logits of my experts
        {
            const int wsz = a.wr_bf16 ? 2 : 4;
            const int q = warp & 3;
            const int nrb = (E + G - 1) / G, e0 = cta * nrb;  // my experts: e0 .. e0 + nr - 1
            const int nr = E - e0 < nrb ? (E - e0 > 0 ? E - e0 : 0) : nrb;
            const float *const rscale = Ly.router_scale;
            auto xf = [&](int t, int h, float v[8]) {
                if (XF32 && !a.stack)
                    load_w8<float>(reinterpret_cast<const float *>(a.x) + (size_t)t * H + h, v);
                else
                    bf16x8_to_f32(*reinterpret_cast<const uint4 *>(xs + (size_t)t * ldx + h), v);
                if (OPTS && rscale) {
                    // the scaled router input x_h * s_h, rounded to fp32
                    float sc[8];
                    load_w8<float>(rscale + h, sc);
#pragma unroll
                    for (int j = 0; j < 8; ++j) v[j] *= sc[j];
                }
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
            // publish the logits of my experts (contiguous words of each token row), or,
            // owning none, a flag (its own 32-byte sector), tagged l + 1; the test hook
            // leaves CTA 0's out at fault_layer
            const int Ep = (E + 31) & ~31;  // token rows of the tagged logits padded to 32
            unsigned long long *lgt = a.lg_t + (size_t)(l & 1) * ((size_t)T * Ep + 4 * kMaxGrid);
            const bool publish = !(a.fault_layer == l && cta == 0);
            if (tid < nr * T) {
                const int r = tid / T, t = tid % T;
                const int e = e0 + r;
                const float v = combine_router4(&s.rpart[r][t][0]) + (Ly.bias ? s.bias[l & 1][r] : 0.f);
                if (publish) st_relaxed_u64(lgt + (size_t)t * Ep + e, tagged(l + 1, __float_as_uint(v)));
                if (a.logits) a.logits[(size_t)t * E + e] = v;
                if (a.trace_logits) a.trace_logits[((size_t)l * T + t) * E + e] = v;
            }
            if (nr == 0 && tid == 0 && publish) st_relaxed_u64(lgt + (size_t)T * Ep + 4 * cta, tagged(l + 1, 1u));
        }
        // ------------------------------------------------ T: top-K and the plan (every CTA)
        {
            // ord keys of the logits; token rows are padded to Ep (a multiple of 32)
            // with "no candidate" entries, so a warp's 32 entries and every segment
            // belong to one token
            const int Ep = (E + 31) & ~31, TE = T * Ep;
            uint32_t *const ords = reinterpret_cast<uint32_t *>(u_region);  // [T][Ep]
            uint32_t *const segmax = ords + TE;                              // [kMaxTok][kMaxSeg]
            unsigned long long *const cand =
                reinterpret_cast<unsigned long long *>(segmax + kMaxTok * kMaxSeg);  // [kMaxTok][kCandCap]
            // segments of `seg` entries, at least K + 2 of them per token where kMaxSeg allows
            int lseg = 5;
            while (lseg > 0 && (Ep >> lseg) < K + 2 && (Ep >> (lseg - 1)) <= kMaxSeg) --lseg;
            const int seg = 1 << lseg, nseg = Ep >> lseg;
            const bool all_cand = E <= kCandCap;  // no threshold: every expert is a candidate
            const unsigned lt = (1u << lane) - 1u;
            // (1) keys and segment maxima (the loop bound is uniform in each warp); the
            // logits are the tagged words every CTA published (tag l + 1), read as soon
            // as they are all there, with the flags of the CTAs (a CTA's flag follows
            // its layer input being read)
            const unsigned long long *lgt = a.lg_t + (size_t)(l & 1) * ((size_t)TE + 4 * kMaxGrid);
            const int c_noexp = (E + (E + G - 1) / G - 1) / ((E + G - 1) / G);  // first CTA owning no expert
            const float inv_ep = __frcp_rn((float)Ep);  // token of flat index i: (int)((i + 0.5) / Ep), exact here
            auto tok = [&](int i) { return (int)(((float)i + 0.5f) * inv_ep); };
            bool fail = false;
            for (int b0 = 0; b0 < TE; b0 += 4 * kPersistThreads) {
                float v[4];
                {
                    // words b0 + u * 512 + tid (u < 4) of the padded rows, and (first
                    // pass) the flag of CTA tid
                    uint32_t vv[5];
                    unsigned m = 0;
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int idx = b0 + u * kPersistThreads + tid, t = tok(idx), e = idx - t * Ep;
                        if (idx < TE && e < E) m |= 1u << u;
                    }
                    if (b0 == 0 && c_noexp + tid < G) m |= 1u << 4;
                    const unsigned long long *base = lgt + b0 + tid, *flag = lgt + TE + 4 * (c_noexp + tid);
                    if (!fail)
                        fail = !wait_tagged<5>(
                            [&](int u) { return u < 4 ? base + u * kPersistThreads : flag; }, m, (unsigned)(l + 1), vv,
                            Waiter{a.bar + 1, a.status});
#pragma unroll
                    for (int u = 0; u < 4; ++u) v[u] = __uint_as_float(vv[u]);
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int idx = b0 + u * kPersistThreads + tid, t = tok(idx), e = idx - t * Ep;
                    if (idx - lane < TE) {
                        const bool valid = e < E;
                        const uint32_t o = valid ? topk_ord(v[u]) : 0u;
                        if (valid && !isfinite(v[u])) s.misc[4 + t] = 1;
                        ords[idx] = o;
                        if (!all_cand) {
                            uint32_t m;
                            if (seg == 32) {
                                m = __reduce_max_sync(0xffffffffu, o);
                            } else {
                                m = o;
                                for (int d = 1; d < seg; d <<= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, d));
                            }
                            if ((lane & (seg - 1)) == 0) segmax[t * kMaxSeg + (e >> lseg)] = m;
                        }
                    }
                }
            }
            if (__syncthreads_or(fail)) break;
            // (2) threshold of each token: the K-th largest segment maximum, counted
            // with multiplicity = the smallest maximum that fewer than K maxima
            // exceed. Each maximum is a distinct entry, so at least K entries reach
            // it and every top-K entry does. A warp ranks one maximum against all
            // (shared-memory broadcasts and a ballot: warp shuffles are slow here).
            // One token with at most 32 segments: every warp finds the threshold itself
            // (lane i ranks maximum i against the others), so no barrier is needed
            // before the candidates.
            const bool warp_theta = T == 1 && nseg <= 32 && !all_cand;
            uint32_t theta_w = 0u;
            if (warp_theta) {
                const uint32_t mine = lane < nseg ? segmax[lane] : 0u;
                int rank = 0;
#pragma unroll
                for (int j = 0; j < 32; ++j) rank += (j < nseg) & (__shfl_sync(0xffffffffu, mine, j) > mine);
                theta_w = __reduce_min_sync(0xffffffffu, (lane < nseg && rank < K) ? mine : 0xFFFFFFFFu);
            } else {
                if (!all_cand) {
                    for (int t = 0; t < T; ++t) {
                        const uint32_t *sm = segmax + t * kMaxSeg;
                        for (int i = warp; i < nseg; i += kPWarps) {
                            const uint32_t mi = sm[i];
                            int rank = 0;
                            for (int j = lane; j - lane < nseg; j += 32)
                                rank += __popc(__ballot_sync(0xffffffffu, j < nseg && sm[j] > mi));
                            if (lane == 0 && rank < K) atomicMin(&s.theta[t], mi);
                        }
                    }
                }
                __syncthreads();
            }
            // (3) candidates: the entries at or above the threshold
            for (int b0 = 0; b0 < TE; b0 += kPersistThreads) {
                if (b0 + warp * 32 >= TE) break;
                const int idx = b0 + tid, t = tok(idx), e = idx - t * Ep;
                const uint32_t o = ords[idx];
                const bool c = e < E && o >= (all_cand ? 0u : warp_theta ? theta_w : s.theta[t]);
                const unsigned bal = __ballot_sync(0xffffffffu, c);
                int base = 0;
                if (lane == 0 && bal) base = atomicAdd(&s.ncand[t], __popc(bal));
                base = __shfl_sync(0xffffffffu, base, 0);
                if (c) {
                    const int pos = base + __popc(bal & lt);
                    if (pos < kCandCap) cand[t * kCandCap + pos] = topk_key_of(o, e);
                }
            }
            __syncthreads();
            // (4) rank of each candidate among its token's candidates = its place in
            // the top-K (keys are distinct); s.sel[t][k] = the k-th key. A warp ranks
            // one candidate against all (broadcast + ballot).
            int maxn = 0;
            for (int t = 0; t < T; ++t) maxn = max(maxn, s.ncand[t]);
            if (maxn <= kCandCap) {
                for (int t = 0; t < T; ++t) {
                    const int n = s.ncand[t];
                    const unsigned long long *ct = cand + t * kCandCap;
                    for (int i = warp; i < n; i += kPWarps) {
                        const unsigned long long ki = ct[i];
                        int rank = 0;
                        for (int j = lane; j - lane < n; j += 32)
                            rank += __popc(__ballot_sync(0xffffffffu, j < n && ct[j] > ki));
                        if (lane == 0 && rank < K) s.sel[t][rank] = ki;
                    }
                }
            } else {
                // too many candidates (e.g. many equal logits)
                topk_sort_merge(lgt, T, E, reinterpret_cast<unsigned long long *>(u_region), s.sel);
            }
            __syncthreads();
            // down units (expert-major: unit j = expert j / dt, row tile j % dt) split
            // over the CTAs by down bytes: CTA c takes the units whose byte midpoint
            // falls in [c D / G, (c + 1) D / G) (single-precision arithmetic: CTA c and
            // CTA c + 1 evaluate the same boundary with the same operations, so the
            // ranges tile [0, n_units)); called by one thread
            auto set_units = [&](int nu) {
                const bool sh = Ly.shared != nullptr;
                const int nr_units = nu * dt;
                const int n_units = nr_units + (sh ? dt : 0);
                const float dr = (float)L.d_tile_bytes, dsb = sh ? (float)a.LS.d_tile_bytes : 0.f;
                const float Dr = (float)nr_units * dr, Dtot = Dr + (float)dt * dsb;
                auto first_unit = [&](int c) -> int {
                    if (c <= 0) return 0;
                    const float b = __fdividef(Dtot * (float)c, (float)G);
                    const float x = b - 0.5f * dr;  // routed: j*dr + dr/2 >= b
                    const int j = x <= 0.f ? 0 : (int)ceilf(__fdividef(x, dr));
                    if (j < nr_units || !sh) return j < nr_units ? j : nr_units;
                    const float y = b - Dr - 0.5f * dsb;  // shared: Dr + k*dsb + dsb/2 >= b
                    const int jj = nr_units + (y <= 0.f ? 0 : (int)ceilf(__fdividef(y, dsb)));
                    return jj < n_units ? jj : n_units;
                };
                s.misc[12] = first_unit(cta);
                s.misc[13] = cta == G - 1 ? n_units : first_unit(cta + 1);
            };
            if (T == 1 && !OPTS) {
                // one token (K <= 32 pairs of distinct experts): weights, the order by
                // expert and the plan in warp 0's registers, the same arithmetic as the
                // steps below (the softmax sum in k order)
                if (warp == 0) {
                    const unsigned long long key = s.sel[0][lane];
                    const int si = lane < K ? topk_key_index(key) : 0x7FFFFFFF;
                    const float sv = topk_key_value(key);
                    const float m = __shfl_sync(0xffffffffu, sv, 0);
                    const bool bad = s.misc[4] != 0;
                    const float ex = (lane < K && !bad) ? expf(sv - m) : 0.f;
                    // loops unrolled to 32 so that every shuffle is issued up front (lanes
                    // k >= K hold ex = 0: adding them leaves the sum's bits unchanged)
                    float exk[32];
#pragma unroll
                    for (int k = 0; k < 32; ++k) exk[k] = __shfl_sync(0xffffffffu, ex, k);
                    float sum = 0.f;
#pragma unroll
                    for (int k = 0; k < 32; ++k) sum += exk[k];
                    const float wk = bad ? __int_as_float(0x7fc00000) : ex / sum;
                    int rank = 0;  // place in expert order (the K experts are distinct)
#pragma unroll
                    for (int q = 0; q < 32; ++q) rank += __shfl_sync(0xffffffffu, si, q) < si;
                    int slot = -1;
                    bool absent = false, oob = false, live = false;
                    if (lane < K) {
                        slot = tab[si];
                        if (slot < 0) absent = true;
                        else if (slot >= Ly.capacity) oob = true;
                        else live = wk != 0.f;
                        s.ids[lane] = si;
                        s.w[lane] = wk;
                        s.live[lane] = live;
                        if (a.ids_out && cta == 0) a.ids_out[lane] = si;
                    }
                    const unsigned lm = __ballot_sync(0xffffffffu, live);
                    int pos = 0;  // place among the live pairs in expert order
#pragma unroll
                    for (int q = 0; q < 32; ++q) {
                        const int rq = __shfl_sync(0xffffffffu, rank, q);
                        pos += (int)((lm >> q) & 1u) & (rq < rank);
                    }
                    if (live) {
                        s.cols[pos] = lane;
                        s.cexp[pos] = s.uexp[pos] = si;
                        s.cslot[pos] = s.uslot[pos] = slot;
                        s.ustart[pos] = pos;
                    }
                    absent = __any_sync(0xffffffffu, absent);
                    oob = __any_sync(0xffffffffu, oob);
                    if (cta == 0 && lane == 0) {
                        if (bad) set_status(a.status, MOE_STATUS_NONFINITE);
                        if (absent) set_status(a.status, MOE_STATUS_EXPERT_ABSENT);
                        if (oob) set_status(a.status, MOE_STATUS_BOUNDS);
                    }
                    if (lane == 0) {
                        const int nlive = __popc(lm);
                        s.ustart[nlive] = nlive;
                        s.misc[0] = nlive;
                        s.misc[1] = nlive;
                        set_units(nlive);
                    }
                }
            } else {
                // (5) weights of token t (warp t)
                if (warp < T) {
                    const int t = warp;
                    const unsigned long long key = s.sel[t][lane];
                    const int si = topk_key_index(key);
                    const float sv = topk_key_value(key);
                    const bool bad = s.misc[4 + t] != 0;
                    const float m = topk_key_value(s.sel[t][0]);
                    float wk;
                    if (bad) {
                        wk = __int_as_float(0x7fc00000);
                        if (OPTS && lane == 0 && cta == 0 && Ly.route.omitted) Ly.route.omitted[t] = 0.f;
                    } else if constexpr (OPTS) {
                        wk = route_weight(Ly.route, sv, m, si, K, lane, s.wex[t],
                                          reinterpret_cast<int *>(u_region) + t * 64,
                                          cta == 0 ? Ly.route.omitted : nullptr, t);
                    } else {
                        wk = topk_weight_smem(sv, m, K, lane, s.wex[t]);
                    }
                    if (lane < K) {
                        s.ids[t * K + lane] = si;
                        s.w[t * K + lane] = wk;
                        if (a.ids_out && cta == 0) a.ids_out[(size_t)t * K + lane] = si;
                    }
                    if (bad && lane == 0 && cta == 0) set_status(a.status, MOE_STATUS_NONFINITE);
                }
                // (6) stable order of pairs by expert: rank = #{q : (id_q, q) < (id_p, p)}
                if (T == 1 && P <= 32) {
                    // one token: its pairs are warp 0's lanes
                    if (warp == 0) {
                        __syncwarp();
                        const int ep = lane < P ? s.ids[lane] : 0x7FFFFFFF;
                        int r = 0;
                        for (int q = 0; q < P; ++q) {
                            const int eq = s.ids[q];
                            r += (eq < ep) | ((eq == ep) & (q < lane));
                        }
                        if (lane < P) s.sorted[r] = lane;
                        __syncwarp();
                    }
                } else {
                    __syncthreads();
                    if (tid < P) {
                        const int ep = s.ids[tid];
                        int r0 = 0, r1 = 0, r2 = 0, r3 = 0;
    #pragma unroll 2
                        for (int q4 = 0; q4 < P; q4 += 4) {
                            const int4 v4 = *reinterpret_cast<const int4 *>(s.ids + q4);
                            r0 += (q4 < P) & ((v4.x < ep) | ((v4.x == ep) & (q4 < tid)));
                            r1 += (q4 + 1 < P) & ((v4.y < ep) | ((v4.y == ep) & (q4 + 1 < tid)));
                            r2 += (q4 + 2 < P) & ((v4.z < ep) | ((v4.z == ep) & (q4 + 2 < tid)));
                            r3 += (q4 + 3 < P) & ((v4.w < ep) | ((v4.w == ep) & (q4 + 3 < tid)));
                        }
                        s.sorted[(r0 + r1) + (r2 + r3)] = tid;
                    }
                    __syncthreads();
                }
                if (warp == 0) {
                    int running = 0;
                    bool absent = false, oob = false;
                    for (int base = 0; base < P; base += 32) {
                        const int r = base + lane;
                        int p = -1, e = -1, slot = -1, live = 0;
                        if (r < P) {
                            p = s.sorted[r];
                            e = s.ids[p];
                            slot = tab[e];
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
                        set_units(nu);
                    }
                }
            }
            __syncthreads();
        }
        const int nU = s.misc[0];
        const bool has_shared = Ly.shared != nullptr;
        const int tilesF = L.gu_tiles, tilesS = has_shared ? a.LS.gu_tiles : 0;
        const int n_items = nU * tilesF + tilesS;
        const int j0 = s.misc[12], j1 = s.misc[13];
        // ------------------------------------------------ weight copies of this warp
        // gate/up groups of S warps; warps past NG * S (16 % S of them) take no gate/up
        // work (they would be a group short of S warps at its named barrier)
        const int grp = warp / S_GU, q = warp % S_GU;
        const bool gu_warp = grp < NG;
        const int n_ch = L.gu_chunks;  // the shared expert has the same H chunks
        const int cb0 = gu_chunk_begin(q, n_ch, S_GU), cb1 = gu_chunk_begin(q + 1, n_ch, S_GU);
        // a group with one item this layer takes its part in one piece when it fits in
        // three quarters of the ring (fewer copies to issue: the copy unit takes them one
        // at a time); otherwise two pieces of each kind fit in the ring at once
        const bool one_item = cta + G * (grp + NG) >= n_items;
        const bool one_piece = one_item && cb1 > cb0 && (cb1 - cb0) * L.gu_chunk_bytes * 4 <= 3 * a.geom.ring_bytes;
        const int pcg = one_piece ? cb1 - cb0 : pcg2;
        const int dw = kPWarps - 1 - warp;  // down units go to the last warps first
        auto gu_tile = [&](int j) -> const uint8_t * {
            if (j >= nU * tilesF) return Ly.shared + (long long)(j - nU * tilesF) * a.LS.gu_tile_bytes;
            return Ly.arena + (long long)s.uslot[j / tilesF] * Ly.stride + (long long)(j % tilesF) * L.gu_tile_bytes;
        };
        auto d_tile = [&](int j) -> const uint8_t * {
            const int ti = j / dt, r = j % dt;
            if (ti >= nU) return Ly.shared + a.LS.d_offset + (long long)r * a.LS.d_tile_bytes;
            return Ly.arena + (long long)s.uslot[ti] * Ly.stride + L.d_offset + (long long)r * L.d_tile_bytes;
        };
        int pphase = 0, pm = 0, pch = cb0, pd = 0, pdch = 0;
        auto produce = [&]() {
            for (;;) {
                if (pphase == 0) {
                    if (pch >= cb1) {
                        ++pm;
                        pch = cb0;
                    }
                    const int j = cta + G * (grp + NG * pm);
                    if (!gu_warp || cb0 >= cb1 || j >= n_items) {
                        pphase = 1;
                        continue;
                    }
                    const int nc = cb1 - pch < pcg ? cb1 - pch : pcg;
                    const int bytes = piece_bytes(L.gu_chunk_bytes, L.gu_half, n_ch, pch, nc);
                    if (!ring_push(ring, gu_tile(j) + (long long)pch * L.gu_chunk_bytes, bytes, lane)) return;
                    pch += nc;
                } else if (pphase == 1) {
                    const int j = j0 + dw + kPWarps * pd;
                    if (j >= j1) {
                        pphase = 2;
                        return;
                    }
                    const QLayout &LL = j / dt >= nU ? a.LS : L;
                    if (pdch >= LL.d_chunks) {
                        ++pd;
                        pdch = 0;
                        continue;
                    }
                    const int nc = LL.d_chunks - pdch < pcd ? LL.d_chunks - pdch : pcd;
                    const int bytes = piece_bytes(LL.d_chunk_bytes, LL.d_half, LL.d_chunks, pdch, nc);
                    if (!ring_push(ring, d_tile(j) + (long long)pdch * LL.d_chunk_bytes, bytes, lane)) return;
                    pdch += nc;
                } else {
                    return;
                }
            }
        };
        produce();
        // ------------------------------------------------ GU: gate/up + activation
        {
            float *gred = red + (size_t)grp * S_GU * 32 * 8;
            for (int m = 0; gu_warp; ++m) {
                const int j = cta + G * (grp + NG * m);
                if (j >= n_items) break;
                const bool shared = j >= nU * tilesF;
                int ncols, col0 = 0, rt;
                if (!shared) {
                    const int u = j / tilesF;
                    rt = j % tilesF;
                    col0 = s.ustart[u];
                    ncols = s.ustart[u + 1] - col0;
                } else {
                    rt = j - nU * tilesF;
                    ncols = T;
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
                const Unpack un = shared ? a.un_s : a.un;  // in registers for the item's chunks
                float acc[2][1][4] = {};
                const uint8_t *pbase = nullptr;
                int pnc = 0, pbytes = 0;
                for (int ch = cb0; ch < cb1; ++ch) {
                    const int k = (ch - cb0) % pcg;
                    if (k == 0) {
                        pnc = cb1 - ch < pcg ? cb1 - ch : pcg;
                        pbytes = piece_bytes(L.gu_chunk_bytes, L.gu_half, n_ch, ch, pnc);
                        pbase = ring_front(ring, pbytes, a.status, a.bar);
                    }
                    const bool half = L.gu_half && ch == n_ch - 1;
                    const int cbh = half ? L.cb / 2 : L.cb, sbh = half ? L.sb / 2 : L.sb;
                    const uint8_t *p = pbase + k * L.gu_chunk_bytes;
                    ChunkRegs<KIND> rg[2];
                    load_chunk_s<KIND>(p, p + 2 * cbh, half, lane, rg[0]);
                    load_chunk_s<KIND>(p + cbh, p + 2 * cbh + sbh, half, lane, rg[1]);
                    if (k == pnc - 1) {
                        ring_pop(ring, pbytes);
                        produce();
                    }
                    mma_chunk<KIND, 2, 1>(rg, half, bt, ch * 128, un, acc);
                }
                // the group adds the S parts in part order (as the multi-kernel k_gateup)
#pragma unroll
                for (int m2 = 0; m2 < 2; ++m2)
#pragma unroll
                    for (int e4 = 0; e4 < 4; ++e4) gred[(q * 32 + lane) * 8 + m2 * 4 + e4] = acc[m2][0][e4];
                asm volatile("bar.sync %0, %1;" ::"r"(grp + 1), "r"(S_GU * 32) : "memory");
                if (q == 0) {
                    float v[8];
#pragma unroll
                    for (int e8 = 0; e8 < 8; ++e8) {
                        float sum = gred[lane * 8 + e8];
#pragma unroll
                        for (int w = 1; w < S_GU; ++w) sum += gred[(w * 32 + lane) * 8 + e8];
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
                    // the item's h is written: count it for its expert (release: the
                    // warp's stores, ordered before by __syncwarp, come first)
                    __syncwarp();
                    if (lane == 0) {
                        int *cnt = a.gu_cnt + (size_t)l * kMaxUnits + (shared ? nU : j / tilesF);
                        asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(cnt) : "memory");
                    }
                }
                asm volatile("bar.sync %0, %1;" ::"r"(grp + 1), "r"(S_GU * 32) : "memory");
            }
        }
        // ------------------------------------------------ D: down projection + combine
        {
            const int n_tasks = nU + (has_shared ? 1 : 0);
            produce();
            // h limbs of the experts of this CTA's units, staged once: routed plan
            // columns [c_lo, c_hi) at hst + (i - c_lo)*ldh (hi) and hst + lo_off + ...
            // (lo; lo_off puts hi and lo rows on different banks); the shared
            // expert's tokens after them at hss
            const int ldh = L.F + 8, ldhs = a.LS.F + 8;
            int c_lo = 0, c_hi = 0;
            bool need_sh = false;
            if (j1 > j0) {
                const int ti_lo = j0 / dt, ti_hi = (j1 - 1) / dt;
                if (ti_lo < nU) {
                    c_lo = s.ustart[ti_lo];
                    c_hi = s.ustart[(ti_hi < nU ? ti_hi : nU - 1) + 1];
                }
                need_sh = ti_hi >= nU;
            }
            // wait until every gate/up item of the experts of my units is done (down
            // units need the expert's whole h); thread i waits for the i-th expert
            {
                bool fail = false;
                if (j1 > j0) {
                    const int u = j0 / dt + tid;
                    if (u <= (j1 - 1) / dt)
                        fail = !wait_count(a.gu_cnt + (size_t)l * kMaxUnits + u, u < nU ? tilesF : tilesS,
                                           Waiter{a.bar + 1, a.status});
                }
                if (__syncthreads_or(fail)) break;
            }
            const int nrow = c_hi - c_lo;
            const int lo_off = ((nrow * ldh + 63) & ~63) + 32;
            const int hss_off = (lo_off + nrow * ldh + 63) & ~63;
            const int lo_off_s = ((T * ldhs + 63) & ~63) + 32;
            const size_t need = (size_t)(hss_off + (need_sh ? lo_off_s + T * ldhs : 0)) * 2;
            const bool staged = need <= a.geom.hst_bytes;
            __nv_bfloat16 *const hss = hst + hss_off;
            if (staged) {
                const int vpr = L.F / 8;  // 16-byte vectors per routed row
                for (int idx = tid; idx < nrow * 2 * vpr; idx += kPersistThreads) {
                    const int i = idx / (2 * vpr), rem = idx % (2 * vpr), limb = rem / vpr, v = rem % vpr;
                    const __nv_bfloat16 *src = (limb ? a.h_lo : a.h_hi) + (size_t)s.cols[c_lo + i] * a.h_ld + v * 8;
                    *reinterpret_cast<uint4 *>(hst + (limb ? lo_off : 0) + i * ldh + v * 8) =
                        __ldcg(reinterpret_cast<const uint4 *>(src));
                }
                if (need_sh) {
                    const int vps = a.LS.F / 8;
                    for (int idx = tid; idx < T * 2 * vps; idx += kPersistThreads) {
                        const int t = idx / (2 * vps), rem = idx % (2 * vps), limb = rem / vps, v = rem % vps;
                        const __nv_bfloat16 *src = (limb ? a.h_lo : a.h_hi) + (size_t)(P + t) * a.h_ld + v * 8;
                        *reinterpret_cast<uint4 *>(hss + (limb ? lo_off_s : 0) + t * ldhs + v * 8) =
                            __ldcg(reinterpret_cast<const uint4 *>(src));
                    }
                }
            }
            __syncthreads();
            // the next layer's router rows (their buffer is free since barrier 1); warp 0
            // gets the last down units, so it has the most slack here
            if (warp == 0 && l + 1 < a.n_layers) {
                prefetch_router(a, l + 1, wr_s, tab_s + ((l + 1) & 1) * tab_ld, s.bias[(l + 1) & 1], &s.rbar);
                r_issued = l + 2;
            }
            for (int di = 0;; ++di) {
                const int j = j0 + dw + kPWarps * di;
                if (j >= j1) break;
                const int ti = j / dt, r = j % dt;
                const bool shared = ti >= nU;
                const QLayout &LL = shared ? a.LS : L;
                int ncols, col0 = 0;
                if (!shared) {
                    col0 = s.ustart[ti];
                    ncols = s.ustart[ti + 1] - col0;
                } else {
                    ncols = T;
                }
                const Unpack un = shared ? a.un_s : a.un;  // in registers for the unit's chunks
                // B tiles: columns nb*4 + (g & 3); lanes g < 4 read hi limbs, g >= 4 lo limbs
                // staged: B rows in shared memory (the pointer provably shared, so the
                // loads are shared-memory loads); otherwise h limbs in global memory
                auto make_bt = [&](int nb, auto staged_tag) {
                    constexpr bool STAGED = decltype(staged_tag)::value;
                    const int jc = nb * 4 + (g & 3);
                    BTile b{STAGED ? hst : a.h_hi, false};
                    if (jc < ncols) {
                        if constexpr (STAGED) {
                            b.row = shared ? hss + (g < 4 ? 0 : lo_off_s) + jc * ldhs + 2 * c
                                           : hst + (g < 4 ? 0 : lo_off) + (col0 + jc - c_lo) * ldh + 2 * c;
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
                                st_relaxed_u64(a.yp_t + (size_t)row * H + r * 16 + rr,
                                               tagged(l + 1, __float_as_uint(v[e4])));
                            }
                        }
                    }
                };
                const int nchk = LL.d_chunks;
                auto run = [&](auto nb_tag, auto staged_tag) {
                    constexpr int NB = decltype(nb_tag)::value;
                    BTile bt[NB];
#pragma unroll
                    for (int nb = 0; nb < NB; ++nb) bt[nb] = make_bt(nb, staged_tag);
                    float acc[1][NB][4] = {};
                    const uint8_t *pbase = nullptr;
                    int pnc = 0, pbytes = 0;
                    for (int ch = 0; ch < nchk; ++ch) {
                        const int k = ch % pcd;
                        if (k == 0) {
                            pnc = nchk - ch < pcd ? nchk - ch : pcd;
                            pbytes = piece_bytes(LL.d_chunk_bytes, LL.d_half, nchk, ch, pnc);
                            pbase = ring_front(ring, pbytes, a.status, a.bar);
                        }
                        const bool half = LL.d_half && ch == nchk - 1;
                        const int cbh = half ? LL.cb / 2 : LL.cb;
                        const uint8_t *p = pbase + k * LL.d_chunk_bytes;
                        ChunkRegs<KIND> rg[1];
                        load_chunk_s<KIND>(p, p + cbh, half, lane, rg[0]);
                        if (k == pnc - 1) {
                            ring_pop(ring, pbytes);
                            produce();
                        }
                        mma_chunk<KIND, 1, NB>(rg, half, bt, ch * 128, un, acc);
                    }
#pragma unroll
                    for (int nb = 0; nb < NB; ++nb) emit(nb, acc[0][nb]);
                };
                if (staged) {
                    if (ncols > 4)
                        run(std::integral_constant<int, 2>{}, std::true_type{});
                    else
                        run(std::integral_constant<int, 1>{}, std::true_type{});
                } else {
                    if (ncols > 4)
                        run(std::integral_constant<int, 2>{}, std::false_type{});
                    else
                        run(std::integral_constant<int, 1>{}, std::false_type{});
                }
            }
            // the combine: row tile r is summed by the warp that ran the last task's unit
            // of that tile (the shared expert's, else the last routed expert's), after all
            // of its own units; it reads every pair's y rows of the tile as tagged words
            // as soon as they are all there, then adds them in k order (+ the shared
            // expert). With no task at all, warp 0 of CTA c writes tiles c, c + G, ...
            float *cs = reinterpret_cast<float *>(ring.base);  // the combine's scratch
            if (n_tasks > 0) {
                for (int di = 0;; ++di) {
                    const int j = j0 + dw + kPWarps * di;
                    if (j >= j1) break;
                    if (j / dt == n_tasks - 1) combine_tile(a, s.live, s.w, cs, j % dt, l, has_shared, lane);
                }
            } else if (warp == 0) {
                for (int r = cta; r < dt; r += G) combine_tile(a, s.live, s.w, cs, r, l, has_shared, lane);
            }
            // no warp starts polling for the next layer's input before the CTA's own
            // combines are done (polling warps of the same SM delay the combiners'
            // loads)
            __syncthreads();
        }
    }
    ring_drain(ring);
    // a router prefetch still in flight (the loop stopped early)
    if (r_issued > r_done) mbar_wait(&s.rbar, (unsigned)(r_issued - 1) & 1u);
    cp_async_wait_all();
}

}  // namespace

PersistGeom persist_geom(int kind, int T, int H, int E, int K, int F, int F_shared, int wr_bytes, int x_f32, int G,
                         size_t max_smem) {
    (void)K;
    (void)F;
    (void)F_shared;
    PersistGeom g;
    auto al = [](size_t v) { return (v + 127) & ~size_t(127); };
    const int nr = (E + G - 1) / G;
    const size_t stat = sizeof(Plan);
    g.tab_ld = (E + 3) & ~3;
    g.off_wr = 0;
    g.off_tab = al((size_t)nr * H * wr_bytes);
    g.off_xs = g.off_tab + al((size_t)2 * g.tab_ld * 4);
    const int xs_rows = x_f32 ? 8 : T;
    const size_t xs_bytes = (size_t)xs_rows * (H + 8) * 2;
    g.off_red = g.off_xs + al(xs_bytes);
    g.off_hst = g.off_xs;
    g.hst_bytes = al(xs_bytes) + kRedBytes;  // h staging reuses xs + red
    g.off_ring = g.off_xs + g.hst_bytes;
    g.off_u = g.off_ring;
    const size_t topk_fast =
        (size_t)T * ((E + 31) & ~31) * 4 + (size_t)kMaxTok * kMaxSeg * 4 + (size_t)T * kCandCap * 8;
    const size_t topk_sort = (size_t)T * ((E + 31) / 32) * 32 * 8;
    const size_t norm = (size_t)T * H * 4;
    size_t u = topk_fast > topk_sort ? topk_fast : topk_sort;
    if (norm > u) u = norm;
    const int gu_chunk = kind == MOE_Q2_64 ? 1152 : 2304;  // the largest piece is one gate/up chunk or more
    const long long room = (long long)max_smem - (long long)stat - (long long)g.off_ring;
    long long per_warp = room / (kPersistThreads / 32);
    if (per_warp > kMaxRingBytes) per_warp = kMaxRingBytes;
    per_warp &= ~15LL;
    if (per_warp < gu_chunk) {  // cannot hold one gate/up chunk per warp
        g.ring_bytes = 0;
        g.dyn_bytes = g.bytes = (size_t)-1;
        return g;
    }
    g.ring_bytes = (int)per_warp;
    size_t tail = (size_t)g.ring_bytes * (kPersistThreads / 32);
    if (u > tail) tail = u;
    g.dyn_bytes = g.off_ring + al(tail);
    g.bytes = g.dyn_bytes + stat;
    if (g.bytes > max_smem) {
        g.ring_bytes = 0;
        g.dyn_bytes = g.bytes = (size_t)-1;
    }
    return g;
}

int launch_decode_persistent(const PersistArgs &a, int G, cudaStream_t s) {
    bool opts = false;
    for (int l = 0; l < a.n_layers; ++l) {
        const PersistLayer &L = a.layers[l];
        opts |= L.router_scale != nullptr || L.route.kind != MOE_ROUTER_SOFTMAX || L.route.down_scale != nullptr ||
                L.route.drop_eligible != nullptr || L.route.omitted != nullptr;
    }
    const void *kern;
#define MOE_PICK(KD, XF) (opts ? (const void *)k_decode<KD, XF, true> : (const void *)k_decode<KD, XF, false>)
    if (a.L.kind == MOE_Q2_64)
        kern = a.x_f32 ? MOE_PICK(MOE_Q2_64, true) : MOE_PICK(MOE_Q2_64, false);
    else
        kern = a.x_f32 ? MOE_PICK(MOE_Q4_32, true) : MOE_PICK(MOE_Q4_32, false);
#undef MOE_PICK
    if (G > kMaxGrid) return set_error(MOE_ERR_UNSUPPORTED, "persistent decode: %d CTAs > %d", G, kMaxGrid);
    MOE_CUDA_TRY(cudaMemsetAsync(a.bar, 0, a.sync_bytes, s));
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
    int per_sm = 0, per_sm2 = 0;
    const int dyn = smem_bytes - (int)sizeof(Plan);
    MOE_CUDA_TRY(
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_decode<MOE_Q2_64, false, true>, kPersistThreads, dyn));
    MOE_CUDA_TRY(
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm2, k_decode<MOE_Q4_32, false, true>, kPersistThreads, dyn));
    if (per_sm2 < per_sm) per_sm = per_sm2;
    *G = per_sm >= 1 ? sms : 0;
    return MOE_OK;
}

int init_persist_attributes(int max_smem) {
    const void *ks[] = {(const void *)k_decode<MOE_Q2_64, true, false>, (const void *)k_decode<MOE_Q2_64, false, false>,
                        (const void *)k_decode<MOE_Q4_32, true, false>, (const void *)k_decode<MOE_Q4_32, false, false>,
                        (const void *)k_decode<MOE_Q2_64, true, true>,  (const void *)k_decode<MOE_Q2_64, false, true>,
                        (const void *)k_decode<MOE_Q4_32, true, true>,  (const void *)k_decode<MOE_Q4_32, false, true>};
    for (const void *k : ks) {
        int rc = set_max_dynamic_smem(k, max_smem);
        if (rc) return rc;
    }
    return MOE_OK;
}

}  // namespace moe
