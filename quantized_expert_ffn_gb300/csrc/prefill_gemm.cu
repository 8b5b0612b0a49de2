// prefill_gemm.cu -- the routed experts for prefill-sized windows as grouped GEMMs
// on the 5th-generation tensor cores (tcgen05.mma, fp16 x fp16 -> fp32 in TMEM).
//
// kairos-engine README, "Prefill and decode are different machines": prefill
// dequantises the expert weights and runs tensor-core GEMMs over the tokens routed
// to each expert; Krasis white paper sec. 5.3: gate/up, activation, down, weighted
// reduce. Here the dequantisation is fused into the staging of each K-slice:
//
//   D[128 weight rows][<=256 tokens] += A[128][64] * B[<=256][64]^T per stage
//
//   A  128 rows of Q4 weights: one TMA warp brings each 128-k chunk of the packed
//      layout (codes + per-32 fp16 scales) in with bulk copies; 8 dequant warps turn
//      it into fp16 w = fp16(d * (q - 8)) (one rounding; q - 8 is exact) and store
//      it with stmatrix, K-major with the 128-byte swizzle the MMA descriptor names;
//   B  the group's rows, 64 fp16 each per stage, loaded by the TMA warp through a
//      tensor map in the smallest box (16 to 256 rows) that holds the group
//      (gate/up: x gathered into plan order and converted to fp16 once per layer;
//      down: h in plan order);
//   MMA one thread waits on the stage's "full" barrier (the B bytes and the dequant
//      warps' arrivals on one barrier), issues 4 x tcgen05.mma (K = 16 each) and
//      commits to the stage's "empty" barrier (which frees the A and the B slot);
//      after the last stage it commits the tile to an "accumulator full" barrier;
//      two accumulators of 256 TMEM columns alternate. This thread's instructions
//      sit on every stage's critical path, so its loop is kept short;
//   epilogue 4 warps read the accumulator with tcgen05.ld (warp q: TMEM lanes
//      32q..32q+31). Gate/up tiles hold rows [gate 16 | up 16] x 4, so a warp pairs
//      gate and up of the same row with one shuffle, applies the activation and
//      writes h as fp16 (row = plan column); down tiles write fp32 y_pair rows.
//
// A tile is (column group of <= 256 live pairs of one expert, 128-row M-tile);
// CTAs (one per SM) take tiles round-robin. Every barrier wait gives up after about
// a second (MOE_STATUS_TIMEOUT) and the CTA stops; the TMEM it allocated is
// released on every path.
#include <cudaTypedefs.h>

#include "decode_common.cuh"
#include "prefill_gemm.cuh"

namespace moe {

namespace {

constexpr int kBM = 128, kBN = 256, kBK = 64;
constexpr int kPSlots = 3;     // packed ring: one 128-k chunk per slot
constexpr int kABoxRows = 128; // rows per router A box
constexpr int kRN = 64;        // router tiles: tokens per tile (and rows per router B box)
// two groups of 8 dequant warps take alternate stages (two stages in flight)
// one TMA warp for the packed weights, one for the B rows (each blocks only on its own
// barriers)
constexpr int kDqWarps = 16, kTmaWarp = 16, kTmaBWarp = 17, kMmaWarp = 18, kEpiWarps = 4;
constexpr int kThreads = 32 * (kDqWarps + 3 + kEpiWarps);  // 736
constexpr int kATile = kBM * kBK * 2;      // 16 KB
constexpr int kPacked = 9216;              // packed codes + scales of one 128-k chunk (Q4, 128 rows)
constexpr int kTmemCols = 512;             // two 256-column fp32 accumulators
constexpr long long kSpin = 2000000000LL;  // about 1 s

// Shared-memory plan: A and B rings of 4 stages, a B stage holding the tile's 256
// columns (32 KB), and the packed-weight ring.
struct Plan {
    static constexpr int kAStages = 4, kBStages = 4;
    static constexpr int kBoxRows = kBN;  // rows of the largest B box
    static constexpr int kBTile = kBoxRows * kBK * 2;
    static constexpr int kTileCache = 96;  // tile descriptors staged per CTA
    static constexpr size_t kSmemA = 0;
    static constexpr size_t kSmemB = kSmemA + (size_t)kAStages * kATile;
    static constexpr size_t kSmemP = kSmemB + (size_t)kBStages * kBTile;
    static constexpr size_t kSmemBytes = kSmemP + (size_t)kPSlots * kPacked;  // 219,136
    static_assert(kSmemB % 1024 == 0 && kSmemP % 16 == 0, "swizzled tiles need 1024-byte alignment");
};

__device__ __forceinline__ unsigned su32(const void *p) { return (unsigned)__cvta_generic_to_shared(p); }

// Byte offset of element (r, k), k < 64, in a K-major tile of 128-byte rows with
// the 128-byte swizzle (16-byte unit index XOR row % 8).
__device__ __forceinline__ unsigned sw128(int r, int k) {
    return (unsigned)(r * 128 + ((((k >> 3) ^ (r & 7)) & 7) << 4) + (k & 7) * 2);
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups 1024
// bytes apart (start address and offsets in 16-byte units; version 1).
__device__ __forceinline__ uint64_t sdesc(unsigned addr) {
    return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor, kind::f16: fp32 accumulator, A and B both fp16 (bf16 when
// `bf16`), both K-major, M = m (128), N = n (multiple of 16, <= 256).
__device__ __forceinline__ uint32_t idesc_f16(int n, bool bf16, int m) {
    const uint32_t ab = bf16 ? 1u : 0u;
    return (1u << 4) | (ab << 7) | (ab << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void mbar_init(uint64_t *m, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(m)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *m) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(m)) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint64_t *m, unsigned parity) {
    unsigned ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(su32(m)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *m, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(m)), "r"(bytes) : "memory");
}
// One box (64 elements x the map's box rows, 128-byte swizzle) of a 2-D tensor map at column
// c0 (a multiple of 64) and row c1.
__device__ __forceinline__ void tma_box(void *dst, const CUtensorMap *map, int c0, int c1, uint64_t *m) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(su32(dst)),
        "l"(map), "r"(c0), "r"(c1), "r"(su32(m))
        : "memory");
}
// One box of a 3-D tensor map at (c0, c1, c2).
__device__ __forceinline__ void tma_box3(void *dst, const CUtensorMap *map, int c0, int c1, int c2, uint64_t *m) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(su32(dst)),
        "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(su32(m))
        : "memory");
}

// Four 8x8 matrices of 16-bit elements, one register of each per lane in the
// mma fragment layout; lane l gives the address of row l % 8 of matrix l / 8.
__device__ __forceinline__ void stmatrix4(void *row_addr, uint32_t r0, uint32_t r1, uint32_t r2, uint32_t r3) {
    asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1, %2, %3, %4};" ::"r"(su32(row_addr)), "r"(r0),
                 "r"(r1), "r"(r2), "r"(r3)
                 : "memory");
}

__device__ __forceinline__ uint32_t lop_or(uint32_t a, uint32_t mask, uint32_t orv) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(mask), "r"(orv));
    return d;
}
__device__ __forceinline__ uint32_t hfma2u(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ uint32_t hmul2u(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// fp16x2 bit patterns
constexpr uint32_t kH1024 = 0x64006400u;     // {1024, 1024}
constexpr uint32_t kHOne = 0x3C003C00u;      // {1, 1}
constexpr uint32_t kHM1032 = 0xE408E408u;    // {-1032, -1032}
constexpr uint32_t kH16th = 0x2C002C00u;     // {1/16, 1/16}
constexpr uint32_t kHM72 = 0xD480D480u;      // {-72, -72}

// Q4 word -> 4 fp16x2 pairs of (q - 8), exactly: pair p holds nibbles (p, low
// half) and (p, high half) of the word (bits 4p and 16 + 4p). A nibble ORed into
// the mantissa of 1024 (fp16 0x6400: 10 mantissa bits, ulp 1) gives 1024 + q, or
// 1024 + 16 q at bits 4..7; the fma removes the offset exactly. Nibbles at bits
// 8..15 would reach the exponent and are shifted down first.
__device__ __forceinline__ void q4_pairs(uint32_t w, uint32_t out[4]) {
    out[0] = hfma2u(lop_or(w, 0x000F000Fu, kH1024), kHOne, kHM1032);
    out[1] = hfma2u(lop_or(w, 0x00F000F0u, kH1024), kH16th, kHM72);
    out[2] = hfma2u(lop_or(w >> 8, 0x000F000Fu, kH1024), kHOne, kHM1032);
    out[3] = hfma2u(lop_or(w >> 12, 0x000F000Fu, kH1024), kHOne, kHM1032);
}

__device__ __forceinline__ int col_row(int cv, int P) { return cv >= 0 ? cv : P + (-cv - 1); }

// The activation of the gate/up epilogue. h is rounded to fp16 right after, so the
// hardware exponential, reciprocal and tanh (errors near 2^-21, 2^-22 and 2^-11
// relative) are used instead of the correctly rounded library forms.
__device__ __forceinline__ float act_fast(int act, float g) {
    if (act == MOE_ACT_GEGLU_TANH) {
        const float k0 = 0.7978845608028654f;  // sqrt(2/pi)
        float t;
        asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(k0 * (g + 0.044715f * g * g * g)));
        return 0.5f * g * (1.0f + t);
    }
    return __fdividef(g, 1.0f + __expf(-g));
}

// The completion of every MMA this thread has issued arrives on `bar`.
__device__ __forceinline__ void commit_to(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(su32(bar))
                 : "memory");
}

// 32 consecutive accumulator columns of this warp's 32 TMEM lanes, waited for.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t v[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
          "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
          "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// One K = 64 stage: four MMAs of K = 16 (descriptor start +2 = +32 bytes per step);
// the first accumulates onto D only when `acc`, the others always.
__device__ __forceinline__ void mma_k64(uint32_t dt, uint64_t da, uint64_t db, uint32_t idesc, bool acc) {
    asm volatile(
        "{ .reg .pred p; setp.ne.b32 p, %4, 0; "
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }" ::"r"(dt),
        "l"(da), "l"(db), "r"(idesc), "r"(acc ? 1u : 0u)
        : "memory");
#pragma unroll
    for (int kk = 1; kk < kBK / 16; ++kk)
        asm volatile("{ .reg .pred p; setp.ne.b32 p, 1, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }" ::"r"(dt),
                     "l"(da + (uint64_t)(2 * kk)), "l"(db + (uint64_t)(2 * kk)), "r"(idesc)
                     : "memory");
}

struct TileInfo {
    Group grp;
    int mt;
    bool shared;
    int nk;  // K stages
};

// Tile t of one launch: t = (group, M-tile), the shared expert's groups first.
__device__ __forceinline__ bool tile_info(const UmmaArgs &a, int n_routed, int t, TileInfo &ti) {
    if (a.mode == 2) {
        // router: tile t = (128 experts mt, kRN tokens nt)
        const int mt = t % a.n_mt, nt = t / a.n_mt;
        ti.grp = Group{-1, kRN * nt, min(kRN, a.T - kRN * nt), 0};
        ti.mt = mt;
        ti.shared = false;
        ti.nk = a.H / kBK;
        return ti.grp.ncols > 0;
    }
    // the shared expert's tiles (all of them full width) first, then the routed
    // groups in the plan's list order (full groups, then partial ones largest first):
    // CTAs take tiles round-robin, so the longest tiles start first
    const int mp = a.n_mt, mps = a.n_mt_s;
    const int ns = a.n_shared * mps;
    int j;
    if (t < ns) {
        ti.grp = a.groups[a.max_routed + t / mps];
        j = t % mps;
        ti.shared = true;
    } else {
        const int t2 = t - ns;
        if (t2 >= n_routed * mp) return false;
        ti.grp = a.groups[t2 / mp];
        j = t2 % mp;
        ti.shared = false;
    }
    ti.mt = j;
    const QLayout &L = ti.shared ? a.src.LS : a.src.L;
    ti.nk = (a.mode == 0 ? L.H : L.F) / kBK;
    return true;
}

__global__ void __launch_bounds__(kThreads, 1) k_umma(const __grid_constant__ UmmaArgs a) {
    using Pl = Plan;
    constexpr int kAS = Pl::kAStages, kBS = Pl::kBStages;
    extern __shared__ uint8_t smem_raw[];
    static_assert(kAS == kBS, "one barrier pair per stage serves both rings");
    __shared__ __align__(8) uint64_t fullA[kAS], emptyA[kAS];
    __shared__ __align__(8) uint64_t accf_bar[2], acce_bar[2];
    __shared__ __align__(8) uint64_t pfull_bar[kPSlots], pempty_bar[kPSlots];
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    __shared__ int epi_rows[kEpiWarps][kBN];        // down epilogue: output row of each column, per warp
    __shared__ TileInfo tiles_s[Pl::kTileCache];  // this CTA's tiles (the first kTileCache of them)
    uint8_t *const sm = reinterpret_cast<uint8_t *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // CTA b takes tiles b, b + G, ...
    const int G = (int)gridDim.x;
    const int wid = (int)blockIdx.x;
    const int n_routed = a.mode == 2 ? 0 : *a.n_groups;
    const int mp = a.n_mt, mps = a.n_mt_s;
    const int n_tiles = a.mode == 2 ? a.n_mt * ((a.T + kRN - 1) / kRN) : n_routed * mp + a.n_shared * mps;
    const int P = a.T * a.K;

    if (tid == 0) {
        for (int s = 0; s < kAS; ++s) {
            // one "full" barrier per stage counts the A and the B side: the B thread's
            // arrival with the stage's bytes, then the dequant group's warps (the
            // router: the A copy's arrival)
            mbar_init(&fullA[s], a.mode == 2 ? 2 : kDqWarps / 2 + 1);
            mbar_init(&emptyA[s], 1);
        }
        for (int s = 0; s < kPSlots; ++s) {
            mbar_init(&pfull_bar[s], 1);
            mbar_init(&pempty_bar[s], kDqWarps);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&accf_bar[b], 1);
            mbar_init(&acce_bar[b], 32 * kEpiWarps);
        }
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // this CTA's tiles: descriptors staged once (one round trip)
    for (int i = tid; i < Pl::kTileCache; i += kThreads) {
        const int t = wid + G * i;
        TileInfo ti;
        if (t < n_tiles && tile_info(a, n_routed, t, ti)) tiles_s[i] = ti;
    }
    if (warp == kMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(&tmem_base)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = tmem_base;

    auto get_tile = [&](int t, TileInfo &ti) -> bool {
        const int i = (t - wid) / G;
        if (i < Pl::kTileCache) {
            ti = tiles_s[i];
            return true;
        }
        return tile_info(a, n_routed, t, ti);
    };

    // bounded wait on a barrier phase; on timeout every role of the CTA stops
    auto wait = [&](uint64_t *m, unsigned parity) -> bool {
        if (mbar_try(m, parity)) return true;
        const long long t0 = clock64();
        while (!mbar_try(m, parity)) {
            if (*(volatile int *)&abort_flag) return false;
            if (clock64() - t0 > kSpin) {
                atomicExch(&abort_flag, 1);
                set_status(a.status, MOE_STATUS_TIMEOUT);
                return false;
            }
        }
        return true;
    };
    // warps that arrive once per warp take their waits' outcome as a warp (a timeout
    // never leaves part of a warp behind at __syncwarp)
    auto wait_warp = [&](uint64_t *m, unsigned parity) -> bool {
        const bool ok = wait(m, parity);
        return __all_sync(0xffffffffu, ok);
    };

    if (warp == kTmaWarp || warp == kTmaBWarp) {
        // ---------------------------------------------------------------- TMA warps
        // warp kTmaWarp: the packed chunk of stages s, s + 1 of each tile (HBM, up to
        // kPSlots chunks ahead); warp kTmaBWarp: the B rows of each stage (L2, up to
        // kBStages ahead) and, for the router, the A rows.
        if (lane == 0) {
            const bool packed = warp == kTmaWarp;
            if (!packed) {
                asm volatile("prefetch.tensormap [%0];" ::"l"(&a.tmap_b) : "memory");
                if (a.mode == 2) asm volatile("prefetch.tensormap [%0];" ::"l"(&a.tmap_a) : "memory");
                else
                    for (int i = 0; i < 4; ++i) asm volatile("prefetch.tensormap [%0];" ::"l"(&a.tmap_bn[i]) : "memory");
            }
            int it = 0, ch = 0;
            int bslot = 0;
            unsigned bphase = 0;
            bool good = !(packed && a.mode == 2);
            for (int t = wid; t < n_tiles && good; t += G) {
                TileInfo ti;
                if (!get_tile(t, ti)) break;
                // B side, per tile: the smallest box holding this CTA's columns of the
                // group (rows past them belong to the next group or read as zeros; the
                // MMA's N stops at round-up(ncols, 16))
                int bi = 4;
                const int r0 = ti.grp.col0;
                if (a.mode != 2) {
                    const int rows = (ti.grp.ncols + 15) & ~15;
                    bi = rows <= 16 ? 0 : rows <= 32 ? 1 : rows <= 64 ? 2 : rows <= 128 ? 3 : 4;
                }
                const CUtensorMap *mb = bi < 4 ? &a.tmap_bn[bi] : &a.tmap_b;
                const int box_rows = a.mode == 2 ? kRN : bi < 4 ? 16 << bi : Pl::kBoxRows;
                const unsigned bbytes = (unsigned)(box_rows * kBK * 2);
                for (int s2 = 0; s2 < ti.nk && good; ++s2, ++it) {
                    if (packed) {
                        if (s2 & 1) continue;
                        const int ps = ch % kPSlots;
                        if (ch >= kPSlots && !wait(&pempty_bar[ps], ((ch / kPSlots) - 1) & 1)) {
                            good = false;
                            break;
                        }
                        // one chunk of the 128-row M-tile: gate/up codes + scales boxes, or
                        // one down box (a half box for a last half chunk)
                        const QLayout &L = ti.shared ? a.src.LS : a.src.L;
                        const CUtensorMap *pk = ti.shared ? &a.pk[2] : &a.pk[0];
                        const int slot = ti.shared ? 0 : ti.grp.slot;
                        const int c = s2 >> 1;
                        uint8_t *dst = sm + Pl::kSmemP + (size_t)ps * kPacked;
                        if (a.mode == 0) {
                            mbar_expect_tx(&pfull_bar[ps], 4u * 2304u);
                            tma_box3(dst, &pk[0], c * 288, 4 * ti.mt, slot, &pfull_bar[ps]);
                            tma_box3(dst + 8192, &pk[1], c * 288 + 256, 4 * ti.mt, slot, &pfull_bar[ps]);
                        } else {
                            const bool half = L.d_half && c == L.d_chunks - 1;
                            mbar_expect_tx(&pfull_bar[ps], half ? 8u * 576u : 8u * 1152u);
                            tma_box3(dst, &pk[half ? 1 : 0], c * 144, 8 * ti.mt, slot, &pfull_bar[ps]);
                        }
                        ++ch;
                    } else {
                        const int bb = bslot;
                        if (it >= kBS && !wait(&emptyA[bb], bphase ^ 1u)) {
                            good = false;
                            break;
                        }
                        uint8_t *dstB = sm + Pl::kSmemB + (size_t)bb * Pl::kBTile;
                        mbar_expect_tx(&fullA[bb], bbytes);
                        tma_box(dstB, mb, s2 * kBK, r0, &fullA[bb]);
                        if (a.mode == 2) {  // the router's A rows, into the same slot
                            mbar_expect_tx(&fullA[bb], (unsigned)(kABoxRows * kBK * 2));
                            tma_box(sm + Pl::kSmemA + (size_t)bb * kATile, &a.tmap_a, s2 * kBK, kBM * ti.mt, &fullA[bb]);
                        }
                        if (++bslot == kBS) {
                            bslot = 0;
                            bphase ^= 1u;
                        }
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp < kDqWarps) {
        // ---------------------------------------------------------------- dequant warps
        // Stage s of a tile dequantises half s & 1 of chunk s / 2 into the A tile; item
        // `it` belongs to group it % 2, and warp w of a group takes one 16-row slice
        // (gate/up tile w / 2, gate if w is even; down tile w). Each warp arrives once
        // per stage.
        const int g = lane >> 2;
        const int grp = warp >> 3, lw = warp & 7;
        // stmatrix row addresses: lane l gives row l % 8 of matrix l / 8 (matrices:
        // rows 0-7 / 8-15 x k 0-7 / 8-15 of a 16 x 16 k-step)
        const int mrow = (lane & 7) + 8 * ((lane >> 3) & 1), mk = 8 * (lane >> 4);
        int it = 0, ch = 0;
        bool good = true;
        for (int t = wid; t < n_tiles && good; t += G) {
            TileInfo ti;
            if (!get_tile(t, ti)) break;
            const QLayout &L = ti.shared ? a.src.LS : a.src.L;
            if (a.mode == 2) break;  // the router has nothing to dequantise
            for (int s2 = 0; s2 < ti.nk; ++s2, ++it) {
                const int b = it % kAS;
                const int ps = ch % kPSlots;
                const bool single = (s2 & 1) == 0 && s2 == ti.nk - 1;  // a chunk of one stage
                const bool chunk_done = (s2 & 1) == 1 || s2 == ti.nk - 1;
                if ((it & 1) != grp) {
                    if (chunk_done) ++ch;
                    continue;
                }
                if (!wait_warp(&pfull_bar[ps], (ch / kPSlots) & 1)) {
                    good = false;
                    break;
                }
                // the A tile of this buffer is free once the MMA of item it - kAStages is done
                if (it >= kAS && !wait_warp(&emptyA[b], ((it / kAS) - 1) & 1)) {
                    good = false;
                    break;
                }
                {
                    const uint8_t *pk = sm + Pl::kSmemP + (size_t)ps * kPacked;
                    uint8_t *sA = sm + Pl::kSmemA + (size_t)b * kATile;
                    const int h = s2 & 1;
                    int row0, off_codes, off_scales;
                    if (a.mode == 0) {
                        // slot: 4 x [gate codes 1024 | up codes 1024], then 4 x [gate scales
                        // 128 | up scales 128]
                        const int j = lw >> 1, jm = lw & 1;
                        row0 = 32 * j + 16 * jm;
                        off_codes = j * 2048 + jm * 1024 + h * 512;
                        off_scales = 8192 + j * 256 + jm * 128 + h * 64;
                    } else {
                        // slot: 8 x [codes 1024 | scales 128] (a half chunk: 8 x [512 | 64])
                        const bool half = L.d_half && (s2 >> 1) == L.d_chunks - 1;
                        row0 = 16 * lw;
                        off_codes = lw * (half ? 576 : 1152) + h * 512;
                        off_scales = lw * (half ? 576 : 1152) + (half ? 512 : 1024) + h * 64;
                    }
                    const uint4 wv = *reinterpret_cast<const uint4 *>(pk + off_codes + 16 * lane);
                    const uint32_t words[4] = {wv.x, wv.y, wv.z, wv.w};
                    // scales of rows g (low half) and g + 8 (high half) for the stage's blocks
                    const uint32_t s0 = *reinterpret_cast<const uint32_t *>(pk + off_scales + 4 * g);
                    const uint32_t s1 = *reinterpret_cast<const uint32_t *>(pk + off_scales + 4 * (8 + g));
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint32_t sw = i < 2 ? s0 : s1;  // block i / 2
                        const uint32_t d_lo = (sw & 0xFFFFu) * 0x10001u, d_hi = (sw >> 16) * 0x10001u;
                        uint32_t q[4];
                        q4_pairs(words[i], q);
                        // q[p] is fragment register p of k-step i: rows g (+8 for odd p),
                        // k = 16 i + 2c (+8 for p >= 2)
                        stmatrix4(sA + sw128(row0 + mrow, 16 * i + mk), hmul2u(q[0], d_lo), hmul2u(q[1], d_hi),
                                  hmul2u(q[2], d_lo), hmul2u(q[3], d_hi));
                    }
                    // generic-proxy writes -> visible to the tensor cores' async proxy
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                }
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&fullA[b]);
                    mbar_arrive(&pempty_bar[ps]);
                    if (single) mbar_arrive(&pempty_bar[ps]);
                }
                if (chunk_done) ++ch;
            }
        }
    } else if (warp == kMmaWarp) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            // The issue loop is on the critical path of every stage (a stage of a narrow
            // group runs in ~180 cycles): ring position as a running slot and phase,
            // descriptors as offsets from per-ring bases.
            const uint64_t dA0 = sdesc(su32(sm + Pl::kSmemA)), dB0 = sdesc(su32(sm + Pl::kSmemB));
            int slot = 0, ti_local = 0, last_slot = -1;
            unsigned phase = 0, last_phase = 0;
            bool good = true;
            for (int t = wid; t < n_tiles && good; t += G, ++ti_local) {
                TileInfo ti;
                if (!get_tile(t, ti)) break;
                const int ab = ti_local & 1;
                if (ti_local >= 2 && !wait(&acce_bar[ab], ((ti_local >> 1) - 1) & 1)) break;
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const int n = (ti.grp.ncols + 15) & ~15;
                const uint32_t idesc = idesc_f16(n, a.mode == 2, kBM);
                const uint32_t dt = tmem + (uint32_t)(256 * ab);
                for (int s = 0; s < ti.nk; ++s) {
                    if (!wait(&fullA[slot], phase)) {
                        good = false;
                        break;
                    }
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                    // descriptor start addresses count 16-byte units; a K step of 16 is 32 bytes
                    const uint64_t da = dA0 + (uint64_t)(slot * (kATile >> 4));
                    const uint64_t db = dB0 + (uint64_t)(slot * (Pl::kBTile >> 4));
                    mma_k64(dt, da, db, idesc, s > 0);
                    // one commit frees the stage's A and B slots (both rings have the
                    // same depth: the B producer waits on the A ring's empty barrier)
                    commit_to(&emptyA[slot]);
                    last_slot = slot;
                    last_phase = phase;
                    if (++slot == kAS) {
                        slot = 0;
                        phase ^= 1u;
                    }
                }
                if (!good) break;
                commit_to(&accf_bar[ab]);
            }
            // every MMA this thread issued has completed before TMEM can be released
            if (last_slot >= 0) {
                const long long t0 = clock64();
                while (!mbar_try(&emptyA[last_slot], last_phase) && clock64() - t0 < kSpin) {
                }
            }
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------------- epilogue
        const int q = warp & 3;  // TMEM lanes 32q .. 32q + 31
        int ti_local = 0;
        for (int t = wid; t < n_tiles; t += G, ++ti_local) {
            TileInfo ti;
            if (!get_tile(t, ti)) break;
            const int ab = ti_local & 1;
            const int ncols = ti.grp.ncols;
            const QLayout &L = ti.shared ? a.src.LS : a.src.L;
            int *rows = epi_rows[q];
            // the down tile's output rows, loaded while its MMAs run
            if (a.mode == 1) {
                for (int j = lane; j < ncols; j += 32) rows[j] = col_row(a.cols[ti.grp.col0 + j], P);
                __syncwarp();
            }
            if (!wait_warp(&accf_bar[ab], (ti_local >> 1) & 1)) break;
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            if (a.mode == 2) {
                // logits[t][e] = acc + bias[e]: lane holds expert 128 mt + 32 q + lane
                const int e = kBM * ti.mt + 32 * q + lane;
                const float be = (a.bias && e < a.E) ? a.bias[e] : 0.f;
                for (int c0 = 0; c0 < ncols; c0 += 32) {
                    uint32_t v[32];
                    tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(256 * ab + c0), v);
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (c0 + j < ncols && e < a.E)
                            a.logits[(size_t)(ti.grp.col0 + c0 + j) * a.E + e] = __uint_as_float(v[j]) + be;
                }
                asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
                mbar_arrive(&acce_bar[ab]);
                continue;
            }
            for (int c0 = 0; c0 < ncols; c0 += 32) {
                uint32_t v[32];
                tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(256 * ab + c0), v);
                if (a.mode == 0) {
                    // lanes 0..15: gate rows, 16..31: up rows of f = 64 mt + 16 q + lane % 16;
                    // lane < 16 forms h for token j, lane >= 16 for token j + 1
                    const int f = 64 * ti.mt + 16 * q + (lane & 15);
                    const bool lo = lane < 16;
#pragma unroll
                    for (int j = 0; j < 32; j += 2) {
                        const float x0 = __uint_as_float(v[j]), x1 = __uint_as_float(v[j + 1]);
                        const float got = __shfl_xor_sync(0xffffffffu, lo ? x1 : x0, 16);
                        const float gate = lo ? x0 : got, up = lo ? got : x1;
                        const int col = c0 + j + (lo ? 0 : 1);
                        if (col < ncols) {
                            const float hv = act_fast(a.act, gate) * up;
                            a.h16[(size_t)(ti.grp.col0 + col) * a.h16_ld + f] = __float2half_rn(hv);
                        }
                    }
                } else {
                    const int hrow = 128 * ti.mt + 32 * q + lane;
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int col = c0 + j;
                        if (col < ncols) a.yp[(size_t)rows[col] * L.H + hrow] = __uint_as_float(v[j]);
                    }
                }
            }
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            mbar_arrive(&acce_bar[ab]);
            __syncwarp();  // the row cache is rewritten for the next tile
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == kMmaWarp) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                     : "memory");
    }
}

// x (bf16 or fp32) -> fp16 rows in plan-column order: one CTA per row; a thread's
// loads of the row (up to kGatherUnits 16-byte output units) are all in flight
// before it converts and stores.
constexpr int kGatherUnits = 4;
__global__ void __launch_bounds__(128) k_gather_f16(const int32_t *__restrict__ cols, const int32_t *__restrict__ n_cols,
                                                    const void *__restrict__ x, int xf32, int K, int H,
                                                    __half *__restrict__ out) {
    const int row = blockIdx.x;
    if (row >= *n_cols) return;
    const int cv = cols[row];
    const int t = cv >= 0 ? cv / K : -cv - 1;
    const int V = H / 8;
    for (int v0 = 0; v0 < V; v0 += kGatherUnits * blockDim.x) {
        float4 a[kGatherUnits][2];
#pragma unroll
        for (int u = 0; u < kGatherUnits; ++u) {
            const int v = v0 + u * blockDim.x + threadIdx.x;
            if (v >= V) continue;
            if (xf32) {
                const float4 *p = reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(x) + (size_t)t * H + 8 * v);
                a[u][0] = p[0];
                a[u][1] = p[1];
            } else {
                const uint4 w =
                    *reinterpret_cast<const uint4 *>(reinterpret_cast<const __nv_bfloat16 *>(x) + (size_t)t * H + 8 * v);
                a[u][0] = make_float4(__uint_as_float(w.x), __uint_as_float(w.y), __uint_as_float(w.z),
                                      __uint_as_float(w.w));
            }
        }
#pragma unroll
        for (int u = 0; u < kGatherUnits; ++u) {
            const int v = v0 + u * blockDim.x + threadIdx.x;
            if (v >= V) continue;
            float f[8];
            if (xf32) {
                f[0] = a[u][0].x; f[1] = a[u][0].y; f[2] = a[u][0].z; f[3] = a[u][0].w;
                f[4] = a[u][1].x; f[5] = a[u][1].y; f[6] = a[u][1].z; f[7] = a[u][1].w;
            } else {
                // bf16 pairs carried as raw words: low half, then high half
                const uint32_t ww[4] = {__float_as_uint(a[u][0].x), __float_as_uint(a[u][0].y),
                                        __float_as_uint(a[u][0].z), __float_as_uint(a[u][0].w)};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    f[2 * j] = __uint_as_float(ww[j] << 16);
                    f[2 * j + 1] = __uint_as_float(ww[j] & 0xFFFF0000u);
                }
            }
            __align__(16) __half o[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) o[j] = __float2half_rn(f[j]);
            __stcs(reinterpret_cast<uint4 *>(out + (size_t)row * H + 8 * v), *reinterpret_cast<const uint4 *>(o));
        }
    }
}

}  // namespace

bool umma_supported(const QLayout &L) { return L.kind == MOE_Q4_32 && L.H % 128 == 0 && L.F % 64 == 0; }

bool umma_router_supported(int H) { return H % kBK == 0; }

int launch_umma(const UmmaArgs &a, int n_ctas, cudaStream_t s) {
    k_umma<<<n_ctas, kThreads, Plan::kSmemBytes + 1024, s>>>(a);
    MOE_CUDA_TRY(cudaGetLastError());
    return MOE_OK;
}

int launch_gather_f16(const int32_t *cols, const int32_t *n_cols, const void *x, int xf32, int K, int H, int max_rows,
                      __half *out, cudaStream_t s) {
    if (max_rows == 0) return MOE_OK;
    k_gather_f16<<<(unsigned)max_rows, 128, 0, s>>>(cols, n_cols, x, xf32, K, H, out);
    MOE_CUDA_TRY(cudaGetLastError());
    return MOE_OK;
}

int make_tmap_2d(CUtensorMap *map, const void *base, bool bf16, unsigned long long rows, unsigned long long cols,
                 unsigned long long row_stride_bytes, int box_rows) {
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    if (!encode) {
        cudaDriverEntryPointQueryResult q;
        void *fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn)
            return set_error(MOE_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
        encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    if ((uintptr_t)base % 16 || row_stride_bytes % 16)
        return set_error(MOE_ERR_ARG, "tensor map base / row stride not 16-byte aligned");
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {row_stride_bytes};
    if (box_rows <= 0) box_rows = kBN;
    const cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = encode(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                              const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return set_error(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return MOE_OK;
}

int make_packed_maps(CUtensorMap maps[2], int mode, const QLayout &L, const uint8_t *base, long long slot_stride,
                     int n_slots) {
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    if (!encode) {
        cudaDriverEntryPointQueryResult q;
        void *fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn)
            return set_error(MOE_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
        encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    const uint8_t *b0 = mode == 0 ? base : base + L.d_offset;
    const long long tile_bytes = mode == 0 ? L.gu_tile_bytes : L.d_tile_bytes;
    const int tiles = mode == 0 ? L.gu_tiles : L.d_tiles;
    if ((uintptr_t)b0 % 16 || tile_bytes % 16 || slot_stride % 16)
        return set_error(MOE_ERR_ARG, "packed weights not 16-byte aligned");
    const cuuint64_t dims[3] = {(cuuint64_t)(tile_bytes / 8), (cuuint64_t)tiles, (cuuint64_t)(n_slots > 0 ? n_slots : 1)};
    const cuuint64_t strides[2] = {(cuuint64_t)tile_bytes, (cuuint64_t)(slot_stride > 0 ? slot_stride : tile_bytes * tiles)};
    const cuuint32_t estr[3] = {1, 1, 1};
    for (int m = 0; m < 2; ++m) {
        cuuint32_t box[3];
        if (mode == 0) {
            box[0] = m == 0 ? 256 : 32;  // 2,048 bytes of codes, 256 bytes of scales
            box[1] = 4;
        } else {
            box[0] = m == 0 ? 144 : 72;  // a whole chunk, a half chunk
            box[1] = 8;
        }
        box[2] = 1;
        const CUresult r = encode(&maps[m], CU_TENSOR_MAP_DATA_TYPE_UINT64, 3, const_cast<uint8_t *>(b0), dims,
                                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return set_error(MOE_ERR_CUDA, "cuTensorMapEncodeTiled (packed) failed (%d)", (int)r);
    }
    return MOE_OK;
}

int init_umma_attributes(int max_smem) {
    // a kernel whose shared memory does not fit is never launched (umma_fits says so)
    return umma_fits(max_smem) ? set_max_dynamic_smem((const void *)k_umma, max_smem) : MOE_OK;
}

bool umma_fits(int max_smem) {
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, (const void *)k_umma) != cudaSuccess) return false;
    const size_t dyn = Plan::kSmemBytes + 1024;
    return dyn + fa.sharedSizeBytes <= (size_t)max_smem;
}

}  // namespace moe
