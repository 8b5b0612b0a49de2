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
//   A  128 rows of Q4 weights, dequantised by 4 producer warps from the packed
//      layout (codes + per-32 fp16 scales, copied in with cp.async) into fp16
//      w = fp16(d * (q - 8)) (one rounding; q - 8 is exact), stored K-major with
//      the 128-byte swizzle the MMA descriptor names;
//   B  the group's token rows, 64 fp16 each per stage, gathered with cp.async
//      (gate/up: rows of x converted to fp16; down: rows of h in plan order);
//   MMA one thread issues 4 x tcgen05.mma (K = 16 each) per stage and commits to
//      the stage's "empty" barrier; after the last stage it commits the tile to an
//      "accumulator full" barrier; two accumulators of 256 TMEM columns alternate;
//   epilogue 4 warps read the accumulator with tcgen05.ld (warp q: TMEM lanes
//      32q..32q+31). Gate/up tiles hold rows [gate 16 | up 16] x 4, so a warp pairs
//      gate and up of the same row with one shuffle, applies the activation and
//      writes h as fp16 (row = plan column); down tiles write fp32 y_pair rows.
//
// A tile is (column group of <= 256 live pairs of one expert, 128-row M-tile);
// CTAs (one per SM) take tiles round-robin. Every barrier wait gives up after
// about a second (MOE_STATUS_TIMEOUT) and the CTA stops; the TMEM it allocated is
// released on every path.
#include "decode_common.cuh"
#include "prefill_gemm.cuh"

namespace moe {

namespace {

constexpr int kBM = 128, kBN = 256, kBK = 64, kStages = 4;  // A/B ring of MMA stages
constexpr int kPStages = 6, kPLead = 4, kBLead = 2;          // packed-weight ring; load lead (items)
constexpr int kProdWarps = 8, kMmaWarp = 8, kEpiWarps = 4;
constexpr int kThreads = 32 * (kProdWarps + 1 + kEpiWarps);  // 416
constexpr int kProdThreads = 32 * kProdWarps;
constexpr int kATile = kBM * kBK * 2;      // 16 KB
constexpr int kBTile = kBN * kBK * 2;      // 32 KB
constexpr int kPacked = 4608;              // packed codes + scales of one stage (Q4, 128 rows x 64)
constexpr int kTmemCols = 512;             // two 256-column fp32 accumulators
constexpr long long kSpin = 2000000000LL;  // about 1 s

constexpr size_t kSmemA = 0;
constexpr size_t kSmemB = kSmemA + (size_t)kStages * kATile;
constexpr size_t kSmemP = kSmemB + (size_t)kStages * kBTile;
constexpr size_t kSmemBytes = kSmemP + (size_t)kPStages * kPacked;  // 224,256
static_assert(kSmemB % 1024 == 0 && kSmemP % 16 == 0, "swizzled tiles need 1024-byte alignment");

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
// `bf16`), both K-major, M = 128, N = n (multiple of 16, <= 256).
__device__ __forceinline__ uint32_t idesc_f16(int n, bool bf16) {
    const uint32_t ab = bf16 ? 1u : 0u;
    return (1u << 4) | (ab << 7) | (ab << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(kBM >> 4) << 24);
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

__device__ __forceinline__ void cp16(void *dst, const void *src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(su32(dst)), "l"(src), "r"(valid ? 16 : 0)
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
__device__ __forceinline__ int col_token(int cv, int K) { return cv >= 0 ? cv / K : -cv - 1; }

struct TileInfo {
    Group grp;
    int mt;
    bool shared;
    int nk;  // K stages
};

__device__ __forceinline__ bool tile_info(const UmmaArgs &a, int n_routed, int t, TileInfo &ti) {
    if (a.mode == 2) {
        // router: tile t = (128 experts mt, 256 tokens nt)
        const int mt = t % a.n_mt, nt = t / a.n_mt;
        ti.grp = Group{-1, kBN * nt, min(kBN, a.T - kBN * nt), 0};
        ti.mt = mt;
        ti.shared = false;
        ti.nk = a.H / kBK;
        return ti.grp.ncols > 0;
    }
    const int nr = n_routed * a.n_mt;
    if (t < nr) {
        ti.grp = a.groups[t / a.n_mt];
        ti.mt = t % a.n_mt;
        ti.shared = false;
    } else {
        const int t2 = t - nr;
        if (t2 >= a.n_shared * a.n_mt_s) return false;
        ti.grp = a.groups[a.max_routed + t2 / a.n_mt_s];
        ti.mt = t2 % a.n_mt_s;
        ti.shared = true;
    }
    const QLayout &L = ti.shared ? a.src.LS : a.src.L;
    ti.nk = (a.mode == 0 ? L.H : L.F) / kBK;
    return true;
}

// Where the packed bytes of stage s of tile ti come from: piece i (16 bytes, 0..287)
// of the 4,608-byte stage image.
__device__ __forceinline__ const uint8_t *packed_src(const UmmaArgs &a, const TileInfo &ti, const uint8_t *wbase,
                                                     int s, int i) {
    const QLayout &L = ti.shared ? a.src.LS : a.src.L;
    const int c = s >> 1, h = s & 1;
    if (a.mode == 0) {
        // 4 gate/up row tiles x [gate codes 512 | up codes 512 | gate scales 64 | up scales 64]
        const int j = i / 72, pp = i % 72;
        const uint8_t *ch = wbase + (long long)(4 * ti.mt + j) * L.gu_tile_bytes + (long long)c * L.gu_chunk_bytes;
        if (pp < 32) return ch + h * 512 + 16 * pp;
        if (pp < 64) return ch + L.cb + h * 512 + 16 * (pp - 32);
        if (pp < 68) return ch + 2 * L.cb + h * 64 + 16 * (pp - 64);
        return ch + 2 * L.cb + L.sb + h * 64 + 16 * (pp - 68);
    }
    // down: 8 row tiles x [codes 512 | scales 64]; the last chunk of a row may be half
    const int j = i / 36, pp = i % 36;
    const uint8_t *ch = wbase + L.d_offset + (long long)(8 * ti.mt + j) * L.d_tile_bytes + (long long)c * L.d_chunk_bytes;
    const bool half_chunk = L.d_half && c == L.d_chunks - 1;
    if (pp < 32) return ch + h * 512 + 16 * pp;
    return ch + (half_chunk ? L.cb / 2 : L.cb) + h * 64 + 16 * (pp - 32);
}

__global__ void __launch_bounds__(kThreads, 1) k_umma(const __grid_constant__ UmmaArgs a) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kStages], empty_bar[kStages], accf_bar[2], acce_bar[2];
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    __shared__ int epi_rows[kEpiWarps][kBN];  // down epilogue: output row of each column, per warp
    uint8_t *const sm = reinterpret_cast<uint8_t *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = gridDim.x;
    const int n_routed = a.mode == 2 ? 0 : *a.n_groups;
    const int n_tiles = a.mode == 2 ? a.n_mt * ((a.T + kBN - 1) / kBN) : n_routed * a.n_mt + a.n_shared * a.n_mt_s;
    const int P = a.T * a.K;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full_bar[s], kProdThreads);
            mbar_init(&empty_bar[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&accf_bar[b], 1);
            mbar_init(&acce_bar[b], 32 * kEpiWarps);
        }
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
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

    if (warp < kProdWarps) {
        // ---------------------------------------------------------------- producers
        // Items are the (tile, stage) pairs of this CTA in order. Iteration `it` requests
        // the packed weights of item it + kPLead and the B rows of item it + kBLead (one
        // commit group each, empty groups past the end), then dequantises item it.
        struct Cursor {
            int t, s, nk;
            TileInfo ti;
            bool ok;
        };
        auto first = [&](Cursor &cu) {
            cu.t = blockIdx.x;
            cu.s = 0;
            cu.ok = cu.t < n_tiles && tile_info(a, n_routed, cu.t, cu.ti);
            cu.nk = cu.ok ? cu.ti.nk : 0;
        };
        auto next = [&](Cursor &cu) {
            if (++cu.s < cu.nk) return;
            cu.t += G;
            cu.s = 0;
            cu.ok = cu.t < n_tiles && tile_info(a, n_routed, cu.t, cu.ti);
            cu.nk = cu.ok ? cu.ti.nk : 0;
        };
        auto wbase_of = [&](const TileInfo &ti) -> const uint8_t * {
            return ti.shared ? a.src.shared : a.src.arena_base + (long long)ti.grp.slot * a.src.slot_stride;
        };
        Cursor cpk, cb, cd;
        first(cpk);
        first(cb);
        first(cd);
        int ip = 0, ib = 0;
        const int pc = tid & 7;          // 16-byte piece of a 128-byte B row
        int brow[kBN / 32];              // element offsets of this thread's B rows (-1: zero)
        int brow_tile = -1;
        const uint16_t *bsrc = a.mode == 0   ? reinterpret_cast<const uint16_t *>(a.x16)
                               : a.mode == 1 ? reinterpret_cast<const uint16_t *>(a.h16)
                                             : reinterpret_cast<const uint16_t *>(a.xb);
        auto issue_packed = [&]() {
            if (cpk.ok && a.mode != 2) {
                uint8_t *pk = sm + kSmemP + (size_t)(ip % kPStages) * kPacked;
                const uint8_t *wb = wbase_of(cpk.ti);
                for (int i = tid; i < kPacked / 16; i += kProdThreads)
                    cp16(pk + 16 * i, packed_src(a, cpk.ti, wb, cpk.s, i), true);
                next(cpk);
            }
            asm volatile("cp.async.commit_group;" ::: "memory");
            ++ip;
        };
        auto issue_b = [&]() -> bool {
            if (cb.ok) {
                const int b = ib % kStages;
                if (ib >= kStages && !wait(&empty_bar[b], ((ib / kStages) - 1) & 1)) return false;
                if (cb.t != brow_tile) {
                    const TileInfo &ti = cb.ti;
                    const QLayout &L = ti.shared ? a.src.LS : a.src.L;
#pragma unroll
                    for (int r = 0; r < kBN / 32; ++r) {
                        const int n = (tid >> 3) + 32 * r;
                        int off = -1;
                        if (n < ti.grp.ncols)
                            off = a.mode == 0   ? col_token(a.cols[ti.grp.col0 + n], a.K) * L.H
                                  : a.mode == 1 ? (ti.grp.col0 + n) * a.h16_ld
                                                : (ti.grp.col0 + n) * a.H;
                        brow[r] = off;
                    }
                    brow_tile = cb.t;
                }
                uint8_t *sB = sm + kSmemB + (size_t)b * kBTile;
#pragma unroll
                for (int r = 0; r < kBN / 32; ++r) {
                    const int n = (tid >> 3) + 32 * r;
                    const int off = brow[r];
                    cp16(sB + sw128(n, 8 * pc), bsrc + (off < 0 ? 0 : off) + cb.s * kBK + 8 * pc, off >= 0);
                }
                if (a.mode == 2) {
                    // router rows 128 mt .. + 127 (A), copied as they are (bf16)
                    uint8_t *sA = sm + kSmemA + (size_t)b * kATile;
#pragma unroll
                    for (int r = 0; r < kBM / 32; ++r) {
                        const int n = (tid >> 3) + 32 * r, e = kBM * cb.ti.mt + n;
                        const bool valid = e < a.E;
                        cp16(sA + sw128(n, 8 * pc), a.wr + (size_t)(valid ? e : 0) * a.H + cb.s * kBK + 8 * pc, valid);
                    }
                }
                next(cb);
            }
            asm volatile("cp.async.commit_group;" ::: "memory");
            ++ib;
            return true;
        };
        bool good = true;
        // prologue: the groups of iterations -kPLead .. -1
        for (int j = -kPLead; j < 0 && good; ++j) {
            issue_packed();
            if (j + kBLead >= 0) good = issue_b();
            else asm volatile("cp.async.commit_group;" ::: "memory");
        }
        for (int it = 0; cd.ok && good; ++it) {
            issue_packed();
            if (!issue_b()) break;
            // B rows of item `it` were the second group of iteration it - kBLead (its
            // packed weights are older): they have landed once at most the 2 * kBLead
            // newer groups are pending; every producer thread reads packed bytes that
            // others copied, so all of them wait
            asm volatile("cp.async.wait_group %0;" ::"n"(2 * kBLead) : "memory");
            asm volatile("bar.sync 1, %0;" ::"n"(kProdThreads) : "memory");
            const int b = it % kStages;
            if (a.mode == 2) {  // nothing to dequantise
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                mbar_arrive(&full_bar[b]);
                next(cd);
                continue;
            }
            const uint8_t *pk = sm + kSmemP + (size_t)(it % kPStages) * kPacked;
            uint8_t *sA = sm + kSmemA + (size_t)b * kATile;
            const int g = lane >> 2, c = lane & 3;
            // warp w dequantises one 16-row slice: gate/up tile w/2 (gate if w even, up if
            // odd), or down tile w
            int row0, off_codes, off_scales;
            if (a.mode == 0) {
                const int j = warp >> 1, jm = warp & 1;
                row0 = 32 * j + 16 * jm;
                off_codes = j * 1152 + jm * 512;
                off_scales = j * 1152 + 1024 + jm * 64;
            } else {
                row0 = 16 * warp;
                off_codes = warp * 576;
                off_scales = warp * 576 + 512;
            }
            const uint4 wv = *reinterpret_cast<const uint4 *>(pk + off_codes + 16 * lane);
            const uint32_t words[4] = {wv.x, wv.y, wv.z, wv.w};
            // scales of rows g (low half) and g + 8 (high half) for the stage's two blocks
            const uint32_t s0 = *reinterpret_cast<const uint32_t *>(pk + off_scales + 4 * g);
            const uint32_t s1 = *reinterpret_cast<const uint32_t *>(pk + off_scales + 4 * (8 + g));
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t sw = i < 2 ? s0 : s1;  // block i / 2
                const uint32_t d_lo = (sw & 0xFFFFu) * 0x10001u, d_hi = (sw >> 16) * 0x10001u;
                uint32_t q[4];
                q4_pairs(words[i], q);
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    // nibble pair p: row g + 8 (p & 1), k = 16 i + 2 c + 8 (p >> 1) (+1)
                    const int r = row0 + g + 8 * (p & 1);
                    const int k = 16 * i + 2 * c + 8 * (p >> 1);
                    *reinterpret_cast<uint32_t *>(sA + sw128(r, k)) = hmul2u(q[p], (p & 1) ? d_hi : d_lo);
                }
            }
            // the generic-proxy writes (dequantised A, cp.async B) become visible to the
            // tensor cores' async proxy before the stage is marked full
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            mbar_arrive(&full_bar[b]);
            next(cd);
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
    } else if (warp == kMmaWarp) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            int it = 0, ti_local = 0;
            bool good = true;
            int last_b = -1;
            unsigned last_par = 0;
            for (int t = blockIdx.x; t < n_tiles && good; t += G, ++ti_local) {
                TileInfo ti;
                if (!tile_info(a, n_routed, t, ti)) break;
                const int ab = ti_local & 1;
                if (ti_local >= 2 && !wait(&acce_bar[ab], ((ti_local >> 1) - 1) & 1)) break;
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const int n = (ti.grp.ncols + 15) & ~15;
                const uint32_t idesc = idesc_f16(n, a.mode == 2);
                const uint32_t dt = tmem + (uint32_t)(256 * ab);
                for (int s = 0; s < ti.nk; ++s, ++it) {
                    const int b = it % kStages;
                    if (!wait(&full_bar[b], (it / kStages) & 1)) {
                        good = false;
                        break;
                    }
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                    const unsigned aa = su32(sm + kSmemA + (size_t)b * kATile);
                    const unsigned bb = su32(sm + kSmemB + (size_t)b * kBTile);
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk) {
                        const uint64_t da = sdesc(aa + 32 * kk), db = sdesc(bb + 32 * kk);
                        const uint32_t acc = (s > 0 || kk > 0) ? 1u : 0u;
                        asm volatile(
                            "{ .reg .pred p; setp.ne.b32 p, %4, 0; "
                            "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }" ::"r"(dt),
                            "l"(da), "l"(db), "r"(idesc), "r"(acc)
                            : "memory");
                    }
                    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                                     su32(&empty_bar[b]))
                                 : "memory");
                    last_b = b;
                    last_par = (unsigned)(it / kStages) & 1u;
                }
                if (!good) break;
                asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                                 su32(&accf_bar[ab]))
                             : "memory");
            }
            // every MMA this thread issued has completed before TMEM can be released
            if (last_b >= 0) {
                const long long t0 = clock64();
                while (!mbar_try(&empty_bar[last_b], last_par) && clock64() - t0 < kSpin) {
                }
            }
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------------- epilogue
        const int q = warp & 3;  // TMEM lanes 32q .. 32q + 31
        int ti_local = 0;
        for (int t = blockIdx.x; t < n_tiles; t += G, ++ti_local) {
            TileInfo ti;
            if (!tile_info(a, n_routed, t, ti)) break;
            const int ab = ti_local & 1;
            if (!wait(&accf_bar[ab], (ti_local >> 1) & 1)) break;
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const int ncols = ti.grp.ncols;
            const QLayout &L = ti.shared ? a.src.LS : a.src.L;
            int *rows = epi_rows[q];
            if (a.mode == 2) {
                // logits[t][e] = acc + bias[e]: lane holds expert 128 mt + 32 q + lane
                const int e = kBM * ti.mt + 32 * q + lane;
                const float be = (a.bias && e < a.E) ? a.bias[e] : 0.f;
                for (int c0 = 0; c0 < ncols; c0 += 32) {
                    uint32_t v[32];
                    const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(256 * ab + c0);
                    asm volatile(
                        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
                        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
                          "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
                          "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]),
                          "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]),
                          "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
                        : "r"(taddr));
                    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (c0 + j < ncols && e < a.E)
                            a.logits[(size_t)(ti.grp.col0 + c0 + j) * a.E + e] = __uint_as_float(v[j]) + be;
                }
                asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
                mbar_arrive(&acce_bar[ab]);
                continue;
            }
            if (a.mode == 1) {
                for (int j = lane; j < ncols; j += 32) rows[j] = col_row(a.cols[ti.grp.col0 + j], P);
                __syncwarp();
            }
            for (int c0 = 0; c0 < ncols; c0 += 32) {
                uint32_t v[32];
                const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(256 * ab + c0);
                asm volatile(
                    "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                    "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
                    : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
                      "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
                      "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]),
                      "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]),
                      "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
                    : "r"(taddr));
                asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
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
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
}

// x (bf16 or fp32) -> fp16 rows
__global__ void k_to_f16(const void *x, int xf32, size_t n, __half *out) {
    const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const float v = xf32 ? reinterpret_cast<const float *>(x)[i]
                         : __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(x)[i]);
    out[i] = __float2half_rn(v);
}

}  // namespace

bool umma_supported(const QLayout &L) { return L.kind == MOE_Q4_32 && L.H % 128 == 0 && L.F % 64 == 0; }

bool umma_router_supported(int H) { return H % kBK == 0; }

int launch_umma(const UmmaArgs &a, int n_ctas, cudaStream_t s) {
    k_umma<<<n_ctas, kThreads, kSmemBytes + 1024, s>>>(a);
    MOE_CUDA_TRY(cudaGetLastError());
    return MOE_OK;
}

int launch_to_f16(const void *x, int xf32, size_t n, __half *out, cudaStream_t s) {
    if (n == 0) return MOE_OK;
    k_to_f16<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(x, xf32, n, out);
    MOE_CUDA_TRY(cudaGetLastError());
    return MOE_OK;
}

int init_umma_attributes(int max_smem) {
    if ((size_t)max_smem < kSmemBytes + 1024 + 256) return MOE_OK;  // too little shared memory: never launched
    return set_max_dynamic_smem((const void *)k_umma, max_smem);
}

size_t umma_smem_bytes() { return kSmemBytes + 1024; }

}  // namespace moe
