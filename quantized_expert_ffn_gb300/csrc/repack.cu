// repack.cu -- canonical expert blob -> device layout (see moe_internal.cuh).
//
// Canonical blob: gate [F][H], up [F][H], down [H][F]; each row a run of 18-byte
// blocks (fp16 scale, then 16 code bytes) along the reduction index. One CTA
// rewrites one 16-row tile: it stages the tile's canonical rows in shared
// memory, then every thread assembles 32-bit words of the device tile.
#include "moe_internal.cuh"

namespace moe {

namespace {

// code of weight n (0-based within its block) from a block's 16 code bytes
__device__ __forceinline__ uint32_t canon_code(int kind, const uint8_t *codes, int n) {
    if (kind == MOE_Q2_64) return (codes[n >> 2] >> (2 * (n & 3))) & 3u;
    return (codes[n >> 1] >> (4 * (n & 1))) & 15u;
}

// Staged rows: srows[m][row][block*18 .. ] for matrix m of the tile.
struct Staged {
    const uint8_t *base;  // shared memory
    int row_bytes;        // bytes of one canonical row (n_blocks * 18)
    int rows;             // 16
};

__device__ __forceinline__ const uint8_t *staged_block(const Staged &s, int m, int row, int blk) {
    return s.base + ((size_t)m * s.rows + row) * s.row_bytes + (size_t)blk * kBlockBytes;
}

// One 32-bit word of the codes of matrix m for chunk `chunk` (k0 = 128*chunk),
// lane-local word index i, lane l.
__device__ uint32_t code_word(const QLayout &L, const Staged &s, int m, int k0, int lane, int i) {
    const int g = lane >> 2, c = lane & 3;
    uint32_t w = 0;
    if (L.kind == MOE_Q2_64) {
        for (int p = 0; p < 8; ++p)
            for (int hb = 0; hb < 2; ++hb) {
                const int kstep = 2 * i + (p >> 2), a = p & 3;
                const int row = g + 8 * (a & 1);
                const int k = k0 + 16 * kstep + 2 * c + hb + 8 * (a >> 1);
                const uint8_t *blk = staged_block(s, m, row, k / 64);
                w |= canon_code(L.kind, blk + 2, k % 64) << (16 * hb + 2 * p);
            }
    } else {
        for (int p = 0; p < 4; ++p)
            for (int hb = 0; hb < 2; ++hb) {
                const int kstep = i, a = p;
                const int row = g + 8 * (a & 1);
                const int k = k0 + 16 * kstep + 2 * c + hb + 8 * (a >> 1);
                const uint8_t *blk = staged_block(s, m, row, k / 32);
                w |= canon_code(L.kind, blk + 2, k % 32) << (16 * hb + 4 * p);
            }
    }
    return w;
}

// Scale word wi of matrix m's scale part in the chunk starting at block b0.
__device__ uint32_t scale_word(const Staged &s, int m, int b0, int wi) {
    const int b = wi / 8, g = wi % 8;
    const uint8_t *lo = staged_block(s, m, g, b0 + b);
    const uint8_t *hi = staged_block(s, m, g + 8, b0 + b);
    return (uint32_t)lo[0] | ((uint32_t)lo[1] << 8) | ((uint32_t)hi[0] << 16) | ((uint32_t)hi[1] << 24);
}

// Word at byte offset `o` of a matrix's code part in a (full or half) chunk.
__device__ uint32_t code_word_at(const QLayout &L, const Staged &s, int m, int k0, bool half, int o) {
    int lane, i;
    if (L.kind == MOE_Q2_64) {
        if (!half) { lane = o / 16; i = (o % 16) / 4; }
        else { lane = o / 8; i = (o % 8) / 4; }
    } else {
        if (!half) { const int part = o / 512; lane = (o % 512) / 16; i = 4 * part + (o % 16) / 4; }
        else { lane = o / 16; i = (o % 16) / 4; }
    }
    return code_word(L, s, m, k0, lane, i);
}

// Rewrite one tile with `nmat` matrices (2: gate/up, 1: down) whose reduction
// length is Kd. src_rows[m] points at row 0 of the tile of matrix m in the blob.
__global__ void k_repack_tile(QLayout L, const uint8_t *blob, uint8_t *dst, int section) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int tile = blockIdx.x;
    const int nmat = section == 0 ? 2 : 1;
    const int Kd = section == 0 ? L.H : L.F;        // reduction length
    const int rows_total = section == 0 ? L.F : L.H; // rows of each matrix
    const int nblk = Kd / L.bw;
    const int row_bytes = nblk * kBlockBytes;
    const long long mat_bytes = (long long)rows_total * row_bytes;
    Staged s{smem, row_bytes, 16};
    // stage: for gate/up, matrices 0 (gate) and 1 (up); for down, matrix 2
    for (int m = 0; m < nmat; ++m) {
        const int msrc = section == 0 ? m : 2;
        const uint8_t *src = blob + msrc * mat_bytes + (long long)tile * 16 * row_bytes;
        uint8_t *d = smem + (size_t)m * 16 * row_bytes;
        for (int b = threadIdx.x; b < 16 * row_bytes; b += blockDim.x) d[b] = src[b];
    }
    __syncthreads();
    const int full_chunks = Kd / 128;
    const bool has_half = (Kd % 128) != 0;
    const int n_chunks = full_chunks + (has_half ? 1 : 0);
    const int chunk_bytes = nmat * (L.cb + L.sb);
    uint8_t *tile_dst = dst + (section == 0 ? 0 : L.d_offset) +
                        (long long)tile * (section == 0 ? L.gu_tile_bytes : L.d_tile_bytes);
    for (int ch = 0; ch < n_chunks; ++ch) {
        const bool half = ch == full_chunks;
        const int cb = half ? L.cb / 2 : L.cb, sb = half ? L.sb / 2 : L.sb;
        const int bytes = nmat * (cb + sb);
        uint32_t *out = (uint32_t *)(tile_dst + (long long)ch * chunk_bytes);
        const int k0 = ch * 128, b0 = k0 / L.bw;
        for (int wi = threadIdx.x; wi < bytes / 4; wi += blockDim.x) {
            const int o = wi * 4;
            uint32_t v;
            if (o < nmat * cb) {
                const int m = o / cb;
                v = code_word_at(L, s, m, k0, half, o % cb);
            } else {
                const int o2 = o - nmat * cb;
                const int m = o2 / sb;
                v = scale_word(s, m, b0, (o2 % sb) / 4);
            }
            out[wi] = v;
        }
    }
}

}  // namespace

int init_repack_attributes(int max_smem) {
    return set_max_dynamic_smem((const void *)k_repack_tile, max_smem);
}

int repack_expert(const QLayout &L, const uint8_t *blob, uint8_t *dst, cudaStream_t stream) {
    const int row_gu = L.H / L.bw * kBlockBytes, row_d = L.F / L.bw * kBlockBytes;
    const size_t smem_gu = (size_t)2 * 16 * row_gu, smem_d = (size_t)16 * row_d;
    const size_t smem_max = smem_gu > smem_d ? smem_gu : smem_d;
    if (smem_max > 200 * 1024)
        return set_error(MOE_ERR_SHAPE, "repack: expert rows too long (H=%d F=%d)", L.H, L.F);
    k_repack_tile<<<L.gu_tiles, 256, smem_gu, stream>>>(L, blob, dst, 0);
    MOE_CUDA_TRY(cudaGetLastError());
    k_repack_tile<<<L.d_tiles, 256, smem_d, stream>>>(L, blob, dst, 1);
    MOE_CUDA_TRY(cudaGetLastError());
    return MOE_OK;
}

}  // namespace moe
