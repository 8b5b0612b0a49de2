// synth_dev.cu -- CUDA twin of synth.expert_blobs: fills canonical expert blobs
// on the device (SplitMix64, Steele, Lea and Flood, OOPSLA 2014). Input
// generation only: it knows the block layout (fp16 scale, 16 code bytes) but
// nothing of what the codes mean.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

__device__ __forceinline__ uint64_t sm64(uint64_t seed, uint64_t idx) {
    return mix64(seed + (idx + 1ull) * 0x9E3779B97F4A7C15ull);
}

__global__ void k_blobs(uint8_t *dst, long long n_blocks_total, long long blocks_per_expert, uint64_t seed,
                        long long first_tag, double d_lo, double d_span) {
    for (long long b = blockIdx.x * (long long)blockDim.x + threadIdx.x; b < n_blocks_total;
         b += (long long)gridDim.x * blockDim.x) {
        const long long e = b / blocks_per_expert, bl = b % blocks_per_expert;
        const uint64_t s = sm64(seed, (uint64_t)(first_tag + e));
        const uint64_t w0 = sm64(s, 3ull * bl), w1 = sm64(s, 3ull * bl + 1ull);
        const double u = (double)(sm64(s, 3ull * bl + 2ull) >> 11) * 0x1p-53;
        const double d = __dadd_rn(d_lo, __dmul_rn(d_span, u));
        const uint16_t dh = __half_as_ushort(__double2half(d));
        uint16_t *out = reinterpret_cast<uint16_t *>(dst + b * 18);
        out[0] = dh;
        for (int i = 0; i < 4; ++i) out[1 + i] = (uint16_t)(w0 >> (16 * i));
        for (int i = 0; i < 4; ++i) out[5 + i] = (uint16_t)(w1 >> (16 * i));
    }
}

}  // namespace

extern "C" __attribute__((visibility("default"))) int synth_expert_blobs(void *dst, long long n_experts,
                                                                         long long blocks_per_expert,
                                                                         unsigned long long seed, long long first_tag,
                                                                         double d_lo, double d_span, void *stream) {
    if (!dst || n_experts < 0 || blocks_per_expert <= 0 || ((uintptr_t)dst & 1)) return -1;
    const long long n = n_experts * blocks_per_expert;
    if (n == 0) return 0;
    long long grid = (n + 255) / 256;
    if (grid > 65536) grid = 65536;
    k_blobs<<<(unsigned)grid, 256, 0, (cudaStream_t)stream>>>((uint8_t *)dst, n, blocks_per_expert, seed, first_tag,
                                                              d_lo, d_span);
    return cudaGetLastError() == cudaSuccess ? 0 : -4;
}
