// static_scratch.cu -- moe_layer_forward_static: the whole layer with the library's
// own fixed scratch area in place of a caller-provided workspace.
//
// Some callers cannot allocate device memory for a workspace: a host framework
// that owns every byte of the GPU through its own pool and gives plugins no
// allocator, a latency-critical decode loop that must never call cudaMalloc
// (it can synchronise the device and stall other streams), or a thin binding
// that has no way to size and keep a buffer. For them the scratch lives in one
// file-scope device array below. Every GPU that loads this library holds the
// array until the process exits.
#include <mutex>

#include "moe_internal.cuh"

namespace moe {
int ctx_device(const moe_ctx *ctx);
}

namespace {

// The scratch. In host code this name is only a stand-in for the device
// symbol, not an address: kernels get the address obtained below.
static __device__ __align__(256) uint8_t g_scratch[MOE_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void *g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of g_scratch on `device`, looked up once per device with that
// device current.
int scratch_address(int device, void **out) {
    if (device < 0 || device >= kMaxDevices) return moe::set_error(MOE_ERR_ARG, "device %d out of range", device);
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[device]) {
        // the lookup needs `device` current; the caller's current device is put
        // back on every path, and a failure to put it back is reported
        int prev = 0;
        cudaError_t e = cudaGetDevice(&prev);
        if (e != cudaSuccess) return moe::cuda_error(e, "cudaGetDevice");
        if (prev != device) {
            e = cudaSetDevice(device);
            if (e != cudaSuccess) return moe::cuda_error(e, "cudaSetDevice (static scratch lookup)");
        }
        void *p = nullptr;
        const cudaError_t el = cudaGetSymbolAddress(&p, g_scratch);
        if (prev != device) {
            e = cudaSetDevice(prev);
            if (e != cudaSuccess) return moe::cuda_error(e, "cudaSetDevice (restoring the caller's device)");
        }
        if (el != cudaSuccess) return moe::cuda_error(el, "cudaGetSymbolAddress(static scratch)");
        g_scratch_ptr[device] = p;
    }
    *out = g_scratch_ptr[device];
    return MOE_OK;
}

}  // namespace

extern "C" int moe_layer_forward_static(moe_ctx *ctx, const moe_layer_desc *desc, const void *x, moe_dtype xt,
                                        int T, float *y, float *logits_out, int32_t *ids_out,
                                        moe_stream_t stream) {
    if (!ctx) return moe::set_error(MOE_ERR_ARG, "null context");
    size_t need = 0;
    int rc = moe_layer_workspace(desc, T < 0 ? 0 : T, &need);
    if (rc) return rc;
    if (need > (size_t)MOE_STATIC_SCRATCH_BYTES)
        return moe::set_error(MOE_ERR_WORKSPACE,
                              "T=%d needs %zu bytes of scratch; the static scratch holds %d bytes "
                              "(use moe_layer_forward with a workspace)",
                              T, need, MOE_STATIC_SCRATCH_BYTES);
    void *scratch = nullptr;
    rc = scratch_address(moe::ctx_device(ctx), &scratch);
    if (rc) return rc;
    return moe_layer_forward(ctx, desc, x, xt, T, y, logits_out, ids_out, scratch,
                             (size_t)MOE_STATIC_SCRATCH_BYTES, stream);
}
