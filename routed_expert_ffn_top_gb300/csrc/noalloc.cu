// noalloc.cu -- the decode block for callers that cannot allocate device memory.
//
// Some callers of this library have no way to obtain device memory for a workspace: the
// block is embedded in a host program whose GPU memory is owned entirely by another
// allocator (an inference server's memory pool, a plugin host that only hands over its
// input and output tensors), or in a deployment that forbids any allocation after
// start-up to keep a fixed memory budget.  For them this file keeps the block's scratch
// memory (alignment rows, per-route intermediate p and expert outputs y, device status
// word) in one fixed device array inside the library and runs the ordinary block on it.
#include <mutex>

#include "moe_internal.cuh"

namespace {

// Scratch for moe_decode_block_noalloc.  Every GPU that loads the library holds these
// bytes until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[MOE_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  In host code the array's
// name is only a host-side stand-in, so the address is looked up once per device (with
// that device current) and cached.
int scratch_on_current_device(void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
            return MOE_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return MOE_OK;
}

}  // namespace

extern "C" int moe_decode_block_noalloc(const void *h, const void *w_router, const float *bias,
                                        const moe_expert_weights_t *w, int M, int k, int b,
                                        const void *residual, void *out, int32_t *topk_ids,
                                        float *topk_weights, void *stream) {
    if (w == nullptr || M < 0) return MOE_ERR_INVALID_ARG;
    const size_t need = moe::workspace_bytes_fixed(w, M, k, moe::block_for(w, M, k, b));
    if (need == 0) return MOE_ERR_UNSUPPORTED;
    if (need > (size_t)MOE_NOALLOC_SCRATCH_BYTES) return MOE_ERR_WORKSPACE;
    if (M == 0) return MOE_OK;
    void *ws = nullptr;
    int rc = scratch_on_current_device(&ws);
    if (rc != MOE_OK) return rc;
    // The array keeps whatever the previous call left in it.  The status word is cleared
    // here; the counters and the one-grid path's routing exchange, which must also start at
    // zero, are zero in the fresh array and every call leaves them zero (no other path writes
    // them); everything else is written before it is read.
    if (cudaMemsetAsync(ws, 0, 64, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return MOE_ERR_CUDA;
    return moe::decode_block(h, w_router, bias, w, M, k, b, residual, out, topk_ids,
                             topk_weights, ws, (size_t)MOE_NOALLOC_SCRATCH_BYTES, stream);
}
