// moe_internal.cuh -- shapes, workspace layout and kernel launchers shared by the .cu files.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

// GEMV-regime tiling (fixed, so every reduction order depends on tile indices only).
constexpr int kNT = 8;          // tokens per sub-block (register tile of the GEMV kernels)
constexpr int kTI = 64;         // gate/up: I columns per tile (128-byte rows in shared memory)
constexpr int kHG = 128;        // gate/up: H rows per unit
constexpr int kTN = 64;         // down: H columns per tile
constexpr int kIG = 128;        // down: I rows per unit
constexpr int kConsumerWarps = 8;
constexpr int kGemvThreads = 32 * (1 + kConsumerWarps);
constexpr int kRouterCluster = 8;  // CTAs per router cluster (split of H)
constexpr int kRouterThreads = 256;

struct Dims {
    int M, k, E, H, I, b;
    int rsub;         // rows per sub-block: b if b <= 8, else 8
    int64_t R;        // routes M*k (also the sentinel value)
    int64_t cap;      // alignment capacity in rows
    int64_t max_sub;  // cap / rsub
    int n_it, n_hg, n_ht, n_ig;
};

struct WsLayout {
    size_t status;   // int32[16]
    size_t sorted;   // int32[cap]
    size_t blocks;   // int32[cap / b]
    size_t npad;     // int32[4]
    size_t p;        // float[R * I]   SiLU(g) * u per route
    size_t y;        // float[R * H]   down-projection output per route
    size_t total;
};

Dims make_dims(int M, int k, int E, int H, int I, int b);
WsLayout ws_layout(const Dims &d);

struct GemvArgs {
    const __nv_bfloat16 *h;
    const int32_t *topk_ids;
    const float *topk_wts;
    const int32_t *sorted;
    const int32_t *blocks;
    const int32_t *npad;
    const __nv_bfloat16 *residual;
    __nv_bfloat16 *out;
    float *p;
    float *y;
    int32_t *status;
    int M, k, E, H, I, b, rsub;
    int n_it, n_hg, n_ht, n_ig;
};

int num_sms();

cudaError_t launch_router(const __nv_bfloat16 *h, const __nv_bfloat16 *w_router,
                          const float *bias, int M, int H, int E, int k, int renormalize,
                          int32_t *topk_ids, float *topk_weights, cudaStream_t stream);

cudaError_t launch_align(const int32_t *topk_ids, int M, int k, int E, int b,
                         int32_t *sorted, int32_t *blocks, int32_t *npad, int64_t cap,
                         int32_t *status, cudaStream_t stream);

cudaError_t launch_gateup_dense(const CUtensorMap &tm_gate, const CUtensorMap &tm_up,
                                const GemvArgs &a, cudaStream_t stream);

cudaError_t launch_down(const CUtensorMap &tm_down, const GemvArgs &a, cudaStream_t stream);

cudaError_t launch_combine(const GemvArgs &a, cudaStream_t stream);

// Shared launch helper: programmatic dependent launch on, optional cluster dims.
cudaLaunchConfig_t launch_config(dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                                 cudaLaunchAttribute *attrs, int cluster_x);

}  // namespace moe
