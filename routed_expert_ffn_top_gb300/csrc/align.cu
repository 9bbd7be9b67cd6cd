// align.cu -- the stand-alone alignment kernel and the plan kernel.
//
// "Route-Block Membership Selects Packed-AWQ Arithmetic", Sections 2.1 and 5.3: the M x k
// expert ids, flattened into route ids, are grouped by expert in ascending route id and
// padded to multiples of b (see align_core.cuh for the atomic-order-free construction).
// The plan kernel turns a caller-supplied alignment into the sub-block table the expert
// kernels read, checking every row against the top-k ids.
#include "align_core.cuh"
#include "moe_internal.cuh"
#include "ptx.cuh"

namespace moe {

// Shared-memory ints the alignment kernel of kThreads threads uses for (E, R, cap, b):
// align_core's tables, the staged ids, and the aligned rows and block vector built in shared
// memory.  Returns 0 when they do not fit (then ids and rows stay in global memory).
template <int kThreads>
static int64_t align_kernel_ints(int E, int64_t R, int64_t cap, int b) {
    const int64_t n = align_smem_ints<kThreads>(E) + R + cap + cap / b + 4;
    return (R <= kAlignStagedRoutes && n * 4 <= kAlignSmemBytes) ? n : 0;
}

template <int kThreads>
__global__ void __launch_bounds__(kThreads)
    align_kernel(const int32_t *__restrict__ ids, int M, int k, int E, int b,
                 int32_t *__restrict__ sorted, int32_t *__restrict__ blocks,
                 int32_t *__restrict__ npad, int64_t cap, SubBlock *sbt, int rsub,
                 int32_t *status, int staged) {
    extern __shared__ __align__(16) int32_t sm[];
    pdl_wait();
    pdl_launch_dependents();
    const int64_t R = (int64_t)M * k;
    if (!staged) {
        align_core<kThreads>(ids, R, k, E, b, rsub, sorted, blocks, npad, cap, sbt, status, sm);
        return;
    }
    // Everything in shared memory: the ids are read once with all loads in flight, the rows
    // and the block vector are built there, then leave with coalesced stores; the sub-block
    // records are formed one per thread from the finished rows.
    int32_t *ids_s = sm + align_smem_ints<kThreads>(E);
    int32_t *rows_s = ids_s + R;
    int32_t *blocks_s = rows_s + cap;
#pragma unroll 8
    for (int64_t r = threadIdx.x; r < R; r += kThreads) ids_s[r] = ids[r];
    __syncthreads();
    align_core<kThreads>(ids_s, R, k, E, b, rsub, rows_s, blocks_s, npad, cap, nullptr, status, sm);
    __syncthreads();
    if (sorted)
        for (int64_t i = threadIdx.x; i < cap; i += kThreads) sorted[i] = rows_s[i];
    if (blocks)
        for (int64_t i = threadIdx.x; i < cap / b; i += kThreads) blocks[i] = blocks_s[i];
    if (sbt) {
        const int64_t total = sm[(3 + kThreads / 32) * E];  // align_core's padded row count
        for (int64_t sb = threadIdx.x; sb < total / rsub; sb += kThreads)
            build_subblock(rows_s, blocks_s, ids_s, sb, rsub, b, E, R, k, false, status, sbt + sb);
    }
}

template <int kThreads>
static cudaError_t launch_align_t(const int32_t *topk_ids, int M, int k, int E, int b,
                                  int32_t *sorted, int32_t *blocks, int32_t *npad, int64_t cap,
                                  SubBlock *sbt, int rsub, int32_t *status, cudaStream_t stream) {
    const int64_t R = (int64_t)M * k;
    const int64_t staged_ints = align_kernel_ints<kThreads>(E, R, cap, b);
    const size_t smem =
        (size_t)(staged_ints ? staged_ints : align_smem_ints<kThreads>(E)) * sizeof(int32_t);
    cudaError_t err = ensure_smem(reinterpret_cast<const void *>(align_kernel<kThreads>), smem);
    if (err != cudaSuccess) return err;
    cudaLaunchAttribute attrs[2];
    cudaLaunchConfig_t cfg = launch_config(dim3(1), dim3(kThreads), smem, stream, attrs, 0);
    return cudaLaunchKernelEx(&cfg, align_kernel<kThreads>, topk_ids, M, k, E, b, sorted, blocks,
                              npad, cap, sbt, rsub, status, staged_ints ? 1 : 0);
}

__global__ void __launch_bounds__(kAlignThreads)
    plan_kernel(const int32_t *__restrict__ ids, const int32_t *__restrict__ sorted,
                const int32_t *__restrict__ blocks, const int32_t *__restrict__ npad, int M,
                int k, int E, int b, int rsub, int64_t max_sub, SubBlock *sbt, int32_t *status) {
    pdl_wait();
    pdl_launch_dependents();
    const int64_t R = (int64_t)M * k;
    int64_t nsub = npad[0] / rsub;
    if (nsub > max_sub) {  // a num_padded larger than the capacity: use what fits
        nsub = max_sub;
        if (threadIdx.x == 0 && blockIdx.x == 0) atomicOr(status, MOE_DEV_BAD_ALIGNMENT);
    }
    for (int64_t sb = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; sb < nsub;
         sb += (int64_t)gridDim.x * blockDim.x)
        build_subblock(sorted, blocks, ids, sb, rsub, b, E, R, k, true, status, sbt + sb);
}

// One CTA of 256 threads, or of 1024 from kAlignWideRoutes routes (the positions are the
// same; more threads shorten the passes over the routes and rows).
constexpr int64_t kAlignWideRoutes = 512;

cudaError_t launch_align(const int32_t *topk_ids, int M, int k, int E, int b, int32_t *sorted,
                         int32_t *blocks, int32_t *npad, int64_t cap, SubBlock *sbt, int rsub,
                         int32_t *status, cudaStream_t stream) {
    if ((int64_t)M * k >= kAlignWideRoutes)
        return launch_align_t<1024>(topk_ids, M, k, E, b, sorted, blocks, npad, cap, sbt, rsub,
                                    status, stream);
    return launch_align_t<kAlignThreads>(topk_ids, M, k, E, b, sorted, blocks, npad, cap, sbt,
                                         rsub, status, stream);
}

// Alignment and row tiles in one launch, for up to kAlignGatherRoutes routes (the tcgen05
// path's tiles): every CTA aligns the routes itself (align_small, one thread per route, the
// same stable order), CTA 0 writes the alignment, and all CTAs copy their share of the
// valid routes' token rows into the K-major 128-byte-swizzle row tiles (16-byte pieces;
// padding rows are left as they are: their columns are dropped by the epilogues).
__global__ void __launch_bounds__(kAlignThreads)
    align_gather_kernel(const int32_t *__restrict__ ids, int M, int k, int E, int b,
                        int32_t *__restrict__ sorted, int32_t *__restrict__ blocks,
                        int32_t *__restrict__ npad, int64_t cap, int32_t *status,
                        const __nv_bfloat16 *__restrict__ x, int H,
                        __nv_bfloat16 *__restrict__ x_tiles, int kn, int tpb,
                        int32_t *__restrict__ ready, int64_t nready) {
    __shared__ int32_t ids_s[kAlignGatherRoutes];
    __shared__ int32_t pos_s[kAlignGatherRoutes];
    __shared__ int32_t scratch[align_small_smem_ints(kAlignThreads)];
    pdl_wait();
    pdl_launch_dependents();
    if (blockIdx.x == 0) zero_counts(ready, nready);  // the next grid's, read after this grid
    const int R = M * k;
    for (int r = threadIdx.x; r < R; r += blockDim.x) ids_s[r] = ids[r];
    __syncthreads();
    const bool first = blockIdx.x == 0;
    align_small(ids_s, R, k, E, b, b, first ? sorted : nullptr, first ? blocks : nullptr,
                first ? npad : nullptr, cap, nullptr, first ? status : nullptr, scratch, pos_s);
    __syncthreads();
    const int pieces = H / 8;  // 16-byte pieces of a token row
    const int64_t chunk_bytes = (int64_t)kn * 128;
    const int64_t tile_bytes = (int64_t)(H / 64) * chunk_bytes;
    unsigned char *xt = reinterpret_cast<unsigned char *>(x_tiles);
    const int64_t total = (int64_t)R * pieces;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    // 4 pieces per thread in flight at once, then their stores
    for (int64_t i0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i0 < total; i0 += 4 * stride) {
        uint4 v[4];
        int64_t dst[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int64_t idx = i0 + u * stride;
            dst[u] = -1;
            if (idx >= total) continue;
            const int r = (int)(idx / pieces), p = (int)(idx - (int64_t)r * pieces);
            const int pos = pos_s[r];
            if (pos < 0) continue;
            const int local = pos % b;
            const int64_t t = (int64_t)(pos / b) * tpb + local / kn;
            const int n = local % kn;
            dst[u] = t * tile_bytes + (p >> 3) * chunk_bytes + tile_offset(n, p & 7);
            v[u] = *reinterpret_cast<const uint4 *>(x + (size_t)(r / k) * H + (size_t)p * 8);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
            if (dst[u] >= 0) *reinterpret_cast<uint4 *>(xt + dst[u]) = v[u];
    }
}

cudaError_t launch_align_gather(const int32_t *topk_ids, int M, int k, int E, int b,
                                int32_t *sorted, int32_t *blocks, int32_t *npad, int64_t cap,
                                int32_t *status, const __nv_bfloat16 *x, int H,
                                const RowTiles &rows, cudaStream_t stream) {
    const int R = M * k;
    if (R < 1 || R > kAlignGatherRoutes || !rows.x_tiles) return cudaErrorInvalidValue;
    const int64_t work = (int64_t)R * (H / 8);
    int grid = (int)((work + 4 * kAlignThreads - 1) / (4 * kAlignThreads));
    grid = grid < 1 ? 1 : (grid > num_sms() ? num_sms() : grid);
    cudaLaunchAttribute attrs[2];
    cudaLaunchConfig_t cfg = launch_config(dim3(grid), dim3(kAlignThreads), 0, stream, attrs, 0);
    return cudaLaunchKernelEx(&cfg, align_gather_kernel, topk_ids, M, k, E, b, sorted, blocks, npad,
                              cap, status, x, H, rows.x_tiles, rows.kn, rows.tpb, rows.ready,
                              rows.nready);
}

cudaError_t launch_plan(const int32_t *topk_ids, const int32_t *sorted, const int32_t *blocks,
                        const int32_t *npad, int M, int k, int E, int b, int rsub,
                        int64_t max_sub, SubBlock *sbt, int32_t *status, cudaStream_t stream) {
    cudaLaunchAttribute attrs[2];
    const int64_t blocks_needed = (max_sub + kAlignThreads - 1) / kAlignThreads;
    const int grid = (int)(blocks_needed < 1 ? 1 : (blocks_needed > 1024 ? 1024 : blocks_needed));
    cudaLaunchConfig_t cfg = launch_config(dim3(grid), dim3(kAlignThreads), 0, stream, attrs, 0);
    return cudaLaunchKernelEx(&cfg, plan_kernel, topk_ids, sorted, blocks, npad, M, k, E, b, rsub,
                              max_sub, sbt, status);
}

}  // namespace moe
