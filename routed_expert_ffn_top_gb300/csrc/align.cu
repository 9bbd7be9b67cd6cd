// align.cu -- deterministic, atomic-order-free block alignment of the routes.
//
// "Route-Block Membership Selects Packed-AWQ Arithmetic", Section 2.1: the top-k router's
// M x k expert ids are flattened row-major into route ids r in [0, M*k); valid routes are
// grouped by expert and each expert's count is padded to a multiple of the block size b,
// with a parallel expert-per-block vector.  Section 5.3: the stable construction orders
// valid routes by (expert id, route id), which makes the result independent of any
// scheduling history; the page's own fix scans the routes with one thread per expert.
//
// Design: one CTA of 256 threads.  (1) per-expert counts in shared memory (integer
// atomics: the counts do not depend on arrival order); (2) one warp scans the padded
// counts into row offsets; (3) routes are scattered chunk by chunk in ascending r: inside
// a warp, __match_any_sync groups lanes with the same expert and a popcount of the lower
// lanes gives each route its rank, warps of the chunk are ranked through a per-warp count
// table, and a per-expert running total carries ranks across chunks.  Every rank, hence
// every output position, is a pure function of the input ids.  (5) Optionally, a table of
// the aligned rows in groups of rsub (expert, routes, tokens) that the expert kernels read
// one record per tile.
#include "moe_internal.cuh"
#include "ptx.cuh"

namespace moe {

constexpr int kAlignThreads = 256;
constexpr int kAlignWarps = kAlignThreads / 32;

__global__ void __launch_bounds__(kAlignThreads)
    align_kernel(const int32_t *__restrict__ ids, int M, int k, int E, int b,
                 int32_t *__restrict__ sorted, int32_t *__restrict__ blocks,
                 int32_t *__restrict__ npad, int64_t cap, SubBlock *sbt, int rsub,
                 int32_t *status) {
    extern __shared__ __align__(16) int32_t sm[];
    int32_t *cnt = sm;                  // [E]
    int32_t *off = cnt + E;             // [E] padded row offsets
    int32_t *running = off + E;         // [E]
    int32_t *warp_cnt = running + E;    // [kAlignWarps][E]
    __shared__ int32_t s_total;
    __shared__ int32_t s_invalid;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t R = (int64_t)M * k;
    const int32_t sentinel = (int32_t)R;

    pdl_wait();
    pdl_launch_dependents();

    for (int i = tid; i < (3 + kAlignWarps) * E; i += kAlignThreads) sm[i] = 0;
    if (tid == 0) s_invalid = 0;
    __syncthreads();

    // (1) counts
    int local_invalid = 0;
    for (int64_t r = tid; r < R; r += kAlignThreads) {
        const int e = ids[r];
        if (e >= 0 && e < E)
            atomicAdd(&cnt[e], 1);
        else
            local_invalid = 1;
    }
    if (local_invalid) atomicOr(&s_invalid, 1);
    __syncthreads();

    // (2) exclusive scan of padded counts (warp 0; lane owns a contiguous run of experts)
    if (warp == 0) {
        const int per = (E + 31) / 32;
        const int e0 = lane * per, e1 = min(E, e0 + per);
        int s = 0;
        for (int e = e0; e < e1; ++e) s += (cnt[e] + b - 1) / b * b;
        int incl = s;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        int run = incl - s;
        for (int e = e0; e < e1; ++e) {
            off[e] = run;
            run += (cnt[e] + b - 1) / b * b;
        }
        if (lane == 31) s_total = incl;
    }
    __syncthreads();
    const int total = s_total;

    // (3) stable scatter in ascending route id
    const unsigned lt_mask = (1u << lane) - 1u;
    for (int64_t base = 0; base < R; base += kAlignThreads) {
        const int64_t r = base + tid;
        const int e = (r < R) ? ids[r] : -1;
        const bool valid = (e >= 0 && e < E);
        const unsigned peers = __match_any_sync(0xffffffffu, valid ? e : -1);
        const int lower = __popc(peers & lt_mask);
        const int wcount = __popc(peers);
        const bool leader = lower == 0;
        if (valid && leader) warp_cnt[warp * E + e] = wcount;
        __syncthreads();
        if (valid) {
            int rank = running[e] + lower;
            for (int w = 0; w < warp; ++w) rank += warp_cnt[w * E + e];
            const int64_t pos = (int64_t)off[e] + rank;
            if (pos < cap) sorted[pos] = (int32_t)r;
        }
        __syncthreads();
        if (valid && leader) {
            // Several warps may hold routes of expert e: integer adds commute, so the
            // total is the same whatever order they land in.
            atomicAdd(&running[e], wcount);
            warp_cnt[warp * E + e] = 0;
        }
        __syncthreads();
    }

    // (4) padding rows, block vector, tail
    for (int e = tid; e < E; e += kAlignThreads) {
        const int n = cnt[e];
        const int padded = (n + b - 1) / b * b;
        for (int q = n; q < padded; ++q)
            if (off[e] + q < cap) sorted[off[e] + q] = sentinel;
        for (int q = 0; q < padded / b; ++q) blocks[off[e] / b + q] = e;
    }
    for (int64_t pos = (int64_t)total + tid; pos < cap; pos += kAlignThreads) sorted[pos] = sentinel;
    for (int64_t q = (int64_t)total / b + tid; q < cap / b; q += kAlignThreads) blocks[q] = -1;
    if (tid == 0) {
        npad[0] = total;
        if (status && s_invalid) atomicOr(status, MOE_DEV_INVALID_EXPERT);
    }
    // (5) the sub-block table the expert kernels stream from
    if (sbt) {
        __syncthreads();
        for (int64_t sb = tid; sb < total / rsub; sb += kAlignThreads)
            build_subblock(sorted, blocks, ids, sb, rsub, b, E, R, k, false, nullptr, sbt + sb);
    }
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

cudaError_t launch_align(const int32_t *topk_ids, int M, int k, int E, int b, int32_t *sorted,
                         int32_t *blocks, int32_t *npad, int64_t cap, SubBlock *sbt, int rsub,
                         int32_t *status, cudaStream_t stream) {
    const size_t smem = (size_t)(3 + kAlignWarps) * E * sizeof(int32_t);
    cudaError_t err = cudaFuncSetAttribute(align_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)smem);
    if (err != cudaSuccess) return err;
    cudaLaunchAttribute attrs[2];
    cudaLaunchConfig_t cfg = launch_config(dim3(1), dim3(kAlignThreads), smem, stream, attrs, 0);
    return cudaLaunchKernelEx(&cfg, align_kernel, topk_ids, M, k, E, b, sorted, blocks, npad,
                              cap, sbt, rsub, status);
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
