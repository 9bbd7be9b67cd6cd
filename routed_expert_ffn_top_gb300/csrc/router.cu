// router.cu -- router GEMV + softmax top-k with renormalised affinities.
//
// "A Multi-Engine Dataflow for MoE Decoding on Scratchpad-Based Tensor Accelerators",
// MoE block background (Figure 2): the router scores the experts for the input h, selects
// k of them and assigns each an affinity a_e.  Read here as softmax over the logits,
// top-k, renormalised over the selected experts; an optional per-expert bias is added to
// the logits before selection.
//
// Design (sm_103a): one thread-block cluster of 8 CTAs per tile of up to 8 tokens.  CTA q
// of the cluster owns rows [q*H/8, (q+1)*H/8) of W_r, which are contiguous in memory and
// arrive with a single bulk copy issued before the programmatic-dependent-launch wait (the
// router weights never depend on the previous kernel).  Each CTA reduces its slice to
// partial logits in shared memory (bf16 h x bf16 W_r into fp32, rows ascending per thread,
// then the row groups in order); after a cluster barrier the CTA of rank t gathers token
// t's 8 partials through distributed shared memory, sums them in rank order, adds the bias,
// and one warp runs the top-k (ties to the lower expert id) and the softmax.  The order
// depends on (H, E) only, so a token's logits are the same for every M.
//
// When one cluster holds every token (M <= 8) the same kernel also runs the alignment
// (align_core.cuh) in the CTA of rank 0 on the ids it gathers from the cluster, which saves
// the alignment launch on the decode path.
#include <float.h>

#include "align_core.cuh"
#include "ptx.cuh"

namespace moe {

struct FusedAlign {
    int enabled;
    int b, rsub;
    int32_t *sorted, *blocks, *npad;
    int64_t cap;
    SubBlock *sbt;
    int32_t *status;
};

// Generic address of `p` (a shared variable of this CTA) in CTA `rank` of the cluster.
__device__ __forceinline__ const float *cluster_peer(const float *p, uint32_t rank) {
    uint64_t out;
    asm("mapa.u64 %0, %1, %2;" : "=l"(out) : "l"(reinterpret_cast<uint64_t>(p)), "r"(rank));
    return reinterpret_cast<const float *>(out);
}
__device__ __forceinline__ const int32_t *cluster_peer(const int32_t *p, uint32_t rank) {
    uint64_t out;
    asm("mapa.u64 %0, %1, %2;" : "=l"(out) : "l"(reinterpret_cast<uint64_t>(p)), "r"(rank));
    return reinterpret_cast<const int32_t *>(out);
}

template <int TM>
__global__ void __launch_bounds__(kRouterThreads)
    router_topk_kernel(const __nv_bfloat16 *__restrict__ h, const __nv_bfloat16 *__restrict__ wr,
                       const float *__restrict__ bias, int M, int H, int E, int k, int renorm,
                       int32_t *__restrict__ topk_ids, float *__restrict__ topk_wts,
                       const FusedAlign fa) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const int tid = threadIdx.x;
    const uint32_t rank = cluster_ctarank();
    const int HS = H / kRouterCluster;
    const int tile = blockIdx.y;
    const int npairs = E / 2;
    const int RG = kRouterThreads / npairs;  // row groups (>= 1 since E <= 512)

    // shared layout: w_s [HS][E] bf16 | x_s [TM][HS] bf16 | red [RG][TM][E] f32 |
    //                part [TM][E] f32 | ids_s [k] | bar | align scratch
    unsigned char *ptr = smem_raw;
    __nv_bfloat16 *w_s = reinterpret_cast<__nv_bfloat16 *>(ptr);
    ptr += (size_t)HS * E * 2;
    __nv_bfloat16 *x_s = reinterpret_cast<__nv_bfloat16 *>(ptr);
    ptr += (size_t)TM * HS * 2;
    float *red = reinterpret_cast<float *>(ptr);
    ptr += (size_t)RG * TM * E * 4;
    float *part = reinterpret_cast<float *>(ptr);
    ptr += (size_t)TM * E * 4;
    int32_t *ids_s = reinterpret_cast<int32_t *>(ptr);  // [8 * 32] gathered ids (rank 0)
    ptr += 8 * 32 * 4;
    uint64_t *bar = reinterpret_cast<uint64_t *>(ptr);
    ptr += 16;
    int32_t *align_sm = reinterpret_cast<int32_t *>(ptr);

    const uint32_t w_bytes = (uint32_t)HS * E * 2;
    if (tid == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0) {
        mbar_arrive_expect_tx(bar, w_bytes);
        bulk_load(w_s, wr + (size_t)rank * HS * E, w_bytes, bar);
    }
    pdl_wait();  // h may come from the previous kernel in the stream
    pdl_launch_dependents();

    // h slices: 16-byte pieces (8 rows) of each token of the tile
    const int pieces = HS / 8;
    for (int idx = tid; idx < TM * pieces; idx += kRouterThreads) {
        const int t = idx / pieces, pc = idx - t * pieces;
        const int m = tile * TM + t;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (m < M) v = *reinterpret_cast<const uint4 *>(h + (size_t)m * H + (size_t)rank * HS + pc * 8);
        *reinterpret_cast<uint4 *>(x_s + (size_t)t * HS + pc * 8) = v;
    }
    __syncthreads();
    const bool ok = mbar_wait_bounded(bar, 0);

    const int pair = tid % npairs, rg = tid / npairs;
    if (ok && rg < RG) {
        const int r0 = rg * HS / RG, r1 = (rg + 1) * HS / RG;
        float acc0[TM], acc1[TM];
#pragma unroll
        for (int t = 0; t < TM; ++t) acc0[t] = acc1[t] = 0.0f;
        const uint32_t *wrow = reinterpret_cast<const uint32_t *>(w_s) + pair;
        const uint32_t *x32 = reinterpret_cast<const uint32_t *>(x_s);
        int r = r0;
        for (; r + 1 < r1 && (r & 1) == 0; r += 2) {  // two rows per step (one bf16 pair of h)
            const uint32_t wa = wrow[(size_t)r * npairs], wb = wrow[(size_t)(r + 1) * npairs];
#pragma unroll
            for (int t = 0; t < TM; ++t) {
                const uint32_t xv = x32[((size_t)t * HS + r) >> 1];
                acc0[t] = fma_bf16<0, 0>(xv, wa, acc0[t]);
                acc1[t] = fma_bf16<0, 1>(xv, wa, acc1[t]);
                acc0[t] = fma_bf16<1, 0>(xv, wb, acc0[t]);
                acc1[t] = fma_bf16<1, 1>(xv, wb, acc1[t]);
            }
        }
        for (; r < r1; ++r) {  // an odd tail row (row groups of odd length)
            const uint32_t wa = wrow[(size_t)r * npairs];
#pragma unroll
            for (int t = 0; t < TM; ++t) {
                const uint32_t xv = x32[((size_t)t * HS + r) >> 1];
                if (r & 1) {
                    acc0[t] = fma_bf16<1, 0>(xv, wa, acc0[t]);
                    acc1[t] = fma_bf16<1, 1>(xv, wa, acc1[t]);
                } else {
                    acc0[t] = fma_bf16<0, 0>(xv, wa, acc0[t]);
                    acc1[t] = fma_bf16<0, 1>(xv, wa, acc1[t]);
                }
            }
        }
#pragma unroll
        for (int t = 0; t < TM; ++t) {
            red[((size_t)rg * TM + t) * E + 2 * pair] = acc0[t];
            red[((size_t)rg * TM + t) * E + 2 * pair + 1] = acc1[t];
        }
    }
    __syncthreads();
    for (int idx = tid; idx < TM * E; idx += kRouterThreads) {
        float s = red[idx];
        for (int g = 1; g < RG; ++g) s += red[(size_t)g * TM * E + idx];
        part[idx] = s;
    }
    cluster_sync();

    // Finalise: CTA of rank t handles token t of the tile (TM <= 8 = cluster size).
    const int warp = tid >> 5, lane = tid & 31;
    const int t = (int)rank;
    const int m = tile * TM + t;
    if (warp == 0 && t < TM && m < M) {
        constexpr int kPerLane = 16;  // E <= 512
        float vals[kPerLane];
#pragma unroll
        for (int i = 0; i < kPerLane; ++i) {
            const int e = lane + 32 * i;
            float v = -FLT_MAX;
            if (e < E) {
                // the 8 partials are loaded together, then summed in rank order
                float pv[kRouterCluster];
#pragma unroll
                for (uint32_t q = 0; q < kRouterCluster; ++q)
                    pv[q] = *cluster_peer(part + (size_t)t * E + e, q);
                v = 0.0f;
#pragma unroll
                for (int q = 0; q < kRouterCluster; ++q) v += pv[q];
                if (bias) v += bias[e];
                if (!ok) v = -FLT_MAX;
            }
            vals[i] = v;
        }
        uint32_t taken = 0;
        int my_e = -1;
        float my_v = -FLT_MAX;
        for (int j = 0; j < k; ++j) {
            float bv = -INFINITY;
            int be = 0x7fffffff;
#pragma unroll
            for (int i = 0; i < kPerLane; ++i) {
                const int e = lane + 32 * i;
                if (e < E && !((taken >> i) & 1u)) {
                    const float v = vals[i];
                    if (v > bv || (v == bv && e < be)) {
                        bv = v;
                        be = e;
                    }
                }
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
                const int oe = __shfl_xor_sync(0xffffffffu, be, off);
                if (ov > bv || (ov == bv && oe < be)) {
                    bv = ov;
                    be = oe;
                }
            }
            if (be >= 0 && be < E && (be & 31) == lane) taken |= 1u << (be >> 5);
            if (lane == j) {
                my_e = be;
                my_v = bv;
            }
        }
        const float l0 = __shfl_sync(0xffffffffu, my_v, 0);
        float denom;
        float ex = 0.0f;
        if (renorm) {
            ex = (lane < k) ? expf(my_v - l0) : 0.0f;
            denom = ex;
        } else {
            float s = 0.0f;
#pragma unroll
            for (int i = 0; i < kPerLane; ++i)
                if (lane + 32 * i < E) s += expf(vals[i] - l0);
            denom = s;
            ex = (lane < k) ? expf(my_v - l0) : 0.0f;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) denom += __shfl_xor_sync(0xffffffffu, denom, off);
        if (lane < k) {
            const int id = ok ? my_e : -1;
            topk_ids[(size_t)m * k + lane] = id;
            topk_wts[(size_t)m * k + lane] = ok ? ex / denom : 0.0f;
            ids_s[lane] = id;
        }
    }
    if (fa.enabled) {
        // every token's ids are in the cluster: rank 0 gathers them and aligns
        cluster_sync();
        if (rank == 0) {
            for (int idx = tid; idx < M * k; idx += kRouterThreads)
                ids_s[idx] = *cluster_peer(ids_s + idx % k, (uint32_t)(idx / k));
            __syncthreads();
            align_core(ids_s, (int64_t)M * k, k, E, fa.b, fa.rsub, fa.sorted, fa.blocks, fa.npad,
                       fa.cap, fa.sbt, fa.status, align_sm);
        }
    }
    cluster_sync();  // keep this CTA's shared memory alive until every peer has read it
}

static size_t router_smem(int TM, int H, int E, bool fuse) {
    const int HS = H / kRouterCluster;
    const int RG = kRouterThreads / (E / 2);
    return (size_t)HS * E * 2 + (size_t)TM * HS * 2 + (size_t)RG * TM * E * 4 +
           (size_t)TM * E * 4 + 8 * 32 * 4 + 16 + (fuse ? (size_t)align_smem_ints(E) * 4 : 0);
}

template <int TM>
static cudaError_t launch_router_tm(const __nv_bfloat16 *h, const __nv_bfloat16 *w_router,
                                    const float *bias, int M, int H, int E, int k, int renorm,
                                    int32_t *ids, float *wts, const FusedAlign &fa,
                                    cudaStream_t stream) {
    const size_t smem = router_smem(TM, H, E, fa.enabled != 0);
    cudaError_t err = cudaFuncSetAttribute(router_topk_kernel<TM>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    cudaLaunchAttribute attrs[2];
    dim3 grid(kRouterCluster, (M + TM - 1) / TM, 1);
    cudaLaunchConfig_t cfg = launch_config(grid, dim3(kRouterThreads), smem, stream, attrs,
                                           kRouterCluster);
    return cudaLaunchKernelEx(&cfg, router_topk_kernel<TM>, h, w_router, bias, M, H, E, k,
                              renorm, ids, wts, fa);
}

static cudaError_t launch_router_any(const __nv_bfloat16 *h, const __nv_bfloat16 *w_router,
                                     const float *bias, int M, int H, int E, int k,
                                     int renormalize, int32_t *topk_ids, float *topk_weights,
                                     const FusedAlign &fa, cudaStream_t stream) {
    if (M <= 0) return cudaSuccess;
    const int renorm = renormalize ? 1 : 0;
    if (M <= 1)
        return launch_router_tm<1>(h, w_router, bias, M, H, E, k, renorm, topk_ids, topk_weights,
                                   fa, stream);
    if (M <= 2)
        return launch_router_tm<2>(h, w_router, bias, M, H, E, k, renorm, topk_ids, topk_weights,
                                   fa, stream);
    if (M <= 4)
        return launch_router_tm<4>(h, w_router, bias, M, H, E, k, renorm, topk_ids, topk_weights,
                                   fa, stream);
    return launch_router_tm<8>(h, w_router, bias, M, H, E, k, renorm, topk_ids, topk_weights, fa,
                               stream);
}

cudaError_t launch_router(const __nv_bfloat16 *h, const __nv_bfloat16 *w_router,
                          const float *bias, int M, int H, int E, int k, int renormalize,
                          int32_t *topk_ids, float *topk_weights, cudaStream_t stream) {
    FusedAlign fa{};
    return launch_router_any(h, w_router, bias, M, H, E, k, renormalize, topk_ids, topk_weights,
                             fa, stream);
}

bool router_can_align(int M, int k) { return M >= 1 && M <= kRouterCluster && M * k <= 8 * 32; }

cudaError_t launch_router_align(const __nv_bfloat16 *h, const __nv_bfloat16 *w_router,
                                const float *bias, int M, int H, int E, int k, int renormalize,
                                int32_t *topk_ids, float *topk_weights, int b, int rsub,
                                int32_t *sorted, int32_t *blocks, int32_t *npad, int64_t cap,
                                SubBlock *sbt, int32_t *status, cudaStream_t stream) {
    FusedAlign fa;
    fa.enabled = 1;
    fa.b = b;
    fa.rsub = rsub;
    fa.sorted = sorted;
    fa.blocks = blocks;
    fa.npad = npad;
    fa.cap = cap;
    fa.sbt = sbt;
    fa.status = status;
    return launch_router_any(h, w_router, bias, M, H, E, k, renormalize, topk_ids, topk_weights,
                             fa, stream);
}

}  // namespace moe
