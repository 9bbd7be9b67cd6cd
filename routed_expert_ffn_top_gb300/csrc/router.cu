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
// When one cluster holds every token (M <= 2 on the decode path) the same kernel also runs
// the alignment (align_core.cuh) in the CTA of rank 0 on the ids it gathers from the
// cluster, which saves the alignment launch.
#include <float.h>

#include "align_core.cuh"
#include "ptx.cuh"
#include "route_core.cuh"

namespace moe {

struct FusedAlign {
    int enabled;
    int b, rsub;
    int32_t *sorted, *blocks, *npad;
    int64_t cap;
    SubBlock *sbt;
    int32_t *status;
    RowTiles rows;  // rows.x_tiles != NULL: every CTA also writes its H slice of the row tiles
};

// Low-rank projections computed in the router's launch (VQ + low-rank gate/up weights):
// clusters blockIdx.y >= lr.first compute z[m][p*r + c] = sum_h h[m][h] D_p[h][c] for
// projection p (0 gate, 1 up) of their token tile, with the same split of H over the
// cluster, the same fixed summation order and no top-k.

// Passes over a CTA's slice of HS weight rows with E columns: the smallest power of two
// that keeps one pass within kRouterPassBytes.
constexpr int kRouterPassBytes = 64 * 1024;
__host__ __device__ inline int router_passes(int HS, int E) {
    int n = 1;
    while ((int64_t)(HS / n) * E * 2 > kRouterPassBytes && n < HS) n *= 2;
    return n;
}

// Generic address of `p` (a shared variable of this CTA) in CTA `rank` of the cluster.
template <typename T>
__device__ __forceinline__ T *cluster_peer_mut(T *p, uint32_t rank) {
    uint64_t out;
    asm("mapa.u64 %0, %1, %2;" : "=l"(out) : "l"(reinterpret_cast<uint64_t>(p)), "r"(rank));
    return reinterpret_cast<T *>(out);
}

// TM tokens per cluster tile; kPerLane experts per lane in the top-k warp (E <= 32 kPerLane).
template <int TM, int kPerLane>
__global__ void __launch_bounds__(kRouterThreads)
    router_topk_kernel(const __nv_bfloat16 *__restrict__ h, const __nv_bfloat16 *__restrict__ wr,
                       const float *__restrict__ bias, int M, int H, int E, int k, int renorm,
                       int32_t *__restrict__ topk_ids, float *__restrict__ topk_wts,
                       const FusedAlign fa, const LowRankProj lr) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const int tid = threadIdx.x;
    const uint32_t rank = cluster_ctarank();
    const int HS = H / kRouterCluster;
    // A cluster either routes its token tile (columns: the E experts of W_r) or computes one
    // low-rank projection of it (columns: the r basis vectors of D_gate or D_up).
    const bool zmode = lr.r > 0 && (int)blockIdx.y >= lr.first;
    const int zi = (int)blockIdx.y - lr.first;
    const int tile = zmode ? zi >> 1 : (int)blockIdx.y;
    const int proj = zi & 1;
    if (zmode) E = lr.r;
    const __nv_bfloat16 *wsrc = zmode ? (proj ? lr.d_up : lr.d_gate) : wr;
    const int npairs = E / 2;
    const int RG = kRouterThreads / npairs;  // row groups (>= 1 since E <= 512)

    // W_r rows of this CTA stream through shared memory in npass passes of HP rows (one
    // pass when the slice is at most kRouterPassBytes), so that two CTAs fit on an SM at
    // every supported shape.  Row group g of pass p is rows p*HP + [g*HP/RG, (g+1)*HP/RG);
    // a thread sums its rows in ascending order over the passes.  The split depends on
    // (H, E) only, never on M.
    const int npass = router_passes(HS, E);
    const int HP = HS / npass;

    // When one cluster aligns every token (routing clusters of the fused launch), every rank
    // receives every token's partial logits and finalises all of them itself, so that the
    // aligned rows are known in every rank without a second cluster barrier.  Otherwise
    // rank t finalises token t of the tile.
    const bool all_ranks = fa.enabled && !zmode;
    const int GT = all_ranks ? TM : 1;  // tokens whose partials this CTA gathers

    // shared layout: w_s [HP][E] bf16 | x_s [TM][HS] bf16 | red [RG][TM][E] f32 |
    //                gath [GT][8][E] f32 (the partial logits of every rank) |
    //                ids_s [8 * 32] | bar | align scratch | aligned row of every route
    unsigned char *ptr = smem_raw;
    __nv_bfloat16 *w_s = reinterpret_cast<__nv_bfloat16 *>(ptr);
    ptr += (size_t)HP * E * 2;
    __nv_bfloat16 *x_s = reinterpret_cast<__nv_bfloat16 *>(ptr);
    ptr += (size_t)TM * HS * 2;
    float *red = reinterpret_cast<float *>(ptr);
    ptr += (size_t)RG * TM * E * 4;
    float *gath = reinterpret_cast<float *>(ptr);
    ptr += (size_t)GT * kRouterCluster * E * 4;
    int32_t *ids_s = reinterpret_cast<int32_t *>(ptr);  // [8 * 32] every token's ids
    ptr += 8 * 32 * 4;
    uint64_t *bar = reinterpret_cast<uint64_t *>(ptr);
    ptr += 16;
    int32_t *align_sm = reinterpret_cast<int32_t *>(ptr);

    const uint32_t w_bytes = (uint32_t)HP * E * 2;
    const __nv_bfloat16 *w_cta = wsrc + (size_t)rank * HS * E;
    if (tid == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0) {
        mbar_arrive_expect_tx(bar, w_bytes);
        bulk_load(w_s, w_cta, w_bytes, bar);
    }
    pdl_wait();  // h may come from the previous kernel in the stream
    pdl_launch_dependents();
    if (fa.enabled && rank == 0 && blockIdx.y == 0) zero_counts(fa.rows.ready, fa.rows.nready);

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

    const int pair = tid % npairs, rg = tid / npairs;
    float acc0[TM], acc1[TM];
#pragma unroll
    for (int t = 0; t < TM; ++t) acc0[t] = acc1[t] = 0.0f;
    const uint32_t *wrow = reinterpret_cast<const uint32_t *>(w_s) + pair;
    const uint32_t *x32 = reinterpret_cast<const uint32_t *>(x_s);
    bool ok = true;
    for (int pass = 0; pass < npass; ++pass) {
        if (pass > 0) {
            __syncthreads();  // every thread is done with the previous pass's rows
            if (tid == 0 && ok) {  // (after a wait that gave up, no further copy is issued)
                mbar_arrive_expect_tx(bar, w_bytes);
                bulk_load(w_s, w_cta + (size_t)pass * HP * E, w_bytes, bar);
            }
        }
        ok = ok && mbar_wait_bounded(bar, (uint32_t)pass & 1u);
        if (!ok || rg >= RG) continue;
        const int base = pass * HP;  // first row of the pass within the CTA's slice
        const int r0 = base + rg * HP / RG, r1 = base + (rg + 1) * HP / RG;
        int r = r0;
        for (; r + 1 < r1 && (r & 1) == 0; r += 2) {  // two rows per step (one bf16 pair of h)
            const uint32_t wa = wrow[(size_t)(r - base) * npairs];
            const uint32_t wb = wrow[(size_t)(r + 1 - base) * npairs];
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
            const uint32_t wa = wrow[(size_t)(r - base) * npairs];
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
    }
    if (ok && rg < RG) {
#pragma unroll
        for (int t = 0; t < TM; ++t) {
            red[((size_t)rg * TM + t) * E + 2 * pair] = acc0[t];
            red[((size_t)rg * TM + t) * E + 2 * pair + 1] = acc1[t];
        }
    }
    __syncthreads();
    // Row groups summed in order, then pushed to the CTAs that finalise the token (rank t, or
    // every rank), into their own shared memory, so that after the cluster barrier all reads
    // are local and no CTA touches another's shared memory.
    for (int idx = tid; idx < TM * E; idx += kRouterThreads) {
        float s = red[idx];
        for (int g = 1; g < RG; ++g) s += red[(size_t)g * TM * E + idx];
        const int t = idx / E, e = idx - t * E;
        if (tile * TM + t >= M) continue;
        if (all_ranks) {
            for (uint32_t q = 0; q < (uint32_t)kRouterCluster; ++q)
                cluster_peer_mut(gath, q)[((size_t)t * kRouterCluster + rank) * E + e] = s;
        } else {
            cluster_peer_mut(gath, (uint32_t)t)[(size_t)rank * E + e] = s;
        }
    }
    cluster_sync();

    if (zmode) {  // the projection: the 8 partials summed in rank order
        const int t = (int)rank;
        const int m = tile * TM + t;
        if (t < TM && m < M)
            for (int c = tid; c < E; c += kRouterThreads) {
                float v = 0.0f;
#pragma unroll
                for (int q = 0; q < kRouterCluster; ++q) v += gath[(size_t)q * E + c];
                lr.z[(size_t)m * 2 * lr.r + (size_t)proj * lr.r + c] = ok ? v : 0.0f;
            }
        return;
    }
    // Tokens finalised here: t0 .. t0 + nt - 1 of the tile.
    const int t0 = all_ranks ? 0 : (int)rank;
    int nt = all_ranks ? TM : ((int)rank < TM ? 1 : 0);
    if (tile * TM + t0 + nt > M) nt = M - tile * TM - t0 > 0 ? M - tile * TM - t0 : 0;
    route_finalize<kPerLane>(gath, nt, E, k, bias, ok, renorm,
                   [&](int i, int j, int id, float wt) {
                       const int t = t0 + i;
                       const int m = tile * TM + t;
                       if (!all_ranks || rank == 0) {
                           topk_ids[(size_t)m * k + j] = id;
                           topk_wts[(size_t)m * k + j] = wt;
                       }
                       if (all_ranks) ids_s[t * k + j] = id;  // every rank aligns them below
                   });
    if (fa.enabled) {
        __syncthreads();
        int32_t *pos_s = align_sm + align_small_smem_ints(kRouterThreads);  // [M * k]
        const int R = M * k;
        if (rank == 0)
            align_small(ids_s, R, k, E, fa.b, fa.rsub, fa.sorted, fa.blocks, fa.npad, fa.cap,
                        fa.sbt, fa.status, align_sm, fa.rows.x_tiles ? pos_s : nullptr);
        else if (fa.rows.x_tiles)  // the same positions, nothing else written
            align_small(ids_s, R, k, E, fa.b, fa.rsub, nullptr, nullptr, nullptr, fa.cap, nullptr,
                        nullptr, align_sm, pos_s);
        if (fa.rows.x_tiles) {
            // The x tile rows of the grouped GEMMs: this CTA's H slice of every valid route's
            // token row (already in x_s, the cluster holds every token) goes to row n of
            // tile t, 16-byte piece by piece in the swizzled image.
            __syncthreads();
            const int kn = fa.rows.kn, tpb = fa.rows.tpb, b = fa.b;
            const int64_t chunk_bytes = (int64_t)kn * 128;
            const int64_t tile_bytes = (int64_t)(H / 64) * chunk_bytes;
            unsigned char *xt = reinterpret_cast<unsigned char *>(fa.rows.x_tiles);
            for (int idx = tid; idx < R * pieces; idx += kRouterThreads) {
                const int r = idx / pieces, q = idx - r * pieces;
                const int pos = pos_s[r];
                if (pos < 0) continue;
                const int p = (int)rank * pieces + q;  // piece of the whole row (8 columns)
                const int local = pos % b;
                const int64_t t = (int64_t)(pos / b) * tpb + local / kn;
                const int n = local % kn;
                *reinterpret_cast<uint4 *>(xt + t * tile_bytes + (p >> 3) * chunk_bytes +
                                           tile_offset(n, p & 7)) =
                    *reinterpret_cast<const uint4 *>(x_s + (size_t)(r / k) * HS + q * 8);
            }
        }
    }
    // No CTA touches another's shared memory after the cluster barrier.
}

static size_t router_smem(int TM, int H, int E, bool fuse) {
    const int HS = H / kRouterCluster;
    const int RG = kRouterThreads / (E / 2);
    const int GT = fuse ? TM : 1;
    return (size_t)(HS / router_passes(HS, E)) * E * 2 + (size_t)TM * HS * 2 + (size_t)RG * TM * E * 4 +
           (size_t)GT * kRouterCluster * E * 4 + 8 * 32 * 4 + 16 +
           (fuse ? (size_t)(align_small_smem_ints(kRouterThreads) + 8 * 32) * 4 : 0);
}

template <int TM, int kPerLane>
static cudaError_t launch_router_tm(const __nv_bfloat16 *h, const __nv_bfloat16 *w_router,
                                    const float *bias, int M, int H, int E, int k, int renorm,
                                    int32_t *ids, float *wts, const FusedAlign &fa,
                                    LowRankProj lr, bool route, cudaStream_t stream) {
    const int ntiles = (M + TM - 1) / TM;
    // the routing clusters and the projection clusters carve shared memory for their own
    // column counts (E, r); the launch gets the larger of the two layouts (not the layout of
    // the larger count: more columns take more, smaller passes)
    size_t smem = route ? router_smem(TM, H, E, fa.enabled != 0) : 0;
    if (lr.r > 0) {
        const size_t zs = router_smem(TM, H, lr.r, false);
        if (zs > smem) smem = zs;
    }
    cudaError_t err =
        ensure_smem(reinterpret_cast<const void *>(router_topk_kernel<TM, kPerLane>), smem);
    if (err != cudaSuccess) return err;
    cudaLaunchAttribute attrs[2];
    lr.first = route ? ntiles : 0;
    dim3 grid(kRouterCluster, lr.first + (lr.r > 0 ? 2 * ntiles : 0), 1);
    cudaLaunchConfig_t cfg = launch_config(grid, dim3(kRouterThreads), smem, stream, attrs,
                                           kRouterCluster);
    return cudaLaunchKernelEx(&cfg, router_topk_kernel<TM, kPerLane>, h, w_router, bias, M, H, E, k,
                              renorm, ids, wts, fa, lr);
}

constexpr int kRouterOwnTileTokens = 32;

template <int kPerLane>
static cudaError_t launch_router_lanes(const __nv_bfloat16 *h, const __nv_bfloat16 *w_router,
                                       const float *bias, int M, int H, int E, int k, int renorm,
                                       int32_t *topk_ids, float *topk_weights,
                                       const FusedAlign &fa, const LowRankProj &lr, bool route,
                                       cudaStream_t stream) {
    // Without the fused alignment (which needs every token in one cluster), up to
    // kRouterOwnTileTokens tokens get a cluster each: a token's arithmetic is the same in any
    // tile, and one token per cluster divides the dot work of a CTA by up to 8.
    if (M <= 1 || (!fa.enabled && M <= kRouterOwnTileTokens))
        return launch_router_tm<1, kPerLane>(h, w_router, bias, M, H, E, k, renorm, topk_ids,
                                             topk_weights, fa, lr, route, stream);
    if (M <= 2)
        return launch_router_tm<2, kPerLane>(h, w_router, bias, M, H, E, k, renorm, topk_ids,
                                             topk_weights, fa, lr, route, stream);
    if (M <= 4)
        return launch_router_tm<4, kPerLane>(h, w_router, bias, M, H, E, k, renorm, topk_ids,
                                             topk_weights, fa, lr, route, stream);
    return launch_router_tm<8, kPerLane>(h, w_router, bias, M, H, E, k, renorm, topk_ids,
                                         topk_weights, fa, lr, route, stream);
}

static cudaError_t launch_router_any(const __nv_bfloat16 *h, const __nv_bfloat16 *w_router,
                                     const float *bias, int M, int H, int E, int k,
                                     int renormalize, int32_t *topk_ids, float *topk_weights,
                                     const FusedAlign &fa, const LowRankProj *lr_in,
                                     cudaStream_t stream) {
    if (M <= 0) return cudaSuccess;
    const int renorm = renormalize ? 1 : 0;
    LowRankProj lr{};
    if (lr_in) lr = *lr_in;
    if (E <= 128)
        return launch_router_lanes<4>(h, w_router, bias, M, H, E, k, renorm, topk_ids,
                                      topk_weights, fa, lr, true, stream);
    if (E <= 256)
        return launch_router_lanes<8>(h, w_router, bias, M, H, E, k, renorm, topk_ids,
                                      topk_weights, fa, lr, true, stream);
    return launch_router_lanes<16>(h, w_router, bias, M, H, E, k, renorm, topk_ids, topk_weights,
                                   fa, lr, true, stream);
}

cudaError_t launch_router(const __nv_bfloat16 *h, const __nv_bfloat16 *w_router,
                          const float *bias, int M, int H, int E, int k, int renormalize,
                          int32_t *topk_ids, float *topk_weights, const LowRankProj *lr,
                          cudaStream_t stream) {
    FusedAlign fa{};
    return launch_router_any(h, w_router, bias, M, H, E, k, renormalize, topk_ids, topk_weights,
                             fa, lr, stream);
}

cudaError_t launch_lowrank_proj(const __nv_bfloat16 *h, int M, int H, const LowRankProj &lr,
                                cudaStream_t stream) {
    if (M <= 0 || lr.r <= 0) return cudaSuccess;
    FusedAlign fa{};
    return launch_router_lanes<4>(h, nullptr, nullptr, M, H, lr.r, 0, 0, nullptr, nullptr, fa, lr,
                                  false, stream);
}

// The router runs the alignment in its own launch for up to 2 tokens.  From 3 tokens on,
// a cluster per token (kRouterOwnTileTokens) and the alignment with the row tiles in one
// launch of its own (up to 128 routes) were faster: same-box A/B, -1.0 us per layer at 4
// tokens, -1.6 us at 8, +0.9 us at 2.
bool router_can_align(int M, int k) { return M >= 1 && M <= 2 && M * k <= 8 * 32; }

cudaError_t launch_router_align(const __nv_bfloat16 *h, const __nv_bfloat16 *w_router,
                                const float *bias, int M, int H, int E, int k, int renormalize,
                                int32_t *topk_ids, float *topk_weights, int b, int rsub,
                                int32_t *sorted, int32_t *blocks, int32_t *npad, int64_t cap,
                                SubBlock *sbt, int32_t *status, const LowRankProj *lr,
                                const RowTiles &rows, cudaStream_t stream) {
    FusedAlign fa;
    fa.rows = rows;
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
                             fa, lr, stream);
}

}  // namespace moe
