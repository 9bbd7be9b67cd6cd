// decode_small.cu -- the whole decode block for a few tokens in one persistent grid: router,
// alignment, gate/up + SiLU, down and the affinity-weighted combine.
//
// The block is the one of "A Multi-Engine Dataflow for MoE Decoding on Scratchpad-Based
// Tensor Accelerators" (MoE block background; stage-3 activation; Section 4.3) with the
// alignment of "Route-Block Membership Selects Packed-AWQ Arithmetic" (Sections 2.1, 5.3).
// At one or two tokens the expert weights are the only real traffic (75 MB per layer at one
// token), and every step of a chain of kernels costs a launch boundary on the critical path
// before the weight stream starts and after it ends.  So one grid does it all:
//
//  1. Routing.  The router kernel's 8 slices of W_r's rows, each cut into row groups with one
//     chain per (token, expert) (the same groups, rows and orders, so the logits and the
//     selection are bitwise those of the multi-kernel path), are spread over 64 CTAs at
//     E = 128: CTA (slice q, chunk c) holds the slice's rows of 16 experts, copied before
//     the wait for the previous grid, and runs one group and expert pair per thread.  It adds
//     its groups in order and publishes the slice's partial logits of its experts with a
//     release count.  Every CTA acquires them and runs the router's own finalisation (logits
//     in slice order, the warp arg-max top-k, softmax) and the alignment itself (one warp,
//     at most 32 routes): no CTA waits for another's result.
//  2. Experts.  Units as in the fused grid (gemm_tc05.cu): gate/up units (tile, 64 channels
//     of I) first, then down units (tile, 128 channels of H), CTA c taking units c, c + G ...
//     The weight boxes come by TMA (warp 0); the tile's few token rows (gate/up: h; down:
//     p) are copied into the stage's swizzled B slot by warp 6 with cp.async, which then
//     fences the generic writes for the tensor cores' async proxy and arrives on the stage's
//     barrier.  A down unit's weight boxes stream at once; its p rows wait for the tile's
//     ready count (release by each gate/up unit once its p rows are stored).  Each output
//     element is one K-ordered MMA chain, as in the multi-kernel path.
//  3. Combine.  A down unit stores y for its routes and counts them, per token and 128-channel
//     tile of H; the unit whose count completes a token's valid routes forms that token's
//     output for its channels: out = bf16(residual + sum_j a_j y_j), slots in order, the
//     combine kernel's arithmetic.
//
// The counters live in a control region of the workspace that is zero between calls: the
// last CTA to finish (an exit count) restores it.  Every wait is bounded; a wait that gives
// up sets MOE_DEV_WAIT_TIMEOUT and the grid drains and exits.
#include "align_core.cuh"
#include "gemm_core.cuh"
#include "route_core.cuh"
#include "small_route.cuh"

namespace moe {

using GS = GTile<16>;
// producer, MMA, 4 epilogue warps, row loader; 9 more warps that only help with the routing
// (512 threads, so that the router's dot products run one row group and expert pair per
// thread, as in the router kernel)
constexpr int kSThreads = kRouterThreads;
constexpr int kSLoaderWarp = 6;
static_assert(kSmallMaxRoutes <= 32, "the alignment runs in one warp");

struct SmallState {
    int32_t ids[kSmallMaxRoutes];
    float wts[kSmallMaxRoutes];
    int32_t tile_e[kSmallMaxRoutes];                     // expert of each tile (block)
    int32_t tile_n[kSmallMaxRoutes];                     // rows holding a route (the first ones)
    int32_t tile_r[kSmallMaxRoutes][kSmallMaxTokens];    // their routes
    int32_t nvalid[kSmallMaxTokens];                     // valid routes of each token
    int32_t comb[kSmallMaxTokens];                       // per row of the down unit: token to combine, or -1
    int32_t ntiles;
    int32_t last;  // this CTA took the last exit ticket
};

__device__ __forceinline__ int32_t atom_add_acq_rel_gpu(int32_t *p, int32_t v) {
    int32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// Bounded wait until *p >= need (acquire, GPU scope), polling every few tens of ns.
__device__ __forceinline__ bool count_wait(const int32_t *p, int need, GCtl &ctl) {
    if (ld_acquire_gpu(p) >= need) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        __nanosleep(32);
        if (ld_acquire_gpu(p) >= need) return true;
        if (ctl.abort) return false;
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
            ctl.abort = 1;
            return false;
        }
    }
}

struct SmallUnits {
    int64_t Tgu, T;
    int n_gu, n_dn, nks_gu, nks_dn;
    __device__ __forceinline__ void at(int64_t u, bool &gu, int &tile, int &ct, int &nks) const {
        gu = u < Tgu;
        const uint32_t v = (uint32_t)(gu ? u : u - Tgu);  // units fit 32 bits (few tiles here)
        const uint32_t n = (uint32_t)(gu ? n_gu : n_dn);
        const uint32_t t = v / n;
        tile = (int)t;
        ct = (int)(v - t * n);
        nks = gu ? nks_gu : nks_dn;
    }
};

// Copy issuer (one thread): the weight boxes of every stage.
__device__ void small_producer(const SmallArgs &a, GCtl &ctl, unsigned char *stages,
                               const SmallState &st, const SmallUnits &f,
                               const CUtensorMap *tm_gate, const CUtensorMap *tm_up,
                               const CUtensorMap *tm_down) {
    const uint64_t pol = policy_evict_first();
    int stage = 0;
    uint32_t phase = 0, issued = 0, parity_bits = 0;
    bool stop = false;
    for (int64_t u = blockIdx.x; u < f.T && !stop && !ctl.abort; u += gridDim.x) {
        bool gu;
        int tile, ct, nks;
        f.at(u, gu, tile, ct, nks);
        const int e = st.tile_e[tile];
        for (int s = 0; s < nks; ++s) {
            if (!gwait(&ctl.empty[stage], phase ^ 1u, ctl)) {
                stop = true;
                break;
            }
            uint64_t *bar = &ctl.full[stage];
            unsigned char *dst = stages + stage * GS::kStageBytes;
            mbar_arrive_expect_tx(bar, GS::kABytes);
            if (gu) {
                const int32_t y = e * a.H + s * GS::kK;
                tma_load_2d(dst, tm_gate, ct * 64, y, bar, pol);
                tma_load_2d(dst + GS::kHalfBytes, tm_up, ct * 64, y, bar, pol);
            } else {
                const int32_t y = e * a.I + s * GS::kK;
                tma_load_2d(dst, tm_down, ct * kGM, y, bar, pol);
                tma_load_2d(dst + GS::kHalfBytes, tm_down, ct * kGM + 64, y, bar, pol);
            }
            issued |= 1u << stage;
            parity_bits = (parity_bits & ~(1u << stage)) | (phase << stage);
            gadvance<GS>(stage, phase);
        }
    }
    for (int s = 0; s < GS::kStages; ++s)
        if ((issued >> s) & 1u)
            if (!mbar_wait_bounded(&ctl.full[s], (parity_bits >> s) & 1u)) ctl.abort = 1;
}

// Row loader (one warp): per stage, the 256-deep K slice of every row of the tile that holds a
// route -- h of the route's token (gate/up) or p of the route (down) -- into the stage's B slot
// in the K-major 128-byte-swizzle layout (row n at n * 128 bytes of each 64-wide chunk, 16-byte
// piece j at (j ^ n % 8) * 16), one 16-byte piece per lane.  Rows without a route keep
// whatever the slot held: their columns of the MMA are dropped.  Two stages' copies are in
// flight at a time: a stage is released (proxy fence, arrival) once its copies have landed,
// after the next stage's are issued.  Before a down unit waits for its tile's p, every
// stage still held is released, so that no wait depends on this warp's own arrivals.
__device__ void small_loader(const SmallArgs &a, GCtl &ctl, unsigned char *stages,
                             const SmallState &st, const SmallUnits &f) {
    const int lane = threadIdx.x & 31;
    int stage = 0;
    uint32_t phase = 0;
    int held[2];
    int nheld = 0;
    auto release_oldest = [&](bool all) {
        if (all)
            cp_async_wait_group<0>();
        else
            cp_async_wait_group<1>();
        fence_proxy_async_smem();  // generic writes, read next by the tensor cores
        __syncwarp();
        const int n = all ? nheld : 1;
        if (lane == 0)
            for (int i = 0; i < n; ++i) mbar_arrive(&ctl.full[held[i]]);
        if (!all) held[0] = held[1];
        nheld -= n;
    };
    for (int64_t u = blockIdx.x; u < f.T && !ctl.abort; u += gridDim.x) {
        bool gu;
        int tile, ct, nks;
        f.at(u, gu, tile, ct, nks);
        const int nrow = st.tile_n[tile];
        if (!gu) {  // p of the tile's routes: stored by all I/64 gate/up units of the tile
            if (nheld > 0) release_oldest(true);
            bool ok = true;
            if (lane == 0) ok = count_wait(a.ctl + kSmallCtlReady + tile, f.n_gu, ctl);
            if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) return;
        }
        for (int s = 0; s < nks; ++s) {
            if (!__all_sync(0xffffffffu, gwait(&ctl.empty[stage], phase ^ 1u, ctl))) return;
            unsigned char *bslot = stages + stage * GS::kStageBytes + GS::kBOff;
            for (int n = 0; n < nrow; ++n) {
                const int r = st.tile_r[tile][n];
                const __nv_bfloat16 *src = gu ? a.h + (size_t)(r / a.k) * a.H + (size_t)s * GS::kK
                                              : a.p_rows + (size_t)r * a.I + (size_t)s * GS::kK;
                cp_async_16(bslot + (lane >> 3) * GS::kChunkBytes + tile_offset(n, lane & 7),
                            src + lane * 8);
            }
            cp_async_commit();
            held[nheld++] = stage;
            if (nheld == 2) release_oldest(false);
            gadvance<GS>(stage, phase);
        }
    }
    if (nheld > 0) release_oldest(true);
}

// MMA issuer (one thread): as in the fused grid.
__device__ void small_mma(GCtl &ctl, unsigned char *stages, const SmallUnits &f) {
    constexpr uint32_t idesc = umma_idesc_bf16(kGM, 16, true, false);
    int stage = 0;
    uint32_t phase = 0;
    int local = 0;
    for (int64_t u = blockIdx.x; u < f.T && !ctl.abort; u += gridDim.x, ++local) {
        bool gu;
        int tile, ct, nks;
        f.at(u, gu, tile, ct, nks);
        const int buf = local & 1;
        if (!gwait(&ctl.tempty[buf], ((uint32_t)(local >> 1) & 1u) ^ 1u, ctl)) break;
        tc_fence_after();
        const uint32_t d = ctl.tmem + (uint32_t)(buf * 16);
        bool ok = true;
        for (int s = 0; s < nks; ++s) {
            if (!gwait(&ctl.full[stage], phase, ctl)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t A = smem_u32(stages + stage * GS::kStageBytes);
            const uint32_t B = A + GS::kBOff;
#pragma unroll
            for (int ks = 0; ks < GS::kK / 16; ++ks) {
                const uint64_t ad = umma_smem_desc(A + ks * 2048, GS::kHalfBytes, 1024, 2);
                const uint64_t bd =
                    umma_smem_desc(B + (ks >> 2) * GS::kChunkBytes + (ks & 3) * 32, 16, 1024, 2);
                umma_bf16(d, ad, bd, idesc, s > 0 || ks > 0);
            }
            umma_commit(&ctl.empty[stage]);
            gadvance<GS>(stage, phase);
        }
        if (!ok) break;
        umma_commit(&ctl.tfull[buf]);
    }
    umma_commit(&ctl.done);
    if (!mbar_wait_bounded(&ctl.done, 0)) ctl.abort = 1;
}

// CTA 0, one warp, while the expert phase runs: the alignment as moe_align_block_size gives
// it (rows of tile t: its routes, then sentinels; the block vector; the row count), the
// status bit for invalid routes, and out = residual (or zero) for a token with no valid route.
__device__ void small_write_alignment(const SmallArgs &a, const SmallState &st, int R) {
    const int lane = threadIdx.x & 31, b = a.b, ntiles = st.ntiles;
    for (int64_t i = lane; i < a.cap; i += 32) {
        const int t = (int)(i / b), n = (int)(i - (int64_t)t * b);
        a.sorted[i] = (t < ntiles && n < st.tile_n[t]) ? st.tile_r[t][n] : R;
    }
    for (int64_t q = lane; q < a.cap / b; q += 32) a.blocks[q] = q < ntiles ? st.tile_e[q] : -1;
    int nv = 0;
    for (int t = 0; t < a.M; ++t) nv += st.nvalid[t];
    if (lane == 0) {
        a.npad[0] = ntiles * b;
        if (nv < R) atomicOr(a.status, MOE_DEV_INVALID_EXPERT);
    }
    for (int t = 0; t < a.M; ++t)
        if (st.nvalid[t] == 0)
            for (int n = lane; n < a.H; n += 32)
                a.out[(size_t)t * a.H + n] =
                    a.residual ? a.residual[(size_t)t * a.H + n] : __float2bfloat16(0.0f);
}

__global__ void __launch_bounds__(kSThreads, 1)
    decode_small_kernel(const __grid_constant__ CUtensorMap tm_gate,
                        const __grid_constant__ CUtensorMap tm_up,
                        const __grid_constant__ CUtensorMap tm_down, const SmallArgs a) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *base = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char *stages = base;
    float *gbuf = reinterpret_cast<float *>(base + GS::kStages * GS::kStageBytes);  // [16][64]
    GCtl &ctl = *reinterpret_cast<GCtl *>(base + GS::kStages * GS::kStageBytes + 16 * 64 * 4);
    SmallState &st = *reinterpret_cast<SmallState *>(reinterpret_cast<unsigned char *>(&ctl) +
                                                     ((sizeof(GCtl) + 15) & ~size_t(15)));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int M = a.M, E = a.E, H = a.H, HS = H / kRouterCluster, R = M * a.k;
    const RouterSplit sp = router_split(H, E);
    const bool router = (int)blockIdx.x < sp.NR;

    // routing scratch inside the ring (no stage is in use yet)
    const SmallRouteScratch sc = small_route_scratch(stages, M, H, E);

    if (threadIdx.x == 0) {
        prefetch_tensormap(&tm_gate);
        prefetch_tensormap(&tm_up);
        prefetch_tensormap(&tm_down);
    }
    // full barriers: the producer's expect_tx arrival and the row loader's arrival
    gemm_init<GS>(ctl, warp, 0, 2);
    // W_r never depends on the previous grid: the CTA's block is copied before the wait
    if (router) small_router_copy(a.w_router, sp, sc.w_s);
    pdl_wait();  // h, and the control region, come after the previous grid
    pdl_launch_dependents();

    // ---------------------------------------------------------------- 1. routing
    if (router) small_route_dots(a.h, M, H, E, a.partials, sp, sc);
    small_route_gather(a.partials, M, E, a.bias, sc.part_s, &ctl.abort, a.status);
    int my_id = -1;  // lane j of warp t: the expert of token t's slot j
    route_finalize_any<true>(sc.part_s, M, E, a.k, nullptr, !ctl.abort, 1,
                       [&](int i, int j, int id, float wt) {
                           st.ids[i * a.k + j] = id;
                           st.wts[i * a.k + j] = wt;
                           if (blockIdx.x == 0) {
                               a.topk_ids[(size_t)i * a.k + j] = id;
                               a.topk_wts[(size_t)i * a.k + j] = wt;
                           }
                           my_id = id;
                       });
    // The alignment of the (at most 32) routes -- the order of align_core: experts ascending,
    // routes ascending, each expert padded to a multiple of b with sentinels -- as the tile
    // plan the expert phase reads (CTA 0 writes it out as the workspace's alignment later).
    if (M == 1) {
        // One token: its valid experts are distinct, one route each padded to b rows, so slot
        // j's tile is the rank of its expert among the token's valid experts, taken from the
        // ids warp 0 still holds (lane j: slot j).
        if (warp == 0) {
            const bool valid = lane < a.k && my_id >= 0 && my_id < E;
            const unsigned vmask = __ballot_sync(0xffffffffu, valid);
            int rank = 0;
#pragma unroll
            for (int q = 0; q < 32; ++q) {
                const int eq = __shfl_sync(0xffffffffu, my_id, q);
                rank += ((vmask >> q) & 1u) && eq < my_id ? 1 : 0;
            }
            if (valid) {
                st.tile_e[rank] = my_id;
                st.tile_n[rank] = 1;
                st.tile_r[rank][0] = lane;
            }
            if (lane == 0) st.ntiles = st.nvalid[0] = __popc(vmask);
        }
    } else {
        __syncthreads();
        // In one warp, lane r holding route r: the lanes of one expert find each other
        // (match), and a route's row is the padded rows of the experts below its own plus the
        // routes of its expert before it.
        if (warp == 0) {
            const int b = a.b;
            const int e = lane < R ? st.ids[lane] : -1;
            const bool valid = lane < R && e >= 0 && e < E;
            const unsigned peers = __match_any_sync(0xffffffffu, valid ? e : -1);
            const int lower = __popc(peers & ((1u << lane) - 1u));
            const int n = __popc(peers);
            const bool leader = valid && lower == 0;
            const int ntile = leader ? (n + b - 1) / b : 0;  // tiles of this lane's expert
            int tile_off = 0, total = 0;
#pragma unroll
            for (int q = 0; q < 32; ++q) {
                const int eq = __shfl_sync(0xffffffffu, e, q);
                const int tq = __shfl_sync(0xffffffffu, ntile, q);
                total += tq;
                if (tq != 0 && eq < e) tile_off += tq;
            }
            if (valid) st.tile_r[tile_off + lower / b][lower % b] = lane;  // lower % b < M
            if (leader)
                for (int q = 0; q < ntile; ++q) {
                    st.tile_e[tile_off + q] = e;
                    st.tile_n[tile_off + q] = min(b, n - q * b);
                }
            if (lane == 0) st.ntiles = total;
        }
        if (threadIdx.x < M) {
            int n = 0;
            for (int j = 0; j < a.k; ++j) {
                const int e = st.ids[threadIdx.x * a.k + j];
                n += (e >= 0 && e < E) ? 1 : 0;
            }
            st.nvalid[threadIdx.x] = n;
        }
    }
    __syncthreads();
    const int ntiles = st.ntiles;

    // ---------------------------------------------------------------- 2. experts
    SmallUnits f;
    f.n_gu = a.I / 64;
    f.n_dn = H / kGM;
    f.nks_gu = H / GS::kK;
    f.nks_dn = a.I / GS::kK;
    f.Tgu = (int64_t)ntiles * f.n_gu;
    f.T = f.Tgu + (int64_t)ntiles * f.n_dn;
    if (warp == 0) {
        if (lane == 0) small_producer(a, ctl, stages, st, f, &tm_gate, &tm_up, &tm_down);
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) small_mma(ctl, stages, f);
        __syncwarp();
    } else if (warp == kSLoaderWarp) {
        small_loader(a, ctl, stages, st, f);
    } else if (warp == kSLoaderWarp + 1) {
        if (blockIdx.x == 0) small_write_alignment(a, st, R);
    } else if (warp >= 2 && warp < 6) {  // the epilogue warps (warps 7.. only helped to route)
        const int quad = warp & 3;
        const int row = 32 * quad + lane;  // accumulator row: channel of the unit
        int32_t *done = a.ctl + kSmallCtlReady + a.ntiles_cap;
        int local = 0;
        for (int64_t u = blockIdx.x; u < f.T; u += gridDim.x, ++local) {
            bool gu;
            int tile, ct, nks;
            f.at(u, gu, tile, ct, nks);
            const int buf = local & 1;
            const int nrow = st.tile_n[tile];
            const bool ok_u = gwait(&ctl.tfull[buf], (uint32_t)(local >> 1) & 1u, ctl);
            if (named_bar_or(1, 128, !ok_u)) break;
            float v[16];
            drain_accumulator<16>(ctl, quad, buf, v);
            if (gu) {
                if (quad < 2) {
#pragma unroll
                    for (int n = 0; n < kSmallMaxTokens; ++n)
                        if (n < nrow) gbuf[n * 64 + row] = v[n];
                }
                named_bar_sync(1, 128);
                if (quad >= 2) {
                    const int ch = row - 64;
#pragma unroll
                    for (int n = 0; n < kSmallMaxTokens; ++n) {
                        if (n >= nrow) break;
                        const float pv = silu_f32(gbuf[n * 64 + ch]) * v[n];
                        a.p_rows[(size_t)st.tile_r[tile][n] * a.I + ct * 64 + ch] = __float2bfloat16(pv);
                    }
                }
                named_bar_sync(1, 128);
                if (threadIdx.x == 64) red_release_gpu_add(a.ctl + kSmallCtlReady + tile, 1);
            } else {
#pragma unroll
                for (int n = 0; n < kSmallMaxTokens; ++n)
                    if (n < nrow) a.y[(size_t)st.tile_r[tile][n] * H + ct * kGM + row] = v[n];
                named_bar_sync(1, 128);
                // row n's count is taken by thread 64 + n (the rows' tokens are distinct: a
                // token routes to an expert once); the one completing its token's valid
                // routes marks the token for the combine
                if (threadIdx.x >= 64 && threadIdx.x < 64 + nrow) {
                    const int n = threadIdx.x - 64;
                    const int m = st.tile_r[tile][n] / a.k;
                    const int old = atom_add_acq_rel_gpu(done + m * f.n_dn + ct, 1);
                    st.comb[n] = old + 1 == st.nvalid[m] ? m : -1;
                }
                named_bar_sync(1, 128);
                // out = bf16(residual + sum_j a_j y_j), valid slots in order (the combine)
                for (int c = 0; c < nrow; ++c) {
                    const int m = st.comb[c];
                    if (m < 0) continue;
                    const int col = ct * kGM + row;
                    float acc = 0.0f;
                    for (int j = 0; j < a.k; ++j) {
                        const int e = st.ids[m * a.k + j];
                        if (e < 0 || e >= E) continue;
                        acc = fmaf(st.wts[m * a.k + j], __ldcg(a.y + (size_t)(m * a.k + j) * H + col), acc);
                    }
                    const float res = a.residual ? __bfloat162float(a.residual[(size_t)m * H + col]) : 0.0f;
                    a.out[(size_t)m * H + col] = __float2bfloat16_rn(res + acc);
                }
            }
        }
    }
    gemm_finish<GS>(ctl, warp, a.status);

    // ---------------------------------------------------------------- exit: restore the region
    __syncthreads();
    if (threadIdx.x == 0) st.last = atom_add_acq_rel_gpu(a.ctl + kSmallCtlExit, 1) == (int)gridDim.x - 1;
    __syncthreads();
    if (st.last) {  // every CTA is done with the counters and the partials
        for (int i = threadIdx.x; i < a.ntiles_cap; i += blockDim.x) a.ctl[kSmallCtlReady + i] = 0;
        for (int i = threadIdx.x; i < M * (H / kGM); i += blockDim.x)
            a.ctl[kSmallCtlReady + a.ntiles_cap + i] = 0;
        for (int i = threadIdx.x; i < M * kRouterCluster * E / 4; i += blockDim.x)
            reinterpret_cast<uint4 *>(a.partials)[i] = make_uint4(0u, 0u, 0u, 0u);
        if (threadIdx.x == 0) a.ctl[kSmallCtlExit] = 0;
    }
}

// Dynamic shared memory: the ring (which also holds the routing scratch), the gate/up
// exchange buffer, the control block and the routing results.
static size_t small_smem_bytes() {
    const size_t ring = (size_t)GS::kStages * GS::kStageBytes;
    return 1024 + ring + 16 * 64 * 4 + ((sizeof(GCtl) + 15) & ~size_t(15)) + sizeof(SmallState);
}

bool small_fits(int M, int k, int E, int H, int b) {
    if (M < 1 || M > kSmallMaxTokens || (int64_t)M * k > kSmallMaxRoutes || b < 1 || b > 16)
        return false;
    if ((size_t)(H / kRouterCluster) * E * 2 > 64 * 1024) return false;  // one router pass
    const int64_t R = (int64_t)M * k;
    const int64_t cap = R + (R < E ? R : E) * (b - 1);
    if (small_routing_bytes(M, H, E) > (size_t)GS::kStages * GS::kStageBytes) return false;
    return small_smem_bytes() <= 227 * 1024 && (int64_t)M * (H / kGM) <= kSmallCtlDone &&
           cap / b <= kSmallMaxRoutes;
}

cudaError_t launch_decode_small(const CUtensorMap &tm_gate, const CUtensorMap &tm_up,
                                const CUtensorMap &tm_down, const SmallArgs &a,
                                cudaStream_t stream) {
    const size_t smem = small_smem_bytes();
    cudaError_t err = ensure_smem(reinterpret_cast<const void *>(decode_small_kernel), smem);
    if (err != cudaSuccess) return err;
    cudaLaunchAttribute attrs[2];
    cudaLaunchConfig_t cfg = launch_config(dim3(num_sms()), dim3(kSThreads), smem, stream, attrs, 0);
    return cudaLaunchKernelEx(&cfg, decode_small_kernel, tm_gate, tm_up, tm_down, a);
}

}  // namespace moe
