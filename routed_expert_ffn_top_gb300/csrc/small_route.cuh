// small_route.cuh -- the routing of the one-grid paths for one or two tokens (dense weights in
// decode_small.cu, VQ weights in gemv.cu): the router kernel's arithmetic spread over 64 CTAs,
// the partial logits exchanged through the workspace, and gathered by every CTA.
//
// "A Multi-Engine Dataflow for MoE Decoding on Scratchpad-Based Tensor Accelerators", MoE
// block background: the router scores the experts for h; the logits here are the router
// kernel's, bit for bit (route_core.cuh finalises them).
#pragma once

#include "moe_internal.cuh"
#include "ptx.cuh"

namespace moe {

// The router kernel's split of W_r: CTA q of its cluster holds slice q (HS = H/8 rows), cuts
// it into RG = 512 / (E/2) row groups (rows [rg*HS/RG, (rg+1)*HS/RG) of the slice) with one
// chain per (token, expert) and group, rows ascending, and adds the groups in order.  Here
// each slice is cut further by experts into C chunks of expert pairs, one CTA per (slice,
// chunk): every thread runs one (group, pair) chain of the router kernel, and the CTA adds
// the groups of its experts in the same order.  A CTA reads only its own block of W_r, and
// every CTA gathers 8 partials per token and expert, as after the router kernel.
struct RouterSplit {
    int HS, RG, npairs, C, NR;  // NR = 8 * C CTAs hold the router
    int q, p0, PC;              // this CTA's slice and pairs [p0, p0 + PC)
};
__device__ __forceinline__ RouterSplit router_split(int H, int E) {
    RouterSplit r;
    r.HS = H / kRouterCluster;
    r.npairs = E / 2;
    r.RG = router_row_groups(E);
    r.C = min(min(8, r.npairs), (int)gridDim.x / kRouterCluster);
    r.NR = kRouterCluster * r.C;
    const int c = (int)blockIdx.x % r.C;
    r.q = (int)blockIdx.x / r.C;
    r.p0 = c * r.npairs / r.C;
    r.PC = (c + 1) * r.npairs / r.C - r.p0;
    return r;
}

// Row group of slice row r (rows [g*HS/RG, (g+1)*HS/RG) form group g).
__device__ __forceinline__ int router_group_of(int r, int HS, int RG) {
    return ((r + 1) * RG + HS - 1) / HS - 1;
}

// Copies this CTA's block of W_r (the slice's HS rows, pairs [p0, p0 + PC)) into w_s as rows
// of PC bf16 pairs, one empty row after each row group: the threads of a warp read the same
// row of up to four groups at a time, and the shift puts them in different banks.
__device__ inline void small_router_copy(const __nv_bfloat16 *w_router, const RouterSplit &sp, uint32_t *w_s) {
    const uint32_t *w32 = reinterpret_cast<const uint32_t *>(w_router) +
                          (size_t)sp.q * sp.HS * sp.npairs + sp.p0;
    if (sp.PC % 4 == 0 && sp.p0 % 4 == 0) {  // 16-byte pieces
        const int per_row = sp.PC / 4;
        for (int i = threadIdx.x; i < sp.HS * per_row; i += blockDim.x) {
            const int r = i / per_row, j = i - r * per_row;
            cp_async_16(w_s + (size_t)(r + router_group_of(r, sp.HS, sp.RG)) * sp.PC + 4 * j,
                        w32 + (size_t)r * sp.npairs + 4 * j);
        }
    } else {
        for (int i = threadIdx.x; i < sp.HS * sp.PC; i += blockDim.x) {
            const int r = i / sp.PC, j = i - r * sp.PC;
            cp_async_4(w_s + (size_t)(r + router_group_of(r, sp.HS, sp.RG)) * sp.PC + j,
                       w32 + (size_t)r * sp.npairs + j);
        }
    }
}

// This CTA's partial logits: thread (group rg, pair pl) chains over the group's rows (one
// fused multiply-add per row) into red[(rg * TM + t) * 2PC + 2 pl (+1)]; then the groups of
// each (token, expert) added in order into partials[(q * M + t) * E + e].
template <int TM>
__device__ void small_router_chunk(float *partials, int E, const RouterSplit &sp,
                                   const uint32_t *w_s, const __nv_bfloat16 *x_s, float *red) {
    const int PC = sp.PC, HS = sp.HS, RG = sp.RG;
    const uint32_t *x32 = reinterpret_cast<const uint32_t *>(x_s);
    const int item = threadIdx.x;
    if (item < RG * PC) {
        const int rg = item / PC, pl = item - rg * PC;
        const uint32_t *wrow = w_s + (size_t)rg * PC + pl;  // row r at wrow[r * PC]
        const int r0 = rg * HS / RG, r1 = (rg + 1) * HS / RG;
        float acc0[TM], acc1[TM];
#pragma unroll
        for (int t = 0; t < TM; ++t) acc0[t] = acc1[t] = 0.0f;
        int r = r0;
        // eight rows per step: their weights and h pairs are all loaded before the first
        // multiply-add, which then run in row order
        for (; r + 7 < r1 && (r & 1) == 0; r += 8) {
            uint32_t w8[8], x4[TM][4];
#pragma unroll
            for (int u = 0; u < 8; ++u) w8[u] = wrow[(r + u) * PC];
#pragma unroll
            for (int t = 0; t < TM; ++t)
#pragma unroll
                for (int u = 0; u < 4; ++u) x4[t][u] = x32[(t * HS + r + 2 * u) >> 1];
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int t = 0; t < TM; ++t) {
                    acc0[t] = fma_bf16<0, 0>(x4[t][u], w8[2 * u], acc0[t]);
                    acc1[t] = fma_bf16<0, 1>(x4[t][u], w8[2 * u], acc1[t]);
                    acc0[t] = fma_bf16<1, 0>(x4[t][u], w8[2 * u + 1], acc0[t]);
                    acc1[t] = fma_bf16<1, 1>(x4[t][u], w8[2 * u + 1], acc1[t]);
                }
        }
        for (; r + 1 < r1 && (r & 1) == 0; r += 2) {
            const uint32_t wa = wrow[r * PC];
            const uint32_t wb = wrow[(r + 1) * PC];
#pragma unroll
            for (int t = 0; t < TM; ++t) {
                const uint32_t xv = x32[(t * HS + r) >> 1];
                acc0[t] = fma_bf16<0, 0>(xv, wa, acc0[t]);
                acc1[t] = fma_bf16<0, 1>(xv, wa, acc1[t]);
                acc0[t] = fma_bf16<1, 0>(xv, wb, acc0[t]);
                acc1[t] = fma_bf16<1, 1>(xv, wb, acc1[t]);
            }
        }
        for (; r < r1; ++r) {  // an odd row at either end of a group
            const uint32_t wa = wrow[r * PC];
#pragma unroll
            for (int t = 0; t < TM; ++t) {
                const uint32_t xv = x32[(t * HS + r) >> 1];
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
            red[((size_t)rg * TM + t) * 2 * PC + 2 * pl] = acc0[t];
            red[((size_t)rg * TM + t) * 2 * PC + 2 * pl + 1] = acc1[t];
        }
    }
    __syncthreads();
    // stored complemented: arithmetic never produces the all-ones NaN (NaN results are the
    // canonical 0x7fffffff), so a zero word means "not written yet" to the readers
    uint32_t *dst = reinterpret_cast<uint32_t *>(partials);
    for (int idx = threadIdx.x; idx < TM * 2 * PC; idx += blockDim.x) {
        float s = red[idx];
        for (int g = 1; g < RG; ++g) s += red[(size_t)g * TM * 2 * PC + idx];
        const int t = idx / (2 * PC), el = idx - t * 2 * PC;
        dst[((size_t)sp.q * TM + t) * E + 2 * sp.p0 + el] = ~__float_as_uint(s);
    }
}

// Shared-memory bytes the routing carves out of the one-grid kernels' rings (before any stage
// is used): the CTA's block of W_r (a slice's rows, one padding row per row group, at most all
// E columns), the slice's h rows, the row-group sums, and the 8 partials of every token.
__host__ __device__ constexpr size_t small_routing_bytes(int M, int H, int E) {
    return (size_t)(H / kRouterCluster + router_row_groups(E)) * E * 2 + 16 +  // W_r block
           (size_t)M * (H / kRouterCluster) * 2 + 16 +                           // h rows
           (size_t)router_row_groups(E) * M * E * 4 + 16 +                       // group sums
           (size_t)M * kRouterCluster * E * 4 + 16;                              // partials
}

// Where the routing scratch lies in `p` (shared memory, 16-byte aligned).
struct SmallRouteScratch {
    uint32_t *w_s;
    __nv_bfloat16 *x_s;
    float *red, *part_s;  // part_s [M][E]: the gathered logits (room for [M][8][E])
};
__device__ __forceinline__ SmallRouteScratch small_route_scratch(unsigned char *p, int M, int H,
                                                                 int E) {
    SmallRouteScratch r;
    const int HS = H / kRouterCluster, RG = router_row_groups(E);
    r.w_s = reinterpret_cast<uint32_t *>(p);
    p += ((size_t)(HS + RG) * E * 2 + 15) & ~size_t(15);
    r.x_s = reinterpret_cast<__nv_bfloat16 *>(p);
    p += ((size_t)M * HS * 2 + 15) & ~size_t(15);
    r.red = reinterpret_cast<float *>(p);
    p += ((size_t)RG * M * E * 4 + 15) & ~size_t(15);
    r.part_s = reinterpret_cast<float *>(p);
    return r;
}

// After the dependency wait, in a router CTA (every thread; the CTA's block of W_r was
// copied before the wait): the slice's h rows, then the partial logits of the CTA's experts,
// published complemented in `partials`.
__device__ inline void small_route_dots(const __nv_bfloat16 *h, int M, int H, int E, float *partials,
                                 const RouterSplit &sp, const SmallRouteScratch &sc) {
    const int HS = H / kRouterCluster;
    for (int idx = threadIdx.x; idx < M * (HS / 8); idx += blockDim.x) {
        const int t = idx / (HS / 8), pc = idx - t * (HS / 8);
        *reinterpret_cast<uint4 *>(sc.x_s + (size_t)t * HS + pc * 8) =
            *reinterpret_cast<const uint4 *>(h + (size_t)t * H + (size_t)sp.q * HS + pc * 8);
    }
    cp_async_wait_all();
    __syncthreads();
    if (M == 1)
        small_router_chunk<1>(partials, E, sp, sc.w_s, sc.x_s, sc.red);
    else
        small_router_chunk<2>(partials, E, sp, sc.w_s, sc.x_s, sc.red);
}

// Every CTA: the logits of every token from the 8 slices' partials, polled where they lie.
// Thread t < M * E/4 takes token t / (E/4) and experts 4 (t % (E/4)) .. +3: its 8 slices'
// loads all in flight at once, reloaded until no word is zero (not written yet), then each
// logit summed in slice order from zero and the bias added -- the router kernel's order --
// into logits [M][E].  A wait past the limit sets *abort and MOE_DEV_WAIT_TIMEOUT.  Ends
// with a barrier.
__device__ inline void small_route_gather(const float *partials, int M, int E, const float *bias,
                                          float *logits, volatile int *abort, int32_t *status) {
    const int e4n = E / 4;
    const int t = threadIdx.x;
    if (t < M * e4n) {
        const int m = t / e4n, e4 = t - m * e4n;
        const uint4 *src = reinterpret_cast<const uint4 *>(partials);
        uint4 v[kRouterCluster];
        unsigned pending = 0;
#pragma unroll
        for (int q = 0; q < kRouterCluster; ++q) {
            v[q] = __ldcg(src + ((size_t)q * M + m) * e4n + e4);
            pending |= 1u << q;
        }
        const uint64_t t0 = globaltimer_ns();
        while (true) {
#pragma unroll
            for (int q = 0; q < kRouterCluster; ++q)
                if ((pending >> q) & 1u)
                    if (v[q].x != 0u && v[q].y != 0u && v[q].z != 0u && v[q].w != 0u)
                        pending &= ~(1u << q);
            if (pending == 0u || *abort) break;
            if (globaltimer_ns() - t0 > kWaitLimitNs) {
                *abort = 1;
                atomicOr(status, MOE_DEV_WAIT_TIMEOUT);
                break;
            }
            __nanosleep(32);
#pragma unroll
            for (int q = 0; q < kRouterCluster; ++q)
                if ((pending >> q) & 1u) v[q] = __ldcg(src + ((size_t)q * M + m) * e4n + e4);
        }
        float l[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int q = 0; q < kRouterCluster; ++q) {
            l[0] += __uint_as_float(~v[q].x);
            l[1] += __uint_as_float(~v[q].y);
            l[2] += __uint_as_float(~v[q].z);
            l[3] += __uint_as_float(~v[q].w);
        }
        if (bias)
#pragma unroll
            for (int c = 0; c < 4; ++c) l[c] += bias[4 * e4 + c];
        *reinterpret_cast<float4 *>(logits + (size_t)m * E + 4 * e4) = make_float4(l[0], l[1], l[2], l[3]);
    }
    __syncthreads();
}

}  // namespace moe
