// align_core.cuh -- the stable alignment as a device function for one 256-thread CTA, shared
// by the stand-alone alignment kernel and the router (which runs it when one cluster holds
// every token).
//
// "Route-Block Membership Selects Packed-AWQ Arithmetic", Section 2.1: route r = m*k + j;
// valid routes grouped by expert, each expert padded to a multiple of b, and a parallel
// expert-per-block vector.  Section 5.3: valid routes ordered by (expert id, route id).
//
// (1) per-expert counts in shared memory (integer atomics commute, so the counts do not
// depend on arrival order); (2) one warp scans the padded counts into row offsets; (3) the
// routes are scattered chunk by chunk in ascending r: inside a warp __match_any_sync groups
// the lanes of one expert and a popcount of the lower lanes ranks them, a per-warp count
// table ranks the warps of a chunk, and per-expert running totals carry ranks across chunks;
// (4) padding rows, the block vector, the tail, and the sub-block records (expert, routes in
// row order, their tokens) that the expert kernels read one per tile.  Every position is a
// pure function of the input ids.
#pragma once

#include "moe_internal.cuh"

namespace moe {

constexpr int kAlignThreads = 256;
constexpr int kAlignWarps = kAlignThreads / 32;
// The stand-alone alignment works in shared memory (ids, aligned rows, block vector) when
// they fit in kAlignSmemBytes.
constexpr int kAlignStagedRoutes = 32768;
constexpr int kAlignSmemBytes = 200 * 1024;

// Shared-memory ints align_core needs for E experts, in a CTA of kThreads threads.
template <int kThreads = kAlignThreads>
__host__ __device__ constexpr int align_smem_ints(int E) { return (3 + kThreads / 32) * E + 4; }

// ids: M*k expert ids (global or shared memory); outputs may be NULL except npad.
// Requires blockDim.x == kThreads and every thread of the CTA to call it.  The positions do
// not depend on kThreads (a route's rank counts the routes of its expert before it, however
// the chunks are cut).
// n rounded up to a multiple of b (mask arithmetic when b is a power of two).
__device__ __forceinline__ int pad_to(int n, int b) {
    return (b & (b - 1)) == 0 ? (n + b - 1) & ~(b - 1) : (n + b - 1) / b * b;
}

template <int kThreads = kAlignThreads>
__device__ inline void align_core(const int32_t *ids, int64_t R, int k, int E, int b, int rsub,
                                  int32_t *sorted, int32_t *blocks, int32_t *npad, int64_t cap,
                                  SubBlock *sbt, int32_t *status, int32_t *sm) {
    constexpr int kWarps = kThreads / 32;
    int32_t *cnt = sm;                          // [E]
    int32_t *off = cnt + E;                     // [E] padded row offsets
    int32_t *running = off + E;                 // [E]
    int32_t *warp_cnt = running + E;            // [kWarps][E]
    int32_t *misc = warp_cnt + kWarps * E;      // [0] total, [1] invalid flag
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int32_t sentinel = (int32_t)R;

    for (int i = tid; i < (3 + kWarps) * E; i += kThreads) sm[i] = 0;
    if (tid == 0) misc[1] = 0;
    __syncthreads();

    // (1) counts
    int local_invalid = 0;
    for (int64_t r = tid; r < R; r += kThreads) {
        const int e = ids[r];
        if (e >= 0 && e < E)
            atomicAdd(&cnt[e], 1);
        else
            local_invalid = 1;
    }
    if (local_invalid) atomicOr(&misc[1], 1);
    __syncthreads();

    // (2) exclusive scan of padded counts (warp 0; lane owns a contiguous run of experts)
    if (warp == 0) {
        const int per = (E + 31) / 32;
        const int e0 = lane * per, e1 = min(E, e0 + per);
        int s = 0;
        for (int e = e0; e < e1; ++e) s += pad_to(cnt[e], b);
        int incl = s;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        int run = incl - s;
        for (int e = e0; e < e1; ++e) {
            off[e] = run;
            run += pad_to(cnt[e], b);
        }
        if (lane == 31) misc[0] = incl;
    }
    __syncthreads();
    const int total = misc[0];
    // Every row starts as a sentinel (coalesced, all threads); the scatter below overwrites
    // the rows of valid routes, so the padding rows and the tail need no per-expert loops.
    if (sorted) {
        for (int64_t pos = tid; pos < cap; pos += kThreads) sorted[pos] = sentinel;
        __syncthreads();
    }

    // (3) stable scatter in ascending route id
    const unsigned lt_mask = (1u << lane) - 1u;
    for (int64_t base = 0; base < R; base += kThreads) {
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
            int w = 0;
            for (; w + 4 <= warp; w += 4)  // four counts loaded before they are added
                rank += warp_cnt[w * E + e] + warp_cnt[(w + 1) * E + e] +
                        warp_cnt[(w + 2) * E + e] + warp_cnt[(w + 3) * E + e];
            for (; w < warp; ++w) rank += warp_cnt[w * E + e];
            const int64_t pos = (int64_t)off[e] + rank;
            if (pos < cap) {
                if (sorted) sorted[pos] = (int32_t)r;
                if (sbt) {
                    SubBlock *rec = sbt + pos / rsub;
                    rec->routes[pos % rsub] = (int32_t)r;
                    rec->tokens[pos % rsub] = (int32_t)(r / k);
                }
            }
        }
        __syncthreads();
        if (valid && leader) {
            // several warps may hold routes of expert e: integer adds commute
            atomicAdd(&running[e], wcount);
            warp_cnt[warp * E + e] = 0;
        }
        __syncthreads();
    }

    // (4) block vector, sub-block records, tail of the block vector
    for (int e = tid; e < E; e += kThreads) {
        const int n = cnt[e];
        if (n == 0) continue;
        const int padded = pad_to(n, b);
        if (blocks)
            for (int q = 0; q < padded / b; ++q) blocks[off[e] / b + q] = e;
        if (sbt)
            for (int s = off[e] / rsub; s < (off[e] + padded) / rsub; ++s) {
                const int first = s * rsub - off[e];
                const int ntok = max(0, min(rsub, n - first));
                SubBlock *rec = sbt + s;
                rec->e = e;
                rec->ntok = ntok;
                for (int q = ntok; q < kNT; ++q) rec->routes[q] = rec->tokens[q] = -1;
            }
    }
    if (blocks)
        for (int64_t q = (int64_t)total / b + tid; q < cap / b; q += kThreads) blocks[q] = -1;
    if (tid == 0) {
        npad[0] = total;
        if (status && misc[1]) atomicOr(status, MOE_DEV_INVALID_EXPERT);
    }
}

// The same alignment for at most 256 routes (and at most blockDim.x) whose ids are already in shared
// memory, with one thread per route and no per-expert tables: thread r counts the routes of
// its expert (n_e) and those of them before r, the first route of each expert publishes
// ceil(n_e / b) * b, and the padded offset of an expert is the sum published by the experts
// below it.  Positions, padding, block vector, sub-block records and tail are the same
// function of the ids as in align_core.  Every output may be NULL; pos_out (shared memory,
// R entries) receives each route's aligned row, -1 for an invalid route.
__host__ __device__ constexpr int align_small_smem_ints(int nthreads) { return nthreads + 4; }

__device__ inline void align_small(const int32_t *ids, int R, int k, int E, int b, int rsub,
                                   int32_t *sorted, int32_t *blocks, int32_t *npad, int64_t cap,
                                   SubBlock *sbt, int32_t *status, int32_t *sm,
                                   int32_t *pos_out = nullptr) {
    int32_t *pub = sm;  // [blockDim.x] padded count published by each expert's first route
    const int nthr = blockDim.x;
    const int tid = threadIdx.x;
    const int32_t sentinel = R;
    int e = -1, n = 0, lower = 0;
    bool valid = false;
    if (tid < R) {
        e = ids[tid];
        valid = e >= 0 && e < E;
        if (valid)
            for (int q0 = 0; q0 < R; q0 += 8) {  // eight ids loaded before they are compared
                int iq[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) iq[u] = q0 + u < R ? ids[q0 + u] : -1;
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    if (iq[u] == e && q0 + u < R) {
                        ++n;
                        lower += q0 + u < tid;
                    }
            }
    }
    const int padded = valid ? pad_to(n, b) : 0;
    const bool leader = valid && lower == 0;
    pub[tid] = leader ? padded : 0;
    // every row starts as a sentinel; the routes' rows are written after the barrier
    if (sorted)
        for (int64_t pos = tid; pos < cap; pos += nthr) sorted[pos] = sentinel;
    const int any_invalid = __syncthreads_or(tid < R && !valid);

    int off = 0, total = 0;
    for (int q0 = 0; q0 < R; q0 += 8) {  // eight entries loaded before they are added
        int pq[8], iq[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            pq[u] = q0 + u < R ? pub[q0 + u] : 0;
            iq[u] = q0 + u < R ? ids[q0 + u] : 0;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            total += pq[u];
            if (pq[u] != 0 && iq[u] < e) off += pq[u];
        }
    }
    if (pos_out && tid < R) pos_out[tid] = (valid && off + lower < cap) ? off + lower : -1;
    if (valid) {
        const int64_t pos = (int64_t)off + lower;
        if (pos < cap) {
            if (sorted) sorted[pos] = tid;
            if (sbt) {
                SubBlock *rec = sbt + pos / rsub;
                rec->routes[pos % rsub] = tid;
                rec->tokens[pos % rsub] = tid / k;
            }
        }
    }
    if (leader) {
        if (blocks)
            for (int q = 0; q < padded / b; ++q) blocks[off / b + q] = e;
        if (sbt)
            for (int s = off / rsub; s < (off + padded) / rsub; ++s) {
                const int first = s * rsub - off;
                const int ntok = max(0, min(rsub, n - first));
                SubBlock *rec = sbt + s;
                rec->e = e;
                rec->ntok = ntok;
                for (int q = ntok; q < kNT; ++q) rec->routes[q] = rec->tokens[q] = -1;
            }
    }
    if (blocks)
        for (int64_t q = (int64_t)total / b + tid; q < cap / b; q += nthr) blocks[q] = -1;
    if (tid == 0) {
        if (npad) npad[0] = total;
        if (status && any_invalid) atomicOr(status, MOE_DEV_INVALID_EXPERT);
    }
}

}  // namespace moe
