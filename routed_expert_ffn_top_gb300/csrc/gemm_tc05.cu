// gemm_tc05.cu -- the expert projections of dense weights as grouped GEMMs on the
// fifth-generation tensor cores (tcgen05.mma, accumulators in tensor memory), at every
// batch size.
//
// The computation is the expert step of "A Multi-Engine Dataflow for MoE Decoding on
// Scratchpad-Based Tensor Accelerators" (stage-3 activation; Section 4.3), for the rows of
// the aligned blocks of "Route-Block Membership Selects Packed-AWQ Arithmetic" (Section
// 2.1): every block holds routes of one expert, so a block is a dense GEMM tile.  A block
// of b rows is cut into tiles of kN rows (kN = 16 for b <= 16, else 64; the MMA's N).
//
// Orientation ("swap AB"): the expert weights are the MMA's A operand (M = 128 output
// channels) and the tile's kN rows are the N side, so the weights stream through HBM once
// per tile and the routes ride along:
//   gate/up:  D[128][kN] = [W_gate[e][:, i0:i0+64] | W_up[e][:, i0:i0+64]]^T  x  X^T
//             (lanes 0-63 accumulate g, lanes 64-127 accumulate u, of channels i0..i0+63)
//   down:     D[128][kN] = W_down[e][:, h0:h0+128]^T  x  P^T
// A comes straight from the [E,H,I] / [E,I,H] weights: TMA boxes of 64 columns x 256 rows
// (32 KB) with 128-byte swizzle form the MN-major canonical layout, one 64-wide M half per
// box.  One SM's TMA unit keeps only a few copies in flight, so copies are made as large
// as the swizzled layout allows.
//
// B is read from "tiled" row buffers: for every tile, K is cut into 64-wide chunks and each
// chunk is stored as the K-major 128-byte-swizzle image of its kN rows (row n at n*128
// bytes, 16-byte piece j at (j ^ n%8)*16).  A stage of 256 K is then one contiguous bulk
// copy that lands in shared memory already in the MMA layout.
//   x tiles: the token rows of h, written per aligned row by gather_rows_kernel, or by the
//            router when one router cluster holds every token;
//   p tiles: p = SiLU(g) * u in bf16, written by the gate/up epilogue, read by down.
// Rows of padding, and tile rows past their block's b rows, are never given a route: their
// columns of D are independent of the others and are dropped by the epilogues, so whatever
// the memory holds there cannot reach a result.
//
// Per CTA (6 warps): warp 0 issues the copies, one thread of warp 1 issues the MMAs
// (K = 16 each) into one of two tensor-memory accumulators, and warps 2-5 drain the
// finished accumulator (a warp reads the TMEM lanes of its rank modulo 4).  Persistent CTAs
// take units (tile, channel tile) round-robin, channel tile fastest, so the units of one
// tile run side by side and share its row tiles in L2.
//
// Each output element is one K-ordered chain of MMAs into its accumulator: 16 K-steps per
// 256-row stage, stages in ascending K, whatever kN is.  A tcgen05 MMA's element does not
// depend on the other columns of B, on N or on its row of the tile (checked bitwise on this
// GPU for N = 16..64, column shifts and row rotations), so a route's bits do not depend on
// the grid, on M, on the other routes of its tile, on its block position or on kN.
#include "gemm_core.cuh"

namespace moe {

// The route of aligned row `pos` of a block of expert e, or -1 for padding and for a row
// whose route does not belong to e (flagged, then skipped like padding).
__device__ __forceinline__ int gemm_route(const GemmArgs &a, int64_t pos, int e, bool flag) {
    const int r = a.sorted[pos];
    if (r < 0 || r >= a.R) return -1;
    if (e < 0 || e >= a.E || a.ids[r] != e) {
        if (flag) atomicOr(a.status, MOE_DEV_BAD_ALIGNMENT);
        return -1;
    }
    return r;
}

// The block vector entry of this CTA's first unit (unit blockIdx.x), read before the unit
// count is known so that the two loads overlap; the index is clamped into the array and
// the value is used only when the unit exists.
// The expert of block blk, and whether the expert spans more than one tile (several tiles
// per block, or a neighbouring block of the same expert): then other units read the same
// weight boxes at about the same time, and the boxes stay in L2 at normal priority for them;
// weights read by one tile only are marked first to evict.
struct UnitExpert {
    int e;
    bool shared;
};
// With at most b tokens and distinct experts per token no expert fills two blocks, and the
// neighbours are not read.
__device__ __forceinline__ UnitExpert unit_expert(const GemmArgs &a, int64_t blk) {
    const int64_t nblk = a.cap / a.b;
    if (blk >= nblk) blk = nblk - 1;
    const int e = a.blocks[blk];
    if (a.tpb > 1) return {e, true};
    if (a.M <= a.b) return {e, false};
    const int before = blk > 0 ? a.blocks[blk - 1] : -1;
    const int after = blk + 1 < nblk ? a.blocks[blk + 1] : -1;
    return {e, before == e || after == e};
}

__device__ __forceinline__ UnitExpert first_unit_expert(const GemmArgs &a, int n_ct) {
    return unit_expert(a, ((int64_t)blockIdx.x / n_ct) / a.tpb);
}

__device__ __forceinline__ int64_t gemm_blocks(const GemmArgs &a) {
    const int64_t n = a.npad[0] / a.b;
    const int64_t cap_blocks = a.cap / a.b;
    return n < 0 ? 0 : (n > cap_blocks ? cap_blocks : n);
}

// Aligned row held by row n of tile t, or -1 when that tile row lies past its block's b rows.
__device__ __forceinline__ int64_t tile_row(const GemmArgs &a, int64_t t, int n) {
    const int local = (int)(t % a.tpb) * a.kn + n;
    return local < a.b ? (t / a.tpb) * a.b + local : -1;
}

// The route of row n of tile t of expert e, or -1 (past the block, padding, or flagged).
__device__ __forceinline__ int tile_route(const GemmArgs &a, int64_t t, int n, int e, bool flag) {
    const int64_t pos = tile_row(a, t, n);
    return pos < 0 ? -1 : gemm_route(a, pos, e, flag);
}

// ------------------------------------------------------------------------ row gather
// x tiles of every valid aligned row: one warp per row, 8 lanes per 64-wide K chunk.
__global__ void __launch_bounds__(256) gather_rows_kernel(const GemmArgs a) {
    pdl_wait();
    pdl_launch_dependents();
    if (blockIdx.x == 0) zero_counts(a.ready, a.nready);  // the fused grid's, read after this grid
    const int lane = threadIdx.x & 31;
    const int64_t nrows = gemm_blocks(a) * a.b;
    const int nchunk = a.H / 64;
    const int64_t chunk_bytes = (int64_t)a.kn * 128;
    const int64_t warp0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t pos = warp0; pos < nrows; pos += nwarps) {
        const int64_t blk = pos / a.b;
        const int local = (int)(pos % a.b);
        const int64_t t = blk * a.tpb + local / a.kn;
        const int n = local % a.kn;
        const int r = gemm_route(a, pos, a.blocks[blk], lane == 0);
        if (r < 0) continue;
        const uint4 *src = reinterpret_cast<const uint4 *>(a.x + (int64_t)(r / a.k) * a.H);
        unsigned char *dst = reinterpret_cast<unsigned char *>(a.x_tiles) + t * nchunk * chunk_bytes;
        const int j = lane & 7;
        const uint32_t off = tile_offset(n, j);
        // 8 pieces per lane in flight at once (chunks c, c+4, ..., c+28), then their stores
        for (int c0 = lane >> 3; c0 < nchunk; c0 += 32) {
            uint4 v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (c0 + 4 * i < nchunk) v[i] = src[(c0 + 4 * i) * 8 + j];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (c0 + 4 * i < nchunk)
                    *reinterpret_cast<uint4 *>(dst + (int64_t)(c0 + 4 * i) * chunk_bytes + off) = v[i];
        }
    }
}

// ------------------------------------------------------------------- pipeline roles
// Copies of one unit (tile, channel tile): per stage the two 32 KB weight boxes (issue_a)
// and the tile's K slice of rows (btiles + (tile * nks + s) * kBBytes).  After a row
// gather the weights depend only on the alignment, which was complete before this grid
// started; the row tiles are written by the previous grid, so the first stages' tile
// copies wait for it (griddepcontrol) while their weight copies are already in flight.
// already_waited: the kernel waited for the previous grid before this point (the gate/up
// kernel when the router wrote the alignment and the x tiles).
template <typename G, typename IssueA>
__device__ void gemm_producer(const GemmArgs &a, GCtl &ctl, unsigned char *stages,
                              const unsigned char *btiles, int64_t T, int n_ct, int nks,
                              bool already_waited, int e_first, IssueA issue_a) {
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued = 0, parity_bits = 0;
    bool waited = already_waited;
    int npend = 0;
    const unsigned char *pend_src[G::kStages];
    int pend_stage[G::kStages];
    for (int64_t u = blockIdx.x; u < T && !ctl.abort; u += gridDim.x) {
        const int64_t tile = u / n_ct;
        const int ct = (int)(u % n_ct);
        int e = u == (int64_t)blockIdx.x ? e_first : a.blocks[tile / a.tpb];
        if (e < 0 || e >= a.E) {
            atomicOr(a.status, MOE_DEV_BAD_ALIGNMENT);
            e = 0;  // keep the pipeline in step; every row of such a block is dropped
        }
        for (int s = 0; s < nks; ++s) {
            if (!gwait(&ctl.empty[stage], phase ^ 1u, ctl)) break;
            uint64_t *bar = &ctl.full[stage];
            unsigned char *st = stages + stage * G::kStageBytes;
            if (G::kSplitB) {
                mbar_arrive_expect_tx(bar, G::kTxBytes - G::kBBytes);
                mbar_arrive_expect_tx(&ctl.bfull[stage], G::kBBytes);
            } else {
                mbar_arrive_expect_tx(bar, G::kTxBytes);
            }
            issue_a(st, bar, e, ct, s);
            const unsigned char *src = btiles + (tile * nks + s) * (int64_t)G::kBBytes;
            if (waited) {
                bulk_load(st + G::kBOff, src, G::kBBytes, G::kSplitB ? &ctl.bfull[stage] : bar);
            } else {
                pend_src[npend] = src;
                pend_stage[npend] = stage;
                if (++npend == G::kDefer) {
                    pdl_wait();
                    waited = true;
                    for (int q = 0; q < npend; ++q)
                        bulk_load(stages + pend_stage[q] * G::kStageBytes + G::kBOff, pend_src[q],
                                  G::kBBytes, G::kSplitB ? &ctl.bfull[pend_stage[q]] : &ctl.full[pend_stage[q]]);
                    npend = 0;
                }
            }
            issued |= 1u << stage;
            parity_bits = (parity_bits & ~(1u << stage)) | (phase << stage);
            gadvance<G>(stage, phase);
        }
    }
    if (!waited) {
        pdl_wait();
        for (int q = 0; q < npend; ++q)
            bulk_load(stages + pend_stage[q] * G::kStageBytes + G::kBOff, pend_src[q], G::kBBytes,
                      G::kSplitB ? &ctl.bfull[pend_stage[q]] : &ctl.full[pend_stage[q]]);
    }
    // every copy has landed before the CTA can exit
    for (int s = 0; s < G::kStages; ++s)
        if ((issued >> s) & 1u) {
            if (!mbar_wait_bounded(&ctl.full[s], (parity_bits >> s) & 1u)) ctl.abort = 1;
            if (G::kSplitB && !mbar_wait_bounded(&ctl.bfull[s], (parity_bits >> s) & 1u))
                ctl.abort = 1;
        }
}

// MMA issuer (one thread): for each unit, nks stages x 16 MMAs of K = 16 into accumulator
// buffer (unit parity); each stage is released when its MMAs complete.
template <typename G>
__device__ void gemm_mma(GCtl &ctl, unsigned char *stages, int64_t T, int nks) {
    constexpr int kN = G::kTileN;
    constexpr uint32_t idesc = umma_idesc_bf16(kGM, kN, true, false);
    int stage = 0;
    uint32_t phase = 0;
    int local = 0;
    for (int64_t u = blockIdx.x; u < T && !ctl.abort; u += gridDim.x, ++local) {
        const int buf = local & 1;
        const uint32_t tph = (uint32_t)(local >> 1) & 1u;
        if (!gwait(&ctl.tempty[buf], tph ^ 1u, ctl)) break;
        tc_fence_after();
        const uint32_t d = ctl.tmem + (uint32_t)(buf * kN);
        bool ok = true;
        for (int s = 0; s < nks; ++s) {
            if (!gwait(&ctl.full[stage], phase, ctl)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t A = smem_u32(stages + stage * G::kStageBytes);
            const uint32_t B = A + G::kBOff;
#pragma unroll
            for (int ks = 0; ks < G::kK / 16; ++ks) {
                // A: MN-major, M halves 32 KB apart, 8-row K atoms 1 KB apart, 16 K rows per MMA
                const uint64_t ad = umma_smem_desc(A + ks * 2048, G::kHalfBytes, 1024, 2);
                // B: K-major, 64-wide K chunks kChunkBytes apart, 32 bytes per K step, 8-row
                // atoms 1 KB apart
                const uint64_t bd =
                    umma_smem_desc(B + (ks >> 2) * G::kChunkBytes + (ks & 3) * 32, 16, 1024, 2);
                umma_bf16(d, ad, bd, idesc, s > 0 || ks > 0);
            }
            umma_commit(&ctl.empty[stage]);
            gadvance<G>(stage, phase);
        }
        if (!ok) break;
        umma_commit(&ctl.tfull[buf]);
    }
    // every issued MMA has completed before the CTA frees its tensor memory
    umma_commit(&ctl.done);
    if (!mbar_wait_bounded(&ctl.done, 0)) ctl.abort = 1;
}

// ------------------------------------------------------------- gate/up and down, one grid
// Dense weights run both projections in one persistent grid.  Units are numbered gate/up
// first -- (tile, 64-channel tile of I), u < Tgu -- then down -- (tile, 128-channel tile of H),
// v = u - Tgu -- and CTA c takes units c, c + G, c + 2G ... (G = grid size).  So every CTA
// runs all its gate/up units before its first down unit, and a down unit only ever waits for
// gate/up units, which wait for nothing but their own copies: with the CTAs resident (one per
// SM) no wait can close a cycle, and every wait is bounded in any case.
//
// A down unit's weight boxes do not depend on p, so the producer issues them as soon as ring
// slots free up, while other SMs still run gate/up (the overlap of the down-projection DMA
// with the gate/up computation in "A Multi-Engine Dataflow for MoE Decoding on
// Scratchpad-Based Tensor Accelerators", Section 4).  Only the unit's p slices wait: for the
// tile's ready count, to which every gate/up unit of the tile adds one (release, GPU scope)
// once its p is stored.  The count is zeroed by the kernel before this one (the one that
// wrote the x tiles), read with acquire, and followed by a proxy fence before the bulk copies
// of p, which go through the async proxy.
//
// Both unit kinds keep the arithmetic of the separate kernels: one K-ordered MMA chain per
// output element into its own accumulator column.
struct FusedShape {
    int64_t Tgu, T;            // gate/up units; all units
    int n_gu, n_dn;            // channel tiles per tile: I / 64 (gate/up), H / 128 (down)
    int nks_gu, nks_dn;        // 256-deep stages per unit
};

__device__ __forceinline__ FusedShape fused_shape(const GemmArgs &a, int kK) {
    FusedShape f;
    const int64_t tiles = gemm_blocks(a) * a.tpb;
    f.n_gu = a.I / 64;
    f.n_dn = a.H / kGM;
    f.nks_gu = a.H / kK;
    f.nks_dn = a.I / kK;
    f.Tgu = tiles * f.n_gu;
    f.T = f.Tgu + tiles * f.n_dn;
    return f;
}

struct FusedUnit {
    bool gu;
    int64_t tile;
    int ct, nks;
};

__device__ __forceinline__ FusedUnit fused_unit(const FusedShape &f, int64_t u) {
    FusedUnit x;
    x.gu = u < f.Tgu;
    const int64_t v = x.gu ? u : u - f.Tgu;
    const int n = x.gu ? f.n_gu : f.n_dn;
    x.tile = v / n;
    x.ct = (int)(v % n);
    x.nks = x.gu ? f.nks_gu : f.nks_dn;
    return x;
}

// Bounded wait until `need` gate/up units of `tile` have stored their p.
__device__ __forceinline__ bool tile_ready_wait(const int32_t *ready, int64_t tile, int need,
                                                GCtl &ctl) {
    if (ld_acquire_gpu(ready + tile) >= need) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (ld_acquire_gpu(ready + tile) >= need) return true;
        if (ctl.abort) return false;
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
            ctl.abort = 1;
            return false;
        }
    }
}

// Unit queue.  A CTA's first unit is unit blockIdx.x; each later one is taken from a grid-wide
// counter (units are handed out in increasing order, so every CTA runs its gate/up units
// before its down units and a down unit never waits behind a unit of its own CTA), which keeps
// the SMs busy to the end when units take different times.  The producer passes each unit to
// the MMA issuer and the epilogue warps through an 8-slot ring of unit ids in shared memory;
// -1 ends the sequence.
constexpr int kUQSlots = 8;
struct UnitQueue {
    uint64_t full[kUQSlots];   // the producer wrote the slot
    uint64_t empty[kUQSlots];  // the MMA thread and the 4 epilogue warps read it
    int64_t u[kUQSlots];
};

__device__ __forceinline__ void uq_init(UnitQueue &q) {
    for (int s = 0; s < kUQSlots; ++s) {
        mbar_init(&q.full[s], 1);
        mbar_init(&q.empty[s], 5);
    }
}

__device__ __forceinline__ bool uq_push(UnitQueue &q, GCtl &ctl, int i, int64_t u) {
    const int slot = i % kUQSlots;
    if (!gwait(&q.empty[slot], ((uint32_t)(i / kUQSlots) & 1u) ^ 1u, ctl)) return false;
    q.u[slot] = u;
    mbar_arrive(&q.full[slot]);
    return true;
}

// The i-th unit of this CTA, or -1 (the end, or a wait that gave up).
__device__ __forceinline__ int64_t uq_pop(UnitQueue &q, GCtl &ctl, int i) {
    const int slot = i % kUQSlots;
    if (!gwait(&q.full[slot], (uint32_t)(i / kUQSlots) & 1u, ctl)) return -1;
    return q.u[slot];
}

// Copy issuer.  Row-slice copies that cannot go yet are held (at most one ring of them):
// a gate/up unit's x slices until the previous grid is complete (they wait for griddepcontrol
// only after the first kDefer weight stages are in flight), a down unit's p slices until the
// tile's ready count is complete (they wait when the ring is full of the unit's stages, or at
// its last stage).  A gate/up slice never waits behind a down unit's readiness: held x slices
// are released before a down unit starts.  The next unit is taken from the counter once the
// previous grid is complete (it zeroes the counter) and while this unit's copies stream.
template <typename G>
__device__ void fused_producer(const GemmArgs &a, GCtl &ctl, UnitQueue &q, unsigned char *stages,
                               const FusedShape &f, UnitExpert first_gu,
                               const CUtensorMap *tm_gate, const CUtensorMap *tm_up,
                               const CUtensorMap *tm_down) {
    const uint64_t pol_once = policy_evict_first(), pol_shared = policy_evict_normal();
    // the row slices are read by every channel tile of their tile: kept before the weights
    const uint64_t pol_rows = policy_evict_last();
    const unsigned char *xt = reinterpret_cast<const unsigned char *>(a.x_tiles);
    const unsigned char *pt = reinterpret_cast<const unsigned char *>(a.p_tiles);
    int32_t *sched = a.ready + a.nready - 1;
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued = 0, parity_bits = 0;
    bool waited = a.wait_first != 0;
    int npend = 0;
    const unsigned char *pend_src[G::kStages];
    int pend_stage[G::kStages];
    auto release_held = [&]() {
        for (int qq = 0; qq < npend; ++qq)
            bulk_load_hint(stages + pend_stage[qq] * G::kStageBytes + G::kBOff, pend_src[qq],
                           G::kBBytes, &ctl.full[pend_stage[qq]], pol_rows);
        npend = 0;
    };
    bool stop = false;
    int i = 0;
    int64_t u = blockIdx.x;
    while (u < f.T && !stop && !ctl.abort) {
        if (!uq_push(q, ctl, i++, u)) break;
        const FusedUnit x = fused_unit(f, u);
        if (!x.gu && npend > 0) {  // x slices of earlier gate/up units still held
            if (!waited) pdl_wait();
            waited = true;
            release_held();
        }
        int64_t next = -1;
        if (waited) next = (int64_t)gridDim.x + atomicAdd(sched, 1);
        const UnitExpert ue =
            (u == (int64_t)blockIdx.x && x.gu) ? first_gu : unit_expert(a, x.tile / a.tpb);
        int e = ue.e;
        const uint64_t pol = ue.shared ? pol_shared : pol_once;
        if (e < 0 || e >= a.E) {
            atomicOr(a.status, MOE_DEV_BAD_ALIGNMENT);
            e = 0;  // keep the pipeline in step; every row of such a block is dropped
        }
        bool ready = x.gu;
        for (int s = 0; s < x.nks; ++s) {
            if (!gwait(&ctl.empty[stage], phase ^ 1u, ctl)) {
                stop = true;
                break;
            }
            uint64_t *bar = &ctl.full[stage];
            unsigned char *st = stages + stage * G::kStageBytes;
            mbar_arrive_expect_tx(bar, G::kTxBytes);
            if (x.gu) {
                const int32_t y = e * a.H + s * G::kK;
                tma_load_2d(st, tm_gate, x.ct * 64, y, bar, pol);
                tma_load_2d(st + G::kHalfBytes, tm_up, x.ct * 64, y, bar, pol);
            } else {
                const int32_t y = e * a.I + s * G::kK;
                tma_load_2d(st, tm_down, x.ct * kGM, y, bar, pol);
                tma_load_2d(st + G::kHalfBytes, tm_down, x.ct * kGM + 64, y, bar, pol);
            }
            const unsigned char *src = (x.gu ? xt : pt) + (x.tile * x.nks + s) * (int64_t)G::kBBytes;
            issued |= 1u << stage;
            parity_bits = (parity_bits & ~(1u << stage)) | (phase << stage);
            if (waited && ready) {
                bulk_load_hint(st + G::kBOff, src, G::kBBytes, bar, pol_rows);
            } else {
                pend_src[npend] = src;
                pend_stage[npend] = stage;
                ++npend;
            }
            gadvance<G>(stage, phase);
            const bool go = x.gu ? npend == G::kDefer
                                 : (npend > 0 && (npend == G::kStages || s == x.nks - 1));
            if (go) {
                if (!waited) pdl_wait();
                waited = true;
                if (!ready) {
                    if (!tile_ready_wait(a.ready, x.tile, f.n_gu, ctl)) {
                        stop = true;
                        break;
                    }
                    fence_proxy_async_global();
                    ready = true;
                }
                release_held();
            }
            if (waited && next < 0) next = (int64_t)gridDim.x + atomicAdd(sched, 1);
        }
        if (next < 0 && !stop) {
            if (!waited) pdl_wait();
            waited = true;
            release_held();
            next = (int64_t)gridDim.x + atomicAdd(sched, 1);
        }
        u = next;
    }
    uq_push(q, ctl, i, -1);  // the end (if this wait gives up, the consumers' own waits do too)
    // Held slices are copied even after an abort (their contents then no longer matter), so
    // that every stage's barrier completes and the drain below ends at once.
    if (npend > 0) {
        if (!waited) pdl_wait();
        release_held();
    }
    for (int s = 0; s < G::kStages; ++s)
        if ((issued >> s) & 1u)
            if (!mbar_wait_bounded(&ctl.full[s], (parity_bits >> s) & 1u)) ctl.abort = 1;
}

// MMA issuer (one thread): per unit its stages x 16 MMAs of K = 16 into the accumulator
// buffer of the unit's parity; each stage is released when its MMAs complete.
template <typename G>
__device__ void fused_mma(GCtl &ctl, UnitQueue &q, unsigned char *stages, const FusedShape &f) {
    constexpr int kN = G::kTileN;
    constexpr uint32_t idesc = umma_idesc_bf16(kGM, kN, true, false);
    int stage = 0;
    uint32_t phase = 0;
    for (int local = 0; !ctl.abort; ++local) {
        const int64_t u = uq_pop(q, ctl, local);
        mbar_arrive(&q.empty[local % kUQSlots]);
        if (u < 0) break;
        const int nks = fused_unit(f, u).nks;
        const int buf = local & 1;
        const uint32_t tph = (uint32_t)(local >> 1) & 1u;
        if (!gwait(&ctl.tempty[buf], tph ^ 1u, ctl)) break;
        tc_fence_after();
        const uint32_t d = ctl.tmem + (uint32_t)(buf * kN);
        bool ok = true;
        for (int s = 0; s < nks; ++s) {
            if (!gwait(&ctl.full[stage], phase, ctl)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t A = smem_u32(stages + stage * G::kStageBytes);
            const uint32_t B = A + G::kBOff;
#pragma unroll
            for (int ks = 0; ks < G::kK / 16; ++ks) {
                const uint64_t ad = umma_smem_desc(A + ks * 2048, G::kHalfBytes, 1024, 2);
                const uint64_t bd =
                    umma_smem_desc(B + (ks >> 2) * G::kChunkBytes + (ks & 3) * 32, 16, 1024, 2);
                umma_bf16(d, ad, bd, idesc, s > 0 || ks > 0);
            }
            umma_commit(&ctl.empty[stage]);
            gadvance<G>(stage, phase);
        }
        if (!ok) break;
        umma_commit(&ctl.tfull[buf]);
    }
    umma_commit(&ctl.done);
    if (!mbar_wait_bounded(&ctl.done, 0)) ctl.abort = 1;
}

template <int kN>
__global__ void __launch_bounds__(kGThreads, 1)
    gemm_fused_kernel(const __grid_constant__ CUtensorMap tm_gate,
                      const __grid_constant__ CUtensorMap tm_up,
                      const __grid_constant__ CUtensorMap tm_down, const GemmArgs a) {
    using G = GTile<kN>;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *base = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char *stages = base;
    float *gbuf = reinterpret_cast<float *>(base + G::kStages * G::kStageBytes);  // [kN][64]
    GCtl &ctl = *reinterpret_cast<GCtl *>(base + G::kStages * G::kStageBytes + kN * 64 * 4);
    UnitQueue &q = *reinterpret_cast<UnitQueue *>(reinterpret_cast<unsigned char *>(&ctl) +
                                                  ((sizeof(GCtl) + 15) & ~size_t(15)));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        prefetch_tensormap(&tm_gate);
        prefetch_tensormap(&tm_up);
        prefetch_tensormap(&tm_down);
        uq_init(q);  // made visible by gemm_init's fence and barrier
    }
    gemm_init<G>(ctl, warp);
    // When the previous kernel wrote the alignment (and the x tiles), wait for it before
    // anything reads them.  The next kernel (the combine) may start at once: it waits for
    // this grid before it reads anything.
    if (a.wait_first) pdl_wait();
    pdl_launch_dependents();

    // the expert of this CTA's first unit if it is a gate/up unit, read beside the unit count
    const int n_gu = a.I / 64;
    const UnitExpert first_gu = threadIdx.x == 0 ? first_unit_expert(a, n_gu) : UnitExpert{0, false};
    const FusedShape f = fused_shape(a, G::kK);

    if (warp == 0) {
        if (lane == 0) fused_producer<G>(a, ctl, q, stages, f, first_gu, &tm_gate, &tm_up, &tm_down);
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) fused_mma<G>(ctl, q, stages, f);
        __syncwarp();
    } else {
        const int quad = warp & 3;           // TMEM lanes [32 quad, 32 quad + 32)
        const int row = 32 * quad + lane;    // accumulator row (gate/up: gate < 64 <= up)
        // the ready counts were zeroed by the previous grid: add to them only after it is done
        if (!a.wait_first) pdl_wait();
        for (int local = 0;; ++local) {
            const int64_t u = uq_pop(q, ctl, local);
            __syncwarp();
            if (lane == 0) mbar_arrive(&q.empty[local % kUQSlots]);
            if (named_bar_or(1, 128, u < 0)) break;
            const FusedUnit x = fused_unit(f, u);
            const int buf = local & 1;
            // Only rows that hold a route get p (gate/up) or y (down); the other columns of
            // the tile are dropped.
            if (row < kN)
                ctl.route[buf][row] = tile_route(a, x.tile, row, a.blocks[x.tile / a.tpb], false);
            const bool ok = gwait(&ctl.tfull[buf], (uint32_t)(local >> 1) & 1u, ctl);
            if (named_bar_or(1, 128, !ok)) break;
            float v[kN];
            drain_accumulator<kN>(ctl, quad, buf, v);
            if (x.gu) {
                if (quad < 2) {
#pragma unroll
                    for (int n = 0; n < kN; ++n)
                        if (ctl.route[buf][n] >= 0) gbuf[n * 64 + row] = v[n];
                }
                named_bar_sync(1, 128);
                if (quad >= 2) {
                    // p of each route row straight into the tile's swizzled chunk: a warp's 32
                    // channels are four 16-byte pieces of the row
                    const int ch = row - 64;
                    unsigned char *dst = reinterpret_cast<unsigned char *>(a.p_tiles) +
                                         (x.tile * f.n_gu + x.ct) * (int64_t)G::kChunkBytes +
                                         (ch & 7) * 2;
#pragma unroll
                    for (int n = 0; n < kN; ++n) {
                        if (ctl.route[buf][n] < 0) continue;
                        const float p = silu_f32(gbuf[n * 64 + ch]) * v[n];
                        *reinterpret_cast<__nv_bfloat16 *>(dst + tile_offset(n, ch >> 3)) =
                            __float2bfloat16(p);
                    }
                    fence_proxy_async_global();  // read next through the async proxy
                }
                named_bar_sync(1, 128);
                if (threadIdx.x == 64) red_release_gpu_add(a.ready + x.tile, 1);
            } else {
                float *ybase = a.y + x.ct * kGM + row;
#pragma unroll
                for (int n = 0; n < kN; ++n) {
                    const int r = ctl.route[buf][n];
                    if (r >= 0) ybase[(int64_t)r * a.H] = v[n];
                }
            }
        }
    }
    gemm_finish<G>(ctl, warp, a.status);
}

// ---------------------------------------------------------------------- VQ gate/up
// Blockwise-VQ gate/up on the tensor cores (16-row tiles).  The weight operand never exists
// in memory: eight decoder warps, one per TMEM lane quadrant and projection (lane = output
// channel of the unit), read their channel's index of every index row q of a 64-row K slot
// from the stage's index box, fetch its code word B[J[q][i]] (kD consecutive K values of row
// i of the weight) from their own repeat of the code book, and write the words to the slot's
// columns with tcgen05.st, software-pipelined: the stores of slot k run while the words of
// slot k+1 are fetched.  The MMA issuer takes A from tensor memory and the row slice from
// the stage.  The chain per element is the dense kernel's (K-ordered, one MMA per 16 K
// rows).  The epilogue thread of a channel holds its gate and up accumulators and writes
// SiLU(g) * u to the p tiles.  14 warps: producer, MMA, 4 epilogue, 8 decoders.
//   Bounds measured on this GPU: an M = 128, K = 16 MMA issues in about 45 cycles for any N
// up to 64 (so the 32 MMAs of a 16-row unit's stage take about 0.7 us), and a warp's
// tcgen05.st with its wait costs about 200 cycles whatever its size; a unit's stage runs in
// about 1.6 us, decoding-bound.  Wider tiles cost the same MMA time per stage.
constexpr int kGVQThreads = 448;
constexpr int kGDecWarp0 = 6;

// Every lane waits; the warp goes on only if all of them got the phase (so that the
// warp-wide tensor-memory instructions after it are never split).
__device__ __forceinline__ bool gwait_warp(uint64_t *bar, uint32_t parity, GCtl &ctl) {
    return __all_sync(0xffffffffu, gwait(bar, parity, ctl));
}

template <int kD, int kN>
__device__ void gemm_mma_vq(GCtl &ctl, unsigned char *stages, int64_t T, int nks) {
    using G = GTileVQ<kD, kN>;
    constexpr uint32_t idesc = umma_idesc_bf16(kGM, kN, false, false);
    constexpr int kStepsPerSlot = G::kSlotK / 16;
    int stage = 0, slot = 0;
    uint32_t phase = 0, sphase = 0;
    int local = 0;
    for (int64_t u = blockIdx.x; u < T && !ctl.abort; u += gridDim.x, ++local) {
        const int buf = local & 1;
        const uint32_t tph = (uint32_t)(local >> 1) & 1u;
        if (!gwait(&ctl.tempty[buf], tph ^ 1u, ctl)) break;
        tc_fence_after();
        const uint32_t dg = ctl.tmem + (uint32_t)(buf * 2 * kN);  // gate, then up
        bool ok = true;
        for (int s = 0; s < nks && ok; ++s) {
            if (!gwait(&ctl.bfull[stage], phase, ctl)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t B = smem_u32(stages + stage * G::kStageBytes) + G::kBOff;
            for (int h = 0; h < G::kSlotsPerStage; ++h) {
                if (!gwait(&ctl.afull[slot], sphase, ctl)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t A = ctl.tmem + G::kSlotCol0 + (uint32_t)slot * G::kSlotCols;
#pragma unroll
                for (int kk = 0; kk < kStepsPerSlot; ++kk) {
                    const int ks = h * kStepsPerSlot + kk;  // K = 16 step within the stage
                    const uint64_t bd =
                        umma_smem_desc(B + (ks >> 2) * G::kChunkBytes + (ks & 3) * 32, 16, 1024, 2);
                    const bool acc = s > 0 || ks > 0;
                    umma_bf16_ts(dg, A + (uint32_t)(kk * 8), bd, idesc, acc);
                    umma_bf16_ts(dg + kN, A + 32 + (uint32_t)(kk * 8), bd, idesc, acc);
                }
                umma_commit(&ctl.aempty[slot]);
                if (++slot == G::kSlots) {
                    slot = 0;
                    sphase ^= 1u;
                }
            }
            if (!ok) break;
            umma_commit(&ctl.empty[stage]);
            gadvance<G>(stage, phase);
        }
        if (!ok) break;
        umma_commit(&ctl.tfull[buf]);
    }
    umma_commit(&ctl.done);
    if (!mbar_wait_bounded(&ctl.done, 0)) ctl.abort = 1;
}

// Decoder warp (TMEM lane quadrant `quad`, projection `p`): the weight operand of every
// stage, slot by slot.
template <int kD, int kN>
struct VQDecoder {
    using G = GTileVQ<kD, kN>;
    static constexpr int kRows = G::kSlotK / kD;  // index rows q per slot: 16 or 8
    GCtl &ctl;
    const unsigned char *jbase;  // this warp's index column in stage 0
    const unsigned char *cb;     // this lane's repeat of its projection's code book
    uint32_t taddr;              // this warp's lanes and columns in slot 0

    // Slot task k (stage k / 4 of the CTA's sequence, quarter k % 4 of its K): waits for the
    // stage's index boxes (first quarter) and for the slot to be free, then gathers the code
    // words of its rows into r; after the last quarter the stage's boxes are released.
    __device__ __forceinline__ bool fetch(int64_t k, uint32_t (&r)[32]) {
        const int64_t gs = k / G::kSlotsPerStage;
        const int h = (int)(k % G::kSlotsPerStage);
        const int stage = (int)(gs % G::kStages);
        if (h == 0 && !gwait_warp(&ctl.full[stage], (uint32_t)(gs / G::kStages) & 1u, ctl)) return false;
        if (!gwait_warp(&ctl.aempty[k % G::kSlots], ((uint32_t)(k / G::kSlots) & 1u) ^ 1u, ctl))
            return false;
        tc_fence_after();
        const unsigned char *jb = jbase + stage * G::kStageBytes + h * kRows * G::kCT;
        uint32_t idx[kRows];
#pragma unroll
        for (int q = 0; q < kRows; ++q) idx[q] = jb[q * G::kCT];
#pragma unroll
        for (int q = 0; q < kRows; ++q) {
            if constexpr (kD == 4) {
                const uint2 w = *reinterpret_cast<const uint2 *>(cb + idx[q] * G::kEntryBytes);
                r[2 * q] = w.x;
                r[2 * q + 1] = w.y;
            } else {
                const uint4 w = *reinterpret_cast<const uint4 *>(cb + idx[q] * G::kEntryBytes);
                r[4 * q] = w.x;
                r[4 * q + 1] = w.y;
                r[4 * q + 2] = w.z;
                r[4 * q + 3] = w.w;
            }
        }
        if (h == G::kSlotsPerStage - 1) {
            __syncwarp();
            if ((threadIdx.x & 31) == 0) mbar_arrive(&ctl.empty[stage]);  // its index boxes are read
        }
        return true;
    }
};

template <int kD, int kN>
__device__ void vq_decode(GCtl &ctl, const unsigned char *stages, const unsigned char *cbs,
                          int64_t T, int nks, int quad, int p, int lane) {
    using G = GTileVQ<kD, kN>;
    using Dec = VQDecoder<kD, kN>;
    const int ch = 32 * quad + lane;  // channel within the unit's 128
    Dec dec{ctl, stages + p * G::kJBytes + ch, cbs + p * G::kCbBytes + (lane % G::kReps) * (kD * 2),
            ctl.tmem + ((uint32_t)(32 * quad) << 16) + G::kSlotCol0 + (uint32_t)(32 * p)};
    const int64_t units = T > blockIdx.x ? (T - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    const int64_t K = units * nks * G::kSlotsPerStage;  // slot tasks of this CTA (even)
    // two register sets, swapped by unrolling by two (never indexed at run time)
    uint32_t r0[32], r1[32];
    auto step = [&](int64_t k, const uint32_t(&cur)[32], uint32_t(&next)[32]) {
        const uint32_t ta = dec.taddr + (uint32_t)(k % G::kSlots) * G::kSlotCols;
        tmem_st16(ta, cur);
        tmem_st16(ta + 16, cur + 16);
        const bool more = k + 1 < K && dec.fetch(k + 1, next);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl.afull[k % G::kSlots]);
        return more;
    };
    if (K == 0 || !dec.fetch(0, r0)) return;
    for (int64_t k = 0; k < K; k += 2)
        if (!step(k, r0, r1) || !step(k + 1, r1, r0)) return;
}

template <int kD, int kN>
__global__ void __launch_bounds__(kGVQThreads, 1)
    gemm_gateup_vq_kernel(const __grid_constant__ CUtensorMap tm_jgate,
                          const __grid_constant__ CUtensorMap tm_jup, const GemmArgs a) {
    using G = GTileVQ<kD, kN>;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *base = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char *stages = base;
    unsigned char *cbs = base + G::kStages * G::kStageBytes;  // gate then up code book
    GCtl &ctl = *reinterpret_cast<GCtl *>(cbs + 2 * G::kCbBytes);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        prefetch_tensormap(&tm_jgate);
        prefetch_tensormap(&tm_jup);
    }
    // the layer-shared code books (weights, not written by an earlier grid), each entry
    // repeated across one 128-byte row of banks
    constexpr int kPieces = 2 * G::kCbBytes / 16;
#pragma unroll 4
    for (int i = threadIdx.x; i < kPieces; i += blockDim.x) {
        const int p = i / (kPieces / 2);
        const int kappa = (i % (kPieces / 2)) / (G::kEntryBytes / 16);
        const int piece = i % (G::kEntryBytes / 16);
        const __nv_bfloat16 *src = (p ? a.cb_up : a.cb_gate) + kappa * kD;
        uint4 v;
        if constexpr (kD == 4) {
            const uint2 w = *reinterpret_cast<const uint2 *>(src);
            v = make_uint4(w.x, w.y, w.x, w.y);
        } else {
            v = *reinterpret_cast<const uint4 *>(src);
        }
        *reinterpret_cast<uint4 *>(cbs + p * G::kCbBytes + kappa * G::kEntryBytes + piece * 16) = v;
    }
    gemm_init<G>(ctl, warp, G::kDecWarps);
    if (a.wait_first) pdl_wait();
    pdl_launch_dependents();

    const int n_ct = a.I / G::kCT;
    const int nks = a.H / G::kK;
    const int nrows = a.H / kD;
    const int e_first = threadIdx.x == 0 ? first_unit_expert(a, n_ct).e : 0;
    const int64_t T = gemm_blocks(a) * a.tpb * n_ct;

    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            gemm_producer<G>(a, ctl, stages, reinterpret_cast<const unsigned char *>(a.x_tiles),
                             T, n_ct, nks, a.wait_first != 0, e_first,
                             [&](unsigned char *st, uint64_t *bar, int e, int ct, int s) {
                const int32_t y = e * nrows + s * G::kJRows;
                tma_load_2d(st, &tm_jgate, ct * G::kCT, y, bar, pol);
                tma_load_2d(st + G::kJBytes, &tm_jup, ct * G::kCT, y, bar, pol);
            });
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) gemm_mma_vq<kD, kN>(ctl, stages, T, nks);
        __syncwarp();
    } else if (warp >= kGDecWarp0) {
        vq_decode<kD, kN>(ctl, stages, cbs, T, nks, warp & 3, (warp - kGDecWarp0) >> 2, lane);
    } else {
        const int quad = warp & 3;
        const int row = 32 * quad + lane;  // channel within the unit
        const uint32_t tl = ctl.tmem + ((uint32_t)(32 * quad) << 16);
        const int64_t chunk_of_tile = a.I / 64;
        int local = 0;
        for (int64_t u = blockIdx.x; u < T; u += gridDim.x, ++local) {
            const int64_t tile = u / n_ct;
            const int ct = (int)(u % n_ct);
            const int buf = local & 1;
            if (row < kN) ctl.route[buf][row] = tile_route(a, tile, row, a.blocks[tile / a.tpb], false);
            const bool ok = gwait(&ctl.tfull[buf], (uint32_t)(local >> 1) & 1u, ctl);
            if (named_bar_or(1, 128, !ok)) break;
            const int c64 = row & 63;  // channel within its 64-wide chunk of p
            unsigned char *dst = reinterpret_cast<unsigned char *>(a.p_tiles) +
                                 (tile * chunk_of_tile + 2 * ct + (row >> 6)) * (int64_t)G::kChunkBytes +
                                 (c64 & 7) * 2;
            tc_fence_after();
#pragma unroll 1
            for (int c0 = 0; c0 < kN; c0 += 16) {  // 16 rows of the tile at a time
                float g[16], up[16];
                tmem_ld16(tl + (uint32_t)(buf * 2 * kN + c0), g);
                tmem_ld16(tl + (uint32_t)(buf * 2 * kN + kN + c0), up);
#pragma unroll
                for (int n = 0; n < 16; ++n) {
                    if (ctl.route[buf][c0 + n] < 0) continue;
                    const float pv = silu_f32(g[n]) * up[n];
                    *reinterpret_cast<__nv_bfloat16 *>(dst + tile_offset(c0 + n, c64 >> 3)) =
                        __float2bfloat16(pv);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl.tempty[buf]);
        }
    }
    gemm_finish<G>(ctl, warp, a.status);
}

// ------------------------------------------------------------------------------- down
template <int kN>
__global__ void __launch_bounds__(kGThreads, 1)
    gemm_down_kernel(const __grid_constant__ CUtensorMap tm_down, const GemmArgs a) {
    using G = GTile<kN>;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *base = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char *stages = base;
    GCtl &ctl = *reinterpret_cast<GCtl *>(base + G::kStages * G::kStageBytes);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) prefetch_tensormap(&tm_down);
    gemm_init<G>(ctl, warp);
    pdl_launch_dependents();

    const int n_ct = a.H / kGM;
    const int nks = a.I / G::kK;
    const int e_first = threadIdx.x == 0 ? first_unit_expert(a, n_ct).e : 0;
    const int64_t T = gemm_blocks(a) * a.tpb * n_ct;

    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            // p tiles come from the gate/up grid: always deferred to this kernel's own wait
            gemm_producer<G>(a, ctl, stages, reinterpret_cast<const unsigned char *>(a.p_tiles),
                              T, n_ct, nks, false, e_first,
                              [&](unsigned char *st, uint64_t *bar, int e, int ct, int s) {
                const int32_t y = e * a.I + s * G::kK;
                tma_load_2d(st, &tm_down, ct * kGM, y, bar, pol);
                tma_load_2d(st + G::kHalfBytes, &tm_down, ct * kGM + 64, y, bar, pol);
            });
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) gemm_mma<G>(ctl, stages, T, nks);
        __syncwarp();
    } else {
        const int quad = warp & 3;
        const int ch = 32 * quad + lane;  // output channel within the 128-channel tile
        int local = 0;
        for (int64_t u = blockIdx.x; u < T; u += gridDim.x, ++local) {
            const int64_t tile = u / n_ct;
            const int ct = (int)(u % n_ct);
            const int buf = local & 1;
            if (ch < kN) ctl.route[buf][ch] = tile_route(a, tile, ch, a.blocks[tile / a.tpb], false);
            const bool ok = gwait(&ctl.tfull[buf], (uint32_t)(local >> 1) & 1u, ctl);
            if (named_bar_or(1, 128, !ok)) break;
            float v[kN];
            drain_accumulator<kN>(ctl, quad, buf, v);
            float *ybase = a.y + ct * kGM + ch;
#pragma unroll
            for (int n = 0; n < kN; ++n) {
                const int r = ctl.route[buf][n];
                if (r >= 0) ybase[(int64_t)r * a.H] = v[n];
            }
        }
    }
    gemm_finish<G>(ctl, warp, a.status);
}

// ------------------------------------------------------------------ bounded-wait self-test
// One CTA shaped like the GEMM kernels takes its tensor memory and then waits on the first
// accumulator's "full" barrier, which no MMA commit ever completes.  The waits and the
// teardown are the GEMM kernels' own: the first elected lane whose wait runs out raises the
// abort flag, the other warps see it and stop waiting, the CTA frees its tensor memory and
// MOE_DEV_WAIT_TIMEOUT lands in the status word.  No copy or MMA is ever in flight.
__global__ void __launch_bounds__(kGThreads, 1) wait_selftest_kernel(int32_t *status) {
    __shared__ GCtl ctl;
    const int warp = threadIdx.x >> 5;
    gemm_init<GTile<kGemmBlock>>(ctl, warp);
    if ((threadIdx.x & 31) == 0) gwait(&ctl.tfull[0], 0, ctl);
    __syncwarp();
    gemm_finish<GTile<kGemmBlock>>(ctl, warp, status);
}

template <int kN>
static size_t gemm_fused_smem() {
    using G = GTile<kN>;
    return 1024 + G::kStages * G::kStageBytes + kN * 64 * 4 + ((sizeof(GCtl) + 15) & ~size_t(15)) +
           sizeof(UnitQueue);
}
template <int kN>
static size_t gemm_down_smem() {
    using G = GTile<kN>;
    return 1024 + G::kStages * G::kStageBytes + sizeof(GCtl);
}

cudaError_t launch_gather_rows(const GemmArgs &a, cudaStream_t stream) {
    cudaLaunchAttribute attrs[2];
    const int64_t want = (a.cap + 7) / 8;  // 8 rows (warps) per CTA
    const int64_t most = 4 * (int64_t)num_sms();
    const int grid = (int)(want < 1 ? 1 : (want > most ? most : want));
    cudaLaunchConfig_t cfg = launch_config(dim3(grid), dim3(256), 0, stream, attrs, 0);
    return cudaLaunchKernelEx(&cfg, gather_rows_kernel, a);
}

template <int kN>
static cudaError_t launch_fused_tiles(const CUtensorMap &tm_gate, const CUtensorMap &tm_up,
                                      const CUtensorMap &tm_down, const GemmArgs &a,
                                      cudaStream_t stream) {
    const size_t smem = gemm_fused_smem<kN>();
    cudaError_t err = ensure_smem(reinterpret_cast<const void *>(gemm_fused_kernel<kN>), smem);
    if (err != cudaSuccess) return err;
    cudaLaunchAttribute attrs[2];
    cudaLaunchConfig_t cfg = launch_config(dim3(num_sms()), dim3(kGThreads), smem, stream, attrs, 0);
    return cudaLaunchKernelEx(&cfg, gemm_fused_kernel<kN>, tm_gate, tm_up, tm_down, a);
}

template <int kN>
static cudaError_t launch_down_tiles(const CUtensorMap &tm_down, const GemmArgs &a,
                                     cudaStream_t stream) {
    const size_t smem = gemm_down_smem<kN>();
    cudaError_t err = ensure_smem(reinterpret_cast<const void *>(gemm_down_kernel<kN>), smem);
    if (err != cudaSuccess) return err;
    cudaLaunchAttribute attrs[2];
    cudaLaunchConfig_t cfg = launch_config(dim3(num_sms()), dim3(kGThreads), smem, stream, attrs, 0);
    return cudaLaunchKernelEx(&cfg, gemm_down_kernel<kN>, tm_down, a);
}

cudaError_t launch_gemm_fused(const CUtensorMap &tm_gate, const CUtensorMap &tm_up,
                              const CUtensorMap &tm_down, const GemmArgs &a, cudaStream_t stream) {
    if (a.kn == 16) return launch_fused_tiles<16>(tm_gate, tm_up, tm_down, a, stream);
    if (a.kn == 64) return launch_fused_tiles<64>(tm_gate, tm_up, tm_down, a, stream);
    return cudaErrorInvalidValue;
}

template <int kD, int kN>
static size_t gemm_gateup_vq_smem() {
    using G = GTileVQ<kD, kN>;
    return 1024 + G::kStages * G::kStageBytes + 2 * G::kCbBytes + sizeof(GCtl);
}

template <int kD, int kN>
static cudaError_t launch_gemm_gateup_vq_t(const CUtensorMap &tm_jgate, const CUtensorMap &tm_jup,
                                           const GemmArgs &a, cudaStream_t stream) {
    const size_t smem = gemm_gateup_vq_smem<kD, kN>();
    cudaError_t err = ensure_smem(reinterpret_cast<const void *>(gemm_gateup_vq_kernel<kD, kN>), smem);
    if (err != cudaSuccess) return err;
    cudaLaunchAttribute attrs[2];
    cudaLaunchConfig_t cfg = launch_config(dim3(num_sms()), dim3(kGVQThreads), smem, stream, attrs, 0);
    return cudaLaunchKernelEx(&cfg, gemm_gateup_vq_kernel<kD, kN>, tm_jgate, tm_jup, a);
}

cudaError_t launch_gemm_gateup_vq(const CUtensorMap &tm_jgate, const CUtensorMap &tm_jup,
                                  const GemmArgs &a, int d, cudaStream_t stream) {
    if (d == 4 && a.kn == 16) return launch_gemm_gateup_vq_t<4, 16>(tm_jgate, tm_jup, a, stream);
    if (d == 4 && a.kn == 64) return launch_gemm_gateup_vq_t<4, 64>(tm_jgate, tm_jup, a, stream);
    if (d == 8 && a.kn == 16) return launch_gemm_gateup_vq_t<8, 16>(tm_jgate, tm_jup, a, stream);
    if (d == 8 && a.kn == 64) return launch_gemm_gateup_vq_t<8, 64>(tm_jgate, tm_jup, a, stream);
    return cudaErrorInvalidValue;
}

cudaError_t launch_gemm_down(const CUtensorMap &tm_down, const GemmArgs &a, cudaStream_t stream) {
    if (a.kn == 16) return launch_down_tiles<16>(tm_down, a, stream);
    if (a.kn == 64) return launch_down_tiles<64>(tm_down, a, stream);
    return cudaErrorInvalidValue;
}

cudaError_t launch_wait_selftest(int32_t *status, cudaStream_t stream) {
    wait_selftest_kernel<<<1, kGThreads, 0, stream>>>(status);
    return cudaGetLastError();
}

}  // namespace moe
