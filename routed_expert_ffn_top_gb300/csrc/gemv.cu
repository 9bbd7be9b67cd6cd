// gemv.cu -- expert kernels of the small-batch (GEMV) regime.
//
// The expert computation of "A Multi-Engine Dataflow for MoE Decoding on Scratchpad-Based
// Tensor Accelerators" (MoE block background; stage-3 activation; Section 4.3):
//   gate/up:  g = h W_gate[e], u = h W_up[e], p = SiLU(g) * u        (per route)
//   down:     y = p W_down[e]
//   combine:  out[m] = residual[m] + sum_j a_{m,j} y_{m,j}   ("accumulated summation")
// and, channel by channel, "Channel Selection for Mixture-of-Experts Decoding Needs No
// Calibration Data" (Background: channel j owns row j of gate/up and column j of down).
//
// At decode batch sizes every weight byte serves only a handful of tokens, so the kernels
// are HBM streams.  The work is cut into tiles over the aligned rows:
//   * a sub-block is `rsub` consecutive aligned rows: at most 8 routes of ONE expert (the
//     alignment pads every expert to a multiple of b and rsub divides b);
//   * gate/up tile = (sub-block, 64-column I tile): all H rows of W_gate[e] and W_up[e] in
//     that column range, streamed as H/128 boxes of 128x64 bf16 per projection;
//   * down tile = (sub-block, 64-column H tile): all I rows of W_down[e] in that range, as
//     I/128 boxes of 128x64 bf16.
// Persistent CTAs (one per SM) own contiguous ranges of whole tiles.  Warp 0 is the
// producer: one thread issues TMA tensor loads of the boxes, plus bulk copies of the
// sub-block's activation slices, into a ring of shared-memory stages guarded by full/empty
// mbarriers.  Warps 1..8 consume: warp w owns rows [16w, 16w+16) of every box, lane l the
// 8 rows [16w + 8(l/16), +8) and the 4 columns [4(l%16), +4), and keeps fp32 accumulators
// for up to 8 tokens in registers across all boxes of the tile (gate/up multiplies the
// bf16 h and weight values directly into fp32; down uses packed fp32 FMAs on fp32 p).  Only at the end of a tile do the 8 warps combine their partial
// sums (shared memory, fixed warp order), and the epilogue writes p (gate/up) or y (down).
// A third small kernel forms out = residual + sum_j a_j y_j in slot order j = 0..k-1.
//
// Reduction order, fixed by tile indices only (never by grid size, CTA, block position,
// batch size or arrival order): per thread, boxes ascending and rows ascending inside its
// 8-row slice; then the two lane halves; then warps 0..7; then, for the combine, slots
// 0..k-1.  So the results are
// bitwise reproducible, a route's bits do not depend on the block it sits in or on the
// other routes of its block, and a token's output does not depend on M.
#include "moe_internal.cuh"
#include "ptx.cuh"

namespace moe {

constexpr int kStagesGU = 5;
constexpr int kStagesDN = 8;
constexpr int kConsumerThreads = 32 * kConsumerWarps;
constexpr int kRowsPerWarp = 16;  // of every 128-row box
static_assert(kHG == kConsumerWarps * kRowsPerWarp && kIG == kConsumerWarps * kRowsPerWarp, "rows");

constexpr int kBoxBytesGU = kHG * kTI * 2;                      // 16 KB per projection
constexpr int kStageBytesGU = 2 * kBoxBytesGU + kNT * kHG * 2;  // + h slices (bf16)
constexpr int kBoxBytesDN = kIG * kTN * 2;                      // 16 KB
constexpr int kStageBytesDN = kBoxBytesDN + kNT * kIG * 4;      // + p slices (fp32)
constexpr int kRedBytesGU = kConsumerWarps * kNT * kTI * 2 * 4;
constexpr int kRedBytesDN = kConsumerWarps * kNT * kTN * 4;
static_assert(kStageBytesGU % 1024 == 0 && kStageBytesDN % 1024 == 0, "stage alignment");

struct StageMeta {
    int ntok;
    int e;
    int routes[kNT];
};

struct Ctl {
    uint64_t full[8];
    uint64_t empty[8];
    StageMeta meta[8];
    volatile int abort;
};

// CTA c owns tiles c, c + G, c + 2G, ... (G = grid size).  Tiles are numbered column
// tile fastest, so at any moment neighbouring CTAs stream neighbouring column ranges of the
// same weight rows, and the DRAM pages those rows live in are read while open.

// Bounded wait that also gives up as soon as another thread of the CTA has aborted.
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, Ctl &ctl) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (ctl.abort) return false;
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
            ctl.abort = 1;
            return false;
        }
    }
}

// Routes of sub-block sb: the valid entries among its rsub aligned rows whose top-k id is
// the block's expert.  Anything else is padding (a mismatch is flagged as a bad alignment).
__device__ void decode_subblock(const GemvArgs &a, int64_t sb, StageMeta &s) {
    const int64_t row0 = sb * a.rsub;
    const int e = a.blocks[row0 / a.b];
    const int64_t R = (int64_t)a.M * a.k;
    s.e = e;
    int n = 0;
    if (e >= 0 && e < a.E) {
        for (int q = 0; q < a.rsub; ++q) {
            const int r = a.sorted[row0 + q];
            if (r < 0 || r >= R) continue;
            if (a.topk_ids[r] != e) {
                atomicOr(a.status, MOE_DEV_BAD_ALIGNMENT);
                continue;
            }
            s.routes[n++] = r;
        }
    }
    s.ntok = n;
}

// Producer (one thread).  A tile with no route is announced by a single stage with
// ntok == 0 and no copies; otherwise `boxes` stages, one per box of the tile.
struct NoFlush {
    __device__ void operator()() const {}
};

// `flush` runs before the producer could block on a stage it issued itself (once every
// stage of the ring has been issued) and after the last stage: the down kernel uses it to
// copy the activations it held back until its dependency wait.
template <int kStages, typename IssueFn, typename FlushFn = NoFlush>
__device__ void producer_loop(const GemvArgs &a, Ctl &ctl, int64_t T, int tiles_per_sub,
                              int boxes, IssueFn issue, FlushFn flush = NoFlush()) {
    int stage = 0;
    uint32_t phase = 0;
    int64_t cur_sb = -1;
    StageMeta cur;
    cur.ntok = 0;
    cur.e = -1;
    uint32_t issued = 0, parity_bits = 0;
    int64_t n_issued = 0;
    for (int64_t t = blockIdx.x; t < T && !ctl.abort; t += gridDim.x) {
        const int64_t sb = t / tiles_per_sub;
        if (sb != cur_sb) {
            decode_subblock(a, sb, cur);
            cur_sb = sb;
        }
        const int nst = cur.ntok > 0 ? boxes : 1;
        for (int bx = 0; bx < nst; ++bx) {
            if (n_issued == kStages) flush();
            if (!wait_or_abort(&ctl.empty[stage], phase ^ 1u, ctl)) break;
            ++n_issued;
            ctl.meta[stage] = cur;
            if (cur.ntok > 0)
                issue(stage, t, bx, cur);
            else
                mbar_arrive(&ctl.full[stage]);
            issued |= 1u << stage;
            parity_bits = (parity_bits & ~(1u << stage)) | (phase << stage);
            if (++stage == kStages) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
    flush();
    // Never leave the CTA while copies may still be landing in its shared memory.
    for (int s = 0; s < kStages; ++s)
        if ((issued >> s) & 1u)
            if (!mbar_wait_bounded(&ctl.full[s], (parity_bits >> s) & 1u)) ctl.abort = 1;
    if (ctl.abort) atomicOr(a.status, MOE_DEV_WAIT_TIMEOUT);
}

template <int kStages>
__device__ __forceinline__ void advance(int &stage, uint32_t &phase) {
    if (++stage == kStages) {
        stage = 0;
        phase ^= 1u;
    }
}

// ---------------------------------------------------------------------------- gate/up
__global__ void __launch_bounds__(kGemvThreads, 1)
    gateup_dense_kernel(const __grid_constant__ CUtensorMap tm_gate,
                        const __grid_constant__ CUtensorMap tm_up, const GemvArgs a) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *base = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char *stages = base;
    float *red = reinterpret_cast<float *>(base + kStagesGU * kStageBytesGU);
    Ctl &ctl = *reinterpret_cast<Ctl *>(base + kStagesGU * kStageBytesGU + kRedBytesGU);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStagesGU; ++s) {
            mbar_init(&ctl.full[s], 1);
            mbar_init(&ctl.empty[s], kConsumerWarps);
        }
        ctl.abort = 0;
        fence_mbar_init();
        prefetch_tensormap(&tm_gate);
        prefetch_tensormap(&tm_up);
    }
    __syncthreads();
    pdl_wait();
    pdl_launch_dependents();

    const int64_t T = (a.npad[0] / a.rsub) * a.n_it;

    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first();
            producer_loop<kStagesGU>(a, ctl, T, a.n_it, a.n_hg,
                                     [&](int stage, int64_t t, int hg, const StageMeta &m) {
                const int it = (int)(t % a.n_it);
                unsigned char *st = stages + stage * kStageBytesGU;
                uint64_t *bar = &ctl.full[stage];
                mbar_arrive_expect_tx(bar, 2 * kBoxBytesGU + m.ntok * kHG * 2);
                const int32_t y = m.e * a.H + hg * kHG;
                tma_load_2d(st, &tm_gate, it * kTI, y, bar, pol_w);
                tma_load_2d(st + kBoxBytesGU, &tm_up, it * kTI, y, bar, pol_w);
                for (int q = 0; q < m.ntok; ++q) {
                    const int tok = m.routes[q] / a.k;
                    bulk_load(st + 2 * kBoxBytesGU + q * kHG * 2,
                              a.h + (size_t)tok * a.H + (size_t)hg * kHG, kHG * 2, bar);
                }
            });
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    // Lane l of consumer warp w: columns 4*(l%16) .. +3 of the tile, rows 16w + 8*(l/16)
    // .. +7 of every box (8 consecutive rows: one 16-byte load of each token's h slice).
    const int ctid = threadIdx.x - 32;
    const int cw = warp - 1;
    const int half = lane >> 4;
    const int c4 = (lane & 15) * 4;
    const int rbase = cw * kRowsPerWarp + half * 8;
    int stage = 0;
    uint32_t phase = 0;
    for (int64_t t = blockIdx.x; t < T; t += gridDim.x) {
        const int it = (int)(t % a.n_it);
        float ag[kNT][4], au[kNT][4];
#pragma unroll
        for (int q = 0; q < kNT; ++q)
#pragma unroll
            for (int j = 0; j < 4; ++j) ag[q][j] = au[q][j] = 0.0f;
        int ntok = 0, r0 = -1, r1 = -1;
        bool failed = false;
        for (int hg = 0; hg < a.n_hg; ++hg) {
            if (failed || !wait_or_abort(&ctl.full[stage], phase, ctl)) {
                failed = true;
                break;
            }
            const StageMeta &mt = ctl.meta[stage];
            if (hg == 0) {
                ntok = mt.ntok;
                const int q0 = ctid / kTI, q1 = (ctid + kConsumerThreads) / kTI;
                r0 = (q0 < ntok) ? mt.routes[q0] : -1;
                r1 = (q1 < ntok) ? mt.routes[q1] : -1;
            }
            if (ntok > 0) {
                const unsigned char *st = stages + stage * kStageBytesGU;
                uint2 gw[8], uw[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    gw[i] = *reinterpret_cast<const uint2 *>(st + (rbase + i) * (kTI * 2) + c4 * 2);
                    uw[i] = *reinterpret_cast<const uint2 *>(st + kBoxBytesGU + (rbase + i) * (kTI * 2) + c4 * 2);
                }
                const unsigned char *xs = st + 2 * kBoxBytesGU + rbase * 2;
#pragma unroll
                for (int q = 0; q < kNT; ++q) {
                    if (q < ntok) {
                        const uint4 xv = *reinterpret_cast<const uint4 *>(xs + q * kHG * 2);
                        const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const uint32_t x2 = xw[i >> 1];
                            if (i & 1) {
                                ag[q][0] = fma_bf16<1, 0>(x2, gw[i].x, ag[q][0]);
                                ag[q][1] = fma_bf16<1, 1>(x2, gw[i].x, ag[q][1]);
                                ag[q][2] = fma_bf16<1, 0>(x2, gw[i].y, ag[q][2]);
                                ag[q][3] = fma_bf16<1, 1>(x2, gw[i].y, ag[q][3]);
                                au[q][0] = fma_bf16<1, 0>(x2, uw[i].x, au[q][0]);
                                au[q][1] = fma_bf16<1, 1>(x2, uw[i].x, au[q][1]);
                                au[q][2] = fma_bf16<1, 0>(x2, uw[i].y, au[q][2]);
                                au[q][3] = fma_bf16<1, 1>(x2, uw[i].y, au[q][3]);
                            } else {
                                ag[q][0] = fma_bf16<0, 0>(x2, gw[i].x, ag[q][0]);
                                ag[q][1] = fma_bf16<0, 1>(x2, gw[i].x, ag[q][1]);
                                ag[q][2] = fma_bf16<0, 0>(x2, gw[i].y, ag[q][2]);
                                ag[q][3] = fma_bf16<0, 1>(x2, gw[i].y, ag[q][3]);
                                au[q][0] = fma_bf16<0, 0>(x2, uw[i].x, au[q][0]);
                                au[q][1] = fma_bf16<0, 1>(x2, uw[i].x, au[q][1]);
                                au[q][2] = fma_bf16<0, 0>(x2, uw[i].y, au[q][2]);
                                au[q][3] = fma_bf16<0, 1>(x2, uw[i].y, au[q][3]);
                            }
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl.empty[stage]);
            advance<kStagesGU>(stage, phase);
            if (ntok == 0) break;  // an empty tile is announced by a single stage
        }
        if (named_bar_or(1, kConsumerThreads, failed)) break;
        if (ntok == 0) continue;
        // rows of the two lane halves: half 0 + half 1 (the same bits on both lanes)
#pragma unroll
        for (int q = 0; q < kNT; ++q)
            if (q < ntok) {
                float g4[4], u4[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    g4[j] = ag[q][j] + __shfl_xor_sync(0xffffffffu, ag[q][j], 16);
                    u4[j] = au[q][j] + __shfl_xor_sync(0xffffffffu, au[q][j], 16);
                }
                if (half == 0) {
                    float *dst = &red[((cw * kNT + q) * kTI + c4) * 2];
                    *reinterpret_cast<float4 *>(dst) = make_float4(g4[0], u4[0], g4[1], u4[1]);
                    *reinterpret_cast<float4 *>(dst + 4) = make_float4(g4[2], u4[2], g4[3], u4[3]);
                }
            }
        named_bar_sync(1, kConsumerThreads);
        const int col0 = it * kTI;
#pragma unroll
        for (int pass = 0; pass < 2; ++pass) {
            const int idx = ctid + pass * kConsumerThreads;
            const int q = idx / kTI, c = idx % kTI;
            const int r = pass ? r1 : r0;
            if (q < ntok) {
                float2 s = *reinterpret_cast<const float2 *>(&red[(q * kTI + c) * 2]);
#pragma unroll
                for (int w = 1; w < kConsumerWarps; ++w) {
                    const float2 v = *reinterpret_cast<const float2 *>(&red[((w * kNT + q) * kTI + c) * 2]);
                    s.x += v.x;
                    s.y += v.y;
                }
                a.p[(int64_t)r * a.I + col0 + c] = silu_f32(s.x) * s.y;
            }
        }
        named_bar_sync(1, kConsumerThreads);
    }
}

// ------------------------------------------------------------------------------- down
__global__ void __launch_bounds__(kGemvThreads, 1)
    down_kernel(const __grid_constant__ CUtensorMap tm_down, const GemvArgs a) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *base = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char *stages = base;
    float *red = reinterpret_cast<float *>(base + kStagesDN * kStageBytesDN);
    Ctl &ctl = *reinterpret_cast<Ctl *>(base + kStagesDN * kStageBytesDN + kRedBytesDN);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStagesDN; ++s) {
            mbar_init(&ctl.full[s], 1);
            mbar_init(&ctl.empty[s], kConsumerWarps);
        }
        ctl.abort = 0;
        fence_mbar_init();
        prefetch_tensormap(&tm_down);
    }
    __syncthreads();
    // The routing and the alignment were complete before the gate/up kernel (the grid this
    // one depends on) started its work, so which down weights to read is already known
    // ("A Multi-Engine Dataflow ...", overlap window of the down-projection DMA): the
    // producer streams W_down boxes into the ring right away and waits for the gate/up
    // grid only before it copies p, which that grid writes.
    const int64_t T = (a.npad[0] / a.rsub) * a.n_ht;

    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first();
            bool waited = false;
            int npend = 0;
            int pend_stage[kStagesDN];
            int pend_ig[kStagesDN];
            StageMeta pend_meta[kStagesDN];
            auto copy_p = [&](int stage, int ig, const StageMeta &m) {
                unsigned char *st = stages + stage * kStageBytesDN;
                for (int q = 0; q < m.ntok; ++q)
                    bulk_load(st + kBoxBytesDN + q * kIG * 4,
                              a.p + (size_t)m.routes[q] * a.I + (size_t)ig * kIG, kIG * 4,
                              &ctl.full[stage]);
            };
            auto flush = [&]() {
                pdl_wait();
                waited = true;
                for (int i = 0; i < npend; ++i) copy_p(pend_stage[i], pend_ig[i], pend_meta[i]);
                npend = 0;
            };
            producer_loop<kStagesDN>(a, ctl, T, a.n_ht, a.n_ig,
                                     [&](int stage, int64_t t, int ig, const StageMeta &m) {
                const int ht = (int)(t % a.n_ht);
                unsigned char *st = stages + stage * kStageBytesDN;
                uint64_t *bar = &ctl.full[stage];
                mbar_arrive_expect_tx(bar, kBoxBytesDN + m.ntok * kIG * 4);
                tma_load_2d(st, &tm_down, ht * kTN, m.e * a.I + ig * kIG, bar, pol_w);
                if (waited) {
                    copy_p(stage, ig, m);
                } else {
                    pend_stage[npend] = stage;
                    pend_ig[npend] = ig;
                    pend_meta[npend] = m;
                    ++npend;
                }
            }, [&]() { if (!waited) flush(); });
        }
        return;
    }
    pdl_launch_dependents();

    // Same lane layout as gate/up: 4 columns x 8 consecutive rows of every box.
    const int ctid = threadIdx.x - 32;
    const int cw = warp - 1;
    const int half = lane >> 4;
    const int c4 = (lane & 15) * 4;
    const int rbase = cw * kRowsPerWarp + half * 8;
    int stage = 0;
    uint32_t phase = 0;
    for (int64_t t = blockIdx.x; t < T; t += gridDim.x) {
        const int ht = (int)(t % a.n_ht);
        float acc[kNT][4];
#pragma unroll
        for (int q = 0; q < kNT; ++q)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[q][j] = 0.0f;
        int ntok = 0, r0 = -1, r1 = -1;
        bool failed = false;
        for (int ig = 0; ig < a.n_ig; ++ig) {
            if (failed || !wait_or_abort(&ctl.full[stage], phase, ctl)) {
                failed = true;
                break;
            }
            const StageMeta &mt = ctl.meta[stage];
            if (ig == 0) {
                ntok = mt.ntok;
                const int q0 = ctid / kTN, q1 = (ctid + kConsumerThreads) / kTN;
                r0 = (q0 < ntok) ? mt.routes[q0] : -1;
                r1 = (q1 < ntok) ? mt.routes[q1] : -1;
            }
            if (ntok > 0) {
                const unsigned char *st = stages + stage * kStageBytesDN;
                float w[8][4];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint2 w2 = *reinterpret_cast<const uint2 *>(st + (rbase + i) * (kTN * 2) + c4 * 2);
                    w[i][0] = bf16_lo(w2.x);
                    w[i][1] = bf16_hi(w2.x);
                    w[i][2] = bf16_lo(w2.y);
                    w[i][3] = bf16_hi(w2.y);
                }
                const float *xs = reinterpret_cast<const float *>(st + kBoxBytesDN) + rbase;
#pragma unroll
                for (int q = 0; q < kNT; ++q) {
                    if (q < ntok) {
                        const float4 p0 = *reinterpret_cast<const float4 *>(xs + q * kIG);
                        const float4 p1 = *reinterpret_cast<const float4 *>(xs + q * kIG + 4);
                        const float x[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            ffma2(acc[q][0], acc[q][1], x[i], w[i][0], w[i][1]);
                            ffma2(acc[q][2], acc[q][3], x[i], w[i][2], w[i][3]);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl.empty[stage]);
            advance<kStagesDN>(stage, phase);
            if (ntok == 0) break;
        }
        if (named_bar_or(1, kConsumerThreads, failed)) break;
        if (ntok == 0) continue;
#pragma unroll
        for (int q = 0; q < kNT; ++q)
            if (q < ntok) {
                float v[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) v[j] = acc[q][j] + __shfl_xor_sync(0xffffffffu, acc[q][j], 16);
                if (half == 0)
                    *reinterpret_cast<float4 *>(&red[(cw * kNT + q) * kTN + c4]) = make_float4(v[0], v[1], v[2], v[3]);
            }
        named_bar_sync(1, kConsumerThreads);
        const int col0 = ht * kTN;
#pragma unroll
        for (int pass = 0; pass < 2; ++pass) {
            const int idx = ctid + pass * kConsumerThreads;
            const int q = idx / kTN, c = idx % kTN;
            const int r = pass ? r1 : r0;
            if (q < ntok) {
                float sum = red[q * kTN + c];
#pragma unroll
                for (int w2 = 1; w2 < kConsumerWarps; ++w2) sum += red[(w2 * kNT + q) * kTN + c];
                a.y[(int64_t)r * a.H + col0 + c] = sum;
            }
        }
        named_bar_sync(1, kConsumerThreads);
    }
}

// ---------------------------------------------------------------------------- combine
// out[m][n] = bf16(residual[m][n] + sum_{j valid} a_{m,j} * y_{m,j}[n]), j ascending.
constexpr int kCombineThreads = 256;

__global__ void __launch_bounds__(kCombineThreads)
    combine_kernel(const float *__restrict__ y, const int32_t *__restrict__ topk_ids,
                   const float *__restrict__ topk_wts, const __nv_bfloat16 *__restrict__ residual,
                   __nv_bfloat16 *__restrict__ out, int M, int k, int E, int H) {
    pdl_wait();
    pdl_launch_dependents();
    const int m = blockIdx.y;
    const int n = (blockIdx.x * kCombineThreads + threadIdx.x) * 4;
    if (m >= M || n >= H) return;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < k; ++j) {
        const int64_t r = (int64_t)m * k + j;
        const int e = topk_ids[r];
        if (e < 0 || e >= E) continue;
        const float aw = topk_wts[r];
        const float4 v = __ldcg(reinterpret_cast<const float4 *>(y + r * H + n));
        acc.x = fmaf(aw, v.x, acc.x);
        acc.y = fmaf(aw, v.y, acc.y);
        acc.z = fmaf(aw, v.z, acc.z);
        acc.w = fmaf(aw, v.w, acc.w);
    }
    const size_t o = (size_t)m * H + n;
    float4 res = make_float4(0.f, 0.f, 0.f, 0.f);
    if (residual) {
        const uint2 rv = *reinterpret_cast<const uint2 *>(residual + o);
        res = make_float4(bf16_lo(rv.x), bf16_hi(rv.x), bf16_lo(rv.y), bf16_hi(rv.y));
    }
    const __nv_bfloat162 o01 = __floats2bfloat162_rn(res.x + acc.x, res.y + acc.y);
    const __nv_bfloat162 o23 = __floats2bfloat162_rn(res.z + acc.z, res.w + acc.w);
    uint2 ov;
    ov.x = *reinterpret_cast<const uint32_t *>(&o01);
    ov.y = *reinterpret_cast<const uint32_t *>(&o23);
    *reinterpret_cast<uint2 *>(out + o) = ov;
}

static size_t gateup_smem() { return 1024 + kStagesGU * kStageBytesGU + kRedBytesGU + sizeof(Ctl); }
static size_t down_smem() { return 1024 + kStagesDN * kStageBytesDN + kRedBytesDN + sizeof(Ctl); }

cudaError_t launch_gateup_dense(const CUtensorMap &tm_gate, const CUtensorMap &tm_up,
                                const GemvArgs &a, cudaStream_t stream) {
    const size_t smem = gateup_smem();
    cudaError_t err = cudaFuncSetAttribute(gateup_dense_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    cudaLaunchAttribute attrs[2];
    cudaLaunchConfig_t cfg = launch_config(dim3(num_sms()), dim3(kGemvThreads), smem, stream, attrs, 0);
    return cudaLaunchKernelEx(&cfg, gateup_dense_kernel, tm_gate, tm_up, a);
}

cudaError_t launch_down(const CUtensorMap &tm_down, const GemvArgs &a, cudaStream_t stream) {
    const size_t smem = down_smem();
    cudaError_t err = cudaFuncSetAttribute(down_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)smem);
    if (err != cudaSuccess) return err;
    cudaLaunchAttribute attrs[2];
    cudaLaunchConfig_t cfg = launch_config(dim3(num_sms()), dim3(kGemvThreads), smem, stream, attrs, 0);
    return cudaLaunchKernelEx(&cfg, down_kernel, tm_down, a);
}

cudaError_t launch_combine(const GemvArgs &a, cudaStream_t stream) {
    cudaLaunchAttribute attrs[2];
    dim3 grid((a.H / 4 + kCombineThreads - 1) / kCombineThreads, a.M);
    cudaLaunchConfig_t cfg = launch_config(grid, dim3(kCombineThreads), 0, stream, attrs, 0);
    return cudaLaunchKernelEx(&cfg, combine_kernel, (const float *)a.y, a.topk_ids, a.topk_wts,
                              a.residual, a.out, a.M, a.k, a.E, a.H);
}

}  // namespace moe
