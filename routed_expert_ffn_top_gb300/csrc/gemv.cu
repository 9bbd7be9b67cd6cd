// gemv.cu -- expert kernels of the small-batch (GEMV) regime.
//
// The expert computation of "A Multi-Engine Dataflow for MoE Decoding on Scratchpad-Based
// Tensor Accelerators" (MoE block background; stage-3 activation; Section 4.3):
//   gate/up:  g = h W_gate[e], u = h W_up[e], p = SiLU(g) * u        (per route)
//   down:     y = p W_down[e];  out[m] = residual[m] + sum_j a_{m,j} y_{m,j}
// and, channel by channel, "Channel Selection for Mixture-of-Experts Decoding Needs No
// Calibration Data" (Background: channel j owns row j of gate/up and column j of down).
//
// At decode batch sizes every weight byte is used by only a handful of tokens, so both
// kernels are HBM streams.  Work is split into fixed tiles over the aligned rows:
//   * a sub-block is `rsub` consecutive aligned rows (<= 8 routes of ONE expert, since the
//     alignment pads every expert to a multiple of b and rsub divides b);
//   * gate/up unit = (sub-block, 64-column I tile, 128-row H group): one 128x64 bf16 box of
//     W_gate and one of W_up (32 KB) plus the sub-block's 128-element h slices;
//   * down unit = (sub-block, 64-column H tile, 128-row I group): one 128x64 bf16 box of
//     W_down (16 KB) plus the sub-block's 128-element p slices.
// Persistent CTAs (one per SM) take contiguous ranges of units.  Warp 0 is the producer:
// one thread issues TMA tensor loads of the weight boxes and bulk copies of the activation
// slices into a ring of shared-memory stages guarded by full/empty mbarriers.  Warps 1..8
// consume: each owns 16 rows of the box, each lane two adjacent columns, and keeps fp32
// accumulators for up to 8 tokens.
//
// Reduction order (fixed by tile indices only -- never by grid size, CTA, block position
// or arrival order; so results are bitwise reproducible and each route's bits do not
// depend on which block it sits in or on M):
//   rows of a warp ascending -> the 8 consumer warps in order -> (per unit) a partial
//   written to global memory at [group][route][column] -> the last unit of a tile to
//   finish (integer ticket) sums the partials over the groups in ascending order.
// Down: y_{m,j} = sum over I groups ascending; out = bf16(residual + sum_j a_j y_j) in
// slot order j = 0..k-1 by the last unit touching (token, H tile).
#include "moe_internal.cuh"
#include "ptx.cuh"

namespace moe {

constexpr int kStagesGU = 4;
constexpr int kStagesDN = 6;
constexpr int kConsumerThreads = 32 * kConsumerWarps;
constexpr int kRowsPerWarpGU = kHG / kConsumerWarps;  // 16
constexpr int kRowsPerWarpDN = kIG / kConsumerWarps;  // 16

constexpr int kBoxBytesGU = kHG * kTI * 2;                      // 16 KB per projection
constexpr int kStageBytesGU = 2 * kBoxBytesGU + kNT * kHG * 2;  // + h slices (bf16)
constexpr int kBoxBytesDN = kIG * kTN * 2;                      // 16 KB
constexpr int kStageBytesDN = kBoxBytesDN + kNT * kIG * 4;      // + p slices (fp32)
constexpr int kRedBytesGU = kConsumerWarps * kNT * kTI * 2 * 4;
constexpr int kRedBytesDN = kConsumerWarps * kNT * kTN * 4;

static_assert(kStageBytesGU % 1024 == 0, "stage alignment");
static_assert(kStageBytesDN % 1024 == 0, "stage alignment");

struct StageMeta {
    int ntok;
    int e;
    int routes[kNT];
};

struct Ctl {
    uint64_t full[8];
    uint64_t empty[8];
    StageMeta meta[8];
    int flag;
    int fin[kNT];
};

__device__ __forceinline__ void unit_range(int64_t U, int64_t &begin, int64_t &end) {
    begin = (int64_t)blockIdx.x * U / gridDim.x;
    end = ((int64_t)blockIdx.x + 1) * U / gridDim.x;
}

// Routes of sub-block sb: the valid entries among its rsub aligned rows whose top-k id
// equals the block's expert.  Anything else is padding (or flagged as a bad alignment).
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

// Producer: one thread.  `units_per_sub` consecutive units share a sub-block.
template <int kStages, typename IssueFn>
__device__ void producer_loop(const GemvArgs &a, Ctl &ctl, int64_t begin, int64_t end,
                              int64_t units_per_sub, IssueFn issue) {
    int stage = 0;
    uint32_t phase = 0;
    int64_t cur_sb = -1;
    StageMeta cur;
    cur.ntok = 0;
    cur.e = -1;
    uint32_t issued_mask = 0, last_parity = 0;
    bool abort = false;
    for (int64_t u = begin; u < end; ++u) {
        const int64_t sb = u / units_per_sub;
        if (sb != cur_sb) {
            decode_subblock(a, sb, cur);
            cur_sb = sb;
        }
        if (!mbar_wait_bounded(&ctl.empty[stage], phase ^ 1u)) {
            atomicOr(a.status, MOE_DEV_WAIT_TIMEOUT);
            abort = true;
            break;
        }
        ctl.meta[stage] = cur;
        if (cur.ntok > 0) {
            issue(stage, u, cur);
        } else {
            mbar_arrive(&ctl.full[stage]);
        }
        issued_mask |= 1u << stage;
        last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
        }
    }
    (void)abort;
    // Never leave the CTA with copies still landing in its shared memory.
    for (int s = 0; s < kStages; ++s)
        if ((issued_mask >> s) & 1u)
            if (!mbar_wait_bounded(&ctl.full[s], (last_parity >> s) & 1u))
                atomicOr(a.status, MOE_DEV_WAIT_TIMEOUT);
}

// ---------------------------------------------------------------------------- gate/up
__global__ void __launch_bounds__(kGemvThreads, 1)
    gateup_dense_kernel(const __grid_constant__ CUtensorMap tm_gate,
                        const __grid_constant__ CUtensorMap tm_up, const GemvArgs a) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *base =
        reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char *stages = base;
    float *red = reinterpret_cast<float *>(base + kStagesGU * kStageBytesGU);
    Ctl &ctl = *reinterpret_cast<Ctl *>(base + kStagesGU * kStageBytesGU + kRedBytesGU);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStagesGU; ++s) {
            mbar_init(&ctl.full[s], 1);
            mbar_init(&ctl.empty[s], kConsumerWarps);
        }
        fence_mbar_init();
        prefetch_tensormap(&tm_gate);
        prefetch_tensormap(&tm_up);
    }
    __syncthreads();
    pdl_wait();
    pdl_launch_dependents();

    const int64_t R = (int64_t)a.M * a.k;
    const int64_t nsub = a.npad[0] / a.rsub;
    const int64_t per_sub = (int64_t)a.n_it * a.n_hg;
    int64_t begin, end;
    unit_range(nsub * per_sub, begin, end);

    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first();
            producer_loop<kStagesGU>(a, ctl, begin, end, per_sub,
                                     [&](int stage, int64_t u, const StageMeta &m) {
                const int hg = (int)(u % a.n_hg);
                const int it = (int)((u / a.n_hg) % a.n_it);
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

    // ------------------------------------------------------------------ consumers
    const int ctid = threadIdx.x - 32;
    const int cw = warp - 1;
    int stage = 0;
    uint32_t phase = 0;
    for (int64_t u = begin; u < end; ++u) {
        const int hg = (int)(u % a.n_hg);
        const int64_t t = u / a.n_hg;
        const int it = (int)(t % a.n_it);
        const int64_t sb = t / a.n_it;
        const bool ok = mbar_wait_bounded(&ctl.full[stage], phase);
        if (named_bar_or(1, kConsumerThreads, !ok)) {
            if (ctid == 0) atomicOr(a.status, MOE_DEV_WAIT_TIMEOUT);
            break;
        }
        const StageMeta &mt = ctl.meta[stage];
        const int ntok = mt.ntok;
        // Route ids this thread needs after the stage is released.
        const int q0 = ctid / kTI, q1 = (ctid + kConsumerThreads) / kTI;
        const int r0 = (q0 < ntok) ? mt.routes[q0] : -1;
        const int r1 = (q1 < ntok) ? mt.routes[q1] : -1;
        if (ntok > 0) {
            const unsigned char *st = stages + stage * kStageBytesGU;
            const uint32_t *gs = reinterpret_cast<const uint32_t *>(st);
            const uint32_t *us = reinterpret_cast<const uint32_t *>(st + kBoxBytesGU);
            const uint16_t *xs = reinterpret_cast<const uint16_t *>(st + 2 * kBoxBytesGU);
            float ag0[kNT], ag1[kNT], au0[kNT], au1[kNT];
#pragma unroll
            for (int q = 0; q < kNT; ++q) ag0[q] = ag1[q] = au0[q] = au1[q] = 0.0f;
#pragma unroll 4
            for (int rr = 0; rr < kRowsPerWarpGU; ++rr) {
                const int row = cw * kRowsPerWarpGU + rr;
                const uint32_t gw = gs[row * (kTI / 2) + lane];
                const uint32_t uw = us[row * (kTI / 2) + lane];
                const float g0 = bf16_lo(gw), g1 = bf16_hi(gw);
                const float u0 = bf16_lo(uw), u1 = bf16_hi(uw);
#pragma unroll
                for (int q = 0; q < kNT; ++q) {
                    if (q < ntok) {
                        const float xv = bf16_to_f32(xs[q * kHG + row]);
                        ag0[q] = fmaf(xv, g0, ag0[q]);
                        ag1[q] = fmaf(xv, g1, ag1[q]);
                        au0[q] = fmaf(xv, u0, au0[q]);
                        au1[q] = fmaf(xv, u1, au1[q]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl.empty[stage]);
#pragma unroll
            for (int q = 0; q < kNT; ++q)
                if (q < ntok)
                    *reinterpret_cast<float4 *>(&red[((cw * kNT + q) * kTI + 2 * lane) * 2]) =
                        make_float4(ag0[q], au0[q], ag1[q], au1[q]);
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
                        const float2 v =
                            *reinterpret_cast<const float2 *>(&red[((w * kNT + q) * kTI + c) * 2]);
                        s.x += v.x;
                        s.y += v.y;
                    }
                    a.part_gu[((int64_t)hg * R + r) * a.I + col0 + c] = s;
                }
            }
            __threadfence();
            named_bar_sync(1, kConsumerThreads);
            if (ctid == 0) {
                int *cnt = &a.cnt_gu[sb * a.n_it + it];
                const int old = atomicAdd(cnt, 1);
                const int last = (old == a.n_hg - 1);
                if (last) atomicExch(cnt, 0);
                ctl.flag = last;
            }
            named_bar_sync(1, kConsumerThreads);
            if (ctl.flag) {
                __threadfence();
#pragma unroll
                for (int pass = 0; pass < 2; ++pass) {
                    const int idx = ctid + pass * kConsumerThreads;
                    const int q = idx / kTI, c = idx % kTI;
                    const int r = pass ? r1 : r0;
                    if (q < ntok) {
                        float g = 0.0f, uu = 0.0f;
                        for (int gi = 0; gi < a.n_hg; ++gi) {
                            const float2 v = __ldcg(&a.part_gu[((int64_t)gi * R + r) * a.I + col0 + c]);
                            g += v.x;
                            uu += v.y;
                        }
                        a.p[(int64_t)r * a.I + col0 + c] = silu_f32(g) * uu;
                    }
                }
            }
        } else {
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl.empty[stage]);
        }
        if (++stage == kStagesGU) {
            stage = 0;
            phase ^= 1u;
        }
    }
}

// ------------------------------------------------------------------------------- down
__global__ void __launch_bounds__(kGemvThreads, 1)
    down_kernel(const __grid_constant__ CUtensorMap tm_down, const GemvArgs a) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *base =
        reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char *stages = base;
    float *red = reinterpret_cast<float *>(base + kStagesDN * kStageBytesDN);
    Ctl &ctl = *reinterpret_cast<Ctl *>(base + kStagesDN * kStageBytesDN + kRedBytesDN);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStagesDN; ++s) {
            mbar_init(&ctl.full[s], 1);
            mbar_init(&ctl.empty[s], kConsumerWarps);
        }
        fence_mbar_init();
        prefetch_tensormap(&tm_down);
    }
    __syncthreads();
    pdl_wait();
    pdl_launch_dependents();

    const int64_t R = (int64_t)a.M * a.k;
    const int64_t nsub = a.npad[0] / a.rsub;
    const int64_t per_sub = (int64_t)a.n_ht * a.n_ig;
    int64_t begin, end;
    unit_range(nsub * per_sub, begin, end);

    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first();
            producer_loop<kStagesDN>(a, ctl, begin, end, per_sub,
                                     [&](int stage, int64_t u, const StageMeta &m) {
                const int ig = (int)(u % a.n_ig);
                const int ht = (int)((u / a.n_ig) % a.n_ht);
                unsigned char *st = stages + stage * kStageBytesDN;
                uint64_t *bar = &ctl.full[stage];
                mbar_arrive_expect_tx(bar, kBoxBytesDN + m.ntok * kIG * 4);
                tma_load_2d(st, &tm_down, ht * kTN, m.e * a.I + ig * kIG, bar, pol_w);
                for (int q = 0; q < m.ntok; ++q)
                    bulk_load(st + kBoxBytesDN + q * kIG * 4,
                              a.p + (size_t)m.routes[q] * a.I + (size_t)ig * kIG, kIG * 4, bar);
            });
        }
        return;
    }

    const int ctid = threadIdx.x - 32;
    const int cw = warp - 1;

    // Tokens without any valid route get the residual (or zero).
    for (int m = blockIdx.x; m < a.M; m += gridDim.x) {
        int nvalid = 0;
        for (int j = 0; j < a.k; ++j) {
            const int e = a.topk_ids[(size_t)m * a.k + j];
            nvalid += (e >= 0 && e < a.E);
        }
        if (nvalid == 0)
            for (int n = ctid; n < a.H; n += kConsumerThreads)
                a.out[(size_t)m * a.H + n] =
                    a.residual ? a.residual[(size_t)m * a.H + n] : __float2bfloat16(0.0f);
    }

    int stage = 0;
    uint32_t phase = 0;
    for (int64_t u = begin; u < end; ++u) {
        const int ig = (int)(u % a.n_ig);
        const int64_t t = u / a.n_ig;
        const int ht = (int)(t % a.n_ht);
        const bool ok = mbar_wait_bounded(&ctl.full[stage], phase);
        if (named_bar_or(1, kConsumerThreads, !ok)) {
            if (ctid == 0) atomicOr(a.status, MOE_DEV_WAIT_TIMEOUT);
            break;
        }
        const StageMeta &mt = ctl.meta[stage];
        const int ntok = mt.ntok;
        const int q0 = ctid / kTN, q1 = (ctid + kConsumerThreads) / kTN;
        const int r0 = (q0 < ntok) ? mt.routes[q0] : -1;
        const int r1 = (q1 < ntok) ? mt.routes[q1] : -1;
        const int rq = (ctid < ntok) ? mt.routes[ctid] : -1;
        if (ntok > 0) {
            const unsigned char *st = stages + stage * kStageBytesDN;
            const uint32_t *ws = reinterpret_cast<const uint32_t *>(st);
            const float *xs = reinterpret_cast<const float *>(st + kBoxBytesDN);
            float a0[kNT], a1[kNT];
#pragma unroll
            for (int q = 0; q < kNT; ++q) a0[q] = a1[q] = 0.0f;
#pragma unroll 4
            for (int rr = 0; rr < kRowsPerWarpDN; ++rr) {
                const int row = cw * kRowsPerWarpDN + rr;
                const uint32_t w2 = ws[row * (kTN / 2) + lane];
                const float w0 = bf16_lo(w2), w1 = bf16_hi(w2);
#pragma unroll
                for (int q = 0; q < kNT; ++q) {
                    if (q < ntok) {
                        const float xv = xs[q * kIG + row];
                        a0[q] = fmaf(xv, w0, a0[q]);
                        a1[q] = fmaf(xv, w1, a1[q]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl.empty[stage]);
#pragma unroll
            for (int q = 0; q < kNT; ++q)
                if (q < ntok)
                    *reinterpret_cast<float2 *>(&red[(cw * kNT + q) * kTN + 2 * lane]) =
                        make_float2(a0[q], a1[q]);
            named_bar_sync(1, kConsumerThreads);
            const int col0 = ht * kTN;
#pragma unroll
            for (int pass = 0; pass < 2; ++pass) {
                const int idx = ctid + pass * kConsumerThreads;
                const int q = idx / kTN, c = idx % kTN;
                const int r = pass ? r1 : r0;
                if (q < ntok) {
                    float s = red[q * kTN + c];
#pragma unroll
                    for (int w = 1; w < kConsumerWarps; ++w) s += red[(w * kNT + q) * kTN + c];
                    a.part_dn[((int64_t)ig * R + r) * a.H + col0 + c] = s;
                }
            }
            __threadfence();
            named_bar_sync(1, kConsumerThreads);
            if (ctid < ntok) {
                const int m = rq / a.k;
                int nvalid = 0;
                for (int j = 0; j < a.k; ++j) {
                    const int e = a.topk_ids[(size_t)m * a.k + j];
                    nvalid += (e >= 0 && e < a.E);
                }
                int *cnt = &a.cnt_dn[(size_t)m * a.n_ht + ht];
                const int old = atomicAdd(cnt, 1);
                const bool last = (old + 1 == nvalid * a.n_ig);
                if (last) atomicExch(cnt, 0);
                ctl.fin[ctid] = last ? m : -1;
            }
            named_bar_sync(1, kConsumerThreads);
            for (int idx = ctid; idx < ntok * kTN; idx += kConsumerThreads) {
                const int q = idx / kTN, c = idx % kTN;
                const int m = ctl.fin[q];
                if (m < 0) continue;
                __threadfence();
                float acc = 0.0f;
                for (int j = 0; j < a.k; ++j) {
                    const int64_t r = (int64_t)m * a.k + j;
                    const int e = a.topk_ids[r];
                    if (e < 0 || e >= a.E) continue;
                    float y = 0.0f;
                    for (int gi = 0; gi < a.n_ig; ++gi)
                        y += __ldcg(&a.part_dn[((int64_t)gi * R + r) * a.H + col0 + c]);
                    acc = fmaf(a.topk_wts[r], y, acc);
                }
                const size_t o = (size_t)m * a.H + col0 + c;
                const float res = a.residual ? __bfloat162float(a.residual[o]) : 0.0f;
                a.out[o] = __float2bfloat16(res + acc);
            }
        } else {
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl.empty[stage]);
        }
        if (++stage == kStagesDN) {
            stage = 0;
            phase ^= 1u;
        }
    }
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

}  // namespace moe
