// gemm_tc05.cu -- expert projections of the large-batch regime as grouped GEMMs on the
// fifth-generation tensor cores (tcgen05.mma, accumulators in tensor memory).
//
// The computation is the expert step of "A Multi-Engine Dataflow for MoE Decoding on
// Scratchpad-Based Tensor Accelerators" (stage-3 activation; Section 4.3), for the rows of
// the aligned 64-row blocks of "Route-Block Membership Selects Packed-AWQ Arithmetic"
// (Section 2.1): every block holds routes of one expert, so a block is a dense GEMM tile.
//
// Orientation ("swap AB"): the expert weights are the MMA's A operand (M = 128 output
// channels) and the block's 64 routes are the N side, so the weights stream through HBM
// once per block and the routes ride along:
//   gate/up:  D[128][64] = [W_gate[e][:, i0:i0+64] | W_up[e][:, i0:i0+64]]^T  x  X^T
//             (lanes 0-63 accumulate g, lanes 64-127 accumulate u, of channels i0..i0+63)
//   down:     D[128][64] = W_down[e][:, h0:h0+128]^T  x  P^T
// A comes straight from the [E,H,I] / [E,I,H] weights: TMA boxes of 64 columns x 128 rows
// with 128-byte swizzle form the MN-major canonical layout (one 64-wide M half per box).
// B (the block's token rows of h, or of p) is gathered by a loader warp with 16-byte
// cp.async copies into the K-major 128-byte-swizzle layout; sentinel rows become zeros.
// Per CTA: warp 0 issues the weight TMA, warp 1 loads B, one thread of warp 2 issues the
// MMAs (K = 16 each) into one of two tensor-memory accumulators, and warps 4-7 drain the
// finished accumulator: gate/up computes p = SiLU(g) * u and writes it as bf16 rows for the
// down GEMM; down writes y per route for the fixed-order combine.  Persistent CTAs take
// units (block, channel tile) round-robin, channel tile fastest, so the units of one block
// and of neighbouring blocks of the same expert run side by side and share weight reads.
//
// Each output element is one K-ordered chain of MMAs into its accumulator, independent of
// the other columns of the block, of the grid and of M: the results are bitwise
// reproducible and a route's bits do not depend on the block position it occupies.
#include "moe_internal.cuh"
#include "ptx.cuh"

namespace moe {

constexpr int kGN = 64;                              // routes per MMA (one aligned block)
constexpr int kGM = 128;                             // output channels per MMA
constexpr int kGK = 128;                             // K per stage
constexpr int kGStages = 4;
constexpr int kGHalfBytes = 64 * kGK * 2;            // one 64-wide M half: 16 KB
constexpr int kGABytes = 2 * kGHalfBytes;            // 32 KB
constexpr int kGBBytes = kGN * kGK * 2;              // 16 KB
constexpr int kGStageBytes = kGABytes + kGBBytes;    // 48 KB
constexpr int kGThreads = 256;                       // 8 warps
constexpr uint32_t kGTmemCols = 2 * kGN;             // two 128 x 64 fp32 accumulators
constexpr int kGEpiWarp0 = 4;

struct GCtl {
    uint64_t full[kGStages];
    uint64_t empty[kGStages];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t done;
    uint32_t tmem;
    volatile int abort;
    int rows[kGN];        // loader: source row of each block row (-1: zeros)
    int route[2][kGN];    // epilogue: route of each block row, per accumulator
};

__device__ __forceinline__ bool gwait(uint64_t *bar, uint32_t parity, GCtl &ctl) {
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

__device__ __forceinline__ void gadvance(int &stage, uint32_t &phase) {
    if (++stage == kGStages) {
        stage = 0;
        phase ^= 1u;
    }
}

// The route of aligned row `pos` of a block of expert e, or -1 for padding and for a row
// whose route does not belong to e (flagged, then skipped like padding).
__device__ __forceinline__ int gemm_route(const GemmArgs &a, int64_t pos, int e, bool flag) {
    const int r = a.sorted[pos];
    if (r < 0 || r >= a.R) return -1;
    if (a.ids[r] != e) {
        if (flag) atomicOr(a.status, MOE_DEV_BAD_ALIGNMENT);
        return -1;
    }
    return r;
}

__device__ __forceinline__ int64_t gemm_blocks(const GemmArgs &a) {
    const int64_t n = a.npad[0] / kGN;
    const int64_t cap_blocks = a.cap / kGN;
    return n < 0 ? 0 : (n > cap_blocks ? cap_blocks : n);
}

// Weight boxes of one unit: `issue(stage_smem, bar, e, ct, s)` copies the A tile of K-step s.
template <typename IssueFn>
__device__ void gemm_producer(const GemmArgs &a, GCtl &ctl, unsigned char *stages, int64_t T,
                              int n_ct, int nks, IssueFn issue) {
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued = 0, parity_bits = 0;
    for (int64_t u = blockIdx.x; u < T && !ctl.abort; u += gridDim.x) {
        const int64_t blk = u / n_ct;
        const int ct = (int)(u % n_ct);
        int e = a.blocks[blk];
        if (e < 0 || e >= a.E) {
            atomicOr(a.status, MOE_DEV_BAD_ALIGNMENT);
            e = 0;  // keep the pipeline in step; the rows of such a block are all padding
        }
        for (int s = 0; s < nks; ++s) {
            if (!gwait(&ctl.empty[stage], phase ^ 1u, ctl)) break;
            uint64_t *bar = &ctl.full[stage];
            mbar_arrive_expect_tx(bar, kGABytes);
            issue(stages + stage * kGStageBytes, bar, e, ct, s);
            issued |= 1u << stage;
            parity_bits = (parity_bits & ~(1u << stage)) | (phase << stage);
            gadvance(stage, phase);
        }
    }
    for (int s = 0; s < kGStages; ++s)
        if ((issued >> s) & 1u)
            if (!mbar_wait_bounded(&ctl.full[s], (parity_bits >> s) & 1u)) ctl.abort = 1;
}

// B tiles: the 64 rows of the unit's block, K-step s, into the K-major swizzled layout
// (element (n, k): 8 KB per 64-wide K half, 1 KB per 8 rows, 16-byte chunk c of row n at
// position c ^ (n % 8)).  Row n comes from src + rows[n] * ld, or is zero when rows[n] < 0.
template <bool kDownB>
__device__ void gemm_loader(const GemmArgs &a, GCtl &ctl, unsigned char *stages, int64_t T,
                            int n_ct, int nks) {
    const int lane = threadIdx.x & 31;
    const __nv_bfloat16 *src = a.x;
    const int64_t ld = kDownB ? a.I : a.H;
    int stage = 0;
    uint32_t phase = 0;
    for (int64_t u = blockIdx.x; u < T && !ctl.abort; u += gridDim.x) {
        const int64_t blk = u / n_ct;
        const int e = a.blocks[blk];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int n = lane + 32 * h;
            int row;
            if (kDownB) {
                row = (int)(blk * kGN + n);  // p rows are stored in aligned-row order
            } else {
                const int r = gemm_route(a, blk * kGN + n, e, u % n_ct == 0);
                row = r >= 0 ? r / a.k : -1;
            }
            ctl.rows[n] = row;
        }
        __syncwarp();
        for (int s = 0; s < nks; ++s) {
            bool ok = true;
            if (lane == 0) ok = gwait(&ctl.empty[stage], phase ^ 1u, ctl);
            if (!__shfl_sync(0xffffffffu, ok, 0)) {
                cp_async_wait_all();
                return;
            }
            unsigned char *B = stages + stage * kGStageBytes + kGABytes;
#pragma unroll 4
            for (int j = 0; j < (kGN * kGK * 2 / 16) / 32; ++j) {
                const int id = j * 32 + lane;
                const int n = id >> 4, c = id & 15;
                const int row = ctl.rows[n];
                const __nv_bfloat16 *g = src + (int64_t)(row >= 0 ? row : 0) * ld + s * kGK + c * 8;
                unsigned char *dst = B + (c >> 3) * 8192 + (n >> 3) * 1024 + (n & 7) * 128 +
                                     (((c & 7) ^ (n & 7)) << 4);
                cp_async_16_zfill(dst, g, row >= 0 ? 16u : 0u);
            }
            cp_async_mbar_arrive(&ctl.full[stage]);
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl.full[stage]);
            gadvance(stage, phase);
        }
        __syncwarp();
    }
    cp_async_wait_all();
}

// MMA issuer (one thread): for each unit, nks stages x 8 MMAs of K = 16 into accumulator
// buffer (unit parity); each stage is released when its MMAs complete.
__device__ void gemm_mma(GCtl &ctl, unsigned char *stages, int64_t T, int nks) {
    constexpr uint32_t idesc = umma_idesc_bf16(kGM, kGN, true, false);
    int stage = 0;
    uint32_t phase = 0;
    int local = 0;
    for (int64_t u = blockIdx.x; u < T && !ctl.abort; u += gridDim.x, ++local) {
        const int buf = local & 1;
        const uint32_t tph = (uint32_t)(local >> 1) & 1u;
        if (!gwait(&ctl.tempty[buf], tph ^ 1u, ctl)) break;
        tc_fence_after();
        const uint32_t d = ctl.tmem + (uint32_t)(buf * kGN);
        bool ok = true;
        for (int s = 0; s < nks; ++s) {
            if (!gwait(&ctl.full[stage], phase, ctl)) {
                ok = false;
                break;
            }
            tc_fence_after();
            fence_proxy_async_smem();  // the B rows arrived through cp.async (generic proxy)
            const uint32_t A = smem_u32(stages + stage * kGStageBytes);
            const uint32_t B = A + kGABytes;
#pragma unroll
            for (int ks = 0; ks < kGK / 16; ++ks) {
                // A: MN-major, M halves 16 KB apart, 8-row K atoms 1 KB apart, 16 K rows per MMA
                const uint64_t ad = umma_smem_desc(A + ks * 2048, kGHalfBytes, 1024, 2);
                // B: K-major, 64-wide K halves 8 KB apart, 32 bytes per K step, 8-row atoms 1 KB
                const uint64_t bd = umma_smem_desc(B + (ks >> 2) * 8192 + (ks & 3) * 32, 16, 1024, 2);
                umma_bf16(d, ad, bd, idesc, s > 0 || ks > 0);
            }
            umma_commit(&ctl.empty[stage]);
            gadvance(stage, phase);
        }
        if (!ok) break;
        umma_commit(&ctl.tfull[buf]);
    }
    // every issued MMA has completed before the CTA frees its tensor memory
    umma_commit(&ctl.done);
    if (!mbar_wait_bounded(&ctl.done, 0)) ctl.abort = 1;
}

__device__ __forceinline__ void gemm_init(GCtl &ctl, int warp) {
    if (threadIdx.x == 0) {
        for (int s = 0; s < kGStages; ++s) {
            mbar_init(&ctl.full[s], 2);  // weight TMA + B loader
            mbar_init(&ctl.empty[s], 1);  // MMA completion
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&ctl.tfull[b], 1);
            mbar_init(&ctl.tempty[b], 4);  // the 4 epilogue warps
        }
        mbar_init(&ctl.done, 1);
        ctl.abort = 0;
        fence_mbar_init();
    }
    if (warp == 2) tmem_alloc(&ctl.tmem, kGTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
}

__device__ __forceinline__ void gemm_finish(GCtl &ctl, int warp, int32_t *status) {
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 2) tmem_dealloc(ctl.tmem, kGTmemCols);
    if (threadIdx.x == 0 && ctl.abort) atomicOr(status, MOE_DEV_WAIT_TIMEOUT);
}

// ---------------------------------------------------------------------------- gate/up
__global__ void __launch_bounds__(kGThreads, 1)
    gemm_gateup_kernel(const __grid_constant__ CUtensorMap tm_gate,
                       const __grid_constant__ CUtensorMap tm_up, const GemmArgs a) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *base = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char *stages = base;
    float *gbuf = reinterpret_cast<float *>(base + kGStages * kGStageBytes);  // [64 rows][64 ch]
    GCtl &ctl = *reinterpret_cast<GCtl *>(base + kGStages * kGStageBytes + 64 * 64 * 4);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        prefetch_tensormap(&tm_gate);
        prefetch_tensormap(&tm_up);
    }
    gemm_init(ctl, warp);
    pdl_wait();
    pdl_launch_dependents();

    const int n_ct = a.I / 64;
    const int nks = a.H / kGK;
    const int64_t T = gemm_blocks(a) * n_ct;

    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            gemm_producer(a, ctl, stages, T, n_ct, nks,
                          [&](unsigned char *st, uint64_t *bar, int e, int ct, int s) {
                const int32_t y = e * a.H + s * kGK;
                tma_load_2d(st, &tm_gate, ct * 64, y, bar, pol);
                tma_load_2d(st + kGHalfBytes, &tm_up, ct * 64, y, bar, pol);
            });
        }
        __syncwarp();
    } else if (warp == 1) {
        gemm_loader<false>(a, ctl, stages, T, n_ct, nks);
    } else if (warp == 2) {
        if (lane == 0) gemm_mma(ctl, stages, T, nks);
        __syncwarp();
    } else if (warp >= kGEpiWarp0) {
        const int ew = warp - kGEpiWarp0;  // TMEM lanes [32 ew, 32 ew + 32)
        const int row = 32 * ew + lane;    // accumulator row: gate channel (< 64) or up channel
        int local = 0;
        for (int64_t u = blockIdx.x; u < T; u += gridDim.x, ++local) {
            const int64_t blk = u / n_ct;
            const int ct = (int)(u % n_ct);
            const int buf = local & 1;
            const uint32_t tph = (uint32_t)(local >> 1) & 1u;
            const bool ok = gwait(&ctl.tfull[buf], tph, ctl);
            if (named_bar_or(2, 128, !ok)) break;
            tc_fence_after();
            float v[kGN];
#pragma unroll
            for (int c0 = 0; c0 < kGN; c0 += 16) {
                float t16[16];
                tmem_ld16(ctl.tmem + ((uint32_t)(32 * ew) << 16) + (uint32_t)(buf * kGN + c0), t16);
#pragma unroll
                for (int i = 0; i < 16; ++i) v[c0 + i] = t16[i];
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl.tempty[buf]);  // accumulator free for the next unit
            if (ew < 2) {
#pragma unroll
                for (int n = 0; n < kGN; ++n) gbuf[n * 64 + row] = v[n];
            }
            named_bar_sync(2, 128);
            if (ew >= 2) {
                const int ch = row - 64;
                __nv_bfloat16 *dst = a.p_rows + (blk * kGN) * a.I + ct * 64 + ch;
#pragma unroll
                for (int n = 0; n < kGN; ++n)
                    dst[(int64_t)n * a.I] = __float2bfloat16(silu_f32(gbuf[n * 64 + ch]) * v[n]);
            }
            named_bar_sync(2, 128);
        }
    }
    gemm_finish(ctl, warp, a.status);
}

// ------------------------------------------------------------------------------- down
__global__ void __launch_bounds__(kGThreads, 1)
    gemm_down_kernel(const __grid_constant__ CUtensorMap tm_down, const GemmArgs a) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *base = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char *stages = base;
    GCtl &ctl = *reinterpret_cast<GCtl *>(base + kGStages * kGStageBytes);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) prefetch_tensormap(&tm_down);
    gemm_init(ctl, warp);
    // The weights of each unit are known from the alignment, which was complete before the
    // gate/up grid started: the weight producer streams right away, the p loader and the
    // epilogue wait for the gate/up grid.
    const int n_ct = a.H / kGM;
    const int nks = a.I / kGK;
    const int64_t T = gemm_blocks(a) * n_ct;

    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            gemm_producer(a, ctl, stages, T, n_ct, nks,
                          [&](unsigned char *st, uint64_t *bar, int e, int ct, int s) {
                const int32_t y = e * a.I + s * kGK;
                tma_load_2d(st, &tm_down, ct * kGM, y, bar, pol);
                tma_load_2d(st + kGHalfBytes, &tm_down, ct * kGM + 64, y, bar, pol);
            });
        }
        __syncwarp();
    } else if (warp == 1) {
        pdl_wait();
        gemm_loader<true>(a, ctl, stages, T, n_ct, nks);
    } else if (warp == 2) {
        if (lane == 0) gemm_mma(ctl, stages, T, nks);
        __syncwarp();
    } else if (warp >= kGEpiWarp0) {
        pdl_wait();
        pdl_launch_dependents();
        const int ew = warp - kGEpiWarp0;
        const int ch = 32 * ew + lane;  // output channel within the 128-channel tile
        int local = 0;
        for (int64_t u = blockIdx.x; u < T; u += gridDim.x, ++local) {
            const int64_t blk = u / n_ct;
            const int ct = (int)(u % n_ct);
            const int buf = local & 1;
            const uint32_t tph = (uint32_t)(local >> 1) & 1u;
            if (ch < kGN) ctl.route[buf][ch] = gemm_route(a, blk * kGN + ch, a.blocks[blk], false);
            const bool ok = gwait(&ctl.tfull[buf], tph, ctl);
            if (named_bar_or(2, 128, !ok)) break;
            tc_fence_after();
            float v[kGN];
#pragma unroll
            for (int c0 = 0; c0 < kGN; c0 += 16) {
                float t16[16];
                tmem_ld16(ctl.tmem + ((uint32_t)(32 * ew) << 16) + (uint32_t)(buf * kGN + c0), t16);
#pragma unroll
                for (int i = 0; i < 16; ++i) v[c0 + i] = t16[i];
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl.tempty[buf]);
            float *ybase = a.y + ct * kGM + ch;
#pragma unroll
            for (int n = 0; n < kGN; ++n) {
                const int r = ctl.route[buf][n];
                if (r >= 0) ybase[(int64_t)r * a.H] = v[n];
            }
            named_bar_sync(2, 128);  // route[buf] may be refilled two units later
        }
    }
    gemm_finish(ctl, warp, a.status);
}

static size_t gemm_gateup_smem() { return 1024 + kGStages * kGStageBytes + 64 * 64 * 4 + sizeof(GCtl); }
static size_t gemm_down_smem() { return 1024 + kGStages * kGStageBytes + sizeof(GCtl); }

cudaError_t launch_gemm_gateup(const CUtensorMap &tm_gate, const CUtensorMap &tm_up,
                               const GemmArgs &a, cudaStream_t stream) {
    const size_t smem = gemm_gateup_smem();
    cudaError_t err = cudaFuncSetAttribute(gemm_gateup_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    cudaLaunchAttribute attrs[2];
    cudaLaunchConfig_t cfg = launch_config(dim3(num_sms()), dim3(kGThreads), smem, stream, attrs, 0);
    return cudaLaunchKernelEx(&cfg, gemm_gateup_kernel, tm_gate, tm_up, a);
}

cudaError_t launch_gemm_down(const CUtensorMap &tm_down, const GemmArgs &a, cudaStream_t stream) {
    const size_t smem = gemm_down_smem();
    cudaError_t err = cudaFuncSetAttribute(gemm_down_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    cudaLaunchAttribute attrs[2];
    cudaLaunchConfig_t cfg = launch_config(dim3(num_sms()), dim3(kGThreads), smem, stream, attrs, 0);
    return cudaLaunchKernelEx(&cfg, gemm_down_kernel, tm_down, a);
}

}  // namespace moe
