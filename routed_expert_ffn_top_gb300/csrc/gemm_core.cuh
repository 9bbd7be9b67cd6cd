// gemm_core.cuh -- the pieces of the tcgen05 grouped-GEMM kernels that every kernel shares:
// tile shapes, the control block (mbarriers of the copy ring and of the two tensor-memory
// accumulators), bounded waits, set-up and teardown, and the accumulator drain.
#pragma once

#include "moe_internal.cuh"
#include "ptx.cuh"

namespace moe {

constexpr int kGM = 128;                             // output channels per MMA
constexpr int kGThreads = 192;                       // 6 warps
constexpr int kGMaxStages = 8;

// The shapes of one tile width kN (the MMA's N: 16 or 64 aligned rows).  A stage is the two
// 32 KB weight boxes (64 columns x 256 rows of K, one per 64-wide M half) and the tile's
// 256-deep slice of rows; narrow tiles keep three stages in flight, wide ones two.  (Stages
// of 128 rows, six in flight, were slower for narrow tiles at 1 to 8 tokens.)
template <int kN>
struct GTile {
    static_assert(kN == 16 || kN == 64, "tile widths: 16 or 64 rows");
    static constexpr int kK = kGemmStageK;                    // K per stage
    static constexpr int kHalfBytes = 64 * kK * 2;            // one M half: 32 KB
    static constexpr int kABytes = 2 * kHalfBytes;            // 64 KB
    static constexpr int kBBytes = kN * kK * 2;               // 8 KB or 32 KB
    static constexpr int kStageBytes = kABytes + kBBytes;     // 72 KB or 96 KB
    static constexpr int kStages = kN == 16 ? 3 : 2;
    static constexpr int kChunkBytes = kN * 64 * 2;         // one 64-wide K chunk: 2 or 8 KB
    static constexpr uint32_t kTmemCols = 2 * kN < 32 ? 32 : 2 * kN;  // two accumulators
    static constexpr int kBOff = kABytes;                   // the row slice after the weights
    static constexpr int kTxBytes = kStageBytes;            // bytes the stage's copies bring
    static constexpr int kTileN = kN;
    static constexpr int kDefer = kStages;  // row-slice copies held back until griddepcontrol
    static constexpr bool kSplitB = false;  // one barrier for the weights and the row slice
};

// The VQ gate/up kernel (tiles of kN = 16 or 64 rows, code words of kD).  A unit is a tile and
// 128 output channels of both projections: two M = 128 MMAs per K step, into a gate and an
// up accumulator.  Its copy ring holds, per 256-deep stage, the gate and up index boxes
// (256 / kD index rows x 128 columns of uint8 each, by TMA: 128-byte rows) and the tile's row
// slice (behind a barrier of its own, so that decoding starts as soon as the index boxes
// land).  The weight operand is decoded into tensor memory: slots of 64 K rows (32 columns
// per projection) after the accumulators, six in flight with 16-row tiles and three with
// 64-row ones (whose accumulators take 256 columns).  The code books sit in shared memory
// with each entry repeated kReps times across the banks, so that the lanes of one wavefront,
// each reading its own repeat, never share a bank.
template <int kD, int kN>
struct GTileVQ {
    static_assert(kD == 4 || kD == 8, "code words of 4 or 8");
    static_assert(kN == 16 || kN == 64, "tile widths: 16 or 64 rows");
    static constexpr int kK = kGemmStageK;
    static constexpr int kCT = 128;                         // channels per unit and projection
    static constexpr int kJRows = kK / kD;
    static constexpr int kJBytes = kJRows * kCT;            // one projection's index box
    static constexpr int kBOff = 2 * kJBytes;
    static constexpr int kBBytes = kN * kK * 2;
    static constexpr int kStageBytes = kBOff + kBBytes;     // 24/16 KB (16 rows), 48/40 KB (64)
    static constexpr int kTxBytes = kStageBytes;
    static constexpr int kStages = kN == 16 ? (kD == 4 ? 6 : 8) : 3;
    static constexpr int kChunkBytes = kN * 64 * 2;
    static constexpr uint32_t kTmemCols = 512;
    static constexpr int kTileN = kN;
    static constexpr int kDefer = 2;
    static constexpr bool kSplitB = true;  // decoders wait for the index boxes only
    static constexpr int kDecWarps = 8;    // per TMEM lane quadrant one gate and one up warp
    static constexpr int kSlotK = 64;                       // K rows per tensor-memory slot
    static constexpr int kSlotsPerStage = kK / kSlotK;
    static constexpr int kSlots = kN == 16 ? 6 : 3;
    static constexpr uint32_t kSlotCols = 64;               // gate 32 columns, then up 32
    static constexpr uint32_t kAccCols = 4 * kN;            // two buffers of gate and up
    static constexpr uint32_t kSlotCol0 = kAccCols < 64 ? 64 : kAccCols;
    static constexpr int kReps = kD == 4 ? 16 : 8;          // 8-byte words: 16 lanes a wavefront
    static constexpr int kEntryBytes = kReps * kD * 2;      // 128
    static constexpr int kCbBytes = 256 * kEntryBytes;      // one projection's code book
    static_assert(kStageBytes % 1024 == 0 && kBOff % 1024 == 0, "stage alignment");
    static_assert(kSlotCol0 + kSlots * kSlotCols <= kTmemCols, "tensor memory");
    static_assert(kSlots <= kGMaxStages && kStages <= kGMaxStages, "barriers");
};

struct GCtl {
    uint64_t full[kGMaxStages];
    uint64_t empty[kGMaxStages];
    uint64_t bfull[kGMaxStages];  // VQ: the stage's row slice has landed
    uint64_t afull[kGMaxStages];   // VQ: a tensor-memory slot of the weight operand is written
    uint64_t aempty[kGMaxStages];  // VQ: the MMAs reading a slot have completed
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t done;
    uint32_t tmem;
    volatile int abort;
    int route[2][kGemmBlock];  // down epilogue: route of each tile row, per accumulator
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

template <typename L>
__device__ __forceinline__ void gadvance(int &stage, uint32_t &phase) {
    if (++stage == L::kStages) {
        stage = 0;
        phase ^= 1u;
    }
}

// decoder_warps (VQ): warps that also read each stage (its index boxes) before it is free,
// and fill the tensor-memory slots of the weight operand.
// full_arrivals: arrivals that complete a stage besides its copies' bytes (the producer's
// expect_tx arrival, and one more when another warp also fills the stage).
template <typename G>
__device__ __forceinline__ void gemm_init(GCtl &ctl, int warp, int decoder_warps = 0,
                                          int full_arrivals = 1) {
    if (threadIdx.x == 0) {
        for (int s = 0; s < G::kStages; ++s) {
            mbar_init(&ctl.full[s], full_arrivals);       // the producer's expect_tx arrival(s)
            mbar_init(&ctl.empty[s], 1 + decoder_warps);  // MMA completion (+ decoders)
        }
        for (int s = 0; s < kGMaxStages && decoder_warps; ++s) {
            mbar_init(&ctl.afull[s], decoder_warps);
            mbar_init(&ctl.aempty[s], 1);
        }
        for (int s = 0; s < G::kStages && G::kSplitB; ++s) mbar_init(&ctl.bfull[s], 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&ctl.tfull[b], 1);
            mbar_init(&ctl.tempty[b], 4);  // the 4 epilogue warps
        }
        mbar_init(&ctl.done, 1);
        ctl.abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(&ctl.tmem, G::kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
}

template <typename G>
__device__ __forceinline__ void gemm_finish(GCtl &ctl, int warp, int32_t *status) {
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(ctl.tmem, G::kTmemCols);
    if (threadIdx.x == 0 && ctl.abort) atomicOr(status, MOE_DEV_WAIT_TIMEOUT);
}

// Epilogue warp: the kN fp32 columns of its 32 TMEM lanes of accumulator `buf`, then the
// accumulator is handed back to the MMA issuer.
template <int kN>
__device__ __forceinline__ void drain_accumulator(GCtl &ctl, int quad, int buf, float (&v)[kN]) {
    tc_fence_after();
#pragma unroll
    for (int c0 = 0; c0 < kN; c0 += 16) {
        float t16[16];
        tmem_ld16(ctl.tmem + ((uint32_t)(32 * quad) << 16) + (uint32_t)(buf * kN + c0), t16);
#pragma unroll
        for (int i = 0; i < 16; ++i) v[c0 + i] = t16[i];
    }
    tc_fence_before();
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&ctl.tempty[buf]);
}

}  // namespace moe
