// gemv.cu -- expert kernels for blockwise-VQ gate/up weights (GEMV streams on CUDA cores):
// VQ (and VQ + low-rank) gate/up, the bf16 down projection and the combine that follow it.
// Dense weights run on the tensor cores instead (gemm_tc05.cu).
//
// The expert computation of "A Multi-Engine Dataflow for MoE Decoding on Scratchpad-Based
// Tensor Accelerators" (MoE block background; stage-3 activation; Section 4.3):
//   gate/up:  g = h W_gate[e], u = h W_up[e], p = SiLU(g) * u        (per route)
//   down:     y = p W_down[e]
//   combine:  out[m] = residual[m] + sum_j a_{m,j} y_{m,j}   ("accumulated summation")
// and, channel by channel, "Channel Selection for Mixture-of-Experts Decoding Needs No
// Calibration Data" (Background: channel j owns row j of gate/up and column j of down).
//
// At decode batch sizes every weight byte serves only a handful of tokens, so both expert
// kernels are HBM streams, and what bounds them is how many bytes each SM keeps in flight.
// An SM's tensor-memory-access unit works on only a few copies at a time, so every weight
// copy here is one large box (256 rows x 64 columns of bf16 = 32 KB), and the small
// activation slices travel separately through 16-byte cp.async copies.
//
// Work is cut into tiles over the aligned rows:
//   * a sub-block is `rsub` consecutive aligned rows: at most 8 routes of ONE expert (the
//     alignment pads every expert to a multiple of b and rsub divides b); its record
//     (expert, routes, tokens) comes from the sub-block table the alignment step wrote;
//   * gate/up tile = (sub-block, 64-column I tile): the index boxes of J_gate[e] and
//     J_up[e] in that column range (each covering 1024 rows of H), alternating gate and up;
//   * down tile = (sub-block, 64-column H tile): all I rows of W_down[e], I/256 boxes.
// Persistent CTAs (one per SM) own tiles c, c + G, c + 2G ... (G = grid size); tiles are
// numbered column tile fastest, so neighbouring SMs stream neighbouring column ranges of
// the same rows.  Warp 0 (one thread) issues the TMA box copies into a ring of stages;
// warp 1 copies each stage's activation slices (h rows for gate/up, p rows for down) with
// cp.async and hangs them on the same full barrier; warps 2..9 consume.  Consumer warp w
// owns rows [32w, 32w+32) of every box; lane l the 16 rows [32w + 16(l/16), +16) and the 4
// columns [4(l%16), +4); fp32 accumulators for up to 8 tokens live in registers across all
// boxes of the tile (gate/up dots h with code words decoded from shared memory; down uses
// packed fp32 FMAs on fp32 p).  At the end of a tile the two lane halves and then the 8
// warps are summed, and the epilogue writes p (gate/up) or y (down).  A third small kernel
// forms out = residual + sum_j a_j y_j in slot order j = 0..k-1.
//
// Reduction order, fixed by tile indices only (never by grid size, CTA, block position,
// batch size or arrival order): per thread, boxes ascending and rows ascending inside its
// 16-row slice; then the two lane halves; then warps 0..7; then, for the combine, slots
// 0..k-1.  So the results are bitwise reproducible, a route's bits do not depend on the
// block it sits in or on the other routes of its block, and a token's output does not
// depend on M.
#include "moe_internal.cuh"
#include "ptx.cuh"
#include "route_core.cuh"
#include "small_route.cuh"

namespace moe {

constexpr int kStages = 5;
constexpr int kConsumerThreads = 32 * kConsumerWarps;
constexpr int kRowsPerWarp = kBoxRows / kConsumerWarps;  // 32
constexpr int kRowsPerThread = kRowsPerWarp / 2;         // 16
constexpr int kFirstConsumerWarp = 2;

constexpr int kBoxBytes = kBoxRows * kTI * 2;                 // 32 KB (also kTN == kTI)
constexpr int kStageBytesDN = kBoxBytes + kNT * kBoxRows * 4;  // + p slices (fp32)
constexpr int kRedBytesGU = kConsumerWarps * kNT * kTI * 4;  // g, then u, through one buffer
// VQ gate/up: a box is 256 rows x 64 columns of uint8 code indices (16 KB), i.e. 1024 rows of
// H; its activation slices are those 1024 h values of each route's token.
// VQ gate/up with code words of kD elements (d = 4 or 8): a box is 1024/kD index rows x 64
// columns of uint8 (16 KB at d = 4, 8 KB at d = 8), i.e. 1024 rows of H either way; its
// activation slices are those 1024 h values of each route's token.
constexpr int kVQHRows = 1024;
__host__ __device__ constexpr int vq_rows(int d) { return kVQHRows / d; }
__host__ __device__ constexpr int vq_box_bytes(int d) { return vq_rows(d) * kTI; }
__host__ __device__ constexpr int vq_stage_bytes(int d) { return vq_box_bytes(d) + kNT * kVQHRows * 2; }
__host__ __device__ constexpr int vq_codebook_bytes(int d) { return 256 * d * 2; }  // one projection
// The VQ-only gate/up kernel keeps kCbReps copies of each code book, entry-major (the copies
// of an entry side by side), and lane l reads copy l % kCbReps: the 32 lanes' random entries
// then meet in at most 4 lanes per bank set instead of up to 8 or more (on this GPU a box's
// decoding was bound by those lookups' bank conflicts).  Same values, same order: same bits.
constexpr int kCbReps = 8;
constexpr int kStageBytesVQ = vq_stage_bytes(4);
// VQ + low-rank gate/up: the ring also carries C boxes (256 rows of r x 64 columns, bf16)
// with fp32 z slices, the shape of a down stage.
constexpr int kStageBytesLR = kStageBytesDN;
constexpr int kRedBytesDN = kConsumerWarps * kNT * kTN * 4;
static_assert(kTI == kTN, "one box shape for both kernels");
static_assert(kStageBytesDN % 1024 == 0 && kStageBytesVQ % 1024 == 0, "stage alignment");
static_assert(vq_rows(4) == kBoxRows && vq_rows(8) * 2 == kBoxRows, "VQ boxes of 256 or 128 rows");

enum TileKind { kDown = 1, kVQGateUp = 2, kVQLRGateUp = 3 };

struct Ctl {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    SubBlock meta[kStages];  // the sub-block record of the tile each stage belongs to
    volatile int abort;
};

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

__device__ __forceinline__ void advance(int &stage, uint32_t &phase) {
    if (++stage == kStages) {
        stage = 0;
        phase ^= 1u;
    }
}

__device__ __forceinline__ void load_record(const SubBlock *src, uint4 (&dst)[5]) {
    const uint4 *s = reinterpret_cast<const uint4 *>(src);
#pragma unroll
    for (int i = 0; i < 5; ++i) dst[i] = s[i];
}

__device__ __forceinline__ void init_ring(Ctl &ctl) {
    for (int s = 0; s < kStages; ++s) {
        mbar_init(&ctl.full[s], 2);  // the box producer and the activation loader
        mbar_init(&ctl.empty[s], kConsumerWarps);
    }
    ctl.abort = 0;
    fence_mbar_init();
}

// Box producer (one thread).  A tile with no route is announced by a single stage that
// carries no copies; otherwise `stages_per_tile` stages.  `issue(stage, tile, j, e)` issues
// the TMA copy of stage j of the tile and arms the stage's full barrier.
template <typename IssueFn>
__device__ void box_producer(const GemvArgs &a, Ctl &ctl, int64_t T, int tiles_per_sub,
                             int stages_per_tile, IssueFn issue) {
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued = 0, parity_bits = 0;
    // The record of the next tile is loaded while the current tile streams.
    uint4 cur[5], nxt[5];
    const int64_t G = gridDim.x;
    if ((int64_t)blockIdx.x < T) load_record(a.sbt + blockIdx.x / tiles_per_sub, nxt);
    for (int64_t t = blockIdx.x; t < T && !ctl.abort; t += G) {
#pragma unroll
        for (int i = 0; i < 5; ++i) cur[i] = nxt[i];
        if (t + G < T) load_record(a.sbt + (t + G) / tiles_per_sub, nxt);
        const int e = (int)cur[0].x;
        const int ntok = (int)cur[0].y;
        const int nst = ntok > 0 ? stages_per_tile : 1;
        for (int j = 0; j < nst; ++j) {
            if (!wait_or_abort(&ctl.empty[stage], phase ^ 1u, ctl)) break;
            uint4 *m = reinterpret_cast<uint4 *>(&ctl.meta[stage]);
#pragma unroll
            for (int i = 0; i < 5; ++i) m[i] = cur[i];
            if (ntok > 0)
                issue(stage, t, j, e);
            else
                mbar_arrive(&ctl.full[stage]);
            issued |= 1u << stage;
            parity_bits = (parity_bits & ~(1u << stage)) | (phase << stage);
            advance(stage, phase);
        }
    }
    // Never leave the CTA while copies may still be landing in its shared memory.
    for (int s = 0; s < kStages; ++s)
        if ((issued >> s) & 1u)
            if (!mbar_wait_bounded(&ctl.full[s], (parity_bits >> s) & 1u)) ctl.abort = 1;
    if (ctl.abort) atomicOr(a.status, MOE_DEV_WAIT_TIMEOUT);
}

// Where a stage's activation slices go: after the stage's box (box_bytes), one slice of
// slice_bytes per route, chunks 16-byte pieces per lane.
struct SliceLayout {
    int box_bytes, slice_bytes, chunks;
};

// Activation loader (one warp).  For every stage j the box producer fills, lane l copies
// its pieces of each route's slice, src(route, token, tile, j, piece) -> the stage's slice
// area (a NULL source writes zeros).  Its arrival on the stage's full barrier completes only
// when its copies have landed.
template <typename LayoutFn, typename SrcFn>
__device__ void slice_loader(const GemvArgs &a, Ctl &ctl, unsigned char *stages, int stage_bytes,
                             int64_t T, int tiles_per_sub, int stages_per_tile, LayoutFn layout,
                             SrcFn src) {
    const int lane = threadIdx.x & 31;
    int stage = 0;
    uint32_t phase = 0;
    const int64_t G = gridDim.x;
    for (int64_t t = blockIdx.x; t < T && !ctl.abort; t += G) {
        const SubBlock *rec = a.sbt + t / tiles_per_sub;
        const int ntok = rec->ntok;
        // lane q (< 8) holds route q and its token
        const int my_route = rec->routes[lane & (kNT - 1)];
        const int my_token = rec->tokens[lane & (kNT - 1)];
        const int nst = ntok > 0 ? stages_per_tile : 1;
        for (int j = 0; j < nst; ++j) {
            if (!wait_or_abort(&ctl.empty[stage], phase ^ 1u, ctl)) {
                cp_async_wait_all();
                return;
            }
            if (ntok > 0) {
                const SliceLayout L = layout(j);
                unsigned char *dst = stages + stage * stage_bytes + L.box_bytes;
                for (int q = 0; q < ntok; ++q) {
                    const int route = __shfl_sync(0xffffffffu, my_route, q);
                    const int token = __shfl_sync(0xffffffffu, my_token, q);
                    for (int c = 0; c < L.chunks; ++c) {
                        const unsigned char *g = src(route, token, t, j, lane * L.chunks + c);
                        cp_async_16_zfill(dst + q * L.slice_bytes + (lane * L.chunks + c) * 16,
                                          g ? g : reinterpret_cast<const unsigned char *>(a.h),
                                          g ? 16u : 0u);
                    }
                }
                cp_async_mbar_arrive(&ctl.full[stage]);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl.full[stage]);
            advance(stage, phase);
        }
    }
    cp_async_wait_all();
}

// Per-thread position inside the consumer warps.
struct Lane {
    int ctid;   // 0..255
    int cw;     // consumer warp 0..7
    int lane;
    int half;   // which 16 rows of the warp's 32
    int c4;     // first of the 4 columns
    int rbase;  // first of the 16 rows
};

// acc[q][c] += sum over this thread's 16 rows of p_q[row] * W[row][c4 + c] for NT routes
// (fp32 p, bf16 weights, packed fp32 FMAs, rows ascending).
template <int NT>
__device__ __forceinline__ void accumulate_f32_box(const unsigned char *st, const Lane &ln,
                                                   float (&acc)[NT][4]) {
    const float *xs = reinterpret_cast<const float *>(st + kBoxBytes) + ln.rbase;
#pragma unroll
    for (int r8 = 0; r8 < kRowsPerThread; r8 += 8) {
        float w[8][4];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint2 w2 = *reinterpret_cast<const uint2 *>(st + (ln.rbase + r8 + i) * (kTN * 2) + ln.c4 * 2);
            w[i][0] = bf16_lo(w2.x);
            w[i][1] = bf16_hi(w2.x);
            w[i][2] = bf16_lo(w2.y);
            w[i][3] = bf16_hi(w2.y);
        }
#pragma unroll
        for (int q = 0; q < NT; ++q) {
            const float4 p0 = *reinterpret_cast<const float4 *>(xs + q * kBoxRows + r8);
            const float4 p1 = *reinterpret_cast<const float4 *>(xs + q * kBoxRows + r8 + 4);
            const float x[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                ffma2(acc[q][0], acc[q][1], x[i], w[i][0], w[i][1]);
                ffma2(acc[q][2], acc[q][3], x[i], w[i][2], w[i][3]);
            }
        }
    }
}

// VQ box ("A Multi-Engine Dataflow ...", Section 2.3: column i of W_e is cut into length-d
// blocks along H, block q holding code word J[e][q][i] of the layer-shared code book):
// acc[q][c] += sum over this thread's index rows r of sum_t x_q[d r + t] * cb[J[r][c]][t]
// (bf16 x bf16 -> fp32, H rows ascending).  `cb` is the code book in shared memory, one
// kD-element code word per 8 (d = 4) or 16 (d = 8) bytes.  A warp owns 1/8 of the box's
// index rows, a lane half 1/16 of them.
template <int NT, int kD, int kReps = 1>
__device__ __forceinline__ void accumulate_vq_box(const unsigned char *st, const void *cb,
                                                  const Lane &ln, float (&acc)[NT][4]) {
    constexpr int kRows = vq_rows(kD) / 16;  // index rows per thread: 16 (d = 4), 8 (d = 8)
    const int rb = ln.cw * (2 * kRows) + ln.half * kRows;
    const unsigned char *xs = st + vq_box_bytes(kD) + rb * kD * 2;
    const int rep = ln.lane % kReps;  // this lane's copy of the code book
#pragma unroll(kD == 4 ? 2 : 1)  // (deeper unrolling spills registers)
    for (int i = 0; i < kRows; ++i) {
        const uint32_t jw = *reinterpret_cast<const uint32_t *>(st + (rb + i) * kTI + ln.c4);
        if constexpr (kD == 4) {
            uint2 cw[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) cw[c] = static_cast<const uint2 *>(cb)[((jw >> (8 * c)) & 0xffu) * kReps + rep];
#pragma unroll
            for (int q = 0; q < NT; ++q) {
                const uint2 xv = *reinterpret_cast<const uint2 *>(xs + q * kVQHRows * 2 + i * 8);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    float v = acc[q][c];
                    v = fma_bf16<0, 0>(xv.x, cw[c].x, v);
                    v = fma_bf16<1, 1>(xv.x, cw[c].x, v);
                    v = fma_bf16<0, 0>(xv.y, cw[c].y, v);
                    v = fma_bf16<1, 1>(xv.y, cw[c].y, v);
                    acc[q][c] = v;
                }
            }
        } else {
            uint4 cw[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) cw[c] = static_cast<const uint4 *>(cb)[((jw >> (8 * c)) & 0xffu) * kReps + rep];
#pragma unroll
            for (int q = 0; q < NT; ++q) {
                const uint4 xv = *reinterpret_cast<const uint4 *>(xs + q * kVQHRows * 2 + i * 16);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    float v = acc[q][c];
                    v = fma_bf16<0, 0>(xv.x, cw[c].x, v);
                    v = fma_bf16<1, 1>(xv.x, cw[c].x, v);
                    v = fma_bf16<0, 0>(xv.y, cw[c].y, v);
                    v = fma_bf16<1, 1>(xv.y, cw[c].y, v);
                    v = fma_bf16<0, 0>(xv.z, cw[c].z, v);
                    v = fma_bf16<1, 1>(xv.z, cw[c].z, v);
                    v = fma_bf16<0, 0>(xv.w, cw[c].w, v);
                    v = fma_bf16<1, 1>(xv.w, cw[c].w, v);
                    acc[q][c] = v;
                }
            }
        }
    }
}

// Releases the stage to the box producer and the loader once this warp is done with it.
__device__ __forceinline__ void release_stage(Ctl &ctl, const Lane &ln, int &stage, uint32_t &phase) {
    __syncwarp();
    if (ln.lane == 0) mbar_arrive(&ctl.empty[stage]);
    advance(stage, phase);
}

// Sums the 8 warps' partials of (route q, column c) in warp order; `red` holds, per warp,
// route and column, the value the warp's two lane halves summed.
__device__ __forceinline__ float sum_warps(const float *red, int q, int c) {
    float v = red[q * kTI + c];
#pragma unroll
    for (int w = 1; w < kConsumerWarps; ++w) v += red[(w * kNT + q) * kTI + c];
    return v;
}

// Writes this thread's lane-half sums of acc into red (lanes of the lower half only).
template <int NT>
__device__ __forceinline__ void stage_partials(float *red, const Lane &ln, float (&acc)[NT][4]) {
#pragma unroll
    for (int q = 0; q < NT; ++q) {
        float v[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) v[c] = acc[q][c] + __shfl_xor_sync(0xffffffffu, acc[q][c], 16);
        if (ln.half == 0)
            *reinterpret_cast<float4 *>(&red[(ln.cw * kNT + q) * kTI + ln.c4]) =
                make_float4(v[0], v[1], v[2], v[3]);
    }
}

// One gate/up tile with NT routes; its first stage has already been waited for.  Returns
// false when the CTA must stop (a bounded wait gave up somewhere in the CTA).
// Stages: a gate and an up index box for every 1024 rows of H; with kLR, then a C_gate and
// a C_up box for every 256 rows of r, multiplied by z = D^T h into the same accumulators
// ([MED]'s joint accumulation of the VQ and low-rank terms).
template <int NT, bool kLR, int kD, int kStride = 0, int kReps = 1>
__device__ bool gateup_tile(const GemvArgs &a, Ctl &ctl, unsigned char *stages, float *red,
                            const uint2 *cbs, const Lane &ln, int it, int r0, int r1, int &stage,
                            uint32_t &phase) {
    // stage stride: the gate/up kernel's own (kStride 0), or a ring shared with down tiles
    constexpr int kSt = kStride ? kStride : (kLR ? kStageBytesLR : vq_stage_bytes(kD));
    float ag[NT][4], au[NT][4];
#pragma unroll
    for (int q = 0; q < NT; ++q)
#pragma unroll
        for (int c = 0; c < 4; ++c) ag[q][c] = au[q][c] = 0.0f;
    bool failed = false;
    const int nvq = 2 * a.n_qb;
    const int nst = nvq + (kLR ? 2 * a.n_rb : 0);
    for (int j = 0; j < nst; ++j) {
        if (j > 0 && !wait_or_abort(&ctl.full[stage], phase, ctl)) {
            failed = true;
            break;
        }
        const unsigned char *st = stages + stage * kSt;
        if (kLR && j >= nvq) {
            if ((j - nvq) & 1)
                accumulate_f32_box<NT>(st, ln, au);
            else
                accumulate_f32_box<NT>(st, ln, ag);
        } else {
            const unsigned char *cb = reinterpret_cast<const unsigned char *>(cbs);
            if (j & 1)
                accumulate_vq_box<NT, kD, kReps>(st, cb + vq_codebook_bytes(kD) * kReps, ln, au);
            else
                accumulate_vq_box<NT, kD, kReps>(st, cb, ln, ag);
        }
        release_stage(ctl, ln, stage, phase);
    }
    if (named_bar_or(1, kConsumerThreads, failed)) return false;
    // the two lane halves (rows), then the warps in order: g first, then u
    float g[2];
    stage_partials<NT>(red, ln, ag);
    named_bar_sync(1, kConsumerThreads);
#pragma unroll
    for (int pass = 0; pass < 2; ++pass) {
        const int idx = ln.ctid + pass * kConsumerThreads;
        g[pass] = (idx / kTI < NT) ? sum_warps(red, idx / kTI, idx % kTI) : 0.0f;
    }
    named_bar_sync(1, kConsumerThreads);
    stage_partials<NT>(red, ln, au);
    named_bar_sync(1, kConsumerThreads);
    const int col0 = it * kTI;
#pragma unroll
    for (int pass = 0; pass < 2; ++pass) {
        const int idx = ln.ctid + pass * kConsumerThreads;
        const int q = idx / kTI, c = idx % kTI;
        if (q < NT)
            a.p[(int64_t)(pass ? r1 : r0) * a.I + col0 + c] = silu_f32(g[pass]) * sum_warps(red, q, c);
    }
    named_bar_sync(1, kConsumerThreads);
    return true;
}

// One down tile with NT routes (first stage already waited for); see gateup_tile.
template <int NT, int kStride = kStageBytesDN>
__device__ bool down_tile(const GemvArgs &a, Ctl &ctl, unsigned char *stages, float *red,
                          const Lane &ln, int ht, int r0, int r1, int &stage, uint32_t &phase) {
    float acc[NT][4];
#pragma unroll
    for (int q = 0; q < NT; ++q)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[q][c] = 0.0f;
    bool failed = false;
    for (int j = 0; j < a.n_ib; ++j) {
        if (j > 0 && !wait_or_abort(&ctl.full[stage], phase, ctl)) {
            failed = true;
            break;
        }
        accumulate_f32_box<NT>(stages + stage * kStride, ln, acc);
        release_stage(ctl, ln, stage, phase);
    }
    if (named_bar_or(1, kConsumerThreads, failed)) return false;
#pragma unroll
    for (int q = 0; q < NT; ++q) {
        float v[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) v[c] = acc[q][c] + __shfl_xor_sync(0xffffffffu, acc[q][c], 16);
        if (ln.half == 0)
            *reinterpret_cast<float4 *>(&red[(ln.cw * kNT + q) * kTN + ln.c4]) = make_float4(v[0], v[1], v[2], v[3]);
    }
    named_bar_sync(1, kConsumerThreads);
    const int col0 = ht * kTN;
#pragma unroll
    for (int pass = 0; pass < 2; ++pass) {
        const int idx = ln.ctid + pass * kConsumerThreads;
        const int q = idx / kTN, c = idx % kTN;
        if (q < NT) {
            float sum = red[q * kTN + c];
#pragma unroll
            for (int w = 1; w < kConsumerWarps; ++w) sum += red[(w * kNT + q) * kTN + c];
            a.y[(int64_t)(pass ? r1 : r0) * a.H + col0 + c] = sum;
        }
    }
    named_bar_sync(1, kConsumerThreads);
    return true;
}

// Consumer loop shared by both kernels: waits for a tile's first stage, reads how many routes
// it has, and runs the tile body specialised for that count.
template <int kKind, int kD = 4>
__device__ void consume_tiles(const GemvArgs &a, Ctl &ctl, unsigned char *stages, float *red,
                              const uint2 *cbs, int64_t T, int tiles_per_sub) {
    const int warp = threadIdx.x >> 5;
    Lane ln;
    ln.ctid = threadIdx.x - 32 * kFirstConsumerWarp;
    ln.cw = warp - kFirstConsumerWarp;
    ln.lane = threadIdx.x & 31;
    ln.half = ln.lane >> 4;
    ln.c4 = (ln.lane & 15) * 4;
    ln.rbase = ln.cw * kRowsPerWarp + ln.half * kRowsPerThread;
    const int cols = kKind == kDown ? kTN : kTI;
    int stage = 0;
    uint32_t phase = 0;
    for (int64_t t = blockIdx.x; t < T; t += gridDim.x) {
        const int ct = (int)(t % tiles_per_sub);
        if (!wait_or_abort(&ctl.full[stage], phase, ctl)) {
            named_bar_or(1, kConsumerThreads, true);
            break;
        }
        const SubBlock &mt = ctl.meta[stage];
        const int ntok = mt.ntok;
        const int q0 = ln.ctid / cols, q1 = (ln.ctid + kConsumerThreads) / cols;
        const int r0 = (q0 < ntok) ? mt.routes[q0] : -1;
        const int r1 = (q1 < ntok) ? mt.routes[q1] : -1;
        bool go = true;
#define MOE_TILE(N)                                                                          \
    case N:                                                                                  \
        if constexpr (kKind == kDown)                                                        \
            go = down_tile<N>(a, ctl, stages, red, ln, ct, r0, r1, stage, phase);            \
        else                                                                                 \
            go = gateup_tile<N, kKind == kVQLRGateUp, kD, 0, kKind == kVQGateUp ? kCbReps : 1>( \
                a, ctl, stages, red, cbs, ln, ct, r0, r1, stage, phase);                     \
        break;
        switch (ntok) {
            MOE_TILE(1)
            MOE_TILE(2)
            MOE_TILE(3)
            MOE_TILE(4)
            MOE_TILE(5)
            MOE_TILE(6)
            MOE_TILE(7)
            MOE_TILE(8)
            default:  // an empty tile is announced by a single stage
                release_stage(ctl, ln, stage, phase);
                go = !named_bar_or(1, kConsumerThreads, false);
        }
#undef MOE_TILE
        if (!go) break;
    }
}

// A VQ gate/up CTA with no tile (small batches: fewer tiles than SMs) warms the routed
// experts' W_down in L2 for the down kernel: the index maps are a quarter of the dense
// gate/up bytes, so HBM has room during gate/up (with dense weights it has not, and the
// prefetch would only slow gate/up down).  Every thread of the idle
// CTAs prefetches 128-byte lines (load-store path, so no copy engine queue is held), the
// lines of each expert's first sub-block dealt out round-robin.
__device__ void prefetch_down_weights(const GemvArgs &a, int64_t T) {
    const int64_t idle = (int64_t)gridDim.x - T;
    if ((int64_t)blockIdx.x < T || idle <= 0) return;
    const int64_t n_sub = num_subblocks(a);
    const int64_t lines = (int64_t)a.I * a.H * 2 / 128;  // per expert
    const int64_t stride = idle * blockDim.x;
    for (int64_t sb = 0; sb < n_sub; ++sb) {
        const int e = a.sbt[sb].e;
        if (e < 0 || e >= a.E || a.sbt[sb].ntok == 0) continue;
        if (sb > 0 && a.sbt[sb - 1].e == e) continue;  // not the expert's first sub-block
        const unsigned char *base = a.w_down + (int64_t)e * lines * 128;
        for (int64_t l = ((int64_t)blockIdx.x - T) * blockDim.x + threadIdx.x; l < lines; l += stride)
            prefetch_l2_line(base + l * 128);
    }
}

// ------------------------------------------------------------------------- VQ gate/up
// tm_jgate / tm_jup: index maps [E*H/4 rows][I] uint8, boxes of 256 index rows x 64
// columns.  With kLR also tm_cgate / tm_cup: C [E][r][I] bf16 as 3-D maps (I, r, E), boxes
// of 64 columns x 256 rows of r x 1 expert (rows past r are read as zeros).
template <bool kLR, int kD>
__global__ void __launch_bounds__(kGemvThreads, 1)
    gateup_vq_kernel(const __grid_constant__ CUtensorMap tm_jgate,
                     const __grid_constant__ CUtensorMap tm_jup,
                     const __grid_constant__ CUtensorMap tm_cgate,
                     const __grid_constant__ CUtensorMap tm_cup, const GemvArgs a) {
    constexpr int kSt = kLR ? kStageBytesLR : vq_stage_bytes(kD);
    constexpr int kBox = vq_box_bytes(kD);
    extern __shared__ unsigned char smem_raw[];
    unsigned char *base = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char *stages = base;
    float *red = reinterpret_cast<float *>(base + kStages * kSt);
    uint2 *cbs = reinterpret_cast<uint2 *>(base + kStages * kSt + kRedBytesGU);
    constexpr int kReps = kLR ? 1 : kCbReps;
    Ctl &ctl = *reinterpret_cast<Ctl *>(base + kStages * kSt + kRedBytesGU +
                                        2 * vq_codebook_bytes(kD) * kReps);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        init_ring(ctl);
        prefetch_tensormap(&tm_jgate);
        prefetch_tensormap(&tm_jup);
        if (kLR) {
            prefetch_tensormap(&tm_cgate);
            prefetch_tensormap(&tm_cup);
        }
    }
    // the layer-shared code books (weights, not produced by an earlier kernel), 8 bytes at
    // a time: gate's K d-element words, then up's, kReps copies of each entry side by side
    constexpr int kCbWords = vq_codebook_bytes(kD) / 8;  // 8-byte words per book
    constexpr int kEntWords = kD / 4;                     // 8-byte words per entry
    for (int i = threadIdx.x; i < 2 * kCbWords * kReps; i += blockDim.x) {
        const int book = i / (kCbWords * kReps), r = i - book * kCbWords * kReps;
        const int ent = r / (kEntWords * kReps), w = r % kEntWords;
        const uint2 *src = book ? a.cb_up : a.cb_gate;
        cbs[i] = src[ent * kEntWords + w];
    }
    __syncthreads();
    pdl_wait();
    pdl_launch_dependents();

    const int64_t T = num_subblocks(a) * a.n_it;
    const int nvq = 2 * a.n_qb;
    const int per_tile = nvq + (kLR ? 2 * a.n_rb : 0);
    prefetch_down_weights(a, T);

    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first();
            box_producer(a, ctl, T, a.n_it, per_tile, [&](int stage, int64_t t, int j, int e) {
                const int it = (int)(t % a.n_it);
                uint64_t *bar = &ctl.full[stage];
                unsigned char *dst = stages + stage * kSt;
                if (kLR && j >= nvq) {
                    const int jj = j - nvq;
                    mbar_arrive_expect_tx(bar, kBoxBytes);
                    tma_load_3d(dst, (jj & 1) ? (const void *)&tm_cup : (const void *)&tm_cgate,
                                it * kTI, (jj >> 1) * kBoxRows, e, bar, pol_w);
                } else {
                    mbar_arrive_expect_tx(bar, kBox);
                    tma_load_2d(dst, (j & 1) ? (const void *)&tm_jup : (const void *)&tm_jgate,
                                it * kTI, e * (a.H / kD) + (j >> 1) * vq_rows(kD), bar, pol_w);
                }
            });
        }
        return;
    }
    if (warp == 1) {
        // VQ stages: h rows [1024 (j/2), +1024) of each token, 2 KB = four 16-byte pieces per
        // lane.  Low-rank stages: z rows [256 (jj/2), +256) of the token's gate or up
        // projection, 1 KB = two pieces per lane; rows past r are zeros.
        slice_loader(a, ctl, stages, kSt, T, a.n_it, per_tile,
                     [&](int j) {
                         return (kLR && j >= nvq) ? SliceLayout{kBoxBytes, kBoxRows * 4, 2}
                                                  : SliceLayout{kBox, kVQHRows * 2, 4};
                     },
                     [&](int route, int token, int64_t t, int j, int piece) -> const unsigned char * {
                         if (kLR && j >= nvq) {
                             const int jj = j - nvq;
                             const int row = (jj >> 1) * kBoxRows + piece * 4;
                             if (row >= a.r) return nullptr;
                             return reinterpret_cast<const unsigned char *>(
                                 a.z + (size_t)token * 2 * a.r + (size_t)(jj & 1) * a.r + row);
                         }
                         return reinterpret_cast<const unsigned char *>(a.h) +
                                ((size_t)token * a.H + (size_t)(j >> 1) * kVQHRows) * 2 + piece * 16;
                     });
        return;
    }
    consume_tiles<kLR ? kVQLRGateUp : kVQGateUp, kD>(a, ctl, stages, red, cbs, T, a.n_it);
}

// ------------------------------------------------------------------------------- down
__global__ void __launch_bounds__(kGemvThreads, 1)
    down_kernel(const __grid_constant__ CUtensorMap tm_down, const GemvArgs a) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *base = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char *stages = base;
    float *red = reinterpret_cast<float *>(base + kStages * kStageBytesDN);
    Ctl &ctl = *reinterpret_cast<Ctl *>(base + kStages * kStageBytesDN + kRedBytesDN);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        init_ring(ctl);
        prefetch_tensormap(&tm_down);
    }
    __syncthreads();
    // The routing and the alignment were complete before the gate/up kernel (the grid this
    // one depends on) started its work, so which down weights to read is already known
    // ("A Multi-Engine Dataflow ...", overlap window of the down-projection DMA): the box
    // producer streams W_down right away; only the loader of p, which the gate/up grid
    // writes, waits for that grid.
    const int64_t T = num_subblocks(a) * a.n_ht;

    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first();
            box_producer(a, ctl, T, a.n_ht, a.n_ib, [&](int stage, int64_t t, int j, int e) {
                const int ht = (int)(t % a.n_ht);
                uint64_t *bar = &ctl.full[stage];
                mbar_arrive_expect_tx(bar, kBoxBytes);
                tma_load_2d(stages + stage * kStageBytesDN, &tm_down, ht * kTN,
                            e * a.I + j * kBoxRows, bar, pol_w);
            });
        }
        return;
    }
    if (warp == 1) {
        pdl_wait();
        // p rows [256 j, +256) of each route: 1 KB = two 16-byte pieces per lane
        slice_loader(a, ctl, stages, kStageBytesDN, T, a.n_ht, a.n_ib,
                     [](int) { return SliceLayout{kBoxBytes, kBoxRows * 4, 2}; },
                     [&](int route, int token, int64_t t, int j, int piece) {
                         return reinterpret_cast<const unsigned char *>(a.p) +
                                ((size_t)route * a.I + (size_t)j * kBoxRows) * 4 + piece * 16;
                     });
        return;
    }
    pdl_launch_dependents();
    consume_tiles<kDown>(a, ctl, stages, red, nullptr, T, a.n_ht);
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
    // 8 slots at a time: ids, affinities and y rows are all loaded before any is used (every
    // route has a y row in the workspace; the rows of invalid routes are simply not added)
    for (int j0 = 0; j0 < k; j0 += 8) {
        int e[8];
        float aw[8];
        float4 v[8];
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
            const int64_t r = (int64_t)m * k + j0 + jj;
            if (j0 + jj < k) {
                e[jj] = topk_ids[r];
                aw[jj] = topk_wts[r];
                v[jj] = __ldcg(reinterpret_cast<const float4 *>(y + r * H + n));
            }
        }
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
            if (j0 + jj < k && e[jj] >= 0 && e[jj] < E) {
                acc.x = fmaf(aw[jj], v[jj].x, acc.x);
                acc.y = fmaf(aw[jj], v[jj].y, acc.y);
                acc.z = fmaf(aw[jj], v[jj].z, acc.z);
                acc.w = fmaf(aw[jj], v[jj].w, acc.w);
            }
        }
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

static size_t down_smem() { return 1024 + kStages * kStageBytesDN + kRedBytesDN + sizeof(Ctl); }

static size_t gateup_vq_smem(bool lr, int d) {
    return 1024 + kStages * (lr ? kStageBytesLR : vq_stage_bytes(d)) + kRedBytesGU +
           2 * vq_codebook_bytes(d) * (lr ? 1 : kCbReps) + sizeof(Ctl);
}

template <bool kLR, int kD>
static cudaError_t launch_vq(const CUtensorMap &tm_jgate, const CUtensorMap &tm_jup,
                             const CUtensorMap &tm_cgate, const CUtensorMap &tm_cup,
                             const GemvArgs &a, cudaStream_t stream) {
    const size_t smem = gateup_vq_smem(kLR, kD);
    cudaError_t err = ensure_smem(reinterpret_cast<const void *>(gateup_vq_kernel<kLR, kD>), smem);
    if (err != cudaSuccess) return err;
    cudaLaunchAttribute attrs[2];
    cudaLaunchConfig_t cfg = launch_config(dim3(num_sms()), dim3(kGemvThreads), smem, stream, attrs, 0);
    return cudaLaunchKernelEx(&cfg, gateup_vq_kernel<kLR, kD>, tm_jgate, tm_jup, tm_cgate, tm_cup, a);
}

cudaError_t launch_gateup_vq(const CUtensorMap &tm_jgate, const CUtensorMap &tm_jup,
                             const CUtensorMap *tm_cgate, const CUtensorMap *tm_cup,
                             const GemvArgs &a, int d, cudaStream_t stream) {
    // without the low-rank term its maps are unused: the index maps stand in for them
    const CUtensorMap &cg = tm_cgate ? *tm_cgate : tm_jgate;
    const CUtensorMap &cu = tm_cup ? *tm_cup : tm_jup;
    if (a.r > 0)
        return d == 8 ? launch_vq<true, 8>(tm_jgate, tm_jup, cg, cu, a, stream)
                      : launch_vq<true, 4>(tm_jgate, tm_jup, cg, cu, a, stream);
    return d == 8 ? launch_vq<false, 8>(tm_jgate, tm_jup, cg, cu, a, stream)
                  : launch_vq<false, 4>(tm_jgate, tm_jup, cg, cu, a, stream);
}

cudaError_t launch_down(const CUtensorMap &tm_down, const GemvArgs &a, cudaStream_t stream) {
    const size_t smem = down_smem();
    cudaError_t err = ensure_smem(reinterpret_cast<const void *>(down_kernel), smem);
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

// The combine of one output element in the one-grid VQ block: out[m][col] = bf16(residual +
// sum_{j valid} a_{m,j} y_{m,j}[col]), slots j ascending (the combine kernel's order), with the
// ids and affinities from shared memory and 8 slots' y loads in flight at once (every route
// has a y row; the rows of invalid routes are loaded but not added).  Against one load per
// slot in turn: one token 24.57 -> 24.15 us per layer, two tokens 32.62 -> 32.15 (same box).
__device__ __forceinline__ void combine_element(const int32_t *ids_s, const float *wts_s,
                                                const float *y, const __nv_bfloat16 *residual,
                                                __nv_bfloat16 *out, int m, int k, int E, int H,
                                                int col) {
    const float res = residual ? __bfloat162float(residual[(size_t)m * H + col]) : 0.0f;
    float acc = 0.0f;
    for (int j0 = 0; j0 < k; j0 += 8) {
        float v[8];
#pragma unroll
        for (int jj = 0; jj < 8; ++jj)
            v[jj] = j0 + jj < k ? __ldcg(y + ((size_t)m * k + j0 + jj) * H + col) : 0.0f;
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
            const int j = j0 + jj;
            if (j >= k) break;
            const int e = ids_s[m * k + j];
            if (e >= 0 && e < E) acc = fmaf(wts_s[m * k + j], v[jj], acc);
        }
    }
    out[(size_t)m * H + col] = __float2bfloat16_rn(res + acc);
}

// ------------------------------------------------------ VQ weights, one or two tokens
// The whole block for VQ-only gate/up weights (code words of 4) in one persistent grid: the
// one-grid routing (small_route.cuh, route_core.cuh), the alignment into sub-blocks in every
// CTA, then units in one ring -- gate/up tiles (sub-block, 64 columns of I) first, then down
// tiles (sub-block, 64 columns of H) -- with the tile bodies of the two kernels above, so the
// arithmetic and the bits are those of the multi-kernel path.  A down tile's W_down boxes
// stream at once; its p slices wait for the sub-block's ready count (each gate/up tile
// releases it once its p columns are stored).  The down tile that completes a token's routes
// for its 64 columns forms out = bf16(residual + sum_j a_j y_j), slots in order: the
// combine kernel's arithmetic.  Counters in the workspace's control region, zero between
// calls (the last CTA to leave restores them and the routing exchange).
// One stride for both kinds of stage, sized for at most kSmallMaxTokens routes per sub-block
// (a sub-block holds one expert, and a token routes to an expert once): a W_down box and two
// p slices, or an index box and two h slices.  The room left holds kCbReps copies of the
// code books, as in the gate/up kernel.
constexpr int kVQSmallStage = 34 * 1024;
constexpr int kVQSmallMaxSub = 32;            // sub-blocks (cap / rsub) the plan holds
constexpr int kVQCtlExit = 1, kVQCtlReady = 32;
static_assert(kBoxBytes + kSmallMaxTokens * kBoxRows * 4 <= kVQSmallStage, "down stage");
static_assert(vq_box_bytes(4) + kSmallMaxTokens * kVQHRows * 2 <= kVQSmallStage, "gate/up stage");
static_assert(kSmallMaxTokens <= 2, "the tile bodies below are instantiated for 1 and 2 routes");

struct VQSmallState {
    SubBlock sbt[kVQSmallMaxSub];
    int32_t ids[kSmallMaxRoutes];
    float wts[kSmallMaxRoutes];
    int32_t nvalid[kSmallMaxTokens];
    int32_t nsub;
    int32_t comb[kNT];  // per route of the down tile: the token to combine, or -1
    int32_t last;
};

__device__ __forceinline__ int32_t atom_add_acq_rel_gpu_vq(int32_t *p, int32_t v) {
    int32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// Bounded wait until *p >= need (acquire, GPU scope).
__device__ __forceinline__ bool vq_count_wait(const int32_t *p, int need, Ctl &ctl) {
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

struct VQUnit {
    bool gu;
    int sub, ct, nst;
};
__device__ __forceinline__ VQUnit vq_unit(const GemvArgs &g, int nsub, int u) {
    VQUnit x;
    const int Tgu = nsub * g.n_it;
    x.gu = u < Tgu;
    const int v = x.gu ? u : u - Tgu;
    const int n = x.gu ? g.n_it : g.n_ht;
    x.sub = v / n;
    x.ct = v - x.sub * n;
    x.nst = x.gu ? 2 * g.n_qb : g.n_ib;
    return x;
}

__global__ void __launch_bounds__(kGemvThreads, 1)
    decode_vq_small_kernel(const __grid_constant__ CUtensorMap tm_jgate,
                           const __grid_constant__ CUtensorMap tm_jup,
                           const __grid_constant__ CUtensorMap tm_down, const VQSmallArgs a) {
    constexpr int kD = 4;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *base = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char *stages = base;
    float *red = reinterpret_cast<float *>(base + kStages * kVQSmallStage);
    uint2 *cbs = reinterpret_cast<uint2 *>(base + kStages * kVQSmallStage + kRedBytesGU);
    Ctl &ctl = *reinterpret_cast<Ctl *>(base + kStages * kVQSmallStage + kRedBytesGU +
                                        2 * vq_codebook_bytes(kD) * kCbReps);
    VQSmallState &st = *reinterpret_cast<VQSmallState *>(reinterpret_cast<unsigned char *>(&ctl) +
                                                         ((sizeof(Ctl) + 15) & ~size_t(15)));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const GemvArgs &g0 = a.g;
    const int M = g0.M, E = g0.E, H = g0.H, k = g0.k, R = M * k;

    const SmallRouteScratch sc = small_route_scratch(stages, M, H, E);
    const RouterSplit sp = router_split(H, E);
    const bool router = (int)blockIdx.x < sp.NR;
    if (threadIdx.x == 0) {
        init_ring(ctl);
        prefetch_tensormap(&tm_jgate);
        prefetch_tensormap(&tm_jup);
        prefetch_tensormap(&tm_down);
    }
    // weights, before the dependency wait: the code books (kCbReps copies of each entry side
    // by side) and this CTA's block of W_r
    constexpr int kCbWords = vq_codebook_bytes(kD) / 8;  // 8-byte words per book
    constexpr int kEntWords = kD / 4;                     // 8-byte words per entry
    for (int i = threadIdx.x; i < 2 * kCbWords * kCbReps; i += blockDim.x) {
        const int book = i / (kCbWords * kCbReps), r = i - book * kCbWords * kCbReps;
        const int ent = r / (kEntWords * kCbReps), w = r % kEntWords;
        cbs[i] = (book ? g0.cb_up : g0.cb_gate)[ent * kEntWords + w];
    }
    if (router) small_router_copy(a.w_router, sp, sc.w_s);
    __syncthreads();
    pdl_wait();  // h, and the control region, come after the previous grid
    pdl_launch_dependents();

    // ---------------------------------------------------------------- routing
    if (router) small_route_dots(g0.h, M, H, E, a.partials, sp, sc);
    small_route_gather(a.partials, M, E, a.bias, sc.part_s, &ctl.abort, g0.status);
    route_finalize_any<true>(sc.part_s, M, E, k, nullptr, !ctl.abort, 1,
                       [&](int i, int j, int id, float wt) {
                           st.ids[i * k + j] = id;
                           st.wts[i * k + j] = wt;
                           if (blockIdx.x == 0) {
                               a.topk_ids[(size_t)i * k + j] = id;
                               a.topk_wts[(size_t)i * k + j] = wt;
                           }
                       });
    __syncthreads();
    // The alignment as sub-blocks (align_core's order: experts ascending, routes ascending,
    // each expert padded to a multiple of b; rsub consecutive rows per sub-block), in one
    // warp with lane r holding route r.
    if (warp == 0) {
        const int b = g0.b, rsub = g0.rsub;
        const int e = lane < R ? st.ids[lane] : -1;
        const bool valid = lane < R && e >= 0 && e < E;
        const unsigned peers = __match_any_sync(0xffffffffu, valid ? e : -1);
        const int lower = __popc(peers & ((1u << lane) - 1u));
        const int n = __popc(peers);
        const bool leader = valid && lower == 0;
        const int padded = leader ? (n + b - 1) / b * b : 0;
        int off = 0, total = 0;
#pragma unroll
        for (int q = 0; q < 32; ++q) {
            const int eq = __shfl_sync(0xffffffffu, e, q);
            const int pq = __shfl_sync(0xffffffffu, padded, q);
            total += pq;
            if (pq != 0 && eq < e) off += pq;
        }
        if (leader)
            for (int sb = off / rsub; sb < (off + padded) / rsub; ++sb) {
                const int first = sb * rsub - off;
                SubBlock &rec = st.sbt[sb];
                rec.e = e;
                rec.ntok = max(0, min(rsub, n - first));
                for (int q = rec.ntok; q < kNT; ++q) rec.routes[q] = rec.tokens[q] = -1;
            }
        __syncwarp();
        if (valid) {
            const int pos = off + lower;
            st.sbt[pos / rsub].routes[pos % rsub] = lane;
            st.sbt[pos / rsub].tokens[pos % rsub] = lane / k;
        }
        if (lane == 0) st.nsub = total / rsub;
        if (lane < M) {
            int nv = 0;
            for (int j = 0; j < k; ++j) {
                const int ej = st.ids[lane * k + j];
                nv += (ej >= 0 && ej < E) ? 1 : 0;
            }
            st.nvalid[lane] = nv;
        }
    }
    __syncthreads();
    const int nsub = st.nsub;
    // CTA 0 leaves the alignment and the sub-block table in the workspace (as
    // moe_align_block_size gives them), and out = residual (or zero) for a token with no route
    if (blockIdx.x == 0) {
        const int rsub = g0.rsub;
        for (int64_t i = threadIdx.x; i < a.cap; i += blockDim.x) {
            const int sb = (int)(i / rsub), q = (int)(i - (int64_t)sb * rsub);
            a.sorted[i] = (sb < nsub && q < st.sbt[sb].ntok) ? st.sbt[sb].routes[q] : R;
        }
        for (int64_t q = threadIdx.x; q < a.cap / g0.b; q += blockDim.x)
            a.blocks[q] = q * g0.b < (int64_t)nsub * rsub ? st.sbt[q * g0.b / rsub].e : -1;
        for (int i = threadIdx.x; i < nsub * (int)(sizeof(SubBlock) / 4); i += blockDim.x)
            reinterpret_cast<int32_t *>(a.sbt_ws)[i] = reinterpret_cast<const int32_t *>(st.sbt)[i];
        if (threadIdx.x == 0) {
            a.npad[0] = nsub * rsub;
            int nv = 0;
            for (int t = 0; t < M; ++t) nv += st.nvalid[t];
            if (nv < R) atomicOr(g0.status, MOE_DEV_INVALID_EXPERT);
        }
        for (int t = 0; t < M; ++t)
            if (st.nvalid[t] == 0)
                for (int c = threadIdx.x; c < H; c += blockDim.x)
                    g0.out[(size_t)t * H + c] =
                        g0.residual ? g0.residual[(size_t)t * H + c] : __float2bfloat16(0.0f);
    }
    GemvArgs ga = g0;
    ga.sbt = st.sbt;
    const int T = nsub * (ga.n_it + ga.n_ht);
    int32_t *ready = a.ctl + kVQCtlReady;
    int32_t *done = ready + kVQSmallMaxSub;

    // ---------------------------------------------------------------- experts
    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first();
            int stage = 0;
            uint32_t phase = 0, issued = 0, parity_bits = 0;
            bool stop = false;
            for (int u = blockIdx.x; u < T && !stop && !ctl.abort; u += gridDim.x) {
                const VQUnit x = vq_unit(ga, nsub, u);
                const SubBlock &rec = st.sbt[x.sub];
                const int nst = rec.ntok > 0 ? x.nst : 1;
                for (int j = 0; j < nst; ++j) {
                    if (!wait_or_abort(&ctl.empty[stage], phase ^ 1u, ctl)) {
                        stop = true;
                        break;
                    }
                    ctl.meta[stage] = rec;
                    uint64_t *bar = &ctl.full[stage];
                    unsigned char *dst = stages + stage * kVQSmallStage;
                    if (rec.ntok == 0) {
                        mbar_arrive(bar);
                    } else if (x.gu) {
                        mbar_arrive_expect_tx(bar, vq_box_bytes(kD));
                        tma_load_2d(dst, (j & 1) ? (const void *)&tm_jup : (const void *)&tm_jgate,
                                    x.ct * kTI, rec.e * (H / kD) + (j >> 1) * vq_rows(kD), bar, pol_w);
                    } else {
                        mbar_arrive_expect_tx(bar, kBoxBytes);
                        tma_load_2d(dst, &tm_down, x.ct * kTN, rec.e * ga.I + j * kBoxRows, bar, pol_w);
                    }
                    issued |= 1u << stage;
                    parity_bits = (parity_bits & ~(1u << stage)) | (phase << stage);
                    advance(stage, phase);
                }
            }
            for (int s2 = 0; s2 < kStages; ++s2)
                if ((issued >> s2) & 1u)
                    if (!mbar_wait_bounded(&ctl.full[s2], (parity_bits >> s2) & 1u)) ctl.abort = 1;
        }
        __syncwarp();
    } else if (warp == 1) {
        int stage = 0;
        uint32_t phase = 0;
        bool stop = false;
        for (int u = blockIdx.x; u < T && !stop && !ctl.abort; u += gridDim.x) {
            const VQUnit x = vq_unit(ga, nsub, u);
            const SubBlock &rec = st.sbt[x.sub];
            const int ntok = rec.ntok;
            const int nst = ntok > 0 ? x.nst : 1;
            if (!x.gu && ntok > 0) {  // p of the sub-block: stored by all its gate/up tiles
                bool ok = true;
                if (lane == 0) ok = vq_count_wait(ready + x.sub, ga.n_it, ctl);
                if (!__shfl_sync(0xffffffffu, ok, 0)) break;
            }
            for (int j = 0; j < nst; ++j) {
                if (!wait_or_abort(&ctl.empty[stage], phase ^ 1u, ctl)) {
                    stop = true;
                    break;
                }
                if (ntok > 0) {
                    unsigned char *dst = stages + stage * kVQSmallStage;
                    for (int q = 0; q < ntok; ++q) {
                        const int route = rec.routes[q], token = rec.tokens[q];
                        if (x.gu) {  // h rows [1024 (j/2), +1024): four 16-byte pieces per lane
                            for (int c = 0; c < 4; ++c) {
                                const int piece = lane * 4 + c;
                                cp_async_16(dst + vq_box_bytes(kD) + q * kVQHRows * 2 + piece * 16,
                                            reinterpret_cast<const unsigned char *>(ga.h) +
                                                ((size_t)token * H + (size_t)(j >> 1) * kVQHRows) * 2 +
                                                piece * 16);
                            }
                        } else {  // p rows [256 j, +256) of the route: two pieces per lane
                            for (int c = 0; c < 2; ++c) {
                                const int piece = lane * 2 + c;
                                cp_async_16(dst + kBoxBytes + q * kBoxRows * 4 + piece * 16,
                                            reinterpret_cast<const unsigned char *>(ga.p) +
                                                ((size_t)route * ga.I + (size_t)j * kBoxRows) * 4 +
                                                piece * 16);
                            }
                        }
                    }
                    cp_async_mbar_arrive(&ctl.full[stage]);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl.full[stage]);
                advance(stage, phase);
            }
        }
        cp_async_wait_all();
    } else {
        Lane ln;
        ln.ctid = threadIdx.x - 32 * kFirstConsumerWarp;
        ln.cw = warp - kFirstConsumerWarp;
        ln.lane = lane;
        ln.half = lane >> 4;
        ln.c4 = (lane & 15) * 4;
        ln.rbase = ln.cw * kRowsPerWarp + ln.half * kRowsPerThread;
        int stage = 0;
        uint32_t phase = 0;
        for (int u = blockIdx.x; u < T; u += gridDim.x) {
            const VQUnit x = vq_unit(ga, nsub, u);
            if (!wait_or_abort(&ctl.full[stage], phase, ctl)) {
                named_bar_or(1, kConsumerThreads, true);
                break;
            }
            const SubBlock &mt = ctl.meta[stage];
            const int ntok = mt.ntok;
            const int cols = x.gu ? kTI : kTN;
            const int q0 = ln.ctid / cols, q1 = (ln.ctid + kConsumerThreads) / cols;
            const int r0 = (q0 < ntok) ? mt.routes[q0] : -1;
            const int r1 = (q1 < ntok) ? mt.routes[q1] : -1;
            // the record's slot is reused once the tile's stages are released: keep what the
            // combine needs (thread q < ntok: the token of route q)
            const int my_token = ln.ctid < ntok ? mt.tokens[ln.ctid] : -1;
            bool go = true;
#define MOE_VQS_TILE(N)                                                                      \
    case N:                                                                                  \
        go = x.gu ? gateup_tile<N, false, kD, kVQSmallStage, kCbReps>(                       \
                        ga, ctl, stages, red, cbs, ln, x.ct, r0, r1, stage, phase)           \
                  : down_tile<N, kVQSmallStage>(ga, ctl, stages, red, ln, x.ct, r0, r1,      \
                                                stage, phase);                               \
        break;
            switch (ntok) {  // (at most kSmallMaxTokens routes per sub-block)
                MOE_VQS_TILE(1)
                MOE_VQS_TILE(2)
                default:  // an empty sub-block is announced by a single stage
                    release_stage(ctl, ln, stage, phase);
                    go = !named_bar_or(1, kConsumerThreads, false);
            }
#undef MOE_VQS_TILE
            if (!go) break;
            if (ntok == 0) continue;
            if (x.gu) {
                // the tile's p columns are stored (the tile body ends with a barrier)
                if (ln.ctid == 0) red_release_gpu_add(ready + x.sub, 1);
            } else {
                // y of the tile's routes is stored: count them per token and 64-column tile;
                // the route completing its token's valid routes marks the token for the combine
                if (ln.ctid < ntok) {
                    const int m = my_token;
                    const int old = atom_add_acq_rel_gpu_vq(done + m * ga.n_ht + x.ct, 1);
                    st.comb[ln.ctid] = old + 1 == st.nvalid[m] ? m : -1;
                }
                named_bar_sync(1, kConsumerThreads);
                // out = bf16(residual + sum_j a_j y_j), valid slots in order (the combine)
                for (int q = 0; q < ntok; ++q) {
                    const int m = st.comb[q];
                    if (m >= 0 && ln.ctid < kTN)
                        combine_element(st.ids, st.wts, ga.y, ga.residual, ga.out, m, k, E, H,
                                        x.ct * kTN + ln.ctid);
                }
                named_bar_sync(1, kConsumerThreads);
            }
        }
    }

    // ---------------------------------------------------------------- exit: restore the region
    __syncthreads();
    if (ctl.abort) atomicOr(g0.status, MOE_DEV_WAIT_TIMEOUT);
    if (threadIdx.x == 0) st.last = atom_add_acq_rel_gpu_vq(a.ctl + kVQCtlExit, 1) == (int)gridDim.x - 1;
    __syncthreads();
    if (st.last) {  // every CTA is done with the counters and the partials
        for (int i = threadIdx.x; i < kVQSmallMaxSub; i += blockDim.x) ready[i] = 0;
        for (int i = threadIdx.x; i < M * ga.n_ht; i += blockDim.x) done[i] = 0;
        for (int i = threadIdx.x; i < M * kRouterCluster * E / 4; i += blockDim.x)
            reinterpret_cast<uint4 *>(a.partials)[i] = make_uint4(0u, 0u, 0u, 0u);
        if (threadIdx.x == 0) a.ctl[kVQCtlExit] = 0;
    }
}

static size_t vq_small_smem() {
    return 1024 + (size_t)kStages * kVQSmallStage + kRedBytesGU + 2 * vq_codebook_bytes(4) * kCbReps +
           ((sizeof(Ctl) + 15) & ~size_t(15)) + sizeof(VQSmallState);
}

bool vq_small_fits(int M, int k, int E, int H, int I, int b, int d) {
    if (d != 4 || M < 1 || M > kSmallMaxTokens || (int64_t)M * k > kSmallMaxRoutes || b < 1 || b > 64)
        return false;
    if ((size_t)(H / kRouterCluster) * E * 2 > 64 * 1024) return false;  // one router pass
    if (small_routing_bytes(M, H, E) > (size_t)kStages * kVQSmallStage) return false;
    const int64_t R = (int64_t)M * k;
    const int64_t cap = R + (R < E ? R : E) * (b - 1);
    const int rsub = b <= kNT ? b : kNT;
    if (cap / rsub > kVQSmallMaxSub) return false;
    if (kVQCtlReady + kVQSmallMaxSub + (int64_t)M * (H / kTN) > kSmallCtlInts) return false;
    return vq_small_smem() <= 227 * 1024;
}

cudaError_t launch_decode_vq_small(const CUtensorMap &tm_jgate, const CUtensorMap &tm_jup,
                                   const CUtensorMap &tm_down, const VQSmallArgs &a,
                                   cudaStream_t stream) {
    const size_t smem = vq_small_smem();
    cudaError_t err = ensure_smem(reinterpret_cast<const void *>(decode_vq_small_kernel), smem);
    if (err != cudaSuccess) return err;
    cudaLaunchAttribute attrs[2];
    cudaLaunchConfig_t cfg = launch_config(dim3(num_sms()), dim3(kGemvThreads), smem, stream, attrs, 0);
    return cudaLaunchKernelEx(&cfg, decode_vq_small_kernel, tm_jgate, tm_jup, tm_down, a);
}

}  // namespace moe
