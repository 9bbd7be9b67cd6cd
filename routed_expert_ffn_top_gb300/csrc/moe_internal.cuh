// moe_internal.cuh -- shapes, workspace layout and kernel launchers shared by the .cu files.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

// GEMV-regime tiling (fixed, so every reduction order depends on tile indices only).
constexpr int kNT = 8;          // tokens per sub-block (register tile of the GEMV kernels)
constexpr int kTI = 64;         // gate/up: I columns per tile (128-byte rows in shared memory)
constexpr int kTN = 64;         // down: H columns per tile
constexpr int kBoxRows = 256;   // rows (of H for gate/up, of I for down) per weight box
constexpr int kConsumerWarps = 8;
constexpr int kGemvThreads = 32 * (2 + kConsumerWarps);  // producer, loader, consumers
constexpr int kRouterCluster = 8;  // CTAs per router cluster (split of H)
constexpr int kRouterThreads = 512;
// Row groups per slice of the router's split of H: RG = 512 / (E/2) (every thread of a
// router CTA one group and expert pair).
__host__ __device__ constexpr int router_row_groups(int E) { return kRouterThreads / (E / 2); }

struct Dims {
    int M, k, E, H, I, b;
    bool gemm;        // every projection runs as tcgen05 tiles of kn rows (dense weights,
                      // or VQ gate/up decoded on the tensor-core path)
    int kn, tpb;      // tile width (16 or 64 aligned rows) and tiles per aligned block
    int rsub;         // rows per sub-block: b if b <= 8, else 8
    int64_t R;        // routes M*k (also the sentinel value)
    int64_t cap;      // alignment capacity in rows
    int64_t max_sub;  // cap / rsub
    int n_it, n_hb, n_ht, n_ib;  // column tiles and 256-row boxes of gate/up and down
    int r = 0;        // rank of the low-rank gate/up term (0: none)
    bool ttable = false;  // VQ gate/up through projected code books
    int vqd = 0;          // VQ code-word length d
    bool vq_tc = false;   // VQ gate/up on the tensor cores (16-row tiles)
};

// One sub-block of the alignment (rsub consecutive aligned rows of one expert), as the
// expert kernels consume it: the expert, its valid routes in row order, and their tokens.
struct __align__(16) SubBlock {
    int e;
    int ntok;
    int routes[kNT];
    int tokens[kNT];
    int pad[2];
};
static_assert(sizeof(SubBlock) == 80, "SubBlock layout");

struct WsLayout {
    size_t status;   // int32[16]
    size_t ctl;      // int32[kSmallCtlInts]  counters of the one-kernel path, zero between calls
    size_t sorted;   // int32[cap]
    size_t blocks;   // int32[cap / b]
    size_t npad;     // int32[4]
    size_t sbt;      // SubBlock[max_sub]
    size_t p;        // float[R * I]   SiLU(g) * u per route
    size_t y;        // float[R * H]   down-projection output per route
    size_t z;        // float[M * 2r]  low-rank projections z = D^T h (gate, then up)
    size_t x_tiles;  // bf16[tile rows * H]  dense weights: token rows per tile row
    size_t p_tiles;  // bf16[tile rows * I]  dense weights: p per tile row
    size_t ready;    // int32[tiles]  dense weights: gate/up units of each tile whose p is stored
    size_t partials; // uint32[kSmallPartialInts]  one-kernel path: the router's partials, zero between calls
    size_t p_rows;   // bf16[R * I]  one-kernel path: p per route
    size_t tt_part;  // float[slices * M*k * 2 * I]  VQ through projected code books
    size_t total;
};

Dims make_dims(int M, int k, int E, int H, int I, int b, int kind);
WsLayout ws_layout(const Dims &d);

struct GemvArgs {
    const __nv_bfloat16 *h;
    const int32_t *topk_ids;
    const float *topk_wts;
    const SubBlock *sbt;
    const int32_t *npad;
    const __nv_bfloat16 *residual;
    __nv_bfloat16 *out;
    float *p;
    float *y;
    int32_t *status;
    const unsigned char *w_down;  // W_down [E, I, H] bf16 (idle gate/up CTAs warm it in L2)
    const float *z;        // VQ + low rank: z = D^T h [M, 2r] (gate, then up); else NULL
    int r, n_rb;           // rank of the low-rank term (0: none); its 256-row boxes
    const uint2 *cb_gate;  // VQ code books [256][d] bf16 read 8 bytes at a time (NULL: dense)
    const uint2 *cb_up;
    int M, k, E, H, I, b, rsub;
    int n_it, n_hb, n_ht, n_ib;
    int n_qb;              // VQ: index-map boxes of 256 rows (1024 rows of H) per projection
    int64_t max_sub;       // rows of the sub-block table
};

// Dense weights (and VQ decoded on the tensor cores): grouped GEMMs on tcgen05 over tiles
// of kn aligned rows of one expert.  An aligned block of b rows is cut into tpb = ceil(b / kn)
// tiles, kn = 16 for b <= 16, else 64.  The library picks 16- or 64-row blocks by routes per
// expert when the caller passes b = 0 (library_block in api.cu).
constexpr int kGemmBlock = 64;
constexpr int kGemmNarrow = 16;

__host__ __device__ constexpr int gemm_tile_width(int b) { return b <= kGemmNarrow ? kGemmNarrow : kGemmBlock; }
constexpr int kGemmStageK = 256;  // K rows per pipeline stage and per weight box
__host__ __device__ constexpr int gemm_tiles_per_block(int b) {
    return (b + gemm_tile_width(b) - 1) / gemm_tile_width(b);
}

// Row tiles hold, for every 64-wide K chunk, the K-major 128-byte-swizzle image of the
// tile's kn rows: row n at n * 128 bytes, its 16-byte piece j at (j ^ n % 8) * 16.
__host__ __device__ constexpr uint32_t tile_offset(int n, int j) {
    return (uint32_t)(n * 128 + ((j ^ (n & 7)) << 4));
}

// Where row tiles of h are written by the router when it also aligns (NULL x_tiles: not).
// The kernel that writes them also zeroes the per-tile ready counts of the grouped GEMM that
// reads them (`ready`, `nready` entries; NULL: none).
struct RowTiles {
    __nv_bfloat16 *x_tiles;
    int kn, tpb;
    int32_t *ready;
    int64_t nready;
};

// Zeroes n counts with the threads of one CTA.
__device__ __forceinline__ void zero_counts(int32_t *p, int64_t n) {
    if (p)
        for (int64_t i = threadIdx.x; i < n; i += blockDim.x) p[i] = 0;
}

struct GemmArgs {
    const __nv_bfloat16 *x;   // h [M,H] (read by the row gather)
    const int32_t *ids;       // topk_ids [M*k]: a row whose route disagrees is skipped
    const int32_t *sorted;    // aligned rows (route ids, sentinel = M*k)
    const int32_t *blocks;    // expert of each b-row block
    const int32_t *npad;
    __nv_bfloat16 *x_tiles;   // token rows of h per tile row, [tiles][H/64][kn * 128 B]
    __nv_bfloat16 *p_tiles;   // SiLU(g) * u per tile row, bf16, [tiles][I/64][kn * 128 B]
    float *y;                 // down output per route [M*k, H]
    int32_t *status;
    int M, k, E, H, I;
    int b, kn, tpb;           // aligned block rows, tile width, tiles per block
    int wait_first;           // the previous kernel wrote the x tiles (and the alignment)
    const __nv_bfloat16 *cb_gate, *cb_up;  // VQ on the tensor cores: the code books
    int64_t R, cap;
    int32_t *ready;           // [tiles] gate/up units done per tile, then the fused grid's unit
    int64_t nready;           // counter: nready = tiles + 1 ints, zeroed by the previous kernel
};

// The whole block for a few tokens in one persistent grid (decode_small.cu): router,
// alignment, gate/up, down and combine.  Its counters live in the workspace's control region
// (zero between calls; the grid's last CTA restores it).
// Up to 2 tokens (same-box A/B on GB300, H=2048, I=768, E=128, k=8, us per layer, one grid
// against router + fused expert grid + combine: M=1 28.6 / 29.8, M=2 40.5 / 40.8, M=3
// 49.2 / 47.9, M=4 58.8 / 56.9: from three tokens the routing every CTA repeats costs more
// than the launches it saves).
constexpr int kSmallMaxTokens = 2;
constexpr int kSmallMaxRoutes = 32;
constexpr int kSmallCtlExit = 1;    // CTAs finished
constexpr int kSmallCtlReady = 32;  // ready[tiles], then done[M][H / 128]
constexpr int kSmallCtlInts = 512;
// The one-grid path's routing exchange: the partial logits [8][M][E] of the router's slices,
// stored complemented (a zero word: not written yet), in a region of fixed size right after
// the control region in every workspace layout, zero between calls like it.
constexpr int kSmallPartialInts = kRouterCluster * kSmallMaxTokens * 512;
constexpr int kSmallCtlDone = kSmallCtlInts - kSmallCtlReady - kSmallMaxRoutes;

struct SmallArgs {
    const __nv_bfloat16 *h, *w_router, *residual;
    const float *bias;
    int M, k, E, H, I, b;
    int64_t cap;
    int32_t *topk_ids;
    float *topk_wts;
    __nv_bfloat16 *out;
    float *partials;                  // [8][M][E], complemented bits, zero between calls
    int32_t *ctl;                     // the control region
    int32_t *sorted, *blocks, *npad;  // the alignment, left in the workspace
    __nv_bfloat16 *p_rows;            // [M*k][I]
    float *y;                         // [M*k][H]
    int32_t *status;
    int ntiles_cap;                   // cap / b
};
// Whether the one-kernel path takes (M, k, E, H, b): dense weights, 1 <= M <= 2, M*k <= 32,
// b <= 16, one router pass per slice of H.
bool small_fits(int M, int k, int E, int H, int b);
cudaError_t launch_decode_small(const CUtensorMap &tm_gate, const CUtensorMap &tm_up,
                                const CUtensorMap &tm_down, const SmallArgs &a,
                                cudaStream_t stream);

// The whole block for VQ-only gate/up weights (code words of 4) and one or two tokens in one
// persistent grid (gemv.cu).
struct VQSmallArgs {
    GemvArgs g;  // sbt, p, y, status: the workspace's (sbt is replaced by each CTA's own plan)
    const __nv_bfloat16 *w_router;
    const float *bias;
    int32_t *topk_ids;
    float *topk_wts;
    float *partials;  // the routing exchange
    int32_t *ctl;     // [kVQCtlExit], ready [kVQCtlReady + s], then done [M][H / 64]
    int32_t *sorted, *blocks, *npad;
    SubBlock *sbt_ws;  // the workspace's sub-block table (CTA 0 writes the plan there)
    int64_t cap;
};

bool vq_small_fits(int M, int k, int E, int H, int I, int b, int d);
cudaError_t launch_decode_vq_small(const CUtensorMap &tm_jgate, const CUtensorMap &tm_jup,
                                   const CUtensorMap &tm_down, const VQSmallArgs &a,
                                   cudaStream_t stream);

cudaError_t launch_gather_rows(const GemmArgs &a, cudaStream_t stream);
// Gate/up + SiLU and down for dense weights in one persistent grid: a down unit's weights
// stream while gate/up runs; its p waits on the tile's ready count.
cudaError_t launch_gemm_fused(const CUtensorMap &tm_gate, const CUtensorMap &tm_up,
                              const CUtensorMap &tm_down, const GemmArgs &a, cudaStream_t stream);
cudaError_t launch_gemm_down(const CUtensorMap &tm_down, const GemmArgs &a, cudaStream_t stream);
// Blockwise-VQ gate/up on the tensor cores (16-row tiles, d = 4 or 8): index maps by TMA,
// decoded through the code books into the MMA's A operand.
cudaError_t launch_gemm_gateup_vq(const CUtensorMap &tm_jgate, const CUtensorMap &tm_jup,
                                  const GemmArgs &a, int d, cudaStream_t stream);
constexpr int kReaderMaxCand = 16384;  // k * I candidate channels per token the selection holds
constexpr int kReaderMaxRank = 32;
// Blockwise VQ gate/up through projected code books (vq_ttable.cu), for at most
// kTTMaxTokens tokens: per route the SiLU(g) * u rows p [M*k][I] fp32 the down kernel reads.
constexpr int kTTMaxTokens = 4;
struct VQTableArgs {
    const __nv_bfloat16 *h;
    const uint8_t *j_gate, *j_up;
    const __nv_bfloat16 *cb_gate, *cb_up;
    const int32_t *ids;
    int M, k, E, H, I, d;
    float *partial;  // [slices][M*k][2][I]
    float *p;        // [M*k][I]
};
int vq_ttable_slices(int H, int d);
cudaError_t launch_vq_ttable(const VQTableArgs &a, cudaStream_t stream);

// The channel reader's data (see reader.cu for the layout) and one call's workspace.
struct ReaderArgs {
    int H, I, E, rank;
    const int8_t *signs;                    // [H] +1 / -1
    const __nv_bfloat16 *g_rows, *v_rows;   // [E][I][H] channel-major gate / up rows
    const __nv_bfloat16 *w_down;            // [E][I][H]
    const uint32_t *g_codes, *v_codes;      // [E][I][H/128][8] two-bit ternary codes
    const float *g_scales, *v_scales;       // [E][I][H/128]
    const float *dnorm;                     // [E][I]
    const float *U;                         // [H][rank]
    const __nv_bfloat16 *coef;              // [E][I][rank]
};
struct ReaderWs {
    size_t status, ctl, xr, ahat, score, keep, sel, nsel, partial, zpart, total;
    int nchunk;
};
ReaderWs reader_ws_layout(const ReaderArgs &r, int M, int k, int K);
// Records the caller's trace event i (moe_set_trace_events) on s, when tracing is on.
void trace_point(int i, cudaStream_t s);
cudaError_t launch_reader_build(const ReaderArgs &r, const __nv_bfloat16 *w_gate,
                                const __nv_bfloat16 *w_up, cudaStream_t stream);
cudaError_t launch_reader_decode(const ReaderArgs &r, const __nv_bfloat16 *h, int M, int k,
                                 const int32_t *ids, const float *wts, int K, int nscan,
                                 const __nv_bfloat16 *residual, __nv_bfloat16 *out,
                                 unsigned char *ws, cudaStream_t stream);
// One CTA whose bounded wait runs out on purpose (sets MOE_DEV_WAIT_TIMEOUT in *status).
cudaError_t launch_wait_selftest(int32_t *status, cudaStream_t stream);

// Sub-blocks to process: num_padded / rsub, never more than the table holds.
__device__ __forceinline__ int64_t num_subblocks(const GemvArgs &a) {
    const int64_t n = a.npad[0] / a.rsub;
    return n < 0 ? 0 : (n > a.max_sub ? a.max_sub : n);
}

int num_sms();
int l2_bytes();  // this device's L2 size in bytes (0 when it cannot be read)

// Record of sub-block sb: expert of its block, valid routes (0 <= r < R) of its rsub rows in
// row order, token of each route.  With `check`, a route whose top-k id is not the block's
// expert is left out and flagged as a bad alignment.
__device__ __forceinline__ void build_subblock(const int32_t *sorted, const int32_t *blocks,
                                               const int32_t *topk_ids, int64_t sb, int rsub,
                                               int b, int E, int64_t R, int k, bool check,
                                               int32_t *status, SubBlock *out) {
    const int64_t row0 = sb * rsub;
    const int e = blocks[row0 / b];
    SubBlock rec;
    rec.e = e;
    int n = 0;
#pragma unroll 1
    for (int q = 0; q < kNT; ++q) rec.routes[q] = rec.tokens[q] = -1;
    rec.pad[0] = rec.pad[1] = 0;
    if (e >= 0 && e < E) {
#pragma unroll 1
        for (int q = 0; q < rsub; ++q) {
            const int r = sorted[row0 + q];
            if (r < 0 || r >= R) continue;
            if (check && topk_ids[r] != e) {
                if (status) atomicOr(status, MOE_DEV_BAD_ALIGNMENT);
                continue;
            }
            rec.routes[n] = r;
            rec.tokens[n] = r / k;
            ++n;
        }
    }
    rec.ntok = n;
    *out = rec;
}

// Low-rank projections z = D^T h of VQ + low-rank gate/up weights, computed by extra
// clusters of the router's launch (see router.cu).
struct LowRankProj {
    const __nv_bfloat16 *d_gate, *d_up;  // [H, r] bf16, layer-shared
    int r;                               // 0: no projection
    int first;                           // set by the launcher
    float *z;                            // [M, 2r] fp32: gate then up
};

cudaError_t launch_router(const __nv_bfloat16 *h, const __nv_bfloat16 *w_router,
                          const float *bias, int M, int H, int E, int k, int renormalize,
                          int32_t *topk_ids, float *topk_weights, const LowRankProj *lr,
                          cudaStream_t stream);

// The projections alone (callers that bring their own routing).
cudaError_t launch_lowrank_proj(const __nv_bfloat16 *h, int M, int H, const LowRankProj &lr,
                                cudaStream_t stream);

// Router that also aligns the routes (and writes the sub-block table) in the same launch;
// possible when one router cluster holds every token.
bool router_can_align(int M, int k);
cudaError_t launch_router_align(const __nv_bfloat16 *h, const __nv_bfloat16 *w_router,
                                const float *bias, int M, int H, int E, int k, int renormalize,
                                int32_t *topk_ids, float *topk_weights, int b, int rsub,
                                int32_t *sorted, int32_t *blocks, int32_t *npad, int64_t cap,
                                SubBlock *sbt, int32_t *status, const LowRankProj *lr,
                                const RowTiles &rows, cudaStream_t stream);

// Alignment; when `sbt` is not NULL it also writes the sub-block table of rsub-row blocks.
cudaError_t launch_align(const int32_t *topk_ids, int M, int k, int E, int b,
                         int32_t *sorted, int32_t *blocks, int32_t *npad, int64_t cap,
                         SubBlock *sbt, int rsub, int32_t *status, cudaStream_t stream);

// Alignment and the row tiles of the tcgen05 path in one launch (M * k <= 128 routes: above
// that the per-CTA alignment, quadratic in the routes, costs more than the launch it saves).
constexpr int kAlignGatherRoutes = 128;
cudaError_t launch_align_gather(const int32_t *topk_ids, int M, int k, int E, int b,
                                int32_t *sorted, int32_t *blocks, int32_t *npad, int64_t cap,
                                int32_t *status, const __nv_bfloat16 *x, int H,
                                const RowTiles &rows, cudaStream_t stream);

// Sub-block table from a caller-supplied alignment, checking each row against topk_ids.
cudaError_t launch_plan(const int32_t *topk_ids, const int32_t *sorted, const int32_t *blocks,
                        const int32_t *npad, int M, int k, int E, int b, int rsub,
                        int64_t max_sub, SubBlock *sbt, int32_t *status, cudaStream_t stream);


// Blockwise-VQ gate/up (d = 4 or 8, K = 256): index maps through TMA (boxes of 1024/d index
// rows x 64 columns), code books in shared memory; with a.r > 0 also the low-rank term (C
// maps through TMA, z slices from a.z).
cudaError_t launch_gateup_vq(const CUtensorMap &tm_jgate, const CUtensorMap &tm_jup,
                             const CUtensorMap *tm_cgate, const CUtensorMap *tm_cup,
                             const GemvArgs &a, int d, cudaStream_t stream);

cudaError_t launch_down(const CUtensorMap &tm_down, const GemvArgs &a, cudaStream_t stream);

cudaError_t launch_combine(const GemvArgs &a, cudaStream_t stream);

// The decode block (b == 0: the library's block size) and the workspace one resolved b
// needs: the allocation-free entry, whose scratch has a fixed size, runs through these.
int decode_block(const void *h, const void *w_router, const float *bias,
                 const moe_expert_weights_t *w, int M, int k, int b, const void *residual,
                 void *out, int32_t *topk_ids, float *topk_weights, void *workspace,
                 size_t ws_bytes, void *stream);
size_t workspace_bytes_fixed(const moe_expert_weights_t *w, int M, int k, int b);
int block_for(const moe_expert_weights_t *w, int M, int k, int b);  // b, or the library's (b == 0)

// Raises `func`'s dynamic shared-memory limit to at least `bytes` on the current device.
// The attribute is set once per (kernel, device) and remembered: repeating the runtime call
// on every launch costs host time that small decode blocks cannot hide.
cudaError_t ensure_smem(const void *func, size_t bytes);

// Shared launch helper: programmatic dependent launch on, optional cluster dims.
cudaLaunchConfig_t launch_config(dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                                 cudaLaunchAttribute *attrs, int cluster_x);

}  // namespace moe
