/*
 * moe.h -- C ABI of the GB300 (sm_103a) small-batch MoE decode block.
 *
 * The block, as the pages define it:
 *   * router: logits = h W_r (+ bias), softmax, top-k experts, affinities a renormalised
 *     over the k selected experts ("A Multi-Engine Dataflow for MoE Decoding on
 *     Scratchpad-Based Tensor Accelerators", MoE block background around Figure 2);
 *   * alignment: the M x k expert ids flattened row-major into route ids r = m*k + j,
 *     valid routes grouped by expert in ascending route id, each expert padded to a
 *     multiple of b rows, plus a parallel expert-per-block vector ("Route-Block Membership
 *     Selects Packed-AWQ Arithmetic", Sections 2.1 and 5.3);
 *   * expert FFN: p = SiLU(h W_gate[e]) * (h W_up[e]), y = p W_down[e] (Multi-Engine
 *     Dataflow page, stage-3 activation and Section 4.3; "Channel Selection for
 *     Mixture-of-Experts Decoding Needs No Calibration Data", Background);
 *   * combine: out[m] = residual[m] + sum_j a_{m,j} y_{m,j} (Multi-Engine Dataflow page,
 *     Section 4.3, "accumulated summation");
 *   * optional blockwise-VQ gate/up: column i of W_e cut into length-d blocks along H,
 *     block q replaced by code word J_e[q][i] of a layer-shared code book
 *     (Multi-Engine Dataflow page, Section 2.3).
 *
 * Conventions shared by every entry point
 *   * Pointers named h, w_*, j_*, cb_*, bias, topk_*, sorted_route_ids, expert_block_ids,
 *     num_padded, residual, out and workspace are DEVICE pointers, row-major and
 *     contiguous, each 16-byte aligned.  The caller owns and allocates every buffer;
 *     the library allocates no device or host memory.
 *   * bf16 tensors are IEEE bfloat16 (uint16 storage).  Accumulation is fp32.
 *   * `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).
 *     Calls are stream-ordered and asynchronous: they never synchronise, except
 *     moe_read_device_status and the *_host entry point, which say so.
 *   * Argument errors are reported synchronously, before anything is launched.  Shapes
 *     the kernels do not support fail closed with MOE_ERR_UNSUPPORTED.
 *   * Conditions found on the device (an expert id outside [0, E), a bounded device wait
 *     that gave up) never trap: they set bits in a status word inside the workspace, read
 *     back with moe_read_device_status.
 *   * Every reduction runs in an order fixed by tile indices only (never by grid size,
 *     block position or atomic arrival order), so results are bitwise reproducible run
 *     to run, and a route's output bits do not depend on which aligned block it lands in.
 *
 * Supported shapes: 1 <= k <= min(E, 32); 8 <= E <= 512, E % 8 == 0; H and I multiples of
 * 256 up to 8192 (moe_route_topk alone: H a multiple of 128); (H/8) * E * 2 <= 131072
 * bytes (router slice); b >= 1 and (b <= 8 or b % 8 == 0), or b == 0 where an entry point
 * says the library picks it; 0 <= M; M * k < 2^24.
 * VQ: d in {4, 8}, K == 256, H a multiple of 1024 (vq_form 0 and 2: any M; vq_form 1: at
 * most 4 tokens); VQ + low rank: r a multiple of 128 up to 512.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum moe_status {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,   /* NULL or misaligned pointer, negative size, bad enum */
    MOE_ERR_UNSUPPORTED = 2,   /* a shape outside the supported range (fails closed) */
    MOE_ERR_WORKSPACE = 3,     /* workspace or alignment capacity smaller than required */
    MOE_ERR_CUDA = 4,          /* a CUDA runtime or driver call failed */
    MOE_ERR_DEVICE = 5         /* moe_read_device_status: the device set a status bit */
} moe_status_t;

/* Bits of the device status word. */
#define MOE_DEV_INVALID_EXPERT 0x1  /* a route's expert id was outside [0, E): excluded */
#define MOE_DEV_WAIT_TIMEOUT   0x2  /* a bounded device wait gave up; outputs undefined */
#define MOE_DEV_BAD_ALIGNMENT  0x4  /* an aligned row disagreed with topk_ids: skipped */

/* Weight representations of the gate/up projections. */
#define MOE_W_DENSE_BF16 0
#define MOE_W_VQ_GATEUP  1
#define MOE_W_VQLR_GATEUP 2

/*
 * One MoE layer's expert weights (all device pointers).
 *   kind == MOE_W_DENSE_BF16: w_gate, w_up [E,H,I] bf16 (row h of expert e holds I
 *     contiguous values); j_*, cb_*, d_*, c_* unused.
 *   kind == MOE_W_VQ_GATEUP: j_gate, j_up [E,H/d,I] uint8 index maps (expert-private);
 *     cb_gate, cb_up [K,d] bf16 code books (layer-shared), W[e][d*q+t][i] =
 *     cb[J[e][q][i]][t]; w_gate, w_up unused.
 *   kind == MOE_W_VQLR_GATEUP: the VQ fields above plus a low-rank term per projection
 *     ("A Multi-Engine Dataflow ...", the hybrid representation around its Eq. (1)):
 *     W_e = Q_B(J_e) + D C_e with d_gate, d_up [H,r] bf16 (layer-shared basis) and c_gate,
 *     c_up [E,r,I] bf16 (expert-private coefficients).  z = D^T h is computed once per
 *     token and projection (in the router's launch), then accumulated with the VQ sum.
 *   w_down [E,I,H] bf16 in every case (the down projection stays dense).
 *   vq_form (MOE_W_VQ_GATEUP only): 0 multiplies every index's code word with h in
 *     shared memory (GEMV streams, any M); 1 uses projected code books ("A Multi-Engine
 *     Dataflow ...", Section 2.3): per token and index row q the table
 *     T[q][kappa] = sum_t h[d q + t] B[kappa][t], so that g_i = sum_q T[q][J[e][q][i]] (one
 *     lookup per index instead of d products), for at most 4 tokens (M > 4:
 *     MOE_ERR_UNSUPPORTED); 2 decodes the index maps through the code books into the
 *     tensor cores' weight operand in tensor memory and runs gate/up as the tcgen05 grouped
 *     GEMM of dense weights, over 16- or 64-row tiles of the aligned blocks (any M; b == 0
 *     lets the library pick 16- or 64-row blocks).  The forms add in different orders; each
 *     is bitwise reproducible and independent of M on its own.
 * Fields after w_down were added later; zero them when they do not apply.
 */
typedef struct moe_expert_weights {
    int32_t kind;
    int32_t H, I, E;
    const void *w_gate;
    const void *w_up;
    const uint8_t *j_gate;
    const uint8_t *j_up;
    const void *cb_gate;
    const void *cb_up;
    int32_t d, K;
    const void *w_down;
    const void *d_gate;
    const void *d_up;
    const void *c_gate;
    const void *c_up;
    int32_t r;
    int32_t vq_form;
} moe_expert_weights_t;

/* A short static description of a status code (never NULL). */
const char *moe_status_string(int status);

/*
 * Router: logits = h W_r (+ bias), top-k, affinities.
 *   h [M,H] bf16; w_router [H,E] bf16; bias [E] fp32 or NULL (added to the logits, used
 *   for both selection and affinities).
 *   Outputs topk_ids [M,k] int32 (slot j = j-th largest logit, ties to the lower expert
 *   id) and topk_weights [M,k] fp32: renormalize != 0 gives softmax over the k selected
 *   logits; renormalize == 0 gives the full softmax over E at the selected experts.
 *   Logits accumulate in fp32 in a fixed order (independent of M).
 */
int moe_route_topk(const void *h, const void *w_router, const float *bias, int M, int H,
                   int E, int k, int renormalize, int32_t *topk_ids, float *topk_weights,
                   void *stream);

/* Rows the alignment can need: M*k + min(E, M*k) * (b - 1).  Returns 0 on bad sizes. */
size_t moe_align_capacity(int M, int k, int E, int b);

/*
 * Stable block alignment ("Route-Block Membership ...", Sections 2.1, 3.1, 5.3).
 *   topk_ids [M,k] int32.  Route r = m*k + j is valid when 0 <= topk_ids[r] < E; invalid
 *   routes are excluded.  For each expert e in ascending order with n_e > 0 routes:
 *   its routes in ascending r, then ceil(n_e/b)*b - n_e sentinel rows (value M*k).
 *   Outputs: sorted_route_ids [cap] int32, expert_block_ids [cap/b] int32 (expert of each
 *   b-row block, -1 past the last block), num_padded [1] int32 (rows used).  Rows past
 *   num_padded are sentinels.  cap must be >= moe_align_capacity(M, k, E, b), else
 *   MOE_ERR_WORKSPACE.  Atomic-free ordering: bitwise identical on every run.
 */
int moe_align_block_size(const int32_t *topk_ids, int M, int k, int E, int b,
                         int32_t *sorted_route_ids, int32_t *expert_block_ids,
                         int32_t *num_padded, size_t cap, void *stream);

/*
 * Workspace bytes that moe_expert_ffn / moe_decode_block need for (weights shape, M, k, b)
 * (b == 0: enough for any block size the library may pick).  The workspace holds the
 * alignment (when the library computes it), the per-route intermediates (dense weights:
 * tiles of token rows and of p in bf16, per-tile counters; VQ weights: p [M*k, I] fp32),
 * the expert outputs y [M*k, H] fp32, the device status word (its first 4 bytes) and
 * counters, which must be zero before the first call (allocate it zero-filled, or zero the
 * first zero_bytes of moe_workspace_layout) and which every call leaves zero.  Calls that share a
 * workspace must be ordered on one stream.  Returns 0 on unsupported arguments.
 */
size_t moe_workspace_bytes(const moe_expert_weights_t *w, int M, int k, int b);

/*
 * The block size moe_decode_block (and moe_expert_ffn without an alignment) aligns with for
 * (weights, M, k, b): b itself when b > 0; for b == 0 the library's choice -- 8 for the VQ
 * forms 0 and 1, and for dense weights and VQ form 2 a tcgen05 tile width, 16 or 64 rows,
 * by routes per expert and (dense) by whether one wave of 16-row units' weights fits in
 * this device's L2.  Every route's bits are the same whatever the block size; the choice
 * only affects speed.  Host-only (reads device attributes of the current device, once).
 * Returns 0 on invalid arguments.
 */
int moe_library_block_size(const moe_expert_weights_t *w, int M, int k, int b);

/*
 * Where moe_decode_block (and moe_expert_ffn without a caller alignment) keeps what it
 * computes inside its workspace, so that a caller can read it after the call: byte offsets
 * of sorted_route_ids [cap] int32, expert_block_ids [cap / b] int32, num_padded [1] int32
 * and the status word, for the block size b the call aligns with (as
 * moe_library_block_size resolves it) -- the arrays have the layout and contents that
 * moe_align_block_size gives for the call's topk_ids, E and b -- and the per-route
 * intermediates: y [M*k][H] fp32 (the down projection of every valid route; rows of invalid
 * routes are not written) and, for the tensor-core paths (kn > 0), the p tiles: for each
 * tile of kn aligned rows (tpb tiles per block, tile t of block q holding rows
 * q*b + t*kn ...), per 64-wide chunk of I, kn rows of 128 bytes, 16-byte piece j of row n at
 * byte n*128 + ((j ^ (n % 8)) * 16): p = SiLU(g) * u in bf16 for the rows that hold a route.
 * Host-only; nothing is launched.  MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED on bad
 * arguments.
 */
typedef struct moe_workspace_layout {
    int32_t b;                /* block size the call aligns with */
    int32_t kn;               /* rows per p tile (0: no p tiles, VQ forms 0 and 1) */
    int64_t cap;              /* rows of sorted_route_ids: moe_align_capacity(M, k, E, b) */
    size_t status;            /* byte offsets inside the workspace */
    size_t sorted_route_ids;
    size_t expert_block_ids;
    size_t num_padded;
    size_t y;
    size_t p_tiles;
    int32_t tpb;              /* p tiles per aligned block */
    int32_t zero_bytes;       /* the first zero_bytes bytes (status word, counters, the
                                 one-grid path's routing exchange) must be zero before the
                                 first call; every call leaves them zero */
    int32_t launches;         /* kernels one moe_decode_block call launches (1: the whole
                                 block in one grid) */
    int32_t reserved;
    size_t p_rows;            /* the one-grid path (launches == 1): p [M*k][I] bf16 per route
                                 instead of p tiles (0 otherwise) */
} moe_workspace_layout_t;
int moe_workspace_layout(const moe_expert_weights_t *w, int M, int k, int b,
                         moe_workspace_layout_t *out);

/*
 * Expert FFN + affinity-weighted combine for given routes.
 *   h [M,H] bf16; topk_ids [M,k] int32; topk_weights [M,k] fp32; residual [M,H] bf16 or
 *   NULL; out [M,H] bf16 = bf16(residual + sum_j a_j y_j) (tokens with no valid route get
 *   the residual, or zero).
 *   Alignment: either all three of sorted_route_ids / expert_block_ids / num_padded as
 *   produced by moe_align_block_size for (topk_ids, E, b) -- every valid route exactly
 *   once, b > 0 -- or all three NULL, in which case the alignment is computed into the
 *   workspace with block size b (b == 0: the library's choice, moe_library_block_size).
 *   workspace: ws_bytes >= moe_workspace_bytes(w, M, k, b).
 */
int moe_expert_ffn(const void *h, const moe_expert_weights_t *w, int M, int k,
                   const int32_t *topk_ids, const float *topk_weights,
                   const int32_t *sorted_route_ids, const int32_t *expert_block_ids,
                   const int32_t *num_padded, int b, const void *residual, void *out,
                   void *workspace, size_t ws_bytes, void *stream);

/*
 * The whole block: router (renormalised softmax top-k) -> alignment -> expert FFN ->
 * combine.  Same arguments as above; topk_ids [M,k] and topk_weights [M,k] are outputs.
 * The routes are aligned into blocks of b rows; b == 0 lets the library pick (16 or 64
 * rows for the tensor-core paths, by routes per expert: moe_library_block_size).  Dense
 * weights (and VQ weights with vq_form 2) run as grouped GEMMs on the tensor cores over
 * tiles of the aligned blocks: 16-row tiles for blocks of up to 16 rows, 64-row tiles
 * otherwise.  Dense gate/up and down run in one persistent grid whose down units stream
 * their weights while gate/up runs.  Every route is one K-ordered chain of MMAs per
 * projection, so a token's output bits do not depend on M, on the other tokens, on its block
 * or its position in it, on b or on the tile width.  VQ gate/up weights with vq_form 0 or 1
 * run on the CUDA cores; their results are bitwise reproducible and independent of M and of
 * block membership.  The alignment stays in the workspace (moe_workspace_layout).
 */
int moe_decode_block(const void *h, const void *w_router, const float *bias,
                     const moe_expert_weights_t *w, int M, int k, int b,
                     const void *residual, void *out, int32_t *topk_ids,
                     float *topk_weights, void *workspace, size_t ws_bytes, void *stream);

/*
 * moe_decode_block with HOST input and output: copies h_host [M,H] bf16 (and residual_host
 * if not NULL) into the caller's device staging buffers h_dev / residual_dev, runs the
 * block, copies out_dev [M,H] back to out_host, and synchronises `stream` before returning.
 * Host buffers should be pinned (page-locked) for asynchronous copies.
 */
int moe_decode_block_host(const void *h_host, const void *residual_host, void *out_host,
                          void *h_dev, void *residual_dev, void *out_dev,
                          const void *w_router, const float *bias,
                          const moe_expert_weights_t *w, int M, int k, int b,
                          int32_t *topk_ids, float *topk_weights, void *workspace,
                          size_t ws_bytes, void *stream);

/*
 * Allocation-free variant of moe_decode_block.  (The papers have no counterpart; this is a
 * deployment convenience of this library.)
 *
 * For callers that cannot allocate device memory for a workspace -- a host program whose
 * GPU memory belongs entirely to another allocator (an inference server's pool, a plugin
 * host that only passes its input and output tensors), or a deployment that forbids
 * allocation after start-up to hold a fixed memory budget.  The caller passes the same
 * inputs and outputs as moe_decode_block, minus the workspace: the block's scratch
 * (alignment rows, per-route p and y, status word) lives in one fixed device array inside
 * the library, MOE_NOALLOC_SCRATCH_BYTES per GPU, held by every GPU that loads the library
 * until the process exits.  It calls no cudaMalloc / cudaFree.
 *   * Sizes whose workspace (moe_workspace_bytes) exceeds MOE_NOALLOC_SCRATCH_BYTES return
 *     MOE_ERR_WORKSPACE before anything is launched (for H=2048, I=768, E=128, k=8 that is
 *     M > 150 tokens at b=8, M > 205 at b=16).
 *   * The first call on a device looks up the array's device address (once per device,
 *     with that device current); make that first call before any stream capture.
 *   * Every call on a device uses the same array: calls that overlap on the GPU (other
 *     streams, or unordered host threads) race.  Order them on one stream.
 *   * The array keeps the previous call's contents; each call clears the status word
 *     itself.  Device status cannot be read back through this entry point.
 */
#define MOE_NOALLOC_SCRATCH_BYTES (32u << 20)
int moe_decode_block_noalloc(const void *h, const void *w_router, const float *bias,
                             const moe_expert_weights_t *w, int M, int k, int b,
                             const void *residual, void *out, int32_t *topk_ids,
                             float *topk_weights, void *stream);

/*
 * Tracing.  When `events` is not NULL, each later moe_decode_block / moe_expert_ffn call
 * made from this host thread records the caller's CUDA events (cudaEvent_t passed as
 * void*) on its stream: events[0] before its first kernel, events[1] after the router,
 * events[2] after the alignment (and the row gather of dense weights), events[3] after the
 * gate/up kernel, events[4] after the
 * down kernel, events[5] after the combine kernel (stages a call does not run are not
 * recorded; n must be 6).  moe_reader_ffn records events[0] before its first kernel, then
 * events[1..5] after its scan and sketch scores, selection, exact reads, recovery and final
 * sum (for one token, whose stages run in one kernel, all five after it).  An
 * event between two kernels removes the launch overlap the
 * kernels otherwise get, so traced calls run slightly slower.  Pass NULL (n = 0) to stop.
 */
int moe_set_trace_events(void *const *events, int n);

/*
 * Synchronises `stream`, reads the workspace's device status word into *status_out and
 * clears it.  Returns MOE_OK when the word was zero, MOE_ERR_DEVICE when any bit was set.
 */
int moe_read_device_status(void *workspace, void *stream, int32_t *status_out);

/*
 * Failure-detection self-test.  Launches, on `stream`, one CTA shaped like the grouped-GEMM
 * kernels that takes its tensor memory and then waits on an mbarrier that nothing ever
 * completes.  The kernels' own bounded wait gives up after about one second of %globaltimer.
 * The CTA then stops its other warps, frees its tensor memory and sets MOE_DEV_WAIT_TIMEOUT
 * in the workspace's status word.  No copy, MMA or memory access besides the status word
 * is ever issued, so the CUDA context stays usable.
 *
 * workspace: a device pointer, 256-byte aligned, with ws_bytes >= 4.  Only its status word
 * (the first int32) is written.
 * Returns MOE_ERR_INVALID_ARG for a NULL, misaligned or too small workspace, MOE_ERR_CUDA if
 * the launch fails, else MOE_OK once the launch is enqueued (asynchronous, like every
 * entry point; read the bit back with moe_read_device_status).
 */
int moe_selftest_wait_timeout(void *workspace, size_t ws_bytes, void *stream);

/*
 * Channel-sparse reader ("Channel Selection for Mixture-of-Experts Decoding Needs No
 * Calibration Data", the reader's Stages 1-3), for dense weights.  Per token, over the
 * k * I channels of its routed experts (channel = one row of gate/up, one row of W_down):
 *   1. x is rotated in 128-coordinate blocks by a random Hadamard transform R (signs given);
 *      every channel's rotated gate and up rows are held as ternary sketches (two-bit codes
 *      and one fp32 scale per block: the Ternary Weight Networks threshold 0.7 mean|r|, the
 *      scale the mean |r| of the nonzero codes); per block only the nscan coordinates of
 *      largest |Rx| are scanned; ahat = SiLU(ghat) * vhat;
 *   2. score = w * ||d|| * |ahat| (w the router weight of the channel's expert); the K best
 *      channels across all the token's experts (ties: lower slot * I + channel index) are
 *      read exactly: a = SiLU(g . x) * (v . x);
 *   3. out = residual + sum_{kept} w a d + U sum_{discarded} w ahat b,  b = U^T d.
 * All sums run in fixed orders: outputs are bitwise reproducible and a token's output does
 * not depend on the other tokens.
 *
 * Data (caller-allocated device buffers, 16-byte aligned):
 *   signs   [H] int8 +1/-1;               U [H][rank] fp32 (rank <= 32), orthonormal columns
 *   w_down  [E][I][H] bf16 (the layer's W_down, read in place)
 *   g_rows, v_rows [E][I][H] bf16;  g_codes, v_codes [E][I][H/128][8] uint32 (per block,
 *   words 0-3 the mask of nonzero codes, words 4-7 the mask of negative ones; coordinate c
 *   at bit c%32 of word c/32);  g_scales, v_scales
 *   [E][I][H/128] fp32;  dnorm [E][I] fp32;  coef [E][I][rank] bf16 -- written by
 *   moe_reader_build.
 * Shapes: H a multiple of 128 up to 8192, 1 <= rank <= 32.
 */
typedef struct moe_reader {
    int H, I, E, rank;
    const int8_t *signs;
    void *g_rows, *v_rows;
    const void *w_down;
    void *g_codes, *v_codes;
    float *g_scales, *v_scales;
    float *dnorm;
    const float *U;
    void *coef;
} moe_reader_t;

/*
 * Builds the reader's data from dense weights w (kind MOE_W_DENSE_BF16, same H, I, E) and
 * rd->signs, rd->U: channel-major gate/up rows, their sketches, the down-row norms and
 * coef = U^T d.  Stream-ordered; MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED before launching.
 */
int moe_reader_build(const moe_expert_weights_t *w, const moe_reader_t *rd, void *stream);

/* Workspace bytes of moe_reader_ffn for (rd, M, k, K); 0 on unsupported arguments. */
size_t moe_reader_workspace_bytes(const moe_reader_t *rd, int M, int k, int K);

/*
 * The reader's decode for M tokens with their routes: topk_ids [M,k] int32 (ids outside
 * [0,E) are skipped), topk_weights [M,k] fp32.  K = channels read exactly per token
 * (0 <= K <= k*I; a token with fewer valid channels reads them all), nscan = coordinates
 * scanned per 128-block (0..128), k*I <= 16384.  residual [M,H] bf16 or NULL; out [M,H]
 * bf16.  Optional outputs for inspection: selected [M,K] int32, the kept channels of each
 * token (slot * I + channel, ascending, -1 past the token's count), and xr [M,H] fp32, Rx
 * with the unscanned coordinates set to zero.  workspace: ws_bytes >=
 * moe_reader_workspace_bytes(rd, M, k, K), 256-byte aligned; its first 128 bytes (the
 * status word and the counters of the one-token path) must be zero before the first call
 * (allocate it zero-filled), and every call leaves them zero.  One token runs as one grid
 * (the stages in one persistent kernel, bitwise the same results); several tokens run the
 * stages as five kernels.
 */
int moe_reader_ffn(const void *h, const moe_reader_t *rd, int M, int k, const int32_t *topk_ids,
                   const float *topk_weights, int K, int nscan, const void *residual, void *out,
                   int32_t *selected, float *xr, void *workspace, size_t ws_bytes, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
