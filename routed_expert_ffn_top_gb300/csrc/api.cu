// api.cu -- the C ABI (include/moe.h): argument validation, workspace layout, TMA tensor
// maps and the stream-ordered orchestration of the kernels.
#include <cudaTypedefs.h>
#include <string.h>

#include <map>
#include <mutex>

#include "moe_internal.cuh"

namespace moe {

static size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

Dims make_dims(int M, int k, int E, int H, int I, int b, int kind) {
    Dims d;
    d.M = M;
    d.k = k;
    d.E = E;
    d.H = H;
    d.I = I;
    d.b = b;
    d.gemm = kind == MOE_W_DENSE_BF16;
    d.kn = gemm_tile_width(b);
    d.tpb = gemm_tiles_per_block(b);
    d.rsub = (b <= kNT) ? b : kNT;
    d.R = (int64_t)M * k;
    d.cap = d.R + (int64_t)(d.R < E ? d.R : E) * (b - 1);
    d.max_sub = d.cap / d.rsub;
    d.n_it = I / kTI;
    d.n_hb = H / kBoxRows;
    d.n_ht = H / kTN;
    d.n_ib = I / kBoxRows;
    return d;
}

WsLayout ws_layout(const Dims &d) {
    WsLayout L;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = align_up(off + bytes, 256);
        return at;
    };
    L.status = take(64);
    L.ctl = take((size_t)kSmallCtlInts * 4);  // every layout keeps it (no other path writes it)
    L.partials = take((size_t)kSmallPartialInts * 4);  // likewise
    L.sorted = take((size_t)d.cap * 4);
    L.blocks = take((size_t)(d.cap / d.b) * 4);
    L.npad = take(16);
    // the sub-block table and fp32 p serve the GEMV kernels, the row tiles the tcgen05 ones
    L.sbt = take(d.gemm ? 0 : (size_t)d.max_sub * sizeof(SubBlock));
    L.p = take(d.gemm ? 0 : (size_t)d.R * d.I * 4);
    L.y = take((size_t)d.R * d.H * 4);
    L.z = take((size_t)d.M * 2 * d.r * 4);
    const size_t tile_rows = d.gemm ? (size_t)(d.cap / d.b) * d.tpb * d.kn : 0;
    L.x_tiles = take(tile_rows * d.H * 2);
    L.p_tiles = take(tile_rows * d.I * 2);
    L.ready = take(d.gemm ? ((size_t)(d.cap / d.b) * d.tpb + 1) * 4 : 0);  // + the unit counter
    const bool small = d.gemm && !d.vq_tc && small_fits(d.M, d.k, d.E, d.H, d.b);
    L.p_rows = take(small ? (size_t)d.R * d.I * 2 : 0);
    L.tt_part = take(d.ttable ? (size_t)vq_ttable_slices(d.H, d.vqd) * d.R * 2 * d.I * 4 : 0);
    L.total = off;
    return L;
}

int num_sms() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
    if (cache[dev] == 0) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        cache[dev] = n > 0 ? n : 1;
    }
    return cache[dev];
}

int l2_bytes() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (cache[dev] == 0) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrL2CacheSize, dev);
        cache[dev] = n > 0 ? n : -1;
    }
    return cache[dev] > 0 ? cache[dev] : 0;
}

cudaError_t ensure_smem(const void *func, size_t bytes) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    static std::mutex mu;
    static std::map<std::pair<const void *, int>, size_t> done;
    std::lock_guard<std::mutex> lock(mu);
    auto it = done.find({func, dev});
    if (it != done.end() && it->second >= bytes) return cudaSuccess;
    err = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (err == cudaSuccess) done[{func, dev}] = bytes;
    return err;
}

cudaLaunchConfig_t launch_config(dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                                 cudaLaunchAttribute *attrs, int cluster_x) {
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    int n = 0;
    attrs[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
    if (cluster_x > 0) {
        attrs[n].id = cudaLaunchAttributeClusterDimension;
        attrs[n].val.clusterDim.x = cluster_x;
        attrs[n].val.clusterDim.y = 1;
        attrs[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attrs;
    cfg.numAttrs = n;
    return cfg;
}

// --------------------------------------------------------------------- tensor maps
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 3-D row-major bf16 tensor [d2][d1][d0], box [b2][b1][b0], no swizzle; out-of-range box
// elements read as zeros.
static bool make_tmap_3d_bf16(CUtensorMap *tm, const void *base, uint64_t d0, uint64_t d1,
                              uint64_t d2, uint32_t b0, uint32_t b1, uint32_t b2) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
    cuuint32_t box[3] = {b0, b1, b2};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D row-major tensor [outer][inner] of `elem` bytes, box [box_outer][box_inner].
static bool make_tmap_2d(CUtensorMap *tm, const void *base, CUtensorMapDataType dt, int elem,
                         uint64_t inner, uint64_t outer, uint32_t box_inner, uint32_t box_outer,
                         CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_NONE) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * (uint64_t)elem};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    return fn(tm, dt, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace moe

using namespace moe;

// ------------------------------------------------------------------------------ tracing
constexpr int kTracePoints = 6;
static thread_local cudaEvent_t g_trace[kTracePoints] = {};
static thread_local bool g_tracing = false;

static void trace(int i, cudaStream_t s) {
    if (g_tracing && g_trace[i]) cudaEventRecord(g_trace[i], s);
}

void moe::trace_point(int i, cudaStream_t s) { trace(i, s); }

extern "C" int moe_set_trace_events(void *const *events, int n) {
    if (events == nullptr) {
        g_tracing = false;
        for (int i = 0; i < kTracePoints; ++i) g_trace[i] = nullptr;
        return MOE_OK;
    }
    if (n != kTracePoints) return MOE_ERR_INVALID_ARG;
    for (int i = 0; i < kTracePoints; ++i) g_trace[i] = static_cast<cudaEvent_t>(events[i]);
    g_tracing = true;
    return MOE_OK;
}

// ------------------------------------------------------------------------ validation
static bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

static int check_router_shape(int M, int H, int E, int k) {
    if (M < 0 || H <= 0 || E <= 0 || k <= 0) return MOE_ERR_INVALID_ARG;
    if (E < 8 || E > 512 || E % 8 != 0) return MOE_ERR_UNSUPPORTED;
    if (k > E || k > 32) return MOE_ERR_UNSUPPORTED;
    if (H % 128 != 0 || H < 128 || H > 8192) return MOE_ERR_UNSUPPORTED;
    if ((size_t)(H / kRouterCluster) * E * 2 > 131072) return MOE_ERR_UNSUPPORTED;
    if ((int64_t)M * k >= (1 << 24)) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

static int check_block(int b) {
    if (b <= 0) return MOE_ERR_INVALID_ARG;
    if (b > kNT && b % kNT != 0) return MOE_ERR_UNSUPPORTED;
    if (b > 4096) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

static int check_weights(const moe_expert_weights_t *w) {
    if (!w) return MOE_ERR_INVALID_ARG;
    if (w->H <= 0 || w->I <= 0 || w->E <= 0) return MOE_ERR_INVALID_ARG;
    if (w->I % kBoxRows != 0 || w->I > 8192) return MOE_ERR_UNSUPPORTED;
    if (w->H % kBoxRows != 0 || w->H > 8192) return MOE_ERR_UNSUPPORTED;
    if (w->E < 8 || w->E > 512 || w->E % 8 != 0) return MOE_ERR_UNSUPPORTED;
    if (!w->w_down || !aligned(w->w_down, 16)) return MOE_ERR_INVALID_ARG;
    if (w->vq_form < 0 || w->vq_form > 2) return MOE_ERR_INVALID_ARG;
    if (w->vq_form != 0 && w->kind != MOE_W_VQ_GATEUP) return MOE_ERR_UNSUPPORTED;
    if (w->kind == MOE_W_DENSE_BF16) {
        if (!w->w_gate || !w->w_up || !aligned(w->w_gate, 16) || !aligned(w->w_up, 16))
            return MOE_ERR_INVALID_ARG;
        return MOE_OK;
    }
    if (w->kind == MOE_W_VQ_GATEUP || w->kind == MOE_W_VQLR_GATEUP) {
        if (!w->j_gate || !w->j_up || !w->cb_gate || !w->cb_up) return MOE_ERR_INVALID_ARG;
        if (!aligned(w->j_gate, 16) || !aligned(w->j_up, 16) || !aligned(w->cb_gate, 16) ||
            !aligned(w->cb_up, 16))
            return MOE_ERR_INVALID_ARG;
        if ((w->d != 4 && w->d != 8) || w->K != 256) return MOE_ERR_UNSUPPORTED;
        if (w->H % 1024 != 0) return MOE_ERR_UNSUPPORTED;  // index boxes cover 1024 rows of H
        if (w->kind == MOE_W_VQ_GATEUP) return MOE_OK;
        if (!w->d_gate || !w->d_up || !w->c_gate || !w->c_up || !aligned(w->d_gate, 16) ||
            !aligned(w->d_up, 16) || !aligned(w->c_gate, 16) || !aligned(w->c_up, 16))
            return MOE_ERR_INVALID_ARG;
        if (w->r <= 0) return MOE_ERR_INVALID_ARG;
        // r in multiples of 128 up to 512 (the router's column split; 256-row boxes of C)
        if (w->r % 128 != 0 || w->r > 512) return MOE_ERR_UNSUPPORTED;
        return MOE_OK;
    }
    return MOE_ERR_INVALID_ARG;
}

// Rank of the low-rank term (0 unless the weights are VQ + low rank).
static int lr_rank(const moe_expert_weights_t *w) {
    return (w && w->kind == MOE_W_VQLR_GATEUP) ? w->r : 0;
}

static Dims dims_for(const moe_expert_weights_t *w, int M, int k, int b) {
    Dims d = make_dims(M, k, w->E, w->H, w->I, b, w->kind);
    d.r = lr_rank(w);
    d.ttable = w->kind == MOE_W_VQ_GATEUP && w->vq_form == 1;
    d.vqd = w->d;
    if (w->kind == MOE_W_VQ_GATEUP && w->vq_form == 2) {
        d.gemm = true;  // the tiles of dense weights (16 or 64 rows by b)
        d.vq_tc = true;
    }
    return d;
}

static int cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

extern "C" const char *moe_status_string(int status) {
    switch (status) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_UNSUPPORTED: return "unsupported shape or configuration";
        case MOE_ERR_WORKSPACE: return "workspace or capacity too small";
        case MOE_ERR_CUDA: return "CUDA error";
        case MOE_ERR_DEVICE: return "device status flag set";
        default: return "unknown status";
    }
}

extern "C" int moe_route_topk(const void *h, const void *w_router, const float *bias, int M,
                              int H, int E, int k, int renormalize, int32_t *topk_ids,
                              float *topk_weights, void *stream) {
    int rc = check_router_shape(M, H, E, k);
    if (rc != MOE_OK) return rc;
    if (M == 0) return MOE_OK;
    if (!h || !w_router || !topk_ids || !topk_weights) return MOE_ERR_INVALID_ARG;
    if (!aligned(h, 16) || !aligned(w_router, 16) || !aligned(topk_ids, 4) ||
        !aligned(topk_weights, 4) || (bias && !aligned(bias, 4)))
        return MOE_ERR_INVALID_ARG;
    return cuda_status(launch_router(static_cast<const __nv_bfloat16 *>(h),
                                     static_cast<const __nv_bfloat16 *>(w_router), bias, M, H, E, k,
                                     renormalize, topk_ids, topk_weights, nullptr,
                                     static_cast<cudaStream_t>(stream)));
}

extern "C" size_t moe_align_capacity(int M, int k, int E, int b) {
    if (M < 0 || k <= 0 || E <= 0 || b <= 0) return 0;
    const int64_t R = (int64_t)M * k;
    return (size_t)(R + (int64_t)(R < E ? R : E) * (b - 1));
}

extern "C" int moe_align_block_size(const int32_t *topk_ids, int M, int k, int E, int b,
                                    int32_t *sorted_route_ids, int32_t *expert_block_ids,
                                    int32_t *num_padded, size_t cap, void *stream) {
    if (M < 0 || k <= 0 || E <= 0 || b <= 0) return MOE_ERR_INVALID_ARG;
    if (E > 4096 || (int64_t)M * k >= (1 << 24)) return MOE_ERR_UNSUPPORTED;
    if (cap < moe_align_capacity(M, k, E, b)) return MOE_ERR_WORKSPACE;
    if (!num_padded || (M > 0 && !topk_ids) || (cap > 0 && !sorted_route_ids) ||
        (cap / b > 0 && !expert_block_ids))
        return MOE_ERR_INVALID_ARG;
    if ((topk_ids && !aligned(topk_ids, 4)) || (sorted_route_ids && !aligned(sorted_route_ids, 4)) ||
        (expert_block_ids && !aligned(expert_block_ids, 4)) || !aligned(num_padded, 4))
        return MOE_ERR_INVALID_ARG;
    return cuda_status(launch_align(topk_ids, M, k, E, b, sorted_route_ids, expert_block_ids,
                                    num_padded, (int64_t)cap, nullptr, 0, nullptr,
                                    static_cast<cudaStream_t>(stream)));
}

// The block size the library aligns with when the caller leaves it to the library (b == 0).
// Dense weights, and VQ weights decoded on the tensor cores, run as tcgen05 tiles, so the
// library picks the tile width: 16-row blocks, or 64-row ones from `per_expert` routes per
// expert on average.  Measured on GB300 (16- against 64-row tiles):
//   - dense weights: an expert's 16-row tiles run on neighbouring CTAs at the same time, so
//     the second tile's weights come from L2 while one wave of units' weights fits in it
//     (H = 2048: 16-row tiles faster up to 16 routes per expert, even at 24, slower at 32);
//     when a wave does not fit (H = 4096, I = 1536) 64-row tiles are faster from 8;
//   - VQ decoded on the tensor cores: a unit's MMAs and decoding cost the same for 16 or
//     64 rows; 16-row tiles faster up to 12 routes per expert, 64-row ones from 16.
// The other VQ forms stream sub-blocks of 8 routes: they take b = 8.
static int library_block(const moe_expert_weights_t *w, int M, int k) {
    const bool vq_tc = w && w->kind == MOE_W_VQ_GATEUP && w->vq_form == 2;
    if (!w || (w->kind != MOE_W_DENSE_BF16 && !vq_tc)) return kNT;
    int per_expert = 16;
    if (!vq_tc) {
        const int64_t wave = (int64_t)num_sms() * 2 * 64 * w->H * 2;  // 16-row units' weights
        per_expert = wave <= (int64_t)l2_bytes() ? 24 : 4;
    }
    return (int64_t)M * k >= (int64_t)per_expert * w->E ? kGemmBlock : kGemmNarrow;
}

// The caller's b, or the library's choice when b == 0; -1 for a negative b.
static int resolve_block(const moe_expert_weights_t *w, int M, int k, int b) {
    if (b < 0) return -1;
    return b == 0 ? library_block(w, M, k) : b;
}

int moe::block_for(const moe_expert_weights_t *w, int M, int k, int b) {
    return resolve_block(w, M, k, b);
}

extern "C" int moe_library_block_size(const moe_expert_weights_t *w, int M, int k, int b) {
    if (!w || M < 0 || k <= 0) return 0;
    b = resolve_block(w, M, k, b);
    return check_block(b) == MOE_OK ? b : 0;
}

size_t moe::workspace_bytes_fixed(const moe_expert_weights_t *w, int M, int k, int b) {
    if (!w || M < 0 || k <= 0 || k > 32 || k > w->E || check_block(b) != MOE_OK) return 0;
    if (w->H <= 0 || w->I <= 0 || w->E <= 0) return 0;
    if ((int64_t)M * k >= (1 << 24)) return 0;
    if (w->vq_form < 0 || w->vq_form > 2 || (w->vq_form != 0 && w->kind != MOE_W_VQ_GATEUP))
        return 0;
    Dims d = dims_for(w, M, k, b);
    return ws_layout(d).total;
}

extern "C" size_t moe_workspace_bytes(const moe_expert_weights_t *w, int M, int k, int b) {
    if (!w || b < 0) return 0;
    if (b > 0) return workspace_bytes_fixed(w, M, k, b);
    // b == 0: enough for either block size the library may pick, so that the size does not
    // depend on the device the choice is made on
    const size_t a = workspace_bytes_fixed(w, M, k, library_block(w, M, k));
    if (a == 0) return 0;
    const bool tiles = w->kind == MOE_W_DENSE_BF16 || (w->kind == MOE_W_VQ_GATEUP && w->vq_form == 2);
    if (!tiles) return a;
    const size_t n = workspace_bytes_fixed(w, M, k, kGemmNarrow);
    const size_t wide = workspace_bytes_fixed(w, M, k, kGemmBlock);
    return a > n ? (a > wide ? a : wide) : (n > wide ? n : wide);
}

// Kernels one moe_decode_block call launches for these dimensions.
static bool vq_small_path(const moe_expert_weights_t *w, const Dims &d) {
    return w->kind == MOE_W_VQ_GATEUP && w->vq_form == 0 && !d.gemm &&
           vq_small_fits(d.M, d.k, d.E, d.H, d.I, d.b, w->d);
}

static int block_launches(const moe_expert_weights_t *w, const Dims &d) {
    if (d.gemm && !d.vq_tc && small_fits(d.M, d.k, d.E, d.H, d.b)) return 1;
    if (vq_small_path(w, d)) return 1;
    const bool fused = router_can_align(d.M, d.k);
    int n = 1 + (fused ? 0 : 1);                                   // router, alignment
    n += (d.gemm && !fused && d.R > kAlignGatherRoutes) ? 1 : 0;   // row gather
    if (w->kind == MOE_W_DENSE_BF16) n += 1;                        // gate/up and down, one grid
    else n += 2 + (d.ttable ? 1 : 0);
    return n + 1;                                                   // combine
}

extern "C" int moe_workspace_layout(const moe_expert_weights_t *w, int M, int k, int b,
                                    moe_workspace_layout_t *out) {
    if (!w || !out || M < 0 || k <= 0) return MOE_ERR_INVALID_ARG;
    b = resolve_block(w, M, k, b);
    int rc = check_block(b);
    if (rc != MOE_OK) return rc;
    if (workspace_bytes_fixed(w, M, k, b) == 0) return MOE_ERR_UNSUPPORTED;
    const Dims d = dims_for(w, M, k, b);
    const WsLayout L = ws_layout(d);
    memset(out, 0, sizeof *out);
    out->b = b;
    out->kn = d.gemm ? d.kn : 0;
    out->tpb = d.gemm ? d.tpb : 0;
    out->cap = d.cap;
    out->status = L.status;
    out->sorted_route_ids = L.sorted;
    out->expert_block_ids = L.blocks;
    out->num_padded = L.npad;
    out->y = L.y;
    out->p_tiles = L.p_tiles;
    out->zero_bytes = (int32_t)(L.partials + (size_t)kSmallPartialInts * 4);
    out->launches = block_launches(w, d);
    out->p_rows = out->launches == 1 ? L.p_rows : 0;
    return MOE_OK;
}

// Where the kernel that writes the x tiles puts them, and the ready counts it zeroes.
static RowTiles row_tiles(const Dims &d, unsigned char *ws, const WsLayout &L) {
    RowTiles rows;
    rows.x_tiles = reinterpret_cast<__nv_bfloat16 *>(ws + L.x_tiles);
    rows.kn = d.kn;
    rows.tpb = d.tpb;
    rows.ready = reinterpret_cast<int32_t *>(ws + L.ready);
    rows.nready = (d.cap / d.b) * d.tpb + 1;  // the tiles' counts and the unit counter
    return rows;
}

// Runs gate/up and down for aligned routes (alignment pointers already resolved).
// The low-rank projections of VQ + low-rank weights (z in the workspace), or NULL.
static const LowRankProj *lowrank_proj(const moe_expert_weights_t *w, const Dims &d,
                                       unsigned char *ws, const WsLayout &L, LowRankProj *out) {
    if (w->kind != MOE_W_VQLR_GATEUP) return nullptr;
    out->d_gate = static_cast<const __nv_bfloat16 *>(w->d_gate);
    out->d_up = static_cast<const __nv_bfloat16 *>(w->d_up);
    out->r = d.r;
    out->first = 0;
    out->z = reinterpret_cast<float *>(ws + L.z);
    return out;
}

// Dense weights (or VQ gate/up decoded on the tensor cores): the row gather (unless the
// router wrote the rows), tcgen05 grouped GEMMs over the tiles of the aligned blocks, then
// the fixed-order combine.
static int run_gemm(const void *h, const moe_expert_weights_t *w, const Dims &d,
                    const int32_t *topk_ids, const float *topk_weights, const int32_t *sorted,
                    const int32_t *blocks, const int32_t *npad, const void *residual, void *out,
                    unsigned char *ws, const WsLayout &L, bool rows_ready, cudaStream_t stream) {
    CUtensorMap tm_gate, tm_up, tm_down;
    const CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_128B;
    const int box_rows = kGemmStageK;  // K rows per weight box: one stage's depth
    // VQ: the index maps [E * H/d rows][I] uint8, boxes of one stage's 256/d index rows x 128
    // columns (unswizzled; the decoder warps write the weight operand to tensor memory)
    const bool maps_ok =
        d.vq_tc
            ? make_tmap_2d(&tm_gate, w->j_gate, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, (uint64_t)d.I,
                           (uint64_t)d.E * (d.H / w->d), 128, box_rows / w->d) &&
                  make_tmap_2d(&tm_up, w->j_up, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, (uint64_t)d.I,
                               (uint64_t)d.E * (d.H / w->d), 128, box_rows / w->d)
            : make_tmap_2d(&tm_gate, w->w_gate, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)d.I,
                           (uint64_t)d.E * d.H, 64, box_rows, sw) &&
                  make_tmap_2d(&tm_up, w->w_up, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)d.I,
                               (uint64_t)d.E * d.H, 64, box_rows, sw);
    if (!maps_ok ||
        !make_tmap_2d(&tm_down, w->w_down, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)d.H,
                      (uint64_t)d.E * d.I, 64, box_rows, sw))
        return MOE_ERR_CUDA;
    GemmArgs g;
    g.x = static_cast<const __nv_bfloat16 *>(h);
    g.ids = topk_ids;
    g.sorted = sorted;
    g.blocks = blocks;
    g.npad = npad;
    g.x_tiles = reinterpret_cast<__nv_bfloat16 *>(ws + L.x_tiles);
    g.p_tiles = reinterpret_cast<__nv_bfloat16 *>(ws + L.p_tiles);
    g.y = reinterpret_cast<float *>(ws + L.y);
    g.status = reinterpret_cast<int32_t *>(ws + L.status);
    g.M = d.M;
    g.k = d.k;
    g.E = d.E;
    g.H = d.H;
    g.I = d.I;
    g.b = d.b;
    g.kn = d.kn;
    g.tpb = d.tpb;
    g.wait_first = rows_ready ? 1 : 0;
    g.cb_gate = d.vq_tc ? static_cast<const __nv_bfloat16 *>(w->cb_gate) : nullptr;
    g.cb_up = d.vq_tc ? static_cast<const __nv_bfloat16 *>(w->cb_up) : nullptr;
    g.R = d.R;
    g.cap = d.cap;
    g.ready = reinterpret_cast<int32_t *>(ws + L.ready);
    g.nready = (d.cap / d.b) * d.tpb + 1;  // the tiles' counts, then the unit counter
    cudaError_t err = rows_ready ? cudaSuccess : launch_gather_rows(g, stream);
    if (err != cudaSuccess) return MOE_ERR_CUDA;
    if (!rows_ready) trace(2, stream);  // the row gather counts with the alignment
    if (d.vq_tc) {
        err = launch_gemm_gateup_vq(tm_gate, tm_up, g, w->d, stream);
        if (err != cudaSuccess) return MOE_ERR_CUDA;
        trace(3, stream);
        err = launch_gemm_down(tm_down, g, stream);
        if (err != cudaSuccess) return MOE_ERR_CUDA;
        trace(4, stream);
    } else {
        // gate/up and down in one grid: both trace points after it
        err = launch_gemm_fused(tm_gate, tm_up, tm_down, g, stream);
        if (err != cudaSuccess) return MOE_ERR_CUDA;
        trace(3, stream);
        trace(4, stream);
    }
    GemvArgs c;
    memset(&c, 0, sizeof c);
    c.topk_ids = topk_ids;
    c.topk_wts = topk_weights;
    c.residual = static_cast<const __nv_bfloat16 *>(residual);
    c.out = static_cast<__nv_bfloat16 *>(out);
    c.y = g.y;
    c.M = d.M;
    c.k = d.k;
    c.E = d.E;
    c.H = d.H;
    err = launch_combine(c, stream);
    if (err != cudaSuccess) return MOE_ERR_CUDA;
    trace(5, stream);
    return MOE_OK;
}

// rows_ready: the router already wrote the x tiles of the grouped GEMMs.
static int run_experts(const void *h, const moe_expert_weights_t *w, const Dims &d,
                       const int32_t *topk_ids, const float *topk_weights, const int32_t *sorted,
                       const int32_t *blocks, const int32_t *npad, const void *residual, void *out,
                       unsigned char *ws, const WsLayout &L, cudaStream_t stream,
                       bool rows_ready = false) {
    if (d.gemm)
        return run_gemm(h, w, d, topk_ids, topk_weights, sorted, blocks, npad, residual, out, ws,
                        L, rows_ready, stream);
    // VQ (and VQ + low-rank) gate/up: GEMV streams on the CUDA cores
    const bool lowrank = w->kind == MOE_W_VQLR_GATEUP;
    CUtensorMap tm_cgate, tm_cup;  // C [E][r][I]: boxes of 64 columns x 256 rows of r
    if (lowrank && (!make_tmap_3d_bf16(&tm_cgate, w->c_gate, (uint64_t)d.I, (uint64_t)d.r,
                                       (uint64_t)d.E, kTI, kBoxRows, 1) ||
                    !make_tmap_3d_bf16(&tm_cup, w->c_up, (uint64_t)d.I, (uint64_t)d.r,
                                       (uint64_t)d.E, kTI, kBoxRows, 1)))
        return MOE_ERR_CUDA;
    CUtensorMap tm_gate, tm_up, tm_down;
    // index maps [E * H/d rows][I] uint8, boxes of 1024/d rows x 64 columns
    const bool ok =
        make_tmap_2d(&tm_gate, w->j_gate, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, (uint64_t)d.I,
                     (uint64_t)d.E * (d.H / w->d), kTI, 1024 / w->d) &&
        make_tmap_2d(&tm_up, w->j_up, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, (uint64_t)d.I,
                     (uint64_t)d.E * (d.H / w->d), kTI, 1024 / w->d);
    if (!ok || !make_tmap_2d(&tm_down, w->w_down, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)d.H,
                             (uint64_t)d.E * d.I, kTN, kBoxRows))
        return MOE_ERR_CUDA;
    GemvArgs a;
    a.h = static_cast<const __nv_bfloat16 *>(h);
    a.topk_ids = topk_ids;
    a.topk_wts = topk_weights;
    a.sbt = reinterpret_cast<const SubBlock *>(ws + L.sbt);
    a.npad = npad;
    a.residual = static_cast<const __nv_bfloat16 *>(residual);
    a.out = static_cast<__nv_bfloat16 *>(out);
    a.p = reinterpret_cast<float *>(ws + L.p);
    a.y = reinterpret_cast<float *>(ws + L.y);
    a.status = reinterpret_cast<int32_t *>(ws + L.status);
    a.M = d.M;
    a.k = d.k;
    a.E = d.E;
    a.H = d.H;
    a.I = d.I;
    a.b = d.b;
    a.rsub = d.rsub;
    a.n_it = d.n_it;
    a.n_hb = d.n_hb;
    a.n_ht = d.n_ht;
    a.n_ib = d.n_ib;
    a.max_sub = d.max_sub;
    a.w_down = static_cast<const unsigned char *>(w->w_down);
    a.cb_gate = static_cast<const uint2 *>(w->cb_gate);
    a.cb_up = static_cast<const uint2 *>(w->cb_up);
    a.n_qb = d.H / (4 * kBoxRows);
    a.z = lowrank ? reinterpret_cast<const float *>(ws + L.z) : nullptr;
    a.r = lowrank ? d.r : 0;
    a.n_rb = lowrank ? (d.r + kBoxRows - 1) / kBoxRows : 0;
    cudaError_t err;
    if (d.ttable) {
        VQTableArgs t;
        t.h = a.h;
        t.j_gate = w->j_gate;
        t.j_up = w->j_up;
        t.cb_gate = static_cast<const __nv_bfloat16 *>(w->cb_gate);
        t.cb_up = static_cast<const __nv_bfloat16 *>(w->cb_up);
        t.ids = topk_ids;
        t.M = d.M;
        t.k = d.k;
        t.E = d.E;
        t.H = d.H;
        t.I = d.I;
        t.d = w->d;
        t.partial = reinterpret_cast<float *>(ws + L.tt_part);
        t.p = a.p;
        err = launch_vq_ttable(t, stream);
    } else {
        err = launch_gateup_vq(tm_gate, tm_up, lowrank ? &tm_cgate : nullptr,
                               lowrank ? &tm_cup : nullptr, a, w->d, stream);
    }
    if (err != cudaSuccess) return MOE_ERR_CUDA;
    trace(3, stream);
    err = launch_down(tm_down, a, stream);
    if (err != cudaSuccess) return MOE_ERR_CUDA;
    trace(4, stream);
    err = launch_combine(a, stream);
    if (err != cudaSuccess) return MOE_ERR_CUDA;
    trace(5, stream);
    return MOE_OK;
}

static int check_ffn_common(const void *h, const moe_expert_weights_t *w, int M, int k, int b,
                            const void *residual, const void *out, const void *workspace,
                            size_t ws_bytes) {
    int rc = check_weights(w);
    if (rc != MOE_OK) return rc;
    rc = check_block(b);
    if (rc != MOE_OK) return rc;
    if (M < 0 || k <= 0) return MOE_ERR_INVALID_ARG;
    if (k > 32 || k > w->E || (int64_t)M * k >= (1 << 24)) return MOE_ERR_UNSUPPORTED;
    if (w->vq_form == 1 && M > kTTMaxTokens) return MOE_ERR_UNSUPPORTED;
    if (M == 0) return MOE_OK;
    if (!h || !out || !workspace) return MOE_ERR_INVALID_ARG;
    if (!aligned(h, 16) || !aligned(out, 16) || !aligned(workspace, 256) ||
        (residual && !aligned(residual, 16)))
        return MOE_ERR_INVALID_ARG;
    if (ws_bytes < workspace_bytes_fixed(w, M, k, b)) return MOE_ERR_WORKSPACE;
    return MOE_OK;
}

extern "C" int moe_expert_ffn(const void *h, const moe_expert_weights_t *w, int M, int k,
                              const int32_t *topk_ids, const float *topk_weights,
                              const int32_t *sorted_route_ids, const int32_t *expert_block_ids,
                              const int32_t *num_padded, int b, const void *residual, void *out,
                              void *workspace, size_t ws_bytes, void *stream) {
    if (!w) return MOE_ERR_INVALID_ARG;
    const int b_in = b;
    b = resolve_block(w, M, k, b);
    int rc = check_ffn_common(h, w, M, k, b, residual, out, workspace, ws_bytes);
    if (rc != MOE_OK || M == 0) return rc;
    if (!topk_ids || !topk_weights || !aligned(topk_ids, 4) || !aligned(topk_weights, 4))
        return MOE_ERR_INVALID_ARG;
    const int given = (sorted_route_ids != nullptr) + (expert_block_ids != nullptr) +
                      (num_padded != nullptr);
    if (given != 0 && given != 3) return MOE_ERR_INVALID_ARG;
    if (given == 3 && b_in == 0) return MOE_ERR_INVALID_ARG;  // an alignment has its own b
    Dims d = dims_for(w, M, k, b);
    const WsLayout L = ws_layout(d);
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    trace(0, s);
    const int32_t *npad = num_padded;
    int32_t *status = reinterpret_cast<int32_t *>(ws + L.status);
    SubBlock *sbt = reinterpret_cast<SubBlock *>(ws + L.sbt);
    cudaError_t err;
    bool rows_ready = false;  // the alignment launch also wrote the row tiles
    if (given == 0) {
        int32_t *ws_npad = reinterpret_cast<int32_t *>(ws + L.npad);
        int32_t *ws_sorted = reinterpret_cast<int32_t *>(ws + L.sorted);
        int32_t *ws_blocks = reinterpret_cast<int32_t *>(ws + L.blocks);
        if (d.gemm && (int64_t)M * k <= kAlignGatherRoutes) {
            const RowTiles rows = row_tiles(d, ws, L);
            err = launch_align_gather(topk_ids, M, k, w->E, b, ws_sorted, ws_blocks, ws_npad, d.cap,
                                      status, static_cast<const __nv_bfloat16 *>(h), w->H, rows, s);
            rows_ready = true;
        } else {
            err = launch_align(topk_ids, M, k, w->E, b, ws_sorted, ws_blocks, ws_npad, d.cap,
                               d.gemm ? nullptr : sbt, d.rsub, status, s);
        }
        npad = ws_npad;
    } else {
        if (!aligned(sorted_route_ids, 4) || !aligned(expert_block_ids, 4) || !aligned(num_padded, 4))
            return MOE_ERR_INVALID_ARG;
        err = d.gemm
                  ? cudaSuccess
                  : launch_plan(topk_ids, sorted_route_ids, expert_block_ids, num_padded, M, k,
                                w->E, b, d.rsub, d.max_sub, sbt, status, s);
    }
    if (err != cudaSuccess) return MOE_ERR_CUDA;
    LowRankProj lr_store;
    if (const LowRankProj *lr = lowrank_proj(w, d, ws, L, &lr_store)) {
        // without a router launch to ride along, the projections get one of their own
        if (launch_lowrank_proj(static_cast<const __nv_bfloat16 *>(h), M, w->H, *lr, s) !=
            cudaSuccess)
            return MOE_ERR_CUDA;
    }
    trace(2, s);
    const int32_t *srt = given ? sorted_route_ids : reinterpret_cast<const int32_t *>(ws + L.sorted);
    const int32_t *blk = given ? expert_block_ids : reinterpret_cast<const int32_t *>(ws + L.blocks);
    return run_experts(h, w, d, topk_ids, topk_weights, srt, blk, npad, residual, out, ws, L, s,
                       rows_ready);
}

// The whole block for a few tokens in one grid (decode_small.cu).
static int run_vq_small(const void *h, const void *w_router, const float *bias,
                        const moe_expert_weights_t *w, const Dims &d, const void *residual,
                        void *out, int32_t *topk_ids, float *topk_weights, unsigned char *ws,
                        const WsLayout &L, cudaStream_t s) {
    CUtensorMap tm_gate, tm_up, tm_down;
    // index maps [E * H/d rows][I] uint8, boxes of 1024/d rows x 64 columns; W_down boxes of
    // 64 columns x 256 rows
    if (!make_tmap_2d(&tm_gate, w->j_gate, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, (uint64_t)d.I,
                      (uint64_t)d.E * (d.H / w->d), kTI, 1024 / w->d) ||
        !make_tmap_2d(&tm_up, w->j_up, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, (uint64_t)d.I,
                      (uint64_t)d.E * (d.H / w->d), kTI, 1024 / w->d) ||
        !make_tmap_2d(&tm_down, w->w_down, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)d.H,
                      (uint64_t)d.E * d.I, kTN, kBoxRows))
        return MOE_ERR_CUDA;
    VQSmallArgs a;
    GemvArgs &g = a.g;
    g = GemvArgs{};
    g.h = static_cast<const __nv_bfloat16 *>(h);
    g.topk_ids = topk_ids;
    g.topk_wts = topk_weights;
    g.sbt = reinterpret_cast<const SubBlock *>(ws + L.sbt);
    g.npad = reinterpret_cast<const int32_t *>(ws + L.npad);
    g.residual = static_cast<const __nv_bfloat16 *>(residual);
    g.out = static_cast<__nv_bfloat16 *>(out);
    g.p = reinterpret_cast<float *>(ws + L.p);
    g.y = reinterpret_cast<float *>(ws + L.y);
    g.status = reinterpret_cast<int32_t *>(ws + L.status);
    g.w_down = static_cast<const unsigned char *>(w->w_down);
    g.cb_gate = static_cast<const uint2 *>(w->cb_gate);
    g.cb_up = static_cast<const uint2 *>(w->cb_up);
    g.M = d.M;
    g.k = d.k;
    g.E = d.E;
    g.H = d.H;
    g.I = d.I;
    g.b = d.b;
    g.rsub = d.rsub;
    g.n_it = d.n_it;
    g.n_hb = d.n_hb;
    g.n_ht = d.n_ht;
    g.n_ib = d.n_ib;
    g.n_qb = d.H / (4 * kBoxRows);
    g.max_sub = d.max_sub;
    a.w_router = static_cast<const __nv_bfloat16 *>(w_router);
    a.bias = bias;
    a.topk_ids = topk_ids;
    a.topk_wts = topk_weights;
    a.partials = reinterpret_cast<float *>(ws + L.partials);
    a.ctl = reinterpret_cast<int32_t *>(ws + L.ctl);
    a.sorted = reinterpret_cast<int32_t *>(ws + L.sorted);
    a.blocks = reinterpret_cast<int32_t *>(ws + L.blocks);
    a.npad = reinterpret_cast<int32_t *>(ws + L.npad);
    a.sbt_ws = reinterpret_cast<SubBlock *>(ws + L.sbt);
    a.cap = d.cap;
    if (launch_decode_vq_small(tm_gate, tm_up, tm_down, a, s) != cudaSuccess) return MOE_ERR_CUDA;
    for (int i = 1; i < kTracePoints; ++i) trace(i, s);  // one kernel: every stage ends here
    return MOE_OK;
}

static int run_small(const void *h, const void *w_router, const float *bias,
                     const moe_expert_weights_t *w, const Dims &d, const void *residual, void *out,
                     int32_t *topk_ids, float *topk_weights, unsigned char *ws, const WsLayout &L,
                     cudaStream_t s) {
    CUtensorMap tm_gate, tm_up, tm_down;
    const CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_128B;
    if (!make_tmap_2d(&tm_gate, w->w_gate, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)d.I,
                      (uint64_t)d.E * d.H, 64, kGemmStageK, sw) ||
        !make_tmap_2d(&tm_up, w->w_up, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)d.I,
                      (uint64_t)d.E * d.H, 64, kGemmStageK, sw) ||
        !make_tmap_2d(&tm_down, w->w_down, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)d.H,
                      (uint64_t)d.E * d.I, 64, kGemmStageK, sw))
        return MOE_ERR_CUDA;
    SmallArgs a;
    a.h = static_cast<const __nv_bfloat16 *>(h);
    a.w_router = static_cast<const __nv_bfloat16 *>(w_router);
    a.residual = static_cast<const __nv_bfloat16 *>(residual);
    a.bias = bias;
    a.M = d.M;
    a.k = d.k;
    a.E = d.E;
    a.H = d.H;
    a.I = d.I;
    a.b = d.b;
    a.cap = d.cap;
    a.topk_ids = topk_ids;
    a.topk_wts = topk_weights;
    a.out = static_cast<__nv_bfloat16 *>(out);
    a.partials = reinterpret_cast<float *>(ws + L.partials);
    a.ctl = reinterpret_cast<int32_t *>(ws + L.ctl);
    a.sorted = reinterpret_cast<int32_t *>(ws + L.sorted);
    a.blocks = reinterpret_cast<int32_t *>(ws + L.blocks);
    a.npad = reinterpret_cast<int32_t *>(ws + L.npad);
    a.p_rows = reinterpret_cast<__nv_bfloat16 *>(ws + L.p_rows);
    a.y = reinterpret_cast<float *>(ws + L.y);
    a.status = reinterpret_cast<int32_t *>(ws + L.status);
    a.ntiles_cap = (int)(d.cap / d.b);
    if (launch_decode_small(tm_gate, tm_up, tm_down, a, s) != cudaSuccess) return MOE_ERR_CUDA;
    for (int i = 1; i < kTracePoints; ++i) trace(i, s);  // one kernel: every stage ends here
    return MOE_OK;
}

int moe::decode_block(const void *h, const void *w_router, const float *bias,
                      const moe_expert_weights_t *w, int M, int k, int b, const void *residual,
                      void *out, int32_t *topk_ids, float *topk_weights, void *workspace,
                      size_t ws_bytes, void *stream) {
    if (!w) return MOE_ERR_INVALID_ARG;
    b = resolve_block(w, M, k, b);
    int rc = check_ffn_common(h, w, M, k, b, residual, out, workspace, ws_bytes);
    if (rc != MOE_OK) return rc;
    rc = check_router_shape(M, w->H, w->E, k);
    if (rc != MOE_OK || M == 0) return rc;
    if (!w_router || !topk_ids || !topk_weights || !aligned(w_router, 16) ||
        !aligned(topk_ids, 4) || !aligned(topk_weights, 4) || (bias && !aligned(bias, 4)))
        return MOE_ERR_INVALID_ARG;
    Dims d = dims_for(w, M, k, b);
    const WsLayout L = ws_layout(d);
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    trace(0, s);
    int32_t *ws_sorted = reinterpret_cast<int32_t *>(ws + L.sorted);
    int32_t *ws_blocks = reinterpret_cast<int32_t *>(ws + L.blocks);
    int32_t *ws_npad = reinterpret_cast<int32_t *>(ws + L.npad);
    SubBlock *ws_sbt = reinterpret_cast<SubBlock *>(ws + L.sbt);
    int32_t *ws_status = reinterpret_cast<int32_t *>(ws + L.status);
    // (the one grid puts a router CTA on every slice of H: at least 8 SMs)
    if (d.gemm && !d.vq_tc && small_fits(M, k, w->E, w->H, b) && num_sms() >= kRouterCluster)
        return run_small(h, w_router, bias, w, d, residual, out, topk_ids, topk_weights, ws, L, s);
    if (vq_small_path(w, d) && num_sms() >= kRouterCluster)
        return run_vq_small(h, w_router, bias, w, d, residual, out, topk_ids, topk_weights, ws, L, s);
    LowRankProj lr_store;
    const LowRankProj *lr = lowrank_proj(w, d, ws, L, &lr_store);  // rides in the router launch
    cudaError_t err;
    const bool fused = router_can_align(M, k);
    bool rows_ready = fused && d.gemm;  // x tiles written before the expert kernels
    if (fused) {  // one launch routes, aligns and (dense weights) writes the x tiles
        RowTiles rows{nullptr, d.kn, d.tpb, nullptr, 0};
        if (d.gemm) rows = row_tiles(d, ws, L);
        err = launch_router_align(static_cast<const __nv_bfloat16 *>(h),
                                  static_cast<const __nv_bfloat16 *>(w_router), bias, M, w->H, w->E,
                                  k, 1, topk_ids, topk_weights, b, d.rsub, ws_sorted, ws_blocks,
                                  ws_npad, d.cap, d.gemm ? nullptr : ws_sbt, ws_status, lr, rows, s);
        if (err != cudaSuccess) return MOE_ERR_CUDA;
        trace(1, s);
    } else {
        err = launch_router(static_cast<const __nv_bfloat16 *>(h),
                            static_cast<const __nv_bfloat16 *>(w_router), bias, M, w->H, w->E, k, 1,
                            topk_ids, topk_weights, lr, s);
        if (err != cudaSuccess) return MOE_ERR_CUDA;
        trace(1, s);
        if (d.gemm && (int64_t)M * k <= kAlignGatherRoutes) {
            const RowTiles rows = row_tiles(d, ws, L);
            err = launch_align_gather(topk_ids, M, k, w->E, b, ws_sorted, ws_blocks, ws_npad, d.cap,
                                      ws_status, static_cast<const __nv_bfloat16 *>(h), w->H, rows,
                                      s);
            rows_ready = true;
        } else {
            err = launch_align(topk_ids, M, k, w->E, b, ws_sorted, ws_blocks, ws_npad, d.cap,
                               d.gemm ? nullptr : ws_sbt, d.rsub, ws_status, s);
        }
        if (err != cudaSuccess) return MOE_ERR_CUDA;
    }
    trace(2, s);
    return run_experts(h, w, d, topk_ids, topk_weights, ws_sorted, ws_blocks, ws_npad, residual, out,
                       ws, L, s, rows_ready);
}

extern "C" int moe_decode_block(const void *h, const void *w_router, const float *bias,
                                const moe_expert_weights_t *w, int M, int k, int b,
                                const void *residual, void *out, int32_t *topk_ids,
                                float *topk_weights, void *workspace, size_t ws_bytes,
                                void *stream) {
    return decode_block(h, w_router, bias, w, M, k, b, residual, out, topk_ids, topk_weights,
                        workspace, ws_bytes, stream);
}

extern "C" int moe_decode_block_host(const void *h_host, const void *residual_host,
                                     void *out_host, void *h_dev, void *residual_dev,
                                     void *out_dev, const void *w_router, const float *bias,
                                     const moe_expert_weights_t *w, int M, int k, int b,
                                     int32_t *topk_ids, float *topk_weights, void *workspace,
                                     size_t ws_bytes, void *stream) {
    if (!w || M < 0) return MOE_ERR_INVALID_ARG;
    if (M > 0 && (!h_host || !out_host || !h_dev || !out_dev)) return MOE_ERR_INVALID_ARG;
    if ((residual_host != nullptr) != (residual_dev != nullptr)) return MOE_ERR_INVALID_ARG;
    // Validate everything before the first copy, so an error leaves nothing enqueued.
    int rc = check_ffn_common(h_dev, w, M, k, resolve_block(w, M, k, b), residual_dev, out_dev,
                              workspace, ws_bytes);
    if (rc != MOE_OK) return rc;
    rc = check_router_shape(M, w->H, w->E, k);
    if (rc != MOE_OK || M == 0) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t bytes = (size_t)M * w->H * 2;
    if (cudaMemcpyAsync(h_dev, h_host, bytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (residual_host &&
        cudaMemcpyAsync(residual_dev, residual_host, bytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    rc = moe_decode_block(h_dev, w_router, bias, w, M, k, b, residual_dev, out_dev, topk_ids,
                          topk_weights, workspace, ws_bytes, stream);
    if (rc != MOE_OK) return rc;
    if (cudaMemcpyAsync(out_host, out_dev, bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    return cuda_status(cudaStreamSynchronize(s));
}

extern "C" int moe_read_device_status(void *workspace, void *stream, int32_t *status_out) {
    if (!workspace || !status_out || !aligned(workspace, 256)) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t v = 0;
    if (cudaMemcpyAsync(&v, workspace, sizeof v, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (cudaMemsetAsync(workspace, 0, sizeof v, s) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
    *status_out = v;
    return v == 0 ? MOE_OK : MOE_ERR_DEVICE;
}

extern "C" int moe_selftest_wait_timeout(void *workspace, size_t ws_bytes, void *stream) {
    if (!workspace || ws_bytes < sizeof(int32_t) || !aligned(workspace, 256))
        return MOE_ERR_INVALID_ARG;
    return cuda_status(moe::launch_wait_selftest(static_cast<int32_t *>(workspace),
                                                 static_cast<cudaStream_t>(stream)));
}

// ------------------------------------------------------------------------ channel reader
static int reader_args(const moe_reader_t *rd, ReaderArgs *r) {
    if (!rd) return MOE_ERR_INVALID_ARG;
    if (rd->H <= 0 || rd->I <= 0 || rd->E <= 0 || rd->rank <= 0) return MOE_ERR_INVALID_ARG;
    if (rd->H % 128 != 0 || rd->H > 8192 || rd->rank > kReaderMaxRank) return MOE_ERR_UNSUPPORTED;
    const void *ptrs[] = {rd->signs, rd->g_rows, rd->v_rows, rd->w_down, rd->g_codes, rd->v_codes,
                          rd->g_scales, rd->v_scales, rd->dnorm, rd->U, rd->coef};
    for (const void *p : ptrs)
        if (!p || !aligned(p, 16)) return MOE_ERR_INVALID_ARG;
    r->H = rd->H;
    r->I = rd->I;
    r->E = rd->E;
    r->rank = rd->rank;
    r->signs = rd->signs;
    r->g_rows = static_cast<const __nv_bfloat16 *>(rd->g_rows);
    r->v_rows = static_cast<const __nv_bfloat16 *>(rd->v_rows);
    r->w_down = static_cast<const __nv_bfloat16 *>(rd->w_down);
    r->g_codes = static_cast<const uint32_t *>(rd->g_codes);
    r->v_codes = static_cast<const uint32_t *>(rd->v_codes);
    r->g_scales = rd->g_scales;
    r->v_scales = rd->v_scales;
    r->dnorm = rd->dnorm;
    r->U = rd->U;
    r->coef = static_cast<const __nv_bfloat16 *>(rd->coef);
    return MOE_OK;
}

extern "C" int moe_reader_build(const moe_expert_weights_t *w, const moe_reader_t *rd, void *stream) {
    ReaderArgs r;
    int rc = reader_args(rd, &r);
    if (rc != MOE_OK) return rc;
    rc = check_weights(w);
    if (rc != MOE_OK) return rc;
    if (w->kind != MOE_W_DENSE_BF16) return MOE_ERR_UNSUPPORTED;
    if (w->H != rd->H || w->I != rd->I || w->E != rd->E || w->w_down != rd->w_down)
        return MOE_ERR_INVALID_ARG;
    return cuda_status(launch_reader_build(r, static_cast<const __nv_bfloat16 *>(w->w_gate),
                                           static_cast<const __nv_bfloat16 *>(w->w_up),
                                           static_cast<cudaStream_t>(stream)));
}

static int check_reader_call(const ReaderArgs &r, int M, int k, int K) {
    if (M < 0 || k <= 0 || K < 0) return MOE_ERR_INVALID_ARG;
    if (k > 32 || (int64_t)k * r.I > kReaderMaxCand || K > k * r.I || M > 65535)
        return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

extern "C" size_t moe_reader_workspace_bytes(const moe_reader_t *rd, int M, int k, int K) {
    ReaderArgs r;
    if (reader_args(rd, &r) != MOE_OK || check_reader_call(r, M, k, K) != MOE_OK) return 0;
    return reader_ws_layout(r, M, k, K).total;
}

extern "C" int moe_reader_ffn(const void *h, const moe_reader_t *rd, int M, int k,
                              const int32_t *topk_ids, const float *topk_weights, int K,
                              int nscan, const void *residual, void *out, int32_t *selected,
                              float *xr, void *workspace, size_t ws_bytes, void *stream) {
    ReaderArgs r;
    int rc = reader_args(rd, &r);
    if (rc != MOE_OK) return rc;
    rc = check_reader_call(r, M, k, K);
    if (rc != MOE_OK) return rc;
    if (nscan < 0 || nscan > 128) return MOE_ERR_UNSUPPORTED;
    if (!h || !out || !topk_ids || !topk_weights || !workspace || !aligned(h, 16) ||
        !aligned(out, 16) || !aligned(topk_ids, 4) || !aligned(topk_weights, 4) ||
        !aligned(workspace, 256) || (residual && !aligned(residual, 16)) ||
        (selected && !aligned(selected, 4)) || (xr && !aligned(xr, 4)))
        return MOE_ERR_INVALID_ARG;
    const ReaderWs L = reader_ws_layout(r, M, k, K);
    if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
    if (M == 0) return MOE_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    cudaError_t err = launch_reader_decode(r, static_cast<const __nv_bfloat16 *>(h), M, k, topk_ids,
                                           topk_weights, K, nscan,
                                           static_cast<const __nv_bfloat16 *>(residual),
                                           static_cast<__nv_bfloat16 *>(out), ws, s);
    if (err != cudaSuccess) return MOE_ERR_CUDA;
    if (selected && K > 0 &&
        cudaMemcpyAsync(selected, ws + L.sel, (size_t)M * K * 4, cudaMemcpyDeviceToDevice, s) !=
            cudaSuccess)
        return MOE_ERR_CUDA;
    if (xr && cudaMemcpyAsync(xr, ws + L.xr, (size_t)M * r.H * 4, cudaMemcpyDeviceToDevice, s) !=
                  cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}
