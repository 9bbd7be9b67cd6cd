// vq_ttable.cu -- blockwise-VQ gate/up through projected code books ("T tables").
//
// "A Multi-Engine Dataflow for MoE Decoding on Scratchpad-Based Tensor Accelerators"
// (Section 2.3 and its projection code book): with W[e][d q + t][i] = B[J[e][q][i]][t],
//   g_i = sum_q T[q][J[e][q][i]],   T[q][kappa] = sum_t h[d q + t] B[kappa][t],
// so one table entry (d products) serves every column and every expert that reads code
// word kappa at index row q.  The table does not fit on chip for a whole token (H/d x 256
// entries per projection), so the work is cut along H: a CTA takes a slice of kRB index
// rows and a group of 256 (route, projection, column) entries, builds the slice's tables
// for the tokens (gate and up, in shared memory) and sums T lookups over its rows in
// order; a second kernel adds the slices in slice order and applies SiLU.  The slice size
// is fixed, so a route's bits do not depend on M, on the grid or on the other routes.
// Used for VQ-only weights with vq_form == 1, at most kTTMaxTokens tokens.
#include <algorithm>

#include "moe_internal.cuh"
#include "ptx.cuh"

namespace moe {

constexpr int kTTRows = 16;  // index rows per slice
constexpr int kTTCodes = 256;

// Grid (G, nslice): the CTAs of a slice stride over the (route, projection, column)
// entries 256 at a time, so that a table serves many columns (a table entry costs d
// products; each lookup replaces d).  Shared memory: the slice's gate and up tables of the
// M tokens, 2 x M x kTTRows x 256 floats, then the slice's h values.
template <int kD>
__global__ void __launch_bounds__(256)
    vq_ttable_partial_kernel(const __nv_bfloat16 *__restrict__ h, const uint8_t *__restrict__ j_gate,
                             const uint8_t *__restrict__ j_up, const __nv_bfloat16 *__restrict__ cb_gate,
                             const __nv_bfloat16 *__restrict__ cb_up, const int32_t *__restrict__ ids,
                             int M, int k, int E, int H, int I, float *__restrict__ partial) {
    extern __shared__ float T[];  // [2][M][kTTRows][256], then hs [M][kTTRows * kD]
    pdl_wait();
    pdl_launch_dependents();
    const int nrows = H / kD;
    const int s = blockIdx.y, b0 = s * kTTRows, nb = min(kTTRows, nrows - b0);
    const int tid = threadIdx.x;
    float *hs = T + (size_t)2 * M * kTTRows * kTTCodes;
    for (int q = tid; q < M * kTTRows * kD; q += blockDim.x) {
        const int m = q / (kTTRows * kD), o = q - m * (kTTRows * kD);
        hs[q] = o < nb * kD ? __bfloat162float(h[(size_t)m * H + (size_t)kD * b0 + o]) : 0.0f;
    }
    __syncthreads();
    // thread kappa builds its code word's entries: (projection, token, row), tau ascending
    {
        const int kappa = tid;
        float cg[kD], cu[kD];
#pragma unroll
        for (int t = 0; t < kD; ++t) {
            cg[t] = __bfloat162float(cb_gate[kappa * kD + t]);
            cu[t] = __bfloat162float(cb_up[kappa * kD + t]);
        }
        for (int m = 0; m < M; ++m)
            for (int bb = 0; bb < nb; ++bb) {
                const float *hx = hs + (size_t)m * kTTRows * kD + bb * kD;
                float ag = 0.0f, au = 0.0f;
#pragma unroll
                for (int t = 0; t < kD; ++t) {
                    const float x = hx[t];
                    ag = fmaf(x, cg[t], ag);
                    au = fmaf(x, cu[t], au);
                }
                T[((size_t)(0 * M + m) * kTTRows + bb) * kTTCodes + kappa] = ag;
                T[((size_t)(1 * M + m) * kTTRows + bb) * kTTCodes + kappa] = au;
            }
    }
    __syncthreads();
    const int R = M * k;
    const int64_t C = (int64_t)R * 2 * I;
    for (int64_t c = (int64_t)blockIdx.x * 256 + tid; c < C; c += (int64_t)gridDim.x * 256) {
        const int r = (int)(c / (2 * I)), p = (int)((c / I) & 1), i = (int)(c % I);
        const int e = ids[r];
        float acc = 0.0f;
        if (e >= 0 && e < E) {
            const uint8_t *J = (p ? j_up : j_gate) + ((size_t)e * nrows + b0) * I + i;
            const float *Tp = T + (size_t)(p * M + r / k) * kTTRows * kTTCodes;
            uint8_t jv[kTTRows];  // the slice's indices first, then the lookups in row order
#pragma unroll
            for (int bb = 0; bb < kTTRows; ++bb) jv[bb] = bb < nb ? J[(size_t)bb * I] : 0;
#pragma unroll
            for (int bb = 0; bb < kTTRows; ++bb)
                if (bb < nb) acc += Tp[bb * kTTCodes + jv[bb]];
        }
        partial[(size_t)s * C + c] = acc;
    }
}

// p[r][i] = SiLU(sum_s gate partials) * (sum_s up partials), slices in order.
__global__ void __launch_bounds__(256)
    vq_ttable_reduce_kernel(const float *__restrict__ partial, int nslice, int R, int I,
                            float *__restrict__ p) {
    pdl_wait();
    pdl_launch_dependents();
    const int64_t idx = (int64_t)blockIdx.x * 256 + threadIdx.x;
    if (idx >= (int64_t)R * I) return;
    const int r = (int)(idx / I), i = (int)(idx % I);
    const int64_t C = (int64_t)R * 2 * I;
    const float *pg = partial + (int64_t)r * 2 * I + i;
    float g = 0.0f, u = 0.0f;
    int s = 0;
    for (; s + 8 <= nslice; s += 8) {  // 8 slices' loads in flight, then their sums in order
        float vg[8], vu[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            vg[q] = pg[(s + q) * C];
            vu[q] = pg[(s + q) * C + I];
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            g += vg[q];
            u += vu[q];
        }
    }
    for (; s < nslice; ++s) {
        g += pg[s * C];
        u += pg[s * C + I];
    }
    p[idx] = silu_f32(g) * u;
}

int vq_ttable_slices(int H, int d) { return (H / d + kTTRows - 1) / kTTRows; }

cudaError_t launch_vq_ttable(const VQTableArgs &a, cudaStream_t stream) {
    const int nslice = vq_ttable_slices(a.H, a.d);
    const int R = a.M * a.k;
    const int64_t C = (int64_t)R * 2 * a.I;
    const size_t smem = ((size_t)2 * a.M * kTTRows * kTTCodes + (size_t)a.M * kTTRows * a.d) * 4;
    auto kern = a.d == 4 ? vq_ttable_partial_kernel<4> : vq_ttable_partial_kernel<8>;
    cudaError_t err = ensure_smem(reinterpret_cast<const void *>(kern), smem);
    if (err != cudaSuccess) return err;
    cudaLaunchAttribute attrs[2];
    // about two CTAs per SM over all slices; each CTA strides over the entries
    const int64_t want = (2 * (int64_t)num_sms() + nslice - 1) / nslice;
    const int G = (int)std::max<int64_t>(1, std::min<int64_t>((C + 255) / 256, want));
    cudaLaunchConfig_t cfg = launch_config(dim3(G, nslice), dim3(256), smem, stream, attrs, 0);
    err = cudaLaunchKernelEx(&cfg, kern, a.h, a.j_gate, a.j_up, a.cb_gate, a.cb_up, a.ids, a.M,
                             a.k, a.E, a.H, a.I, a.partial);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg2 = launch_config(dim3((unsigned)(((int64_t)R * a.I + 255) / 256)),
                                            dim3(256), 0, stream, attrs, 0);
    return cudaLaunchKernelEx(&cfg2, vq_ttable_reduce_kernel, (const float *)a.partial, nslice, R,
                              a.I, a.p);
}

}  // namespace moe
