// route_core.cuh -- the router's last step, shared by the router kernel and the one-kernel
// decode path: logits from the partial sums of the 8 slices of H, the top-k, and the
// affinities ("A Multi-Engine Dataflow for MoE Decoding on Scratchpad-Based Tensor
// Accelerators", MoE block background: the router selects k experts and assigns each an
// affinity; read as softmax top-k renormalised over the selected experts).
#pragma once

#include <float.h>

#include "moe_internal.cuh"

namespace moe {

// fp32 -> uint32 with the same order (larger float, larger key; -0 and +0 both map to the
// key of +0, so they tie as floats do).  Every non-NaN float maps above 0.
__device__ __forceinline__ uint32_t order_key(float v) {
    if (v == 0.0f) v = 0.0f;
    const uint32_t u = __float_as_uint(v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Finalises nt tokens, one warp per token (warp i: token i; at least nt warps).
// part[(i * kRouterCluster + q) * E + e] (shared memory) holds the partial logit of token i and
// expert e over slice q of H; lane l owns experts l, l + 32, ... (kPerLane of them,
// E <= 32 * kPerLane).  The logit is the 8 partials summed in slice order from zero, plus the
// bias (NULL: none), or -FLT_MAX for every expert when !ok.  Top-k in k rounds of a warp
// arg-max over order-preserving keys: the largest key, ties to the lower expert id (the
// lowest id among the lanes' candidates at the maximum), so slot j holds the j-th largest
// logit.  Then renorm != 0 gives exp(l_j - l_0) /
// sum_{j'<k} exp(l_j' - l_0), renorm == 0 the softmax over all E at the selected experts.
// emit(i, j, id, weight) runs on lane j < k of warp i.
// kLogits: part holds the finished logits [nt][E] (the 8 partials already summed in slice
// order and the bias added), else the partials as above.
template <int kPerLane, bool kLogits = false, typename Emit>
__device__ void route_finalize(const float *part, int nt, int E, int k, const float *bias,
                               bool ok, int renorm, Emit emit) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp >= nt) return;
    const int i = warp;
    float vals[kPerLane];
    uint32_t key[kPerLane];
#pragma unroll
    for (int q = 0; q < kPerLane; ++q) {
        const int e = lane + 32 * q;
        float v = -FLT_MAX;
        key[q] = 0u;  // no candidate
        if (e < E) {
            if (kLogits) {
                v = part[(size_t)i * E + e];
            } else {
                v = 0.0f;
#pragma unroll
                for (int s = 0; s < kRouterCluster; ++s) v += part[((size_t)i * kRouterCluster + s) * E + e];
                if (bias) v += bias[e];
            }
            if (!ok) v = -FLT_MAX;
            key[q] = order_key(v);
        }
        vals[q] = v;
    }
    // This lane's candidates sorted once, largest key first and the lower expert id first
    // among equal keys; a round then looks only at each lane's head.  The lowest id at the
    // warp's largest key is some lane's head (a lane's other experts at that key come after
    // its head), so the selection is the arg-max described above.
    uint32_t sk[kPerLane];
    int sq[kPerLane];
#pragma unroll
    for (int q = 0; q < kPerLane; ++q) {
        sk[q] = key[q];
        sq[q] = q;
    }
#pragma unroll
    for (int a = 0; a < kPerLane - 1; ++a)
#pragma unroll
        for (int c = 0; c < kPerLane - 1 - a; ++c)
            if (sk[c] < sk[c + 1] || (sk[c] == sk[c + 1] && sq[c] > sq[c + 1])) {
                const uint32_t tk = sk[c];
                sk[c] = sk[c + 1];
                sk[c + 1] = tk;
                const int tq = sq[c];
                sq[c] = sq[c + 1];
                sq[c + 1] = tq;
            }
    int my_e = -1;
    for (int j = 0; j < k; ++j) {
        const uint32_t mk = __reduce_max_sync(0xffffffffu, sk[0]);
        const uint32_t cand =
            (sk[0] != 0u && sk[0] == mk) ? (uint32_t)(lane + 32 * sq[0]) : 0xffffffffu;
        const uint32_t be = __reduce_min_sync(0xffffffffu, cand);
        if (lane == j) my_e = be == 0xffffffffu ? -1 : (int)be;
        if (be != 0xffffffffu && (int)(be & 31) == lane) {  // taken: the next one moves up
#pragma unroll
            for (int q = 0; q < kPerLane - 1; ++q) {
                sk[q] = sk[q + 1];
                sq[q] = sq[q + 1];
            }
            sk[kPerLane - 1] = 0u;
        }
    }
    // the selected logits, from the lanes that own them
    float my_v = -FLT_MAX;
    const int src = my_e >= 0 ? (my_e & 31) : 0;
#pragma unroll
    for (int q = 0; q < kPerLane; ++q) {
        const float t = __shfl_sync(0xffffffffu, vals[q], src);
        if (my_e >= 0 && (my_e >> 5) == q) my_v = t;
    }
    const float l0 = __shfl_sync(0xffffffffu, my_v, 0);
    float denom;
    float ex = 0.0f;
    if (renorm) {
        ex = (lane < k) ? expf(my_v - l0) : 0.0f;
        denom = ex;
    } else {
        float sum = 0.0f;
#pragma unroll
        for (int q = 0; q < kPerLane; ++q)
            if (lane + 32 * q < E) sum += expf(vals[q] - l0);
        denom = sum;
        ex = (lane < k) ? expf(my_v - l0) : 0.0f;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) denom += __shfl_xor_sync(0xffffffffu, denom, off);
    if (lane < k) emit(i, lane, ok ? my_e : -1, ok ? ex / denom : 0.0f);
}

// route_finalize for any supported E (8 <= E <= 512): experts per lane by E.
template <bool kLogits = false, typename Emit>
__device__ void route_finalize_any(const float *part, int nt, int E, int k, const float *bias,
                                   bool ok, int renorm, Emit emit) {
    if (E <= 128)
        route_finalize<4, kLogits>(part, nt, E, k, bias, ok, renorm, emit);
    else if (E <= 256)
        route_finalize<8, kLogits>(part, nt, E, k, bias, ok, renorm, emit);
    else
        route_finalize<16, kLogits>(part, nt, E, k, bias, ok, renorm, emit);
}

}  // namespace moe
