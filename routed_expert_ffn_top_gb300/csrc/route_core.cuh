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

// Finalises nt tokens.  part[(i * kRouterCluster + q) * E + e] (shared memory) holds the
// partial logit of token i and expert e over slice q of H; the logit is the 8 partials
// summed in slice order from zero, plus the bias (NULL: none), or -FLT_MAX for every expert
// when !ok.  The top-k are ranks: expert e's slot is the number of experts before it in the
// order (larger key first, ties to the lower id); the k with a slot below k are the
// selection, already in slot order.  Four threads count a quarter of the experts each (those
// congruent to their part modulo 4: neighbouring words, no bank conflicts) and add by
// shuffles; they are neighbouring lanes, and E % 8 == 0 with blockDim.x % 32 == 0 keeps whole
// warps in or out of the loop.  Then warp i takes token i (lane j holds slot j): renorm != 0
// gives exp(l_j - l_0) / sum_{j'<k} exp(l_j' - l_0), renorm == 0 the softmax over all E at
// the selected experts.  emit(i, j, id, weight) runs on lane j < k of warp i.  Every thread
// of the CTA must call it; scratch key_s, val_s [nt * E] and slot_e, slot_v [nt * 32].
template <typename Emit>
__device__ void route_finalize(const float *part, int nt, int E, int k, const float *bias,
                               bool ok, int renorm, uint32_t *key_s, float *val_s,
                               int32_t *slot_e, float *slot_v, Emit emit) {
    const int tid = threadIdx.x, nthr = blockDim.x;
    for (int idx = tid; idx < nt * E; idx += nthr) {
        const int i = idx / E, e = idx - i * E;
        float v = 0.0f;
#pragma unroll
        for (int q = 0; q < kRouterCluster; ++q) v += part[((size_t)i * kRouterCluster + q) * E + e];
        if (bias) v += bias[e];
        if (!ok) v = -FLT_MAX;
        val_s[idx] = v;
        key_s[idx] = order_key(v);
    }
    for (int idx = tid; idx < nt * 32; idx += nthr) {
        slot_e[idx] = -1;  // no candidate (only when fewer than k logits are numbers)
        slot_v[idx] = -FLT_MAX;
    }
    __syncthreads();
    for (int idx = tid; idx < nt * E * 4; idx += nthr) {
        const int part_q = idx & 3, ie = idx >> 2;
        const int i = ie / E, e = ie - i * E;
        const uint32_t *keys = key_s + (size_t)i * E;
        const uint32_t ke = keys[e];
        int cnt = 0;
        // eight keys per step, all loaded before any is compared (E % 8 == 0)
        for (int f0 = part_q; f0 < E; f0 += 32) {
            uint32_t kk[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) kk[u] = f0 + 4 * u < E ? keys[f0 + 4 * u] : 0u;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int f = f0 + 4 * u;
                cnt += (f < E && (kk[u] > ke || (kk[u] == ke && f < e))) ? 1 : 0;
            }
        }
        cnt += __shfl_xor_sync(0xffffffffu, cnt, 1);
        cnt += __shfl_xor_sync(0xffffffffu, cnt, 2);
        if (part_q == 0 && ke != 0u && cnt < k) {  // key 0: not a candidate
            slot_e[i * 32 + cnt] = e;
            slot_v[i * 32 + cnt] = val_s[ie];
        }
    }
    __syncthreads();
    const int warp = tid >> 5, lane = tid & 31;
    if (warp < nt) {
        const int i = warp;
        const int my_e = lane < k ? slot_e[i * 32 + lane] : -1;
        const float my_v = lane < k ? slot_v[i * 32 + lane] : -FLT_MAX;
        const float l0 = __shfl_sync(0xffffffffu, my_v, 0);
        float denom;
        float ex = 0.0f;
        if (renorm) {
            ex = (lane < k) ? expf(my_v - l0) : 0.0f;
            denom = ex;
        } else {
            float s = 0.0f;
            for (int e = lane; e < E; e += 32) s += expf(val_s[(size_t)i * E + e] - l0);
            denom = s;
            ex = (lane < k) ? expf(my_v - l0) : 0.0f;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) denom += __shfl_xor_sync(0xffffffffu, denom, off);
        if (lane < k) emit(i, lane, ok ? my_e : -1, ok ? ex / denom : 0.0f);
    }
}

}  // namespace moe
