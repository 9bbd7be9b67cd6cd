// reader.cu -- the channel-sparse reader of "Channel Selection for Mixture-of-Experts
// Decoding Needs No Calibration Data" (the reader's Stages 1-3) on this GPU.
//
// For one token, a routed expert's channel j owns row j of gate/up and column j of down
// (Background: channels and retention rules).  The reader
//   Stage 1: rotates x in 128-coordinate blocks by a random Hadamard transform R and dots
//            it with a ternary sketch of every candidate channel's rotated gate and up rows,
//            scanning per block only the nscan coordinates of largest |Rx|:
//            ahat_j = SiLU(ghat_j) * vhat_j;
//   Stage 2: scores score_j = w_j * ||d_j|| * |ahat_j| (w_j the router weight of channel
//            j's expert) and reads the top K channels across all the token's experts
//            exactly: a_j = SiLU(g_j . x) * (v_j . x);
//   Stage 3: adds the discarded channels through a rank-r map:
//            out = residual + sum_{kept} w_j a_j d_j + U sum_{discarded} w_j ahat_j b_j,
//            b_j = U^T d_j.
// Readings (the page's Equations 1 and 2 and its sketch block format are not in the text):
// the ternary code of a rotated block is the Ternary Weight Networks rule (threshold
// 0.7 mean|r|, one scale per block = the mean |r| of the nonzero codes); ties in the scan
// and in the top K go to the lower coordinate / channel index.
//
// Layout of the reader's data (built once from the dense weights by moe_reader_build):
//   rows g, v      [E][I][H] bf16  channel-major gate and up rows (the exact reads);
//   codes          [E][I][H/128][8] uint32 per block: words 0-3 the nonzero mask, words 4-7
//                  the negative mask (coordinate c of the block at bit c%32 of word c/32);
//   scales         [E][I][H/128] fp32;  dnorm [E][I] fp32;
//   U              [H][r] fp32;  coef b [E][I][r] bf16.
// Every sum has an order fixed by indices (never by the grid or by M): a token's output
// is bitwise reproducible and independent of the other tokens.
#include <algorithm>
#include <type_traits>

#include "moe_internal.cuh"
#include "ptx.cuh"

namespace moe {

constexpr int kRB = 128;              // coordinates per rotation block
constexpr int kRWords = kRB / 16;     // uint32 code words per block
constexpr int kExactChunk = 8;        // selected channels per exact-read CTA (one per warp)
constexpr int kSelectThreads = 1024;
constexpr int kSketchWarps = 32;      // one 1024-thread CTA per SM: the scan and the table once
// Nibble table layout: the 16 sums of 4-coordinate group g = 8w + q (word w of a row covers
// groups 8w .. 8w+7) for nibble n sit at nib_index(w, q, n), so that every lookup of the lane
// that reads word w falls in bank w % 32 (one wavefront per warp-wide lookup, whatever the
// nibbles); 4096 floats per 32 words.
__host__ __device__ constexpr int nib_index(int w, int q, int n) {
    return (w >> 5) * 4096 + (n * 8 + q) * 32 + (w & 31);
}
__host__ __device__ constexpr int nib_table_floats(int H) { return ((H / 32 + 31) / 32) * 4096; }

// ------------------------------------------------------------------ rotation in a warp
// A warp holds one 128-coordinate block, lane l coordinates 4l..4l+3 in v[0..3].  The
// Sylvester-Hadamard butterflies of distance 1 and 2 are inside a lane, 4..64 across lanes
// (partner lane l ^ (d/4)); the lower index of a pair takes the sum, the upper the
// difference.  The result is H_128 v / sqrt(128).
__device__ __forceinline__ void fwht128_warp(float (&v)[4], int lane) {
    float a0 = v[0] + v[1], a1 = v[0] - v[1], a2 = v[2] + v[3], a3 = v[2] - v[3];
    v[0] = a0 + a2;
    v[1] = a1 + a3;
    v[2] = a0 - a2;
    v[3] = a1 - a3;
#pragma unroll
    for (int s = 1; s < 32; s <<= 1) {
        const bool upper = (lane & s) != 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float o = __shfl_xor_sync(0xffffffffu, v[q], s);
            v[q] = upper ? o - v[q] : v[q] + o;
        }
    }
    const float inv = 0.08838834764831845f;  // 1 / sqrt(128)
#pragma unroll
    for (int q = 0; q < 4; ++q) v[q] *= inv;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// ------------------------------------------------------------------------------ build
// Channel-major copies of gate and up: rows[e][i][h] = w[e][h][i], 32 x 32 tiles through
// shared memory (both sides coalesced).
__global__ void __launch_bounds__(256)
    reader_transpose_kernel(const __nv_bfloat16 *__restrict__ w, __nv_bfloat16 *__restrict__ rows,
                            int H, int I) {
    __shared__ __nv_bfloat16 tile[32][33];
    const int e = blockIdx.z;
    const int i0 = blockIdx.x * 32, h0 = blockIdx.y * 32;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 8 rows of 32 per pass
    const __nv_bfloat16 *src = w + (size_t)e * H * I;
    for (int r = ty; r < 32; r += 8) {
        const int h = h0 + r, i = i0 + tx;
        if (h < H && i < I) tile[r][tx] = src[(size_t)h * I + i];
    }
    __syncthreads();
    __nv_bfloat16 *dst = rows + (size_t)e * I * H;
    for (int r = ty; r < 32; r += 8) {
        const int i = i0 + r, h = h0 + tx;
        if (h < H && i < I) dst[(size_t)i * H + h] = tile[tx][r];
    }
}

// One warp per channel (e, i): the sketch of its gate and up rows, ||d||, b = U^T d.
__global__ void __launch_bounds__(256)
    reader_sketch_build_kernel(const __nv_bfloat16 *__restrict__ g_rows,
                               const __nv_bfloat16 *__restrict__ v_rows,
                               const __nv_bfloat16 *__restrict__ w_down,
                               const int8_t *__restrict__ signs, const float *__restrict__ U,
                               int rank, int64_t nchan, int H, uint32_t *__restrict__ g_codes,
                               uint32_t *__restrict__ v_codes, float *__restrict__ g_scales,
                               float *__restrict__ v_scales, float *__restrict__ dnorm,
                               __nv_bfloat16 *__restrict__ coef) {
    const int lane = threadIdx.x & 31;
    const int64_t ch = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (ch >= nchan) return;
    const int nb = H / kRB;
    for (int p = 0; p < 2; ++p) {
        const __nv_bfloat16 *row = (p ? v_rows : g_rows) + ch * H;
        uint32_t *codes = (p ? v_codes : g_codes) + ch * nb * kRWords;
        float *scales = (p ? v_scales : g_scales) + ch * nb;
        for (int b = 0; b < nb; ++b) {
            const int c0 = b * kRB + 4 * lane;
            const uint2 raw = *reinterpret_cast<const uint2 *>(row + c0);
            const char4 sg = *reinterpret_cast<const char4 *>(signs + c0);
            float v[4] = {bf16_lo(raw.x) * sg.x, bf16_hi(raw.x) * sg.y, bf16_lo(raw.y) * sg.z,
                          bf16_hi(raw.y) * sg.w};
            fwht128_warp(v, lane);
            const float tau = 0.7f * (warp_sum(fabsf(v[0]) + fabsf(v[1]) + fabsf(v[2]) + fabsf(v[3])) /
                                      (float)kRB);
            uint32_t nz = 0, ng = 0;
            float mag = 0.0f, cnt = 0.0f;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (fabsf(v[q]) > tau) {
                    nz |= 1u << q;
                    if (v[q] < 0.0f) ng |= 1u << q;
                    mag += fabsf(v[q]);
                    cnt += 1.0f;
                }
            }
            mag = warp_sum(mag);
            cnt = warp_sum(cnt);
            // lane l's 4 coordinates sit at bits 4 (l % 8) of word l / 8 of each plane
            uint32_t wz = nz << (4 * (lane & 7)), wn = ng << (4 * (lane & 7));
#pragma unroll
            for (int o = 1; o < 8; o <<= 1) {
                wz |= __shfl_xor_sync(0xffffffffu, wz, o);
                wn |= __shfl_xor_sync(0xffffffffu, wn, o);
            }
            if ((lane & 7) == 0) {
                codes[b * kRWords + (lane >> 3)] = wz;
                codes[b * kRWords + 4 + (lane >> 3)] = wn;
            }
            if (lane == 0) scales[b] = cnt > 0.0f ? mag / cnt : 0.0f;
        }
    }
    // down column: norm and coefficients on U, fixed order (lane slices, then xor tree)
    const __nv_bfloat16 *d = w_down + ch * H;
    float sq = 0.0f;
    for (int h = lane; h < H; h += 32) {
        const float x = __bfloat162float(d[h]);
        sq = fmaf(x, x, sq);
    }
    sq = warp_sum(sq);
    if (lane == 0) dnorm[ch] = sqrtf(sq);
    for (int r = 0; r < rank; ++r) {
        float s = 0.0f;
        for (int h = lane; h < H; h += 32) s = fmaf(__bfloat162float(d[h]), U[(size_t)h * rank + r], s);
        s = warp_sum(s);
        if (lane == 0) coef[ch * rank + r] = __float2bfloat16_rn(s);
    }
}

cudaError_t launch_reader_build(const ReaderArgs &r, const __nv_bfloat16 *w_gate,
                                const __nv_bfloat16 *w_up, cudaStream_t stream) {
    dim3 tg((r.I + 31) / 32, (r.H + 31) / 32, r.E);
    reader_transpose_kernel<<<tg, 256, 0, stream>>>(w_gate, const_cast<__nv_bfloat16 *>(r.g_rows),
                                                    r.H, r.I);
    reader_transpose_kernel<<<tg, 256, 0, stream>>>(w_up, const_cast<__nv_bfloat16 *>(r.v_rows),
                                                    r.H, r.I);
    const int64_t nchan = (int64_t)r.E * r.I;
    const int64_t blocks = (nchan * 32 + 255) / 256;
    reader_sketch_build_kernel<<<(unsigned)blocks, 256, 0, stream>>>(
        r.g_rows, r.v_rows, r.w_down, r.signs, r.U, r.rank, nchan, r.H,
        const_cast<uint32_t *>(r.g_codes), const_cast<uint32_t *>(r.v_codes),
        const_cast<float *>(r.g_scales), const_cast<float *>(r.v_scales),
        const_cast<float *>(r.dnorm), const_cast<__nv_bfloat16 *>(r.coef));
    return cudaGetLastError();
}

// ----------------------------------------------------------------------------- decode
// Stage 1a for block b of token m, by one warp: x rotated, and every coordinate outside the
// block's nscan largest |Rx| (ties: lower coordinate) zeroed, so the sketch products need
// no mask.  The nscan-th largest magnitude is found bit by bit from the top (its bits as
// an unsigned integer order like the non-negative floats), counting with warp ballots; the
// coordinates equal to it are then taken in index order.  xr: where the block's 128 values
// go (shared memory).
__device__ __forceinline__ void scan_block(const __nv_bfloat16 *hm, char4 sg, int b, int nscan,
                                           float *xr, int lane) {
    const int c0 = b * kRB + 4 * lane;
    const uint2 raw = *reinterpret_cast<const uint2 *>(hm + c0);
    float v[4] = {bf16_lo(raw.x) * sg.x, bf16_hi(raw.x) * sg.y, bf16_lo(raw.y) * sg.z,
                  bf16_hi(raw.y) * sg.w};
    fwht128_warp(v, lane);
    uint32_t key[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) key[q] = __float_as_uint(fabsf(v[q]));
    bool keep[4] = {false, false, false, false};
    if (nscan >= kRB) {
        keep[0] = keep[1] = keep[2] = keep[3] = true;
    } else if (nscan > 0) {
        uint32_t t = 0;  // the largest value with at least nscan keys >= it
        for (int bit = 31; bit >= 0; --bit) {
            const uint32_t cand = t | (1u << bit);
            int cnt = 0;
#pragma unroll
            for (int q = 0; q < 4; ++q) cnt += __popc(__ballot_sync(0xffffffffu, key[q] >= cand));
            if (cnt >= nscan) t = cand;
            // exactly nscan keys at or above the candidate: they are the nscan largest and
            // every other key is below them, so the lower bits cannot change the kept set
            if (cnt == nscan) break;  // uniform across the warp (ballot counts)
        }
        int above = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) above += __popc(__ballot_sync(0xffffffffu, key[q] > t));
        // equal keys before this lane's (lower lanes hold lower coordinates)
        int eq = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) eq += key[q] == t;
        int before = eq;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, before, o);
            if (lane >= o) before += u;
        }
        before -= eq;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            if (key[q] > t) keep[q] = true;
            else if (key[q] == t) keep[q] = before++ < nscan - above;
        }
    }
    *reinterpret_cast<float4 *>(xr + 4 * lane) =
        make_float4(keep[0] ? v[0] : 0.0f, keep[1] ? v[1] : 0.0f, keep[2] ? v[2] : 0.0f,
                    keep[3] ? v[3] : 0.0f);
}

// Stage 1 and the score of Stage 2.  The CTA first rotates and scans the token's x (warp w
// takes blocks w, w + 32, ...; every CTA of the token does the same, CTA 0 also stores the
// result for inspection), then tabulates, for every group of 4
// coordinates g and every 4-bit pattern n, T[g][n] = sum of the (scanned) xr of the pattern's
// coordinates, coordinates ascending.  A code word pair (nonzero, negative masks of 32
// coordinates) then dots with xr in 16 table reads: the positive nibbles' sums minus the
// negative nibbles' sums.  One warp per candidate channel f = slot * I + i at a time (warps
// stride over the token's channels); lanes take the 32-coordinate words of a block four at
// a time, and the blocks are summed with their scales in block order.
// Grid (G, M), 32 warps (one CTA per SM and token, so the scan and the table are built once
// per SM); shared memory: the table, (H/4) x 17 floats (one pad float per group spreads
// the lanes' reads over the banks) and xr (H floats).
// Stage 1a in one CTA for token row hm: x rotated and scanned into xr (warp w of W takes
// blocks w, w + W, ...; sg0 is the signs of warp w's first block, loaded early), then the
// nibble table T (see nib_index) from a copy of xr padded to 33 floats per 32-coordinate word.
// T: the shared-memory table, xr at T + nib_table_floats(H), the padded copy after xr.
// xr_out (may be NULL): where the scanned xr is also stored.
__device__ void sketch_prepare(const ReaderArgs &r, const __nv_bfloat16 *hm, int nscan, char4 sg0,
                               float *T, float *xr_out) {
    const int H = r.H, nb = H / kRB;
    float *xr = T + nib_table_floats(H);
    for (int b = threadIdx.x >> 5; b < nb; b += (int)(blockDim.x >> 5)) {
        const char4 sg = b == (int)(threadIdx.x >> 5) ? sg0 : *reinterpret_cast<const char4 *>(
                                                               r.signs + b * kRB + 4 * (threadIdx.x & 31));
        scan_block(hm, sg, b, nscan, xr + b * kRB, threadIdx.x & 31);
    }
    __syncthreads();
    if (xr_out)
        for (int c = threadIdx.x; c < H; c += blockDim.x) xr_out[c] = xr[c];
    // The table from a copy of xr padded to 33 floats per 32-coordinate word: the thread of
    // (word w, group q) reads its 4 coordinates and writes its 16 sums, both bank-distinct
    // across the warp's consecutive words.
    const int W = H / 32;
    float *xp = xr + H;  // [W][33]
    for (int c = threadIdx.x; c < H; c += blockDim.x) xp[(c >> 5) * 33 + (c & 31)] = xr[c];
    __syncthreads();
    for (int t = threadIdx.x; t < 8 * W; t += blockDim.x) {
        const int w = t % W, q = t / W;
        const float *x4 = xp + w * 33 + 4 * q;
        const float a[4] = {x4[0], x4[1], x4[2], x4[3]};
#pragma unroll
        for (int n = 0; n < 16; ++n) {
            float v = 0.0f;
#pragma unroll
            for (int c = 0; c < 4; ++c)
                if (n & (1 << c)) v += a[c];
            T[nib_index(w, q, n)] = v;
        }
    }
    __syncthreads();
}

// The signs of this thread's warp's first rotation block (weights: read before the wait).
__device__ __forceinline__ char4 first_block_signs(const ReaderArgs &r) {
    char4 sg0 = make_char4(0, 0, 0, 0);
    if ((int)(threadIdx.x >> 5) < r.H / kRB)
        sg0 = *reinterpret_cast<const char4 *>(r.signs + (threadIdx.x >> 5) * kRB + 4 * (threadIdx.x & 31));
    return sg0;
}

// Stage 1b and the score of Stage 2 for token m's candidate channels f = f0, f0 + fstep, ...
// (this warp's), against the table T: a code word pair (nonzero, negative masks of 32
// coordinates) dots with xr in 16 table reads, the positive nibbles' sums minus the negative
// nibbles' sums; lanes take the 32-coordinate words of a block four at a time, and the
// blocks are summed with their scales in block order.
template <int kMaxPass>
__device__ void sketch_channels(const ReaderArgs &r, const float *T, int m, int f0, int fstep,
                                const int32_t *__restrict__ ids, const float *__restrict__ wts,
                                int k, float *__restrict__ ahat, float *__restrict__ score) {
    const int I = r.I, nb = r.H / kRB;
    const int N = k * I;
    const int lane = threadIdx.x & 31;
    const int nwords = 4 * nb;              // 32-coordinate words per row
    const int npass = (nwords + 31) / 32;   // words per lane and row, at most kMaxPass
    for (int f = f0; f < N; f += fstep) {
        const int j = f / I, i = f - j * I;
        const int e = ids[(size_t)m * k + j];
        const size_t o = (size_t)m * N + f;
        if (e < 0 || e >= r.E) {
            if (lane == 0) {
                ahat[o] = 0.0f;
                score[o] = -1.0f;
            }
            continue;
        }
        const int64_t ch = (int64_t)e * I + i;
        // every load of the channel first: its code words and block scales for both rows
        uint32_t nzw[2][kMaxPass], ngw[2][kMaxPass];
        float scw[2][kMaxPass];
#pragma unroll
        for (int p = 0; p < 2; ++p) {
            const uint32_t *codes = (p ? r.v_codes : r.g_codes) + ch * nb * kRWords;
            const float *scales = (p ? r.v_scales : r.g_scales) + ch * nb;
#pragma unroll
            for (int ps = 0; ps < kMaxPass; ++ps) {
                const int w = ps * 32 + lane;  // word w of the row: block w / 4, quarter w % 4
                nzw[p][ps] = ngw[p][ps] = 0u;
                scw[p][ps] = 0.0f;
                if (ps < npass && w < nwords) {
                    nzw[p][ps] = codes[(w >> 2) * kRWords + (w & 3)];
                    ngw[p][ps] = codes[(w >> 2) * kRWords + 4 + (w & 3)];
                    scw[p][ps] = scales[w >> 2];
                }
            }
        }
        const float dn = r.dnorm[ch];
        const float wj = wts[(size_t)m * k + j];
        float est[2];
#pragma unroll
        for (int p = 0; p < 2; ++p) {
            float acc = 0.0f;
#pragma unroll
            for (int ps = 0; ps < kMaxPass; ++ps) {
                if (ps >= npass) break;
                const int w = ps * 32 + lane;
                const uint32_t pos = nzw[p][ps] & ~ngw[p][ps], neg = nzw[p][ps] & ngw[p][ps];
                float s = 0.0f;
                if (w < nwords) {
                    const float *Tw = T + nib_index(w, 0, 0);  // groups 8w .. 8w+7, bank w % 32
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        s += Tw[(((pos >> (4 * q)) & 15u) * 8 + q) * 32] -
                             Tw[(((neg >> (4 * q)) & 15u) * 8 + q) * 32];
                }
                // the block's four words, in order, then its scale
                s += __shfl_xor_sync(0xffffffffu, s, 1);
                s += __shfl_xor_sync(0xffffffffu, s, 2);
                if (w < nwords && (lane & 3) == 0) acc = fmaf(scw[p][ps], s, acc);
            }
            est[p] = warp_sum(acc);
        }
        if (lane == 0) {
            const float a = silu_f32(est[0]) * est[1];
            ahat[o] = a;
            score[o] = wj * dn * fabsf(a);
        }
    }
}

// Stage 1 and the score of Stage 2.  Every CTA of token m rotates and scans the token's x and
// builds the table (CTA 0 also stores xr for inspection); then one warp per candidate channel
// at a time (warps stride over the token's channels).  Grid (G, M), 32 warps (one CTA per SM
// and token, so the scan and the table are built once per SM); shared memory: the table, xr
// (H floats) and its padded copy ((H/32) x 33 floats).
template <int kMaxPass>
__global__ void __launch_bounds__(kSketchWarps * 32)
    reader_sketch_kernel(ReaderArgs r, const __nv_bfloat16 *__restrict__ h, int nscan,
                         float *__restrict__ xr_out, const int32_t *__restrict__ ids,
                         const float *__restrict__ wts, int k, float *__restrict__ ahat,
                         float *__restrict__ score) {
    extern __shared__ __align__(16) float T[];
    // the rotation signs of this warp's first block are weights: load them before the wait
    const char4 sg0 = first_block_signs(r);
    pdl_wait();
    pdl_launch_dependents();
    const int m = blockIdx.y;
    sketch_prepare(r, h + (size_t)m * r.H, nscan, sg0, T,
                   blockIdx.x == 0 ? xr_out + (size_t)m * r.H : nullptr);
    sketch_channels<kMaxPass>(r, T, m, blockIdx.x * kSketchWarps + (threadIdx.x >> 5),
                              gridDim.x * kSketchWarps, ids, wts, k, ahat, score);
}

// Inclusive scan over the threads of a block of at most 1024 (values in thread order).
__device__ __forceinline__ int block_scan(int v, int *warp_tot) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += u;
    }
    if (lane == 31) warp_tot[warp] = v;
    __syncthreads();
    if (warp == 0) {
        int t = lane < nwarps ? warp_tot[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o) t += u;
        }
        warp_tot[lane] = t;
    }
    __syncthreads();
    const int add = warp > 0 ? warp_tot[warp - 1] : 0;
    __syncthreads();  // warp_tot is reused by the next scan
    return v + add;
}

// Stage 2 selection: the K largest of a token's N scores (ties: lower channel index), by a
// most-significant-digit radix select on order-preserving keys (integer counts commute, so
// the result does not depend on arrival order), then the kept flags and the kept channels
// in ascending index.  One CTA of 256 to 1024 threads (the result does not depend on the
// count); keys [N] and two sets of 32 warp histograms of 256 bins in shared memory.  On return keys[f] is 1 for a kept channel, else 0 (read after
// a barrier).  Outputs: keep (may be NULL) one byte per channel, sel [K] the kept channels
// then -1, nsel the count.
__device__ void select_token(const float *__restrict__ score, int N, int K, uint32_t *keys,
                             int *whist, uint8_t *keep, int32_t *sel, int32_t *nsel) {
    __shared__ int warp_tot[32];
    __shared__ int s_nvalid, s_digit, s_remaining, s_count;
    __shared__ uint32_t s_and, s_or;
    const int tid = threadIdx.x;
    if (tid == 0) {
        s_nvalid = 0;
        s_and = ~0u;
        s_or = 0u;
    }
    const int nwh = (int)blockDim.x >> 5;  // one histogram per warp
    for (int d = tid; d < nwh * 256; d += (int)blockDim.x) whist[d] = 0;
    __syncthreads();
    int nv = 0;
    uint32_t k_and = ~0u, k_or = 0u;  // over the valid keys: their common leading bits
    const int nthr = (int)blockDim.x;
    for (int f0 = tid; f0 < N; f0 += 8 * nthr) {  // 8 scores' loads in flight at once
        float sv[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) sv[u] = f0 + u * nthr < N ? __ldcg(score + f0 + u * nthr) : -1.0f;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int f = f0 + u * nthr;
            if (f >= N) break;
            const float s = sv[u];
            const uint32_t key = s >= 0.0f ? __float_as_uint(s) + 1u : 0u;  // invalid / NaN: 0
            keys[f] = key;
            nv += key != 0u;
            if (key != 0u) {
                k_and &= key;
                k_or |= key;
            }
        }
    }
    atomicAdd(&s_nvalid, nv);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        k_and &= __shfl_xor_sync(0xffffffffu, k_and, o);
        k_or |= __shfl_xor_sync(0xffffffffu, k_or, o);
    }
    if ((tid & 31) == 0) {
        atomicAnd(&s_and, k_and);
        atomicOr(&s_or, k_or);
    }
    __syncthreads();
    const int Keff = min(K, s_nvalid);
    // Radix select from the first bit where the valid keys differ (the bits above it are the
    // same in all of them: scores of one sign and a narrow exponent range), up to 8 bits a
    // pass.  After a pass, the keys above the prefix are kept, those below dropped, and
    // `remaining` of those under it are still to be kept.  When that is all of them, later
    // passes cannot change the kept set: stop there.  (Invalid keys, 0, are below every
    // valid one and never needed: Keff <= the valid count.)
    const uint32_t diff = s_and ^ s_or;
    int hi = diff ? 31 - __clz(diff) : -1;  // highest differing bit
    uint32_t mask = hi < 0 ? ~0u : ~((2u << hi) - 1u);  // 2u << 31 wraps to 0: mask 0
    uint32_t prefix = s_and & mask;
    int remaining = Keff;
    if (Keff > 0) {
        int buf = 0;
        while (hi >= 0) {
            const int lo = hi >= 7 ? hi - 7 : 0;
            const int nb = 1 << (hi - lo + 1);  // bins of this pass's digit
            const uint32_t dmask = (uint32_t)nb - 1u;
            int *hist = whist + buf * 32 * 256;
            int *next = whist + (buf ^ 1) * 32 * 256;  // (sets spaced for 32 warps)
            const int wbase = (tid >> 5) * 256;
            // each warp counts into its own histogram (integer adds commute); the other set
            // is cleared for the next pass meanwhile
            for (int f = tid; f < N; f += (int)blockDim.x)
                if ((keys[f] & mask) == prefix) atomicAdd(&hist[wbase + ((keys[f] >> lo) & dmask)], 1);
            for (int d = tid; d < nwh * 256; d += (int)blockDim.x) next[d] = 0;
            __syncthreads();
            // thread t < nb owns digit nb - 1 - t: its count over the warps, then a scan in
            // descending digit order finds the digit where the count reaches `remaining`
            int c = 0;
            if (tid < nb)
                for (int w = 0; w < nwh; ++w) c += hist[w * 256 + (nb - 1 - tid)];
            const int incl = block_scan(c, warp_tot);
            if (tid < nb && c > 0 && incl >= remaining && incl - c < remaining) {
                s_digit = nb - 1 - tid;
                s_remaining = remaining - (incl - c);
                s_count = c;
            }
            __syncthreads();
            prefix |= (uint32_t)s_digit << lo;
            mask |= dmask << lo;
            remaining = s_remaining;
            const bool all_kept = remaining == s_count;
            buf ^= 1;
            hi = lo - 1;
            if (all_kept) break;  // uniform: every thread read the same shared values
        }
    }
    // keys above the prefix are kept, and the first `remaining` keys under it in index order;
    // each thread owns a contiguous run of channels
    const uint32_t T = prefix;
    const int per = (N + (int)blockDim.x - 1) / (int)blockDim.x;
    const int f0 = tid * per, f1 = min(N, f0 + per);
    int eq = 0;
    for (int f = f0; f < f1; ++f) eq += (Keff > 0 && (keys[f] & mask) == T);
    int eq_before = block_scan(eq, warp_tot) - eq;
    int kc = 0;
    for (int f = f0; f < f1; ++f) {
        const uint32_t key = keys[f] & mask;
        bool kp = false;
        if (Keff > 0) {
            if (key > T) kp = true;
            else if (key == T) kp = eq_before++ < remaining;
        }
        if (keep) keep[f] = kp ? 1 : 0;
        keys[f] = kp ? 1u : 0u;  // reused as the kept flag
        kc += kp;
    }
    __syncthreads();
    int pos = block_scan(kc, warp_tot) - kc;
    for (int f = f0; f < f1; ++f)
        if (keys[f]) sel[pos++] = f;
    for (int q = Keff + tid; q < K; q += (int)blockDim.x) sel[q] = -1;
    if (tid == 0) *nsel = Keff;
}

// The selection of token m = blockIdx.x, into the workspace.  One 1024-thread CTA per token.
__global__ void __launch_bounds__(kSelectThreads)
    reader_select_kernel(const float *__restrict__ score, int N, int K,
                         uint8_t *__restrict__ keep, int32_t *__restrict__ sel,
                         int32_t *__restrict__ nsel) {
    extern __shared__ uint32_t keys[];  // [N], then two sets of 32 warp histograms of 256 bins
    pdl_wait();
    pdl_launch_dependents();
    const int m = blockIdx.x;
    select_token(score + (size_t)m * N, N, K, keys, reinterpret_cast<int *>(keys + N),
                 keep + (size_t)m * N, sel + (size_t)m * K, nsel + m);
}

// Stage 2 exact reads: chunk c of a token's kept channels (positions 8c .. 8c+7 of the
// ascending list sel, nsel of them), one warp per channel for a = SiLU(g . x) (v . x), then
// the chunk's sum of w a d in channel order into its own partial row out [H].  The work runs
// on the CTA's first 256 threads; every thread of the CTA must call it (it has barriers).
// Shared memory: xs4 the token row (H bf16), wa [8], chs [8].
template <int kDPass>
__device__ void exact_chunk(const ReaderArgs &r, const __nv_bfloat16 *__restrict__ hm,
                            const int32_t *__restrict__ ids_m, const float *__restrict__ wts_m,
                            const int32_t *sel, int nsel, int c, float *__restrict__ out,
                            uint4 *xs4, float *wa, int64_t *chs) {
    const int H = r.H, I = r.I;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const bool act = threadIdx.x < 256;
    const uint4 *hx = reinterpret_cast<const uint4 *>(hm);
    for (int q = threadIdx.x; q < H / 8; q += blockDim.x) xs4[q] = hx[q];
    __syncthreads();
    // the chunk's channels first (one per warp), so that every load below can be issued at once
    const int s = c * kExactChunk + warp;
    if (warp < kExactChunk && lane == 0) {
        int64_t ch = -1;
        float w = 0.0f;
        if (s < nsel) {
            const int f = sel[s];
            const int j = f / I, i = f - j * I;
            const int e = ids_m[j];
            if (e >= 0 && e < r.E) {
                ch = (int64_t)e * I + i;
                w = wts_m[j];
            }
        }
        chs[warp] = ch;
        wa[warp] = w;
    }
    __syncthreads();
    // this thread's pieces of the chunk's down rows are in flight while the warps form a
    const int c0 = threadIdx.x * 8;  // 2048 columns per pass: kDPass = ceil(H / 2048)
    uint4 dv[kDPass][kExactChunk];
    if (act) {
#pragma unroll
        for (int ps = 0; ps < kDPass; ++ps)
#pragma unroll
            for (int q = 0; q < kExactChunk; ++q)
                if (c0 + ps * 2048 < H && chs[q] >= 0)
                    dv[ps][q] = *reinterpret_cast<const uint4 *>(r.w_down + chs[q] * H + c0 + ps * 2048);
    }
    const int64_t ch = warp < kExactChunk ? chs[warp] : -1;
    if (ch >= 0) {
        const uint4 *g = reinterpret_cast<const uint4 *>(r.g_rows + ch * H);
        const uint4 *v = reinterpret_cast<const uint4 *>(r.v_rows + ch * H);
        float gx = 0.0f, vx = 0.0f;
        // 8 pieces of each row per lane in flight, then their products in piece order
        for (int q0 = lane; q0 < H / 8; q0 += 32 * 8) {
            uint4 ga[8], va[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int q = q0 + 32 * u;
                if (q < H / 8) {
                    ga[u] = g[q];
                    va[u] = v[q];
                }
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int q = q0 + 32 * u;
                if (q >= H / 8) break;
                const uint4 xa = xs4[q];
                const uint32_t xw[4] = {xa.x, xa.y, xa.z, xa.w};
                const uint32_t gw[4] = {ga[u].x, ga[u].y, ga[u].z, ga[u].w};
                const uint32_t vw[4] = {va[u].x, va[u].y, va[u].z, va[u].w};
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    gx = fmaf(bf16_lo(gw[t]), bf16_lo(xw[t]), gx);
                    gx = fmaf(bf16_hi(gw[t]), bf16_hi(xw[t]), gx);
                    vx = fmaf(bf16_lo(vw[t]), bf16_lo(xw[t]), vx);
                    vx = fmaf(bf16_hi(vw[t]), bf16_hi(xw[t]), vx);
                }
            }
        }
        gx = warp_sum(gx);
        vx = warp_sum(vx);
        __syncwarp();
        if (lane == 0) wa[warp] = wa[warp] * (silu_f32(gx) * vx);
    }
    __syncthreads();
    if (act) {
#pragma unroll
        for (int ps = 0; ps < kDPass; ++ps) {
            const int cc = c0 + ps * 2048;
            if (cc >= H) break;
            float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
            for (int q = 0; q < kExactChunk; ++q) {
                if (chs[q] < 0) continue;
                const uint32_t dw[4] = {dv[ps][q].x, dv[ps][q].y, dv[ps][q].z, dv[ps][q].w};
                const float a = wa[q];
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    acc[2 * t] = fmaf(a, bf16_lo(dw[t]), acc[2 * t]);
                    acc[2 * t + 1] = fmaf(a, bf16_hi(dw[t]), acc[2 * t + 1]);
                }
            }
            *reinterpret_cast<float4 *>(out + cc) = make_float4(acc[0], acc[1], acc[2], acc[3]);
            *reinterpret_cast<float4 *>(out + cc + 4) = make_float4(acc[4], acc[5], acc[6], acc[7]);
        }
    }
    __syncthreads();  // the shared arrays may be reused by the caller's next chunk
}

// The exact reads of chunk blockIdx.x of token blockIdx.y.  Grid (nchunk, M), 256 threads.
template <int kDPass>
__global__ void __launch_bounds__(256)
    reader_exact_kernel(ReaderArgs r, const __nv_bfloat16 *__restrict__ h,
                        const int32_t *__restrict__ ids, const float *__restrict__ wts, int k,
                        int K, const int32_t *__restrict__ sel, const int32_t *__restrict__ nsel,
                        int nchunk, float *__restrict__ partial) {
    extern __shared__ __align__(16) unsigned char xraw[];  // token row, bf16 [H]
    __shared__ float wa[kExactChunk];
    __shared__ int64_t chs[kExactChunk];
    pdl_wait();
    pdl_launch_dependents();
    const int m = blockIdx.y, c = blockIdx.x;
    exact_chunk<kDPass>(r, h + (size_t)m * r.H, ids + (size_t)m * k, wts + (size_t)m * k,
                        sel + (size_t)m * K, nsel[m], c, partial + ((size_t)m * nchunk + c) * r.H,
                        reinterpret_cast<uint4 *>(xraw), wa, chs);
}

// Stage 3: z_j = sum over the discarded channels i of slot j (ascending within a thread,
// then the lanes by a fixed xor tree, then the warps in order) of w_j ahat b_{e,i}.
// Part p of slot j takes channels [p I/4, (p+1) I/4) of a token; its z goes to zpart.  The
// work runs on the CTA's first 256 threads; every thread must call it (it has a barrier).
// keep: the token's kept flags (global bytes, or the selection's shared-memory flags).
constexpr int kRecParts = 4;
__device__ __forceinline__ bool kept_flag(const uint8_t *keep, size_t f) { return __ldcg(keep + f) != 0; }
__device__ __forceinline__ bool kept_flag(const uint32_t *keep, size_t f) { return keep[f] != 0u; }

template <typename KeepT>
__device__ void recover_part(const ReaderArgs &r, const int32_t *__restrict__ ids_m,
                             const float *__restrict__ wts_m, int k, const float *ahat_m,
                             const KeepT *keep_m, int j, int part, float *__restrict__ zout,
                             float (*red)[kReaderMaxRank]) {
    const int I = r.I, rank = r.rank, tid = threadIdx.x;
    const bool act = tid < 256;
    const int per = (I + kRecParts - 1) / kRecParts;
    const int i0 = part * per, i1 = min(I, i0 + per);
    const int e = ids_m[j];
    float acc[kReaderMaxRank];
#pragma unroll
    for (int q = 0; q < kReaderMaxRank; ++q) acc[q] = 0.0f;
    if (act && e >= 0 && e < r.E) {
        const float w = wts_m[j];
        for (int i = i0 + tid; i < i1; i += 256) {
            const size_t f = (size_t)j * I + i;
            if (kept_flag(keep_m, f)) continue;
            const float cw = w * __ldcg(ahat_m + f);
            const __nv_bfloat16 *b = r.coef + ((int64_t)e * I + i) * rank;
            if ((rank & 7) == 0) {  // whole 16-byte pieces of 8 coefficients
#pragma unroll
                for (int q8 = 0; q8 < kReaderMaxRank / 8; ++q8) {
                    if (q8 * 8 >= rank) break;
                    const uint4 pc = *reinterpret_cast<const uint4 *>(b + q8 * 8);
                    const uint32_t pw[4] = {pc.x, pc.y, pc.z, pc.w};
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        acc[q8 * 8 + 2 * t] = fmaf(cw, bf16_lo(pw[t]), acc[q8 * 8 + 2 * t]);
                        acc[q8 * 8 + 2 * t + 1] = fmaf(cw, bf16_hi(pw[t]), acc[q8 * 8 + 2 * t + 1]);
                    }
                }
            } else {
#pragma unroll
                for (int q = 0; q < kReaderMaxRank; ++q)
                    if (q < rank) acc[q] = fmaf(cw, __bfloat162float(b[q]), acc[q]);
            }
        }
    }
    if (act) {
#pragma unroll
        for (int q = 0; q < kReaderMaxRank; ++q) {
            const float v = warp_sum(acc[q]);
            if ((tid & 31) == 0) red[tid >> 5][q] = v;
        }
    }
    __syncthreads();
    if (tid < rank) {
        float z = 0.0f;
        for (int w = 0; w < 8; ++w) z += red[w][tid];
        zout[tid] = z;
    }
    __syncthreads();  // red may be reused by the caller's next part
}

// It needs only the selection, which was complete before the exact-read grid that precedes
// it could start, so it runs beside that grid (reading the selection from L2) and waits for
// it only before finishing: the final grid, which waits for this one, then sees both.
// Grid (4 k, M), 256 threads.
__global__ void __launch_bounds__(256)
    reader_recover_kernel(ReaderArgs r, const int32_t *__restrict__ ids,
                          const float *__restrict__ wts, int k, const float *__restrict__ ahat,
                          const uint8_t *__restrict__ keep, float *__restrict__ zpart) {
    __shared__ float red[8][kReaderMaxRank];
    pdl_launch_dependents();
    const int j = blockIdx.x / kRecParts, part = blockIdx.x % kRecParts, m = blockIdx.y;
    const size_t N = (size_t)k * r.I;
    recover_part(r, ids + (size_t)m * k, wts + (size_t)m * k, k, ahat + (size_t)m * N,
                 keep + (size_t)m * N, j, part,
                 zpart + (((size_t)m * k + j) * kRecParts + part) * r.rank, red);
    pdl_wait();  // the exact-read grid has finished before this one does
}

// out[n] = bf16(residual + (ex + sum_r U[n][r] z[r])) for the 32 columns of block bx of a
// token: z = sum over slots in order of zpart, ex the chunk partials -- warp w sums chunks
// w, w + 8, ... in order for 32 columns, then the 8 warps' sums are added in warp order.  The
// work runs on the CTA's first 256 threads; every thread must call it (it has barriers).
__device__ void final_block(const ReaderArgs &r, int k, int nchunk, const float *partial_m,
                            const float *zpart_m, const __nv_bfloat16 *res_m,
                            __nv_bfloat16 *out_m, int bx, float *z, float (*red)[32],
                            float *recs) {
    const int H = r.H, rank = r.rank, tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const bool act = tid < 256;
    if (tid < rank) {
        float s = 0.0f;
        for (int q = 0; q < k * kRecParts; ++q) s += __ldcg(zpart_m + (size_t)q * rank + tid);
        z[tid] = s;
    }
    const int n = bx * 32 + lane;
    if (act) {
        float ex = 0.0f;
        if (n < H) {
            const float *pp = partial_m + n;
            int c = warp;
            for (; c + 8 * 7 < nchunk; c += 8 * 8) {  // 8 of the warp's chunks in flight
                float v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) v[u] = __ldcg(pp + (size_t)(c + 8 * u) * H);
#pragma unroll
                for (int u = 0; u < 8; ++u) ex += v[u];
            }
            for (; c < nchunk; c += 8) ex += __ldcg(pp + (size_t)c * H);
        }
        red[warp][lane] = ex;
    }
    __syncthreads();
    // U z for the block's 32 columns: warp w takes columns 4w .. 4w+3, lane q the q-th
    // coefficient of a column's U row (one coalesced row read), then a fixed xor tree
    if (act) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int col = bx * 32 + 4 * warp + u;
            float t = 0.0f;
            if (col < H && lane < rank) t = r.U[(size_t)col * rank + lane] * z[lane];
            t = warp_sum(t);
            if (lane == 0) recs[4 * warp + u] = t;
        }
    }
    __syncthreads();
    if (warp == 0 && n < H) {
        float acc = 0.0f;
        for (int w = 0; w < 8; ++w) acc += red[w][lane];
        acc += recs[lane];
        const float res = res_m ? __bfloat162float(res_m[n]) : 0.0f;
        out_m[n] = __float2bfloat16_rn(res + acc);
    }
    __syncthreads();  // the shared arrays may be reused by the caller's next block
}

// The final sum of column block blockIdx.x of token blockIdx.y.  Grid (ceil(H / 32), M), 256
// threads.
__global__ void __launch_bounds__(256)
    reader_final_kernel(ReaderArgs r, int k, int nchunk, const float *__restrict__ partial,
                        const float *__restrict__ zpart, const __nv_bfloat16 *__restrict__ residual,
                        __nv_bfloat16 *__restrict__ out) {
    __shared__ float z[kReaderMaxRank];
    __shared__ float red[8][32];
    __shared__ float recs[32];
    pdl_wait();
    pdl_launch_dependents();
    const int m = blockIdx.y, H = r.H;
    final_block(r, k, nchunk, partial + (size_t)m * nchunk * H,
                zpart + (size_t)m * k * kRecParts * r.rank,
                residual ? residual + (size_t)m * H : nullptr, out + (size_t)m * H, blockIdx.x, z,
                red, recs);
}

// ------------------------------------------------------------- one token, one grid
// For one token the five stages above run as one persistent grid of 512-thread CTAs, one
// per SM: every stage is the same device function with the same arithmetic, so the output
// is bitwise the multi-kernel path's.  Between the stages:
//   scores   -> every CTA, after a release count of all CTAs: the selection, run by every
//               CTA on its own (the same result everywhere; CTA 0 stores it);
//   items    -> exact chunks c and recovery parts, CTA i taking items i, i + G, ...;
//   partials -> the CTAs of the column blocks, after a second count: the final sum.
// The counters live in the workspace (zero between calls: the last CTA to leave, found with
// an exit ticket, restores them); every wait is bounded and a wait that gives up sets
// MOE_DEV_WAIT_TIMEOUT.
constexpr int kReaderCtlScores = 0, kReaderCtlItems = 1, kReaderCtlExit = 2;
// 512 threads: the exact reads' 122 registers per thread fit.  (1024 threads cap them at 64:
// with the exact reads' loads batched 4 instead of 8 it still spilled, and measured slower,
// 36.5 against 33.1 us per router + reader step.)
constexpr int kOneThreads = 512;

// Bounded wait until *p >= need (acquire, GPU scope).
__device__ __forceinline__ bool reader_count_wait(const int32_t *p, int need) {
    if (ld_acquire_gpu(p) >= need) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        __nanosleep(64);
        if (ld_acquire_gpu(p) >= need) return true;
        if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
    }
}

// Shared-memory floats of the one-grid kernel: the largest of the stages' carves.
__host__ __device__ inline size_t reader_one_smem_floats(int H, int N, int K) {
    const size_t sketch = (size_t)nib_table_floats(H) + H + (size_t)(H / 32) * 33;
    const size_t later = (size_t)N + 2 * 32 * 256 + (((size_t)(K > 0 ? K : 1) + 3) & ~size_t(3)) + H / 2;
    return sketch > later ? sketch : later;
}

template <int kMaxPass, int kDPass>
__global__ void __launch_bounds__(kOneThreads, 1)
    reader_one_kernel(ReaderArgs r, const __nv_bfloat16 *__restrict__ h, int nscan,
                      float *__restrict__ xr_out, const int32_t *__restrict__ ids,
                      const float *__restrict__ wts, int k, int K, float *__restrict__ ahat,
                      float *__restrict__ score, int32_t *__restrict__ sel,
                      int32_t *__restrict__ nsel, int nchunk, float *__restrict__ partial,
                      float *__restrict__ zpart, const __nv_bfloat16 *__restrict__ residual,
                      __nv_bfloat16 *__restrict__ out, int32_t *__restrict__ ctl,
                      int32_t *__restrict__ status) {
    extern __shared__ __align__(16) float smem[];
    __shared__ float wa[kExactChunk];
    __shared__ int64_t chs[kExactChunk];
    __shared__ float red_r[8][kReaderMaxRank];
    __shared__ float zf[kReaderMaxRank], redf[8][32], recs[32];
    __shared__ int32_t nsel_s;
    __shared__ int last_s;
    const int tid = threadIdx.x, G = gridDim.x, H = r.H;
    const int N = k * r.I;
    const char4 sg0 = first_block_signs(r);  // weights: before the wait
    pdl_wait();
    pdl_launch_dependents();

    // Stage 1: scan, table, and the scores of this CTA's share of the channels
    sketch_prepare(r, h, nscan, sg0, smem, blockIdx.x == 0 ? xr_out : nullptr);
    sketch_channels<kMaxPass>(r, smem, 0, blockIdx.x * (kOneThreads / 32) + (tid >> 5),
                              G * (kOneThreads / 32), ids, wts, k, ahat, score);
    __syncthreads();
    if (tid == 0) {
        red_release_gpu_add(ctl + kReaderCtlScores, 1);
        if (!reader_count_wait(ctl + kReaderCtlScores, G)) atomicOr(status, MOE_DEV_WAIT_TIMEOUT);
    }
    __syncthreads();

    // Stage 2 selection, in every CTA
    uint32_t *keys = reinterpret_cast<uint32_t *>(smem);
    int *whist = reinterpret_cast<int *>(keys + N);
    int32_t *sel_s = whist + 2 * 32 * 256;
    uint4 *xs4 = reinterpret_cast<uint4 *>(sel_s + (((K > 0 ? K : 1) + 3) & ~3));
    select_token(score, N, K, keys, whist, nullptr, sel_s, &nsel_s);
    __syncthreads();
    const int nsl = nsel_s;
    if (blockIdx.x == 0) {
        for (int q = tid; q < K; q += blockDim.x) sel[q] = sel_s[q];
        if (tid == 0) nsel[0] = nsl;
    }

    // Stage 2 exact reads and Stage 3 recovery: items i, i + G, ...
    const int nitems = nchunk + k * kRecParts;
    for (int it = blockIdx.x; it < nitems; it += G) {
        if (it < nchunk) {
            exact_chunk<kDPass>(r, h, ids, wts, sel_s, nsl, it, partial + (size_t)it * H, xs4, wa, chs);
        } else {
            const int q = it - nchunk, j = q / kRecParts, part = q % kRecParts;
            recover_part(r, ids, wts, k, ahat, keys, j, part,
                         zpart + ((size_t)j * kRecParts + part) * r.rank, red_r);
        }
    }
    __syncthreads();
    if (tid == 0) red_release_gpu_add(ctl + kReaderCtlItems, 1);

    // the final sum, by the CTAs of the column blocks
    const int nbx = (H + 31) / 32;
    if ((int)blockIdx.x < nbx) {
        if (tid == 0 && !reader_count_wait(ctl + kReaderCtlItems, G))
            atomicOr(status, MOE_DEV_WAIT_TIMEOUT);
        __syncthreads();
        for (int bx = blockIdx.x; bx < nbx; bx += G)
            final_block(r, k, nchunk, partial, zpart, residual, out, bx, zf, redf, recs);
    }

    // exit: the last CTA restores the counters
    __syncthreads();
    if (tid == 0) {
        int32_t old;
        asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(old) : "l"(ctl + kReaderCtlExit) : "memory");
        last_s = old == G - 1;
        if (last_s) {
            ctl[kReaderCtlScores] = 0;
            ctl[kReaderCtlItems] = 0;
            ctl[kReaderCtlExit] = 0;
        }
    }
}

// Workspace of one reader call: status, counters, xr, ahat, score, keep, sel, nsel, partial,
// zpart.
ReaderWs reader_ws_layout(const ReaderArgs &r, int M, int k, int K) {
    ReaderWs L;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = (off + bytes + 255) / 256 * 256;
        return at;
    };
    const size_t N = (size_t)k * r.I;
    L.nchunk = (K + kExactChunk - 1) / kExactChunk;
    L.status = take(64);
    L.ctl = take(64);  // the one-grid path's counters: zero between calls
    L.xr = take((size_t)M * r.H * 4);
    L.ahat = take((size_t)M * N * 4);
    L.score = take((size_t)M * N * 4);
    L.keep = take((size_t)M * N);
    L.sel = take((size_t)M * (K > 0 ? K : 1) * 4);
    L.nsel = take((size_t)M * 4);
    L.partial = take((size_t)M * (L.nchunk > 0 ? L.nchunk : 1) * r.H * 4);
    L.zpart = take((size_t)M * k * kRecParts * r.rank * 4);
    L.total = off;
    return L;
}

cudaError_t launch_reader_decode(const ReaderArgs &r, const __nv_bfloat16 *h, int M, int k,
                                 const int32_t *ids, const float *wts, int K, int nscan,
                                 const __nv_bfloat16 *residual, __nv_bfloat16 *out,
                                 unsigned char *ws, cudaStream_t stream) {
    const ReaderWs L = reader_ws_layout(r, M, k, K);
    float *xr = reinterpret_cast<float *>(ws + L.xr);
    float *ahat = reinterpret_cast<float *>(ws + L.ahat);
    float *score = reinterpret_cast<float *>(ws + L.score);
    uint8_t *keep = ws + L.keep;
    int32_t *sel = reinterpret_cast<int32_t *>(ws + L.sel);
    int32_t *nsel = reinterpret_cast<int32_t *>(ws + L.nsel);
    float *partial = reinterpret_cast<float *>(ws + L.partial);
    float *zpart = reinterpret_cast<float *>(ws + L.zpart);
    const int N = k * r.I;
    cudaLaunchAttribute attrs[2];
    cudaError_t err;
    // trace points: 0 before the first kernel, 1 after the scan and sketch scores, 2 after
    // the selection, 3 after the exact reads, 4 after the recovery, 5 after the final sum
    // (one token: every point after the one grid)
    trace_point(0, stream);
    const size_t one_smem = reader_one_smem_floats(r.H, N, K) * 4;
    if (M == 1 && one_smem <= 200 * 1024) {
        const int npass = (r.H / 32 + 31) / 32;
        const int dp = (r.H + 2047) / 2048;
        auto pick = [&](auto mp) {
            constexpr int kMP = decltype(mp)::value;
            return dp <= 1 ? reader_one_kernel<kMP, 1> : dp <= 2 ? reader_one_kernel<kMP, 2>
                                                                 : reader_one_kernel<kMP, 4>;
        };
        auto kern = npass <= 1 ? pick(std::integral_constant<int, 1>())
                  : npass <= 2 ? pick(std::integral_constant<int, 2>())
                  : npass <= 4 ? pick(std::integral_constant<int, 4>())
                               : pick(std::integral_constant<int, 8>());
        err = ensure_smem(reinterpret_cast<const void *>(kern), one_smem);
        if (err != cudaSuccess) return err;
        cudaLaunchConfig_t cfg =
            launch_config(dim3(num_sms()), dim3(kOneThreads), one_smem, stream, attrs, 0);
        err = cudaLaunchKernelEx(&cfg, kern, r, h, nscan, xr, ids, wts, k, K, ahat, score, sel, nsel,
                                 L.nchunk, partial, zpart, residual, out,
                                 reinterpret_cast<int32_t *>(ws + L.ctl),
                                 reinterpret_cast<int32_t *>(ws + L.status));
        for (int i = 1; i <= 5; ++i) trace_point(i, stream);
        return err;
    }
    {
        // the nibble table and xr
        const size_t smem = ((size_t)nib_table_floats(r.H) + r.H + (size_t)(r.H / 32) * 33) * 4;
        const int npass = (r.H / 32 + 31) / 32;  // 32-coordinate words per lane and row
        auto kern = npass <= 1 ? reader_sketch_kernel<1>
                  : npass <= 2 ? reader_sketch_kernel<2>
                  : npass <= 4 ? reader_sketch_kernel<4> : reader_sketch_kernel<8>;
        err = ensure_smem(reinterpret_cast<const void *>(kern), smem);
        if (err != cudaSuccess) return err;
        const int G = (int)std::min<int64_t>((N + kSketchWarps - 1) / kSketchWarps, num_sms());
        cudaLaunchConfig_t cfg =
            launch_config(dim3(G, M), dim3(kSketchWarps * 32), smem, stream, attrs, 0);
        err = cudaLaunchKernelEx(&cfg, kern, r, h, nscan, xr, ids, wts, k, ahat, score);
        if (err != cudaSuccess) return err;
    }
    trace_point(1, stream);
    {
        const size_t smem = (size_t)N * 4 + 2 * 32 * 256 * 4;  // keys, two histogram sets
        err = ensure_smem(reinterpret_cast<const void *>(reader_select_kernel), smem);
        if (err != cudaSuccess) return err;
        cudaLaunchConfig_t cfg = launch_config(dim3(M), dim3(kSelectThreads), smem, stream, attrs, 0);
        err = cudaLaunchKernelEx(&cfg, reader_select_kernel, (const float *)score, N, K, keep, sel,
                                 nsel);
        if (err != cudaSuccess) return err;
    }
    trace_point(2, stream);
    if (L.nchunk > 0) {
        const size_t smem = (size_t)r.H * 2;
        const int dp = (r.H + 2047) / 2048;
        auto kern = dp <= 1 ? reader_exact_kernel<1>
                  : dp <= 2 ? reader_exact_kernel<2> : reader_exact_kernel<4>;
        cudaLaunchConfig_t cfg = launch_config(dim3(L.nchunk, M), dim3(256), smem, stream, attrs, 0);
        err = cudaLaunchKernelEx(&cfg, kern, r, h, ids, wts, k, K,
                                 (const int32_t *)sel, (const int32_t *)nsel, L.nchunk, partial);
        if (err != cudaSuccess) return err;
    }
    trace_point(3, stream);
    {
        cudaLaunchConfig_t cfg = launch_config(dim3(k * kRecParts, M), dim3(256), 0, stream, attrs, 0);
        err = cudaLaunchKernelEx(&cfg, reader_recover_kernel, r, ids, wts, k, (const float *)ahat,
                                 (const uint8_t *)keep, zpart);
        if (err != cudaSuccess) return err;
    }
    trace_point(4, stream);
    {
        cudaLaunchConfig_t cfg =
            launch_config(dim3((r.H + 31) / 32, M), dim3(256), 0, stream, attrs, 0);
        err = cudaLaunchKernelEx(&cfg, reader_final_kernel, r, k, L.nchunk, (const float *)partial,
                                 (const float *)zpart, residual, out);
    }
    trace_point(5, stream);
    return err;
}

}  // namespace moe
