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
//   codes          [E][I][H/128][8] uint32: 128 two-bit codes per block, code c of a block
//                  at bits 2(c%16) of word c/16; 00 = 0, 01 = +1, 11 = -1;
//   scales         [E][I][H/128] fp32;  dnorm [E][I] fp32;
//   U              [H][r] fp32;  coef b [E][I][r] bf16.
// Every sum has an order fixed by indices (never by the grid or by M): a token's output
// is bitwise reproducible and independent of the other tokens.
#include "moe_internal.cuh"
#include "ptx.cuh"

namespace moe {

constexpr int kRB = 128;              // coordinates per rotation block
constexpr int kRWords = kRB / 16;     // uint32 code words per block
constexpr int kExactChunk = 8;        // selected channels per exact-read CTA (one per warp)
constexpr int kSelectThreads = 1024;

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
            uint32_t bits = 0;
            float mag = 0.0f, cnt = 0.0f;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (fabsf(v[q]) > tau) {
                    bits |= (v[q] < 0.0f ? 3u : 1u) << (2 * q);
                    mag += fabsf(v[q]);
                    cnt += 1.0f;
                }
            }
            mag = warp_sum(mag);
            cnt = warp_sum(cnt);
            // lane l's 8 code bits sit at bits 8 (l % 4) of word l / 4
            uint32_t word = bits << (8 * (lane & 3));
            word |= __shfl_xor_sync(0xffffffffu, word, 1);
            word |= __shfl_xor_sync(0xffffffffu, word, 2);
            if ((lane & 3) == 0) codes[b * kRWords + (lane >> 2)] = word;
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
// Stage 1a: x of token m rotated block by block; every coordinate outside its block's
// nscan largest |Rx| (ties: lower coordinate) is zeroed, so the sketch products below
// need no mask.  Grid (H/128, M), one warp per block.
__global__ void __launch_bounds__(32)
    reader_scan_kernel(const __nv_bfloat16 *__restrict__ h, const int8_t *__restrict__ signs,
                       int H, int nscan, float *__restrict__ xr) {
    __shared__ float av[kRB];
    pdl_wait();
    pdl_launch_dependents();
    const int lane = threadIdx.x, b = blockIdx.x, m = blockIdx.y;
    const int c0 = b * kRB + 4 * lane;
    const uint2 raw = *reinterpret_cast<const uint2 *>(h + (size_t)m * H + c0);
    const char4 sg = *reinterpret_cast<const char4 *>(signs + c0);
    float v[4] = {bf16_lo(raw.x) * sg.x, bf16_hi(raw.x) * sg.y, bf16_lo(raw.y) * sg.z,
                  bf16_hi(raw.y) * sg.w};
    fwht128_warp(v, lane);
#pragma unroll
    for (int q = 0; q < 4; ++q) av[4 * lane + q] = fabsf(v[q]);
    __syncwarp();
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int c = 4 * lane + q;
        const float a = av[c];
        int rank = 0;
        for (int t = 0; t < kRB; ++t) {
            const float o = av[t];
            rank += (o > a) || (o == a && t < c);
        }
        xr[(size_t)m * H + c0 + q] = rank < nscan ? v[q] : 0.0f;
    }
}

// sum over one half block (64 coordinates) of code * xr: lane-rotated start so that the 32
// lanes of a warp read 32 different shared-memory banks.
__device__ __forceinline__ float half_block_dot(uint4 cw, const float *xr, int lane) {
    float s = 0.0f;
#pragma unroll 4
    for (int t = 0; t < 64; ++t) {
        const int tt = (t + lane) & 63;
        const int q = tt >> 4;
        const uint32_t w = q == 0 ? cw.x : (q == 1 ? cw.y : (q == 2 ? cw.z : cw.w));
        const uint32_t bits = (w >> (2 * (tt & 15))) & 3u;
        const float x = xr[tt];
        if (bits & 1u) s += (bits & 2u) ? -x : x;
    }
    return s;
}

// Stage 1b and the score of Stage 2: one warp per candidate channel f = slot * I + i of
// token m.  Grid (ceil(k I / 8), M), 8 warps; xr of the token in shared memory.
__global__ void __launch_bounds__(256)
    reader_sketch_kernel(ReaderArgs r, const float *__restrict__ xr_all,
                         const int32_t *__restrict__ ids, const float *__restrict__ wts, int k,
                         float *__restrict__ ahat, float *__restrict__ score) {
    extern __shared__ float xs[];  // [H]
    pdl_wait();
    pdl_launch_dependents();
    const int m = blockIdx.y, H = r.H, I = r.I, nb = H / kRB;
    const int N = k * I;
    for (int c = threadIdx.x; c < H; c += blockDim.x) xs[c] = xr_all[(size_t)m * H + c];
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int f = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (f >= N) return;
    const int j = f / I, i = f - j * I;
    const int e = ids[(size_t)m * k + j];
    const size_t o = (size_t)m * N + f;
    if (e < 0 || e >= r.E) {
        if (lane == 0) {
            ahat[o] = 0.0f;
            score[o] = -1.0f;
        }
        return;
    }
    const int64_t ch = (int64_t)e * I + i;
    float est[2];
#pragma unroll
    for (int p = 0; p < 2; ++p) {
        const uint32_t *codes = (p ? r.v_codes : r.g_codes) + ch * nb * kRWords;
        const float *scales = (p ? r.v_scales : r.g_scales) + ch * nb;
        float acc = 0.0f;
        for (int base = 0; base < 2 * nb; base += 32) {  // half blocks, 32 per pass
            const int idx = base + lane;
            const bool on = idx < 2 * nb;
            const int b = idx >> 1, half = idx & 1;
            float s = 0.0f;
            if (on)
                s = half_block_dot(*reinterpret_cast<const uint4 *>(codes + b * kRWords + half * 4),
                                   xs + b * kRB + half * 64, lane);
            s += __shfl_xor_sync(0xffffffffu, s, 1);  // the block's two halves
            if (on && half == 0) acc = fmaf(scales[b], s, acc);
        }
        est[p] = warp_sum(acc);
    }
    if (lane == 0) {
        const float a = silu_f32(est[0]) * est[1];
        ahat[o] = a;
        score[o] = wts[(size_t)m * k + j] * r.dnorm[ch] * fabsf(a);
    }
}

// Inclusive scan over the 1024 threads of a block (values in thread order).
__device__ __forceinline__ int block_scan_1024(int v, int *warp_tot) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += u;
    }
    if (lane == 31) warp_tot[warp] = v;
    __syncthreads();
    if (warp == 0) {
        int t = warp_tot[lane];
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

// Stage 2 selection: the K largest scores of token m (ties: lower channel index), by a
// most-significant-digit radix select on order-preserving keys (integer counts commute, so
// the result does not depend on arrival order), then the kept flags and the kept channels
// in ascending index.  One 1024-thread CTA per token; keys in shared memory.
__global__ void __launch_bounds__(kSelectThreads)
    reader_select_kernel(const float *__restrict__ score, int N, int K,
                         uint8_t *__restrict__ keep, int32_t *__restrict__ sel,
                         int32_t *__restrict__ nsel) {
    extern __shared__ uint32_t keys[];  // [N]
    __shared__ int hist[256];
    __shared__ int warp_tot[32];
    __shared__ int s_nvalid, s_digit, s_remaining;
    pdl_wait();
    pdl_launch_dependents();
    const int m = blockIdx.x, tid = threadIdx.x;
    if (tid == 0) s_nvalid = 0;
    __syncthreads();
    int nv = 0;
    for (int f = tid; f < N; f += kSelectThreads) {
        const float s = score[(size_t)m * N + f];
        const uint32_t key = s >= 0.0f ? __float_as_uint(s) + 1u : 0u;  // invalid / NaN: 0
        keys[f] = key;
        nv += key != 0u;
    }
    atomicAdd(&s_nvalid, nv);
    __syncthreads();
    const int Keff = min(K, s_nvalid);
    uint32_t prefix = 0, mask = 0;
    int remaining = Keff;
    if (Keff > 0) {
        for (int shift = 24; shift >= 0; shift -= 8) {
            for (int d = tid; d < 256; d += kSelectThreads) hist[d] = 0;
            __syncthreads();
            for (int f = tid; f < N; f += kSelectThreads)
                if ((keys[f] & mask) == prefix) atomicAdd(&hist[(keys[f] >> shift) & 255u], 1);
            __syncthreads();
            if (tid == 0) {
                int cum = 0, d = 255;
                for (; d > 0; --d) {
                    if (cum + hist[d] >= remaining) break;
                    cum += hist[d];
                }
                s_digit = d;
                s_remaining = remaining - cum;
            }
            __syncthreads();
            prefix |= (uint32_t)s_digit << shift;
            mask |= 255u << shift;
            remaining = s_remaining;
            __syncthreads();
        }
    }
    // keys above the threshold are kept, and the first `remaining` keys equal to it in
    // index order; each thread owns a contiguous run of channels
    const uint32_t T = prefix;
    const int per = (N + kSelectThreads - 1) / kSelectThreads;
    const int f0 = tid * per, f1 = min(N, f0 + per);
    int eq = 0;
    for (int f = f0; f < f1; ++f) eq += (Keff > 0 && keys[f] == T);
    int eq_before = block_scan_1024(eq, warp_tot) - eq;
    int kc = 0;
    for (int f = f0; f < f1; ++f) {
        const uint32_t key = keys[f];
        bool kp = false;
        if (Keff > 0) {
            if (key > T) kp = true;
            else if (key == T) kp = eq_before++ < remaining;
        }
        keep[(size_t)m * N + f] = kp ? 1 : 0;
        keys[f] = kp ? 1u : 0u;  // reused as the kept flag
        kc += kp;
    }
    __syncthreads();
    int pos = block_scan_1024(kc, warp_tot) - kc;
    for (int f = f0; f < f1; ++f)
        if (keys[f]) sel[(size_t)m * K + pos++] = f;
    for (int q = Keff + tid; q < K; q += kSelectThreads) sel[(size_t)m * K + q] = -1;
    if (tid == 0) nsel[m] = Keff;
}

// Stage 2 exact reads: chunk c of token m's kept channels (positions 8c .. 8c+7 of the
// ascending list), one warp per channel for a = SiLU(g . x) (v . x), then the chunk's
// sum of w a d in channel order into its own partial row.  Grid (nchunk, M), 256 threads.
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
    const int m = blockIdx.y, c = blockIdx.x, H = r.H, I = r.I;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint4 *hx = reinterpret_cast<const uint4 *>(h + (size_t)m * H);
    uint4 *xs4 = reinterpret_cast<uint4 *>(xraw);
    for (int q = threadIdx.x; q < H / 8; q += blockDim.x) xs4[q] = hx[q];
    __syncthreads();
    const int s = c * kExactChunk + warp;
    int64_t ch = -1;
    float w = 0.0f;
    if (s < nsel[m]) {
        const int f = sel[(size_t)m * K + s];
        const int j = f / I, i = f - j * I;
        const int e = ids[(size_t)m * k + j];
        if (e >= 0 && e < r.E) {
            ch = (int64_t)e * I + i;
            w = wts[(size_t)m * k + j];
        }
    }
    if (ch >= 0) {
        const uint4 *g = reinterpret_cast<const uint4 *>(r.g_rows + ch * H);
        const uint4 *v = reinterpret_cast<const uint4 *>(r.v_rows + ch * H);
        float gx = 0.0f, vx = 0.0f;
        for (int q = lane; q < H / 8; q += 32) {
            const uint4 xa = xs4[q], ga = g[q], va = v[q];
            const uint32_t xw[4] = {xa.x, xa.y, xa.z, xa.w};
            const uint32_t gw[4] = {ga.x, ga.y, ga.z, ga.w};
            const uint32_t vw[4] = {va.x, va.y, va.z, va.w};
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                gx = fmaf(bf16_lo(gw[t]), bf16_lo(xw[t]), gx);
                gx = fmaf(bf16_hi(gw[t]), bf16_hi(xw[t]), gx);
                vx = fmaf(bf16_lo(vw[t]), bf16_lo(xw[t]), vx);
                vx = fmaf(bf16_hi(vw[t]), bf16_hi(xw[t]), vx);
            }
        }
        gx = warp_sum(gx);
        vx = warp_sum(vx);
        if (lane == 0) wa[warp] = w * (silu_f32(gx) * vx);
    }
    if (lane == 0) chs[warp] = ch;
    __syncthreads();
    float *out = partial + ((size_t)m * nchunk + c) * H;
    for (int c0 = threadIdx.x * 8; c0 < H; c0 += blockDim.x * 8) {
        float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        for (int q = 0; q < kExactChunk; ++q) {
            const int64_t cq = chs[q];
            if (cq < 0) continue;
            const uint4 dv = *reinterpret_cast<const uint4 *>(r.w_down + cq * H + c0);
            const uint32_t dw[4] = {dv.x, dv.y, dv.z, dv.w};
            const float a = wa[q];
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                acc[2 * t] = fmaf(a, bf16_lo(dw[t]), acc[2 * t]);
                acc[2 * t + 1] = fmaf(a, bf16_hi(dw[t]), acc[2 * t + 1]);
            }
        }
        *reinterpret_cast<float4 *>(out + c0) = make_float4(acc[0], acc[1], acc[2], acc[3]);
        *reinterpret_cast<float4 *>(out + c0 + 4) = make_float4(acc[4], acc[5], acc[6], acc[7]);
    }
}

// Stage 3: z_j = sum over the discarded channels i of slot j (ascending within a thread,
// then threads in order) of w_j ahat b_{e,i}.  Grid (k, M), 256 threads.
__global__ void __launch_bounds__(256)
    reader_recover_kernel(ReaderArgs r, const int32_t *__restrict__ ids,
                          const float *__restrict__ wts, int k, const float *__restrict__ ahat,
                          const uint8_t *__restrict__ keep, float *__restrict__ zpart) {
    __shared__ float red[256][33];
    pdl_wait();
    pdl_launch_dependents();
    const int j = blockIdx.x, m = blockIdx.y, I = r.I, rank = r.rank, tid = threadIdx.x;
    const int N = k * I;
    const int e = ids[(size_t)m * k + j];
    float acc[32];
#pragma unroll
    for (int q = 0; q < 32; ++q) acc[q] = 0.0f;
    if (e >= 0 && e < r.E) {
        const float w = wts[(size_t)m * k + j];
        for (int i = tid; i < I; i += 256) {
            const size_t f = (size_t)m * N + (size_t)j * I + i;
            if (keep[f]) continue;
            const float cw = w * ahat[f];
            const __nv_bfloat16 *b = r.coef + ((int64_t)e * I + i) * rank;
#pragma unroll
            for (int q = 0; q < 32; ++q)
                if (q < rank) acc[q] = fmaf(cw, __bfloat162float(b[q]), acc[q]);
        }
    }
#pragma unroll
    for (int q = 0; q < 32; ++q) red[tid][q] = acc[q];
    __syncthreads();
    if (tid < rank) {
        float z = 0.0f;
        for (int t = 0; t < 256; ++t) z += red[t][tid];
        zpart[((size_t)m * k + j) * rank + tid] = z;
    }
}

// out[m][n] = bf16(residual + (sum of the chunk partials in chunk order + sum_r U[n][r] z[r])),
// z = sum over slots in order.  Grid (ceil(H / 256), M).
__global__ void __launch_bounds__(256)
    reader_final_kernel(ReaderArgs r, int k, int nchunk, const float *__restrict__ partial,
                        const float *__restrict__ zpart, const __nv_bfloat16 *__restrict__ residual,
                        __nv_bfloat16 *__restrict__ out) {
    __shared__ float z[32];
    pdl_wait();
    pdl_launch_dependents();
    const int m = blockIdx.y, H = r.H, rank = r.rank, tid = threadIdx.x;
    if (tid < rank) {
        float s = 0.0f;
        for (int j = 0; j < k; ++j) s += zpart[((size_t)m * k + j) * rank + tid];
        z[tid] = s;
    }
    __syncthreads();
    const int n = blockIdx.x * 256 + tid;
    if (n >= H) return;
    const float *pp = partial + (size_t)m * nchunk * H + n;
    float ex = 0.0f;
    int c = 0;
    for (; c + 8 <= nchunk; c += 8) {
        float v[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) v[q] = pp[(size_t)(c + q) * H];
#pragma unroll
        for (int q = 0; q < 8; ++q) ex += v[q];
    }
    for (; c < nchunk; ++c) ex += pp[(size_t)c * H];
    float rec = 0.0f;
    for (int q = 0; q < rank; ++q) rec = fmaf(r.U[(size_t)n * rank + q], z[q], rec);
    const float res = residual ? __bfloat162float(residual[(size_t)m * H + n]) : 0.0f;
    out[(size_t)m * H + n] = __float2bfloat16_rn(res + (ex + rec));
}

// Workspace of one reader call: xr, ahat, score, keep, sel, nsel, partial, zpart.
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
    L.xr = take((size_t)M * r.H * 4);
    L.ahat = take((size_t)M * N * 4);
    L.score = take((size_t)M * N * 4);
    L.keep = take((size_t)M * N);
    L.sel = take((size_t)M * (K > 0 ? K : 1) * 4);
    L.nsel = take((size_t)M * 4);
    L.partial = take((size_t)M * (L.nchunk > 0 ? L.nchunk : 1) * r.H * 4);
    L.zpart = take((size_t)M * k * r.rank * 4);
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
    {
        cudaLaunchConfig_t cfg = launch_config(dim3(r.H / kRB, M), dim3(32), 0, stream, attrs, 0);
        err = cudaLaunchKernelEx(&cfg, reader_scan_kernel, h, r.signs, r.H, nscan, xr);
        if (err != cudaSuccess) return err;
    }
    {
        const size_t smem = (size_t)r.H * 4;
        err = ensure_smem(reinterpret_cast<const void *>(reader_sketch_kernel), smem);
        if (err != cudaSuccess) return err;
        cudaLaunchConfig_t cfg = launch_config(dim3((N + 7) / 8, M), dim3(256), smem, stream, attrs, 0);
        err = cudaLaunchKernelEx(&cfg, reader_sketch_kernel, r, (const float *)xr, ids, wts, k,
                                 ahat, score);
        if (err != cudaSuccess) return err;
    }
    {
        const size_t smem = (size_t)N * 4;
        err = ensure_smem(reinterpret_cast<const void *>(reader_select_kernel), smem);
        if (err != cudaSuccess) return err;
        cudaLaunchConfig_t cfg = launch_config(dim3(M), dim3(kSelectThreads), smem, stream, attrs, 0);
        err = cudaLaunchKernelEx(&cfg, reader_select_kernel, (const float *)score, N, K, keep, sel,
                                 nsel);
        if (err != cudaSuccess) return err;
    }
    if (L.nchunk > 0) {
        const size_t smem = (size_t)r.H * 2;
        cudaLaunchConfig_t cfg = launch_config(dim3(L.nchunk, M), dim3(256), smem, stream, attrs, 0);
        err = cudaLaunchKernelEx(&cfg, reader_exact_kernel, r, h, ids, wts, k, K,
                                 (const int32_t *)sel, (const int32_t *)nsel, L.nchunk, partial);
        if (err != cudaSuccess) return err;
    }
    {
        cudaLaunchConfig_t cfg = launch_config(dim3(k, M), dim3(256), 0, stream, attrs, 0);
        err = cudaLaunchKernelEx(&cfg, reader_recover_kernel, r, ids, wts, k, (const float *)ahat,
                                 (const uint8_t *)keep, zpart);
        if (err != cudaSuccess) return err;
    }
    {
        cudaLaunchConfig_t cfg =
            launch_config(dim3((r.H + 255) / 256, M), dim3(256), 0, stream, attrs, 0);
        err = cudaLaunchKernelEx(&cfg, reader_final_kernel, r, k, L.nchunk, (const float *)partial,
                                 (const float *)zpart, residual, out);
    }
    return err;
}

}  // namespace moe
