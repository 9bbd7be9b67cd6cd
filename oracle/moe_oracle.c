/*
 * moe_oracle.c -- plain, slow, fp64 CPU oracle for the small-batch MoE decode block.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls this
 * file: only the test suite, the package's smoke check and the benchmark's CPU-baseline
 * leg do.  It shares no code, header, table or constant with the CUDA library.
 *
 * Every floating-point input (bf16 bit patterns, fp32 values) is widened exactly to
 * double, and all arithmetic is done in double with no intermediate rounding, except the
 * one place where floating point decides an integer (the top-k selection), which is taken
 * on the logits rounded to fp32, the precision the router kernel decides in.
 *
 * Sources (by page title and section):
 *   [MED] "A Multi-Engine Dataflow for MoE Decoding on Scratchpad-Based Tensor
 *         Accelerators": MoE block background (Figure 2 description): router picks k
 *         experts with affinities a_e, each expert applies gate and up projections,
 *         the activation phi, the down projection, and the block sums a_e-scaled outputs;
 *         Section 2.3 (blockwise VQ: columns cut into length-d blocks replaced by code
 *         words, per-expert index map, layer-shared code book); the stage-3 description of
 *         phi applied to the gate output followed by an elementwise product with the up
 *         output; Section 4.3 (down projection y_e = W_down,e^T p_e and the accumulated
 *         summation sum_e a_e y_e).
 *   [CSM] "Channel Selection for Mixture-of-Experts Decoding Needs No Calibration Data",
 *         "Background: Channels and Retention Rules" (channel j: a_j = phi(g_j.x)(v_j.x),
 *         output = router weight times sum_j a_j d_j).
 *   [RBM] "Route-Block Membership Selects Packed-AWQ Arithmetic", Section 2.1 (M x k
 *         expert ids flattened row-major to route ids, valid routes grouped by expert,
 *         each expert padded to a multiple of b, parallel expert-block vector) and
 *         Section 5.3 (stable construction orders valid routes by (expert id, route id)).
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - the router is softmax over logits, top-k, then renormalised over the k selected
 *     experts (renormalize=1) or left as the full-softmax probabilities (renormalize=0);
 *   - top-k order: descending fp32-rounded logit, ties to the lower expert id; slot j of
 *     token m is the j-th selected expert, giving route id r = m*k + j;
 *   - the optional per-expert bias is added to the logits and used both for selection and
 *     for the affinities;
 *   - phi is SiLU: silu(g) = g / (1 + exp(-g));
 *   - a route whose expert id lies outside [0, E) is invalid: the alignment excludes it
 *     and it contributes nothing to the output;
 *   - padding rows carry the sentinel value M*k; an expert with no route gets no block;
 *     rows past num_padded are sentinels and block entries past the last block are -1;
 *   - VQ (d-length column blocks along H): W[e][d*q + t][i] = B[J[e][q][i]][t];
 *   - VQ+LR (the hybrid representation; the page's Eq. (1) is garbled, its text describes a
 *     sum): per projection W_e = Q_B(J_e) + D C_e, with D [H, r] shared by all experts of the
 *     layer and projection and C_e [r, I] private to the expert; down stays dense bf16.
 */
#include <math.h>
#ifdef _OPENMP
#include <omp.h>
#endif
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_ERR_ARG 1
#define ORACLE_ERR_CAPACITY 2
#define ORACLE_ERR_NOMEM 3

/* Exact widening of a bf16 bit pattern: bf16 is the top half of an IEEE fp32. */
static double bf16_bits_to_double(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round-to-nearest-even of a double to fp32 (the C conversion does exactly that). */
static float to_f32(double v) { return (float)v; }

/*
 * Router logits [MED, MoE block background]:
 *   logits[m][e] = sum_h h[m][h] * W_r[h][e]  (+ bias[e] when a bias is given).
 * h is [M,H] bf16, W_r is [H,E] bf16, bias is [E] fp32 or NULL, logits is [M,E] double.
 */
int oracle_router_logits(const uint16_t *h, const uint16_t *w_router, const float *bias,
                         int M, int H, int E, double *logits)
{
    if (M < 0 || H <= 0 || E <= 0 || (M > 0 && (!h || !w_router || !logits)))
        return ORACLE_ERR_ARG;
    for (int m = 0; m < M; ++m) {
        double *row = logits + (size_t)m * E;
        for (int e = 0; e < E; ++e)
            row[e] = 0.0;
        for (int hh = 0; hh < H; ++hh) {
            double x = bf16_bits_to_double(h[(size_t)m * H + hh]);
            const uint16_t *wrow = w_router + (size_t)hh * E;
            for (int e = 0; e < E; ++e)
                row[e] += x * bf16_bits_to_double(wrow[e]);
        }
        if (bias)
            for (int e = 0; e < E; ++e)
                row[e] += (double)bias[e];
    }
    return ORACLE_OK;
}

/*
 * Softmax top-k with renormalised affinities [MED, MoE block background; reading above].
 * Selection: the k largest fp32-rounded logits, ties to the lower expert id, in that order.
 * renormalize=1: a_j = exp(l_j - l_0) / sum_{j'<k} exp(l_j' - l_0)   (softmax restricted to
 *   the selected experts, equal to softmax over all E followed by renormalisation).
 * renormalize=0: a_j = exp(l_j - l_max) / sum_{e<E} exp(l_e - l_max).
 * gap[m] (if not NULL) = l_(k-1) - l_(k) in double: the margin between the last selected
 *   and the first unselected logit (+inf when k == E).
 */
int oracle_topk_softmax(const double *logits, int M, int E, int k, int renormalize,
                        int32_t *topk_ids, double *topk_weights, double *gap)
{
    if (M < 0 || E <= 0 || k <= 0 || k > E || (M > 0 && (!logits || !topk_ids || !topk_weights)))
        return ORACLE_ERR_ARG;
    unsigned char *taken = (unsigned char *)malloc((size_t)E);
    if (!taken)
        return ORACLE_ERR_NOMEM;
    for (int m = 0; m < M; ++m) {
        const double *l = logits + (size_t)m * E;
        int32_t *ids = topk_ids + (size_t)m * k;
        double *a = topk_weights + (size_t)m * k;
        memset(taken, 0, (size_t)E);
        for (int j = 0; j < k; ++j) {
            int best = -1;
            float bestv = 0.0f;
            for (int e = 0; e < E; ++e) {
                if (taken[e])
                    continue;
                float v = to_f32(l[e]);
                if (best < 0 || v > bestv) { /* strict '>' keeps the lower id on ties */
                    best = e;
                    bestv = v;
                }
            }
            taken[best] = 1;
            ids[j] = best;
        }
        if (gap) {
            if (k == E) {
                gap[m] = INFINITY;
            } else {
                int next = -1;
                float nextv = 0.0f;
                for (int e = 0; e < E; ++e) {
                    if (taken[e])
                        continue;
                    float v = to_f32(l[e]);
                    if (next < 0 || v > nextv) {
                        next = e;
                        nextv = v;
                    }
                }
                gap[m] = l[ids[k - 1]] - l[next];
            }
        }
        if (renormalize) {
            double l0 = l[ids[0]];
            double denom = 0.0;
            for (int j = 0; j < k; ++j)
                denom += exp(l[ids[j]] - l0);
            for (int j = 0; j < k; ++j)
                a[j] = exp(l[ids[j]] - l0) / denom;
        } else {
            double lmax = l[0];
            for (int e = 1; e < E; ++e)
                if (l[e] > lmax)
                    lmax = l[e];
            double denom = 0.0;
            for (int e = 0; e < E; ++e)
                denom += exp(l[e] - lmax);
            for (int j = 0; j < k; ++j)
                a[j] = exp(l[ids[j]] - lmax) / denom;
        }
    }
    free(taken);
    return ORACLE_OK;
}

/*
 * Stable block alignment [RBM, Sections 2.1 and 5.3].
 * Route r = m*k + j is valid when 0 <= topk_ids[r] < E.  For each expert e in ascending
 * order with n_e > 0 valid routes: append its routes in ascending r, then
 * ceil(n_e/b)*b - n_e sentinels (value M*k), and append ceil(n_e/b) copies of e to the
 * expert-block vector.  num_padded = number of rows appended.  Rows num_padded..cap-1 are
 * sentinels; block entries past the last block (up to cap/b) are -1.
 * Returns ORACLE_ERR_CAPACITY when the padded rows do not fit in cap.
 */
int oracle_align(const int32_t *topk_ids, int M, int k, int E, int b,
                 int32_t *sorted_route_ids, int32_t *expert_block_ids, int32_t *num_padded,
                 int64_t cap)
{
    if (M < 0 || k <= 0 || E <= 0 || b <= 0 || cap < 0 || !num_padded ||
        (cap > 0 && (!sorted_route_ids || !expert_block_ids)) || (M > 0 && !topk_ids))
        return ORACLE_ERR_ARG;
    const int64_t R = (int64_t)M * k;
    const int32_t sentinel = (int32_t)R;
    int64_t pos = 0, nblk = 0;
    for (int e = 0; e < E; ++e) {
        int64_t n = 0;
        for (int64_t r = 0; r < R; ++r) {
            if (topk_ids[r] == e) {
                if (pos >= cap)
                    return ORACLE_ERR_CAPACITY;
                sorted_route_ids[pos++] = (int32_t)r;
                ++n;
            }
        }
        if (n == 0)
            continue;
        int64_t blocks = (n + b - 1) / b;
        for (int64_t q = n; q < blocks * b; ++q) {
            if (pos >= cap)
                return ORACLE_ERR_CAPACITY;
            sorted_route_ids[pos++] = sentinel;
        }
        for (int64_t q = 0; q < blocks; ++q)
            expert_block_ids[nblk++] = e;
    }
    *num_padded = (int32_t)pos;
    for (int64_t q = pos; q < cap; ++q)
        sorted_route_ids[q] = sentinel;
    for (int64_t q = nblk; q < cap / b; ++q)
        expert_block_ids[q] = -1;
    return ORACLE_OK;
}

/* Weight representations for the gate/up projections. */
#define ORACLE_W_DENSE 0
#define ORACLE_W_VQ 1
#define ORACLE_W_VQLR 2

typedef struct {
    int kind;                 /* ORACLE_W_DENSE, ORACLE_W_VQ or ORACLE_W_VQLR */
    int H, I, E;
    const uint16_t *w_gate;   /* dense: [E,H,I] bf16 */
    const uint16_t *w_up;     /* dense: [E,H,I] bf16 */
    const uint8_t *j_gate;    /* VQ: [E,H/d,I] uint8 code indices */
    const uint8_t *j_up;      /* VQ: [E,H/d,I] uint8 code indices */
    const uint16_t *cb_gate;  /* VQ: [K,d] bf16 code book, layer-shared */
    const uint16_t *cb_up;    /* VQ: [K,d] bf16 code book, layer-shared */
    int d, K;
    const uint16_t *w_down;   /* [E,I,H] bf16 */
    const uint16_t *d_gate;   /* VQ+LR: [H,r] bf16 low-rank basis, layer-shared */
    const uint16_t *d_up;     /* VQ+LR: [H,r] bf16 */
    const uint16_t *c_gate;   /* VQ+LR: [E,r,I] bf16 low-rank coefficients, per expert */
    const uint16_t *c_up;     /* VQ+LR: [E,r,I] bf16 */
    int r;
} oracle_weights_t;

/*
 * One projection row h of expert e, accumulated into acc[0..I):  acc[i] += x * W[e][h][i].
 * Dense: W[e][h][i] is stored.  VQ [MED, Section 2.3]: the column i of W_e is cut into
 * length-d blocks along H; block q = h / d holds code word J[e][q][i] and row h reads
 * element t = h mod d of that code word.
 */
static void accumulate_row(const oracle_weights_t *w, const uint16_t *dense, const uint8_t *J,
                           const uint16_t *cb, int e, int hh, double x, double *acc)
{
    const int H = w->H, I = w->I;
    if (w->kind == ORACLE_W_DENSE) {
        const uint16_t *row = dense + ((size_t)e * H + hh) * I;
        for (int i = 0; i < I; ++i)
            acc[i] += x * bf16_bits_to_double(row[i]);
    } else {
        const int d = w->d;
        const int q = hh / d, t = hh % d;
        const uint8_t *jrow = J + ((size_t)e * (H / d) + q) * I;
        for (int i = 0; i < I; ++i)
            acc[i] += x * bf16_bits_to_double(cb[(size_t)jrow[i] * d + t]);
    }
}

/*
 * Low-rank half of the hybrid gate/up representation [MED, the hybrid-representation
 * paragraph around its Eq. (1), and "Reuse of shared projections"]: each projection's weight is
 * W_e = Q_B(J_e) + D C_e with the layer-shared basis D [H, r] and the expert's coefficients
 * C_e [r, I], so h^T W_e = h^T Q_B(J_e) + (D^T h)^T C_e.  The product is taken in that
 * factored order: z = D^T h once per token and projection, then acc[i] += sum_rho z[rho]
 * C_e[rho][i] (the same value as h^T (D C_e) in exact arithmetic).
 */
static void add_low_rank(const oracle_weights_t *w, const uint16_t *hrow, int e, double *zg,
                         double *zu, double *g, double *u)
{
    const int H = w->H, I = w->I, R = w->r;
    for (int rho = 0; rho < R; ++rho)
        zg[rho] = zu[rho] = 0.0;
    for (int hh = 0; hh < H; ++hh) {
        const double x = bf16_bits_to_double(hrow[hh]);
        for (int rho = 0; rho < R; ++rho) {
            zg[rho] += x * bf16_bits_to_double(w->d_gate[(size_t)hh * R + rho]);
            zu[rho] += x * bf16_bits_to_double(w->d_up[(size_t)hh * R + rho]);
        }
    }
    for (int rho = 0; rho < R; ++rho) {
        const uint16_t *cg = w->c_gate + ((size_t)e * R + rho) * I;
        const uint16_t *cu = w->c_up + ((size_t)e * R + rho) * I;
        for (int i = 0; i < I; ++i) {
            g[i] += zg[rho] * bf16_bits_to_double(cg[i]);
            u[i] += zu[rho] * bf16_bits_to_double(cu[i]);
        }
    }
}

/*
 * Expert FFN and weighted combine [MED, MoE block background, stage-3 activation, Section
 * 4.3; CSM, channel view]:
 *   g = h W_gate[e], u = h W_up[e], p = silu(g) * u, y = p W_down[e],
 *   out[m] = residual[m] + sum_j a_j * y_{m,j}   (invalid routes skipped).
 * h [M,H] bf16; topk_ids [M,k]; a [M,k] double; residual [M,H] bf16 or NULL; out [M,H]
 * double.  p_out [M*k, I] and y_out [M*k, H] (double, optional) receive the per-route
 * intermediate and expert output; rows of invalid routes are zero.
 */
int oracle_expert_ffn(const uint16_t *h, const oracle_weights_t *w, int M, int k,
                      const int32_t *topk_ids, const double *a, const uint16_t *residual,
                      double *out, double *p_out, double *y_out)
{
    if (!w || M < 0 || k <= 0 || w->H <= 0 || w->I <= 0 || w->E <= 0)
        return ORACLE_ERR_ARG;
    if (M > 0 && (!h || !topk_ids || !a || !out || !w->w_down))
        return ORACLE_ERR_ARG;
    if (w->kind == ORACLE_W_DENSE) {
        if (!w->w_gate || !w->w_up)
            return ORACLE_ERR_ARG;
    } else if (w->kind == ORACLE_W_VQ || w->kind == ORACLE_W_VQLR) {
        if (!w->j_gate || !w->j_up || !w->cb_gate || !w->cb_up || w->d <= 0 || w->K <= 0 ||
            w->H % w->d != 0)
            return ORACLE_ERR_ARG;
        if (w->kind == ORACLE_W_VQLR &&
            (!w->d_gate || !w->d_up || !w->c_gate || !w->c_up || w->r <= 0))
            return ORACLE_ERR_ARG;
    } else {
        return ORACLE_ERR_ARG;
    }
    const int H = w->H, I = w->I, E = w->E;
    const int R = w->kind == ORACLE_W_VQLR ? w->r : 0;
    const int64_t routes = (int64_t)M * k;
    /* y of every route first (routes are independent: with OpenMP each thread takes whole
     * routes, each computed by the single-threaded loop below, unchanged), then the combine
     * of every token in slot order. */
    double *yall = (double *)malloc(sizeof(double) * (size_t)(routes > 0 ? routes : 1) * H);
    if (!yall)
        return ORACLE_ERR_NOMEM;
    int status = ORACLE_OK;
#ifdef _OPENMP
#pragma omp parallel
#endif
    {
        double *g = (double *)malloc(sizeof(double) * (size_t)I);
        double *u = (double *)malloc(sizeof(double) * (size_t)I);
        double *p = (double *)malloc(sizeof(double) * (size_t)I);
        double *zg = (double *)malloc(sizeof(double) * (size_t)(R > 0 ? R : 1));
        double *zu = (double *)malloc(sizeof(double) * (size_t)(R > 0 ? R : 1));
        const int ok = g && u && p && zg && zu;
        if (!ok) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            status = ORACLE_ERR_NOMEM;
        }
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int64_t r = 0; r < routes; ++r) {
            double *y = yall + (size_t)r * H;
            const int e = topk_ids[r];
            if (!ok || e < 0 || e >= E) {
                if (p_out)
                    memset(p_out + (size_t)r * I, 0, sizeof(double) * (size_t)I);
                memset(y, 0, sizeof(double) * (size_t)H);
                continue;
            }
            const int64_t m = r / k;
            for (int i = 0; i < I; ++i)
                g[i] = u[i] = 0.0;
            for (int hh = 0; hh < H; ++hh) {
                const double x = bf16_bits_to_double(h[(size_t)m * H + hh]);
                accumulate_row(w, w->w_gate, w->j_gate, w->cb_gate, e, hh, x, g);
                accumulate_row(w, w->w_up, w->j_up, w->cb_up, e, hh, x, u);
            }
            if (R > 0)
                add_low_rank(w, h + (size_t)m * H, e, zg, zu, g, u);
            for (int i = 0; i < I; ++i)
                p[i] = g[i] / (1.0 + exp(-g[i])) * u[i];
            for (int n = 0; n < H; ++n)
                y[n] = 0.0;
            for (int i = 0; i < I; ++i) {
                const uint16_t *drow = w->w_down + ((size_t)e * I + i) * H;
                for (int n = 0; n < H; ++n)
                    y[n] += p[i] * bf16_bits_to_double(drow[n]);
            }
            if (p_out)
                memcpy(p_out + (size_t)r * I, p, sizeof(double) * (size_t)I);
        }
        free(g); free(u); free(p); free(zg); free(zu);
    }
    for (int m = 0; m < M && status == ORACLE_OK; ++m) {
        double *o = out + (size_t)m * H;
        for (int n = 0; n < H; ++n)
            o[n] = residual ? bf16_bits_to_double(residual[(size_t)m * H + n]) : 0.0;
        for (int j = 0; j < k; ++j) {
            const size_t r = (size_t)m * k + j;
            const int e = topk_ids[r];
            if (e < 0 || e >= E)
                continue;
            for (int n = 0; n < H; ++n)
                o[n] += a[r] * yall[r * H + n];
        }
    }
    if (y_out && status == ORACLE_OK)
        memcpy(y_out, yall, sizeof(double) * (size_t)routes * H);
    free(yall);
    return status;
}

/*
 * Threads the expert loop may use (OpenMP builds; 1 otherwise).  n <= 0 leaves the count
 * as it is.  Returns the count in effect.
 */
int oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
    return omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}

/*
 * The whole block: router logits, softmax top-k, expert FFN and combine.  The alignment
 * does not enter the arithmetic of the definition; it is computed separately by
 * oracle_align.  Outputs: topk_ids [M,k], topk_weights [M,k] double, gap [M] (optional),
 * out [M,H] double.
 */
int oracle_decode_block(const uint16_t *h, const uint16_t *w_router, const float *bias,
                        const oracle_weights_t *w, int M, int k, int renormalize,
                        const uint16_t *residual, int32_t *topk_ids, double *topk_weights,
                        double *gap, double *out)
{
    if (!w || M < 0)
        return ORACLE_ERR_ARG;
    if (M == 0)
        return ORACLE_OK;
    double *logits = (double *)malloc(sizeof(double) * (size_t)M * w->E);
    if (!logits)
        return ORACLE_ERR_NOMEM;
    int rc = oracle_router_logits(h, w_router, bias, M, w->H, w->E, logits);
    if (rc == ORACLE_OK)
        rc = oracle_topk_softmax(logits, M, w->E, k, renormalize, topk_ids, topk_weights, gap);
    free(logits);
    if (rc != ORACLE_OK)
        return rc;
    return oracle_expert_ffn(h, w, M, k, topk_ids, topk_weights, residual, out, NULL, NULL);
}
