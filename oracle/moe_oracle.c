/*
 * moe_oracle.c -- plain, slow, obviously-correct CPU oracle of the MoE layer
 * forward pass (gate -> TopK -> softmax over the K kept logits -> dispatch
 * under capacity -> expert FFN -> combine -> load-balancing loss).
 *
 * TEST INFRASTRUCTURE. Only the test suite, the package smoke check and the
 * benchmark's CPU-baseline leg may load this library. The product path never
 * calls it. It shares no source, header, table or helper with the CUDA path.
 *
 * Arithmetic is IEEE double throughout. The only roundings to narrower types
 * are the storage points the layer defines: routing weights are stored fp32,
 * the expert hidden activation, the expert output, the shared-expert output and
 * the layer output are stored bf16 (round to nearest, ties to even).
 * Compile without -ffast-math.
 *
 * Sources (the MoE web pages this layer is defined by):
 *  [Infra]  lmnt.cn/news/351908, an infrastructure-side walk-through of MoE:
 *           sec. 2.1 (score = Softmax(TopK(W_g x)), TopK before softmax),
 *           sec. 3.1 (dispatch = regroup token order into per-expert blocks),
 *           sec. 3.2 (combine equation; same order as dispatch),
 *           sec. 3.3 (capacity equation; overflow dropped to the residual),
 *           sec. 5.1-5.2 (balance loss alpha*N*sum f_i P_i and its code),
 *           sec. 5.3 (router z-loss beta * mean_t logsumexp_t^2).
 *  [Yunthe] "MoE混合专家模型实战：专家路由与稀疏激活的推理成本优化方案"
 *           (yunthe.com): output equation y = sum_{i in TopK} g_i(x) E_i(x),
 *           the MoELayer listing (expert = Linear -> GELU -> Linear), and the
 *           aux-loss-free per-expert selection bias b_i.
 *  [Wiblog] "MoE 专家路由如何实现稀疏激活：从 Router 到专家并行的工程权衡"
 *           (wiblog.cn): the always-on shared expert.
 *
 * Readings taken where the pages are silent (each is also a test):
 *  - TopK order and ties: experts sorted by (u descending, expert id
 *    ascending); output slot k holds the k-th of that order.
 *  - The selection bias b (optional) is added to the logits only for the
 *    selection; the softmax weights use the unbiased logits.
 *  - Capacity is ceil(T/N * capacity_factor) evaluated in double exactly as
 *    the [Infra] sec. 3.3 equation is written (no factor K); capacity_factor
 *    <= 0 means dropless (capacity = T).
 *  - Which assignments survive capacity: per expert, the first C tokens in
 *    increasing token order (dispatch scans tokens in order).
 *  - A dropped assignment contributes nothing; surviving weights are not
 *    renormalised.
 *  - f_i counts assignments before capacity, divided by T*K; P_i is the mean
 *    over tokens of the softmax over all N unbiased logits.
 *  - GELU is the erf form 0.5 v (1 + erf(v / sqrt 2)) (nn.GELU's default).
 *  - The shared expert's output enters the combine with weight 1, first.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- bf16 */

static double bf16_val(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a double to the nearest bf16 (8 significant bits, ties to even),
 * directly from the double (no intermediate float rounding). */
static uint16_t bf16_round(double v)
{
    if (isnan(v))
        return 0x7FC0;
    double a = fabs(v);
    double r;
    if (a == 0.0) {
        r = 0.0;
    } else {
        int e;
        frexp(a, &e);              /* a = m 2^e, m in [0.5, 1) */
        int E = e - 1;             /* a = 1.xxx 2^E */
        if (E < -126)
            E = -126;              /* subnormal range: fixed ulp 2^-133 */
        /* nearbyint rounds half to even under the default rounding mode */
        r = ldexp(nearbyint(ldexp(a, 7 - E)), E - 7);
        if (r >= 0x1p128)
            r = INFINITY;
    }
    float fr = (float)(signbit(v) ? -r : r); /* exact: r has <= 8 significant bits */
    uint32_t u;
    memcpy(&u, &fr, sizeof u);
    return (uint16_t)(u >> 16);
}

double oracle_bf16_value(uint16_t b) { return bf16_val(b); }
uint16_t oracle_bf16_round(double v) { return bf16_round(v); }

/* ---------------------------------------------------------------- capacity */

/* [Infra] sec. 3.3: capacity = ceil(T / N * capacity_factor). */
int oracle_capacity(int T, int N, double capacity_factor)
{
    if (capacity_factor <= 0.0)
        return T;
    double c = ceil((double)T / (double)N * capacity_factor);
    if (c > (double)T)
        c = (double)T;
    if (c < 0.0)
        c = 0.0;
    return (int)c;
}

/* ---------------------------------------------------------------- gate */

/* [Infra] sec. 2.1: logits = W_g x, one linear map with no bias.
 * s[t*N + e] = sum_j x[t, j] * Wg[e, j]. */
void oracle_gate_logits(int T, int d, int N, const uint16_t *x, const uint16_t *Wg, double *s)
{
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        for (int e = 0; e < N; ++e) {
            double acc = 0.0;
            for (int j = 0; j < d; ++j)
                acc += bf16_val(x[(size_t)t * d + j]) * bf16_val(Wg[(size_t)e * d + j]);
            s[(size_t)t * N + e] = acc;
        }
    }
}

/* ---------------------------------------------------------------- route */

typedef struct {
    double u;
    int e;
} scored_expert;

/* Sort order: larger u first; equal u -> smaller expert id first. */
static int cmp_scored(const void *pa, const void *pb)
{
    const scored_expert *a = (const scored_expert *)pa, *b = (const scored_expert *)pb;
    if (a->u > b->u)
        return -1;
    if (a->u < b->u)
        return 1;
    return (a->e > b->e) - (a->e < b->e);
}

/* [Infra] sec. 2.1 (TopK over the N logits first, then softmax over only the
 * K kept logits) and sec. 5.2 (the balance-loss statistics).
 *   s        [T, N]  unbiased gate logits
 *   sel_bias [N]     optional selection-only bias ([Yunthe], b_i), may be NULL
 * Outputs:
 *   idx      [T, K]  selected experts in rank order
 *   w        [T, K]  softmax of the K unbiased logits, stored fp32
 *   demand   [N]     number of (t, k) with idx == e (before capacity)
 *   P        [N]     mean over t of softmax over all N unbiased logits */
void oracle_route(int T, int N, int K, const double *s, const float *sel_bias,
                  int32_t *idx, float *w, int32_t *demand, double *P)
{
    scored_expert *buf = (scored_expert *)malloc(sizeof(scored_expert) * (size_t)N);
    double *ex = (double *)malloc(sizeof(double) * (size_t)N);
    for (int e = 0; e < N; ++e) {
        demand[e] = 0;
        P[e] = 0.0;
    }
    for (int t = 0; t < T; ++t) {
        const double *st = s + (size_t)t * N;
        for (int e = 0; e < N; ++e) {
            buf[e].u = st[e] + (sel_bias ? (double)sel_bias[e] : 0.0);
            buf[e].e = e;
        }
        qsort(buf, (size_t)N, sizeof(scored_expert), cmp_scored);

        /* softmax over the K kept, unbiased logits */
        double m = -INFINITY;
        for (int k = 0; k < K; ++k)
            if (st[buf[k].e] > m)
                m = st[buf[k].e];
        double z = 0.0;
        for (int k = 0; k < K; ++k)
            z += exp(st[buf[k].e] - m);
        for (int k = 0; k < K; ++k) {
            idx[(size_t)t * K + k] = buf[k].e;
            w[(size_t)t * K + k] = (float)(exp(st[buf[k].e] - m) / z);
            demand[buf[k].e] += 1;
        }

        /* softmax over all N unbiased logits, for P_i */
        double mn = -INFINITY;
        for (int e = 0; e < N; ++e)
            if (st[e] > mn)
                mn = st[e];
        double zn = 0.0;
        for (int e = 0; e < N; ++e) {
            ex[e] = exp(st[e] - mn);
            zn += ex[e];
        }
        for (int e = 0; e < N; ++e)
            P[e] += ex[e] / zn;
    }
    for (int e = 0; e < N; ++e)
        P[e] /= (double)T;
    free(ex);
    free(buf);
}

/* ---------------------------------------------------------------- dispatch */

/* [Infra] sec. 3.1 and 3.3: regroup the (token, rank) assignments into one
 * contiguous block per expert, tokens in increasing order inside a block, and
 * keep only the first C of each expert.
 * Outputs:
 *   kept    [N]      min(demand[e], C)
 *   offsets [N + 1]  exclusive prefix sum of kept (offsets[N] = rows kept, R)
 *   slot_of [T, K]   global row of assignment (t, k) in the regrouped buffer,
 *                    or -1 when it was dropped
 *   row_token [T*K]  token of each kept row (entries >= R are set to -1) */
void oracle_dispatch_ordered(int T, int N, int K, int C, int rank_major, const int32_t *idx,
                             int32_t *kept, int32_t *offsets, int32_t *slot_of, int32_t *row_token);

void oracle_dispatch(int T, int N, int K, int C, const int32_t *idx,
                     int32_t *kept, int32_t *offsets, int32_t *slot_of, int32_t *row_token)
{
    oracle_dispatch_ordered(T, N, K, C, 0, idx, kept, offsets, slot_of, row_token);
}

/* Same dispatch with a choice of priority for the capacity cut: rank_major = 0
 * scans tokens in order (t outer, k inner: the default reading); rank_major =
 * 1 scans every token's first choice before any second choice (k outer, t
 * inner), the loop order of the yunthe.com MoELayer listing's combine. */
void oracle_dispatch_ordered(int T, int N, int K, int C, int rank_major, const int32_t *idx,
                             int32_t *kept, int32_t *offsets, int32_t *slot_of, int32_t *row_token)
{
    int32_t *seen = (int32_t *)calloc((size_t)N, sizeof(int32_t));
    for (int t = 0; t < T; ++t)
        for (int k = 0; k < K; ++k)
            seen[idx[(size_t)t * K + k]] += 1;
    offsets[0] = 0;
    for (int e = 0; e < N; ++e) {
        kept[e] = seen[e] < C ? seen[e] : C;
        offsets[e + 1] = offsets[e] + kept[e];
        seen[e] = 0;
    }
    for (int r = 0; r < T * K; ++r)
        row_token[r] = -1;
    const int outer = rank_major ? K : T, inner = rank_major ? T : K;
    for (int a = 0; a < outer; ++a) {
        for (int b = 0; b < inner; ++b) {
            const int t = rank_major ? b : a, k = rank_major ? a : b;
            int e = idx[(size_t)t * K + k];
            int p = seen[e]++;
            if (p < C) {
                int row = offsets[e] + p;
                slot_of[(size_t)t * K + k] = row;
                row_token[row] = t;
            } else {
                slot_of[(size_t)t * K + k] = -1;
            }
        }
    }
    free(seen);
}

/* ---------------------------------------------------------------- expert FFN */

static double gelu_erf(double v) { return 0.5 * v * (1.0 + erf(v / sqrt(2.0))); }

double oracle_gelu(double v) { return gelu_erf(v); }

/* ---------------------------------------------------- quantised weights */

/* FP8 E4M3 (the "e4m3fn" variant: no infinities; codes 0x7f/0xff are NaN),
 * decoded from its definition: sign bit, 4 exponent bits with bias 7, 3
 * mantissa bits; exponent field 0 holds the subnormals m * 2^-9. */
static double fp8e4m3_val(uint8_t q)
{
    int sgn = q >> 7, ex = (q >> 3) & 15, man = q & 7;
    double v;
    if (ex == 15 && man == 7)
        return NAN;
    if (ex == 0)
        v = ldexp((double)man, -9);
    else
        v = ldexp(1.0 + (double)man / 8.0, ex - 7);
    return sgn ? -v : v;
}

double oracle_fp8_value(uint8_t q) { return fp8e4m3_val(q); }

/* INT4 group-wise (the 4-bit expert weights of the lmnt.cn/news/351908 sec.
 * 4.3 remark; the yunthe.com page measures a 4-bit Mixtral): 4-bit codes, the
 * eight reduction columns 8m .. 8m + 7 of a row in one little-endian 32-bit
 * word (bytes 4m .. 4m + 3 of the row's packed bytes) whose nibble j (bits
 * 4j .. 4j + 3) holds column 8m + 2j and nibble j + 4 holds column
 * 8m + 2j + 1; code c stands for the integer c - 8; one bf16 scale per output
 * row and group of 128 consecutive reduction columns. The dequantised weight
 * is (c - 8) * scale rounded to bf16 (RNE): the bf16 value the matrix product
 * consumes. */
static double int4_dequant(int code, uint16_t scale)
{
    return bf16_val(bf16_round((double)(code - 8) * bf16_val(scale)));
}

double oracle_int4_dequant(int code, uint16_t scale) { return int4_dequant(code, scale); }

/* An expert weight matrix [rows, cols] in nn.Linear layout: bf16 values, or
 * (weight-only quantisation: the lmnt.cn/news/351908 sec. 4.3 remark on
 * storing expert weights in 8 or 4 bits, and the CSDN page's sec. 3.2 FP8
 * weights at one byte per parameter) FP8 E4M3 codes with one fp32 scale per
 * row, i.e. per output channel, whose dequantised value is code * scale. */
typedef struct {
    const uint16_t *bf;
    const uint8_t *q;
    const float *scale;
    /* INT4 group-wise: codes [rows][cols / 2], scales group-major [cols / 128][rows] */
    const uint8_t *q4;
    const uint16_t *gscale;
    size_t rows;
} wmat;

static double wval(const wmat *m, size_t row, size_t col, size_t cols)
{
    if (m->q)
        return fp8e4m3_val(m->q[row * cols + col]) * (double)m->scale[row];
    if (m->q4) {
        const size_t word = col / 8, in_word = col % 8;
        const size_t nibble = in_word / 2 + 4 * (in_word % 2);
        const uint8_t byte = m->q4[row * (cols / 2) + 4 * word + nibble / 2];
        const int code = (nibble & 1) ? (byte >> 4) : (byte & 15);
        return int4_dequant(code, m->gscale[(col / 128) * m->rows + row]);
    }
    return bf16_val(m->bf[row * cols + col]);
}

/* Expert e of a stack of N matrices [N, rows, cols]. */
static wmat wexpert(const wmat *m, int e, size_t rows, size_t cols)
{
    wmat r = *m;
    if (r.q) {
        r.q += (size_t)e * rows * cols;
        r.scale += (size_t)e * rows;
    } else if (r.q4) {
        r.q4 += (size_t)e * rows * (cols / 2);
        r.gscale += (size_t)e * (cols / 128) * rows;
    } else {
        r.bf += (size_t)e * rows * cols;
    }
    return r;
}

/* ---------------------------------------------------------------- FFN */

/* [Yunthe] MoELayer listing: expert = Linear(d_model -> d_ff) -> GELU ->
 * Linear(d_ff -> d_model), nn.Linear layout [out, in] (bf16 or quantised),
 * biases fp32:
 *   h = bf16(GELU(x W1^T + b1)),   out = bf16(h W2^T + b2). */
static void ffn_row(int d, int f, const uint16_t *xrow, const wmat *W1e, const float *b1e,
                    const wmat *W2e, const float *b2e, double *xd, double *h, uint16_t *out)
{
    for (int i = 0; i < d; ++i)
        xd[i] = bf16_val(xrow[i]);
    for (int j = 0; j < f; ++j) {
        double acc = 0.0;
        for (int i = 0; i < d; ++i)
            acc += xd[i] * wval(W1e, (size_t)j, (size_t)i, (size_t)d);
        acc += (double)b1e[j];
        h[j] = bf16_val(bf16_round(gelu_erf(acc)));
    }
    for (int c = 0; c < d; ++c) {
        double acc = 0.0;
        for (int j = 0; j < f; ++j)
            acc += h[j] * wval(W2e, (size_t)c, (size_t)j, (size_t)f);
        acc += (double)b2e[c];
        out[c] = bf16_round(acc);
    }
}

/* One expert FFN on a list of rows: out[i] = E(x[rows[i]]). */
void oracle_expert_rows(int d, int f, int nrows, const int32_t *rows, const uint16_t *x,
                        const uint16_t *W1e, const float *b1e, const uint16_t *W2e,
                        const float *b2e, uint16_t *out)
{
#pragma omp parallel
    {
        double *xd = (double *)malloc(sizeof(double) * (size_t)d);
        double *h = (double *)malloc(sizeof(double) * (size_t)f);
        const wmat w1 = {W1e, NULL, NULL, NULL, NULL, 0}, w2 = {W2e, NULL, NULL, NULL, NULL, 0};
#pragma omp for schedule(dynamic, 1)
        for (int i = 0; i < nrows; ++i)
            ffn_row(d, f, x + (size_t)rows[i] * d, &w1, b1e, &w2, b2e, xd, h, out + (size_t)i * d);
        free(h);
        free(xd);
    }
}

/* The regrouped expert computation: for every kept row r of the dispatch
 * (expert e = the block r lies in, token t = row_token[r]),
 *   y_perm[r] = E_e(x[t]).
 * Rows whose token has want[t] == 0 are skipped (want may be NULL = all). */
static void expert_ffn(int d, int f, int N, const int32_t *offsets, const int32_t *row_token,
                       const uint16_t *x, const wmat *W1, const float *b1, const wmat *W2,
                       const float *b2, const uint8_t *want, uint16_t *y_perm)
{
    int R = offsets[N];
    int *row_expert = (int *)malloc(sizeof(int) * (size_t)(R > 0 ? R : 1));
    for (int e = 0; e < N; ++e)
        for (int r = offsets[e]; r < offsets[e + 1]; ++r)
            row_expert[r] = e;
#pragma omp parallel
    {
        double *xd = (double *)malloc(sizeof(double) * (size_t)d);
        double *h = (double *)malloc(sizeof(double) * (size_t)f);
#pragma omp for schedule(dynamic, 1)
        for (int r = 0; r < R; ++r) {
            int t = row_token[r];
            if (want && !want[t])
                continue;
            int e = row_expert[r];
            wmat w1 = wexpert(W1, e, (size_t)f, (size_t)d), w2 = wexpert(W2, e, (size_t)d, (size_t)f);
            ffn_row(d, f, x + (size_t)t * d, &w1, b1 + (size_t)e * f, &w2, b2 + (size_t)e * d, xd, h,
                    y_perm + (size_t)r * d);
        }
        free(h);
        free(xd);
    }
    free(row_expert);
}

void oracle_expert_ffn(int T, int d, int f, int N, const int32_t *offsets, const int32_t *row_token,
                       const uint16_t *x, const uint16_t *W1, const float *b1, const uint16_t *W2,
                       const float *b2, const uint8_t *want, uint16_t *y_perm)
{
    const wmat w1 = {W1, NULL, NULL, NULL, NULL, 0}, w2 = {W2, NULL, NULL, NULL, NULL, 0};
    (void)T;
    expert_ffn(d, f, N, offsets, row_token, x, &w1, b1, &w2, b2, want, y_perm);
}

/* The same with FP8 E4M3 expert weights: W1q[N][f][d] with scales s1[N][f],
 * W2q[N][d][f] with scales s2[N][d] (one per output channel). */
void oracle_expert_ffn_fp8(int T, int d, int f, int N, const int32_t *offsets, const int32_t *row_token,
                           const uint16_t *x, const uint8_t *W1q, const float *s1, const float *b1,
                           const uint8_t *W2q, const float *s2, const float *b2, const uint8_t *want,
                           uint16_t *y_perm)
{
    const wmat w1 = {NULL, W1q, s1, NULL, NULL, 0}, w2 = {NULL, W2q, s2, NULL, NULL, 0};
    (void)T;
    expert_ffn(d, f, N, offsets, row_token, x, &w1, b1, &w2, b2, want, y_perm);
}

/* The same with INT4 group-wise expert weights: W1q4[N][f][d / 2] with
 * scales g1[N][d / 128][f], W2q4[N][d][f / 2] with scales g2[N][f / 128][d]. */
void oracle_expert_ffn_int4(int T, int d, int f, int N, const int32_t *offsets, const int32_t *row_token,
                            const uint16_t *x, const uint8_t *W1q4, const uint16_t *g1, const float *b1,
                            const uint8_t *W2q4, const uint16_t *g2, const float *b2, const uint8_t *want,
                            uint16_t *y_perm)
{
    const wmat w1 = {NULL, NULL, NULL, W1q4, g1, (size_t)f}, w2 = {NULL, NULL, NULL, W2q4, g2, (size_t)d};
    (void)T;
    expert_ffn(d, f, N, offsets, row_token, x, &w1, b1, &w2, b2, want, y_perm);
}

/* [Wiblog] shared expert: the same FFN applied to every token (want may be NULL). */
static void shared_ffn(int T, int d, int f, const uint16_t *x, const wmat *Ws1, const float *bs1,
                       const wmat *Ws2, const float *bs2, const uint8_t *want, uint16_t *z)
{
#pragma omp parallel
    {
        double *xd = (double *)malloc(sizeof(double) * (size_t)d);
        double *h = (double *)malloc(sizeof(double) * (size_t)f);
#pragma omp for schedule(dynamic, 1)
        for (int t = 0; t < T; ++t) {
            if (want && !want[t])
                continue;
            ffn_row(d, f, x + (size_t)t * d, Ws1, bs1, Ws2, bs2, xd, h, z + (size_t)t * d);
        }
        free(h);
        free(xd);
    }
}

void oracle_shared_ffn(int T, int d, int f, const uint16_t *x, const uint16_t *Ws1, const float *bs1,
                       const uint16_t *Ws2, const float *bs2, const uint8_t *want, uint16_t *z)
{
    const wmat w1 = {Ws1, NULL, NULL, NULL, NULL, 0}, w2 = {Ws2, NULL, NULL, NULL, NULL, 0};
    shared_ffn(T, d, f, x, &w1, bs1, &w2, bs2, want, z);
}

void oracle_shared_ffn_fp8(int T, int d, int f, const uint16_t *x, const uint8_t *Ws1q, const float *ss1,
                           const float *bs1, const uint8_t *Ws2q, const float *ss2, const float *bs2,
                           const uint8_t *want, uint16_t *z)
{
    const wmat w1 = {NULL, Ws1q, ss1, NULL, NULL, 0}, w2 = {NULL, Ws2q, ss2, NULL, NULL, 0};
    shared_ffn(T, d, f, x, &w1, bs1, &w2, bs2, want, z);
}

void oracle_shared_ffn_int4(int T, int d, int f, const uint16_t *x, const uint8_t *Ws1q4, const uint16_t *gs1,
                            const float *bs1, const uint8_t *Ws2q4, const uint16_t *gs2, const float *bs2,
                            const uint8_t *want, uint16_t *z)
{
    const wmat w1 = {NULL, NULL, NULL, Ws1q4, gs1, (size_t)f}, w2 = {NULL, NULL, NULL, Ws2q4, gs2, (size_t)d};
    shared_ffn(T, d, f, x, &w1, bs1, &w2, bs2, want, z);
}

/* ---------------------------------------------------------------- combine */

/* [Infra] sec. 3.2: output[t] = sum_{e in selected(t)} weight[t, e] *
 * expert_output_e, read back through the dispatch table in the same (rank)
 * order the dispatch used. Dropped assignments (slot -1) add nothing. The
 * shared expert's output, when given, enters first with weight 1. */
void oracle_combine(int T, int d, int K, const uint16_t *y_perm, const int32_t *slot_of,
                    const float *w, const uint16_t *z, const uint8_t *want, uint16_t *y)
{
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        if (want && !want[t])
            continue;
        for (int c = 0; c < d; ++c) {
            double acc = z ? bf16_val(z[(size_t)t * d + c]) : 0.0;
            for (int k = 0; k < K; ++k) {
                int r = slot_of[(size_t)t * K + k];
                if (r < 0)
                    continue;
                acc += (double)w[(size_t)t * K + k] * bf16_val(y_perm[(size_t)r * d + c]);
            }
            y[(size_t)t * d + c] = bf16_round(acc);
        }
    }
}

/* ---------------------------------------------------------------- router health */

/* Router health statistics the pages monitor (lmnt.cn/news/351908 sec. 8.2
 * and 9.3: tokens per expert, mean routing weight per expert, token drop
 * rate, gate logit range; the CSDN page's sec. 3.3 expert_util_std):
 *   h[0] util_std     population std over experts of f_e = demand_e / (T K)
 *   h[1] drop_rate    fraction of the T K assignments dropped by capacity
 *   h[2] entropy      mean over tokens of the entropy (nats) of softmax_N(s_t)
 *   h[3] max |s|      largest gate logit magnitude
 *   mean_w[e]         mean routing weight of the assignments to e (0 if none) */
void oracle_health(int T, int N, int K, const double *s, const int32_t *demand, const int32_t *kept,
                   const int32_t *idx, const float *w, double *h, double *mean_w)
{
    const double TK = (double)T * (double)K;
    double mean = 0.0, var = 0.0;
    for (int e = 0; e < N; ++e)
        mean += (double)demand[e] / TK;
    mean /= (double)N;
    for (int e = 0; e < N; ++e) {
        const double df = (double)demand[e] / TK - mean;
        var += df * df;
    }
    h[0] = sqrt(var / (double)N);
    double kept_all = 0.0;
    for (int e = 0; e < N; ++e)
        kept_all += (double)kept[e];
    h[1] = 1.0 - kept_all / TK;
    double ent = 0.0, amax = 0.0;
    for (int t = 0; t < T; ++t) {
        const double *st = s + (size_t)t * N;
        double m = -INFINITY, z = 0.0;
        for (int e = 0; e < N; ++e)
            m = fmax(m, st[e]);
        for (int e = 0; e < N; ++e)
            z += exp(st[e] - m);
        for (int e = 0; e < N; ++e) {
            const double p = exp(st[e] - m) / z;
            if (p > 0.0)
                ent -= p * log(p);
            amax = fmax(amax, fabs(st[e]));
        }
    }
    h[2] = ent / (double)T;
    h[3] = amax;
    for (int e = 0; e < N; ++e)
        mean_w[e] = 0.0;
    for (int t = 0; t < T; ++t)
        for (int k = 0; k < K; ++k)
            mean_w[idx[(size_t)t * K + k]] += (double)w[(size_t)t * K + k];
    for (int e = 0; e < N; ++e)
        mean_w[e] = demand[e] > 0 ? mean_w[e] / (double)demand[e] : 0.0;
}

/* ---------------------------------------------------------------- backward */

static double gelu_grad(double v)
{
    /* d/dv [v Phi(v)] = Phi(v) + v phi(v) */
    const double phi = exp(-0.5 * v * v) / sqrt(2.0 * 3.14159265358979323846);
    return 0.5 * (1.0 + erf(v / sqrt(2.0))) + v * phi;
}

/* One expert row, forward then backward:
 *   a = x W1^T + b1, h = bf16(GELU(a)), o = bf16(h W2^T + b2)   (as the forward)
 *   dw = <dy, o> (returned);  dO = wgt * dy
 *   dh = dO W2,  da = dh * GELU'(a)
 *   dW2 += dO^T h,  db2 += dO,  dW1 += da^T x,  db1 += da,  dxrow = da W1
 * With round_stored, dO and da are rounded to bf16 (the values the GPU keeps
 * between its GEMMs). wgt = 1 and no dw for the shared expert. */
static double expert_row_backward(int d, int f, const uint16_t *xrow, const uint16_t *W1e, const float *b1e,
                                  const uint16_t *W2e, const float *b2e, const uint16_t *dyrow, double wgt,
                                  int round_stored, double *a, double *h, double *dO, double *dh,
                                  double *dW1e, double *db1e, double *dW2e, double *db2e, double *dxrow)
{
    for (int j = 0; j < f; ++j) {
        double acc = 0.0;
        for (int i = 0; i < d; ++i)
            acc += bf16_val(xrow[i]) * bf16_val(W1e[(size_t)j * d + i]);
        a[j] = acc + (double)b1e[j];
        h[j] = bf16_val(bf16_round(gelu_erf(a[j])));
    }
    double dw = 0.0;
    for (int c = 0; c < d; ++c) {
        double acc = 0.0;
        for (int j = 0; j < f; ++j)
            acc += h[j] * bf16_val(W2e[(size_t)c * f + j]);
        const double o = bf16_val(bf16_round(acc + (double)b2e[c]));
        const double g = bf16_val(dyrow[c]);
        dw += g * o;
        dO[c] = round_stored ? bf16_val(bf16_round(wgt * g)) : wgt * g;
    }
    for (int j = 0; j < f; ++j) {
        double acc = 0.0;
        for (int c = 0; c < d; ++c)
            acc += dO[c] * bf16_val(W2e[(size_t)c * f + j]);
        double da = acc * gelu_grad(a[j]);
        if (round_stored)
            da = bf16_val(bf16_round(da));
        dh[j] = da;
    }
    if (dW2e) {  /* NULL: only dx and dw wanted */
        for (int c = 0; c < d; ++c) {
            db2e[c] += dO[c];
            for (int j = 0; j < f; ++j)
                dW2e[(size_t)c * f + j] += dO[c] * h[j];
        }
    }
    for (int i = 0; i < d; ++i)
        dxrow[i] = 0.0;
    for (int j = 0; j < f; ++j) {
        if (dW1e)
            db1e[j] += dh[j];
        for (int i = 0; i < d; ++i) {
            if (dW1e)
                dW1e[(size_t)j * d + i] += dh[j] * bf16_val(xrow[i]);
            dxrow[i] += dh[j] * bf16_val(W1e[(size_t)j * d + i]);
        }
    }
    return dw;
}

/* Routing weights in double: softmax over the K selected, unbiased logits
 * ([Infra] sec. 2.1), w[t*K + k] for the expert in slot k. */
static void routing_weights(int T, int N, int K, const double *s, const int32_t *idx, double *w)
{
    for (int t = 0; t < T; ++t) {
        double m = -INFINITY, z = 0.0;
        for (int k = 0; k < K; ++k)
            m = fmax(m, s[(size_t)t * N + idx[(size_t)t * K + k]]);
        for (int k = 0; k < K; ++k)
            z += exp(s[(size_t)t * N + idx[(size_t)t * K + k]] - m);
        for (int k = 0; k < K; ++k)
            w[(size_t)t * K + k] = exp(s[(size_t)t * N + idx[(size_t)t * K + k]] - m) / z;
    }
}

/* Gradient of the loss with respect to the gate logits, ds [T, N], for the
 * tokens with want[t] != 0 (want may be NULL = all; other rows are left as
 * they are):
 *   ds_t[e] = w_te (dw_te - sum_k w_tk dw_tk) on the TopK set (softmax over
 *             the K kept logits, [Infra] sec. 2.1)
 *           + g_aux alpha N / T p_te (f_e - sum_e' f_e' p_te')   ([Infra] sec. 5.2,
 *             f = demand / (T K) held constant, p_t = softmax over all N)
 *           + g_z 2 beta / T lse_t p_te                           ([Infra] sec. 5.3). */
static void gate_logit_grads(int T, int N, int K, const double *s, const int32_t *idx, const double *w,
                             const double *dw_out, const int32_t *demand, double alpha, double beta,
                             double g_aux, double g_z, const uint8_t *want, double *ds)
{
    const double TK = (double)T * (double)K;
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        if (want && !want[t])
            continue;
        const double *st = s + (size_t)t * N;
        double *dst = ds + (size_t)t * N;
        double m = -INFINITY, z = 0.0;
        for (int e = 0; e < N; ++e)
            m = fmax(m, st[e]);
        for (int e = 0; e < N; ++e)
            z += exp(st[e] - m);
        const double lse = m + log(z);
        double fp = 0.0;
        for (int e = 0; e < N; ++e)
            fp += ((double)demand[e] / TK) * exp(st[e] - m) / z;
        for (int e = 0; e < N; ++e) {
            const double p = exp(st[e] - m) / z;
            dst[e] = g_aux * alpha * (double)N / (double)T * p * ((double)demand[e] / TK - fp)
                   + g_z * 2.0 * beta / (double)T * lse * p;
        }
        double sdw = 0.0;
        for (int k = 0; k < K; ++k)
            sdw += w[(size_t)t * K + k] * dw_out[(size_t)t * K + k];
        for (int k = 0; k < K; ++k)
            dst[idx[(size_t)t * K + k]] += w[(size_t)t * K + k] * (dw_out[(size_t)t * K + k] - sdw);
    }
}

/* dW_g[e, :] = sum_t ds[t, e] x[t, :] (written, not accumulated into). */
static void gate_weight_grads(int T, int d, int N, const double *ds, const uint16_t *x, double *dWg)
{
    memset(dWg, 0, sizeof(double) * (size_t)N * d);
#pragma omp parallel for schedule(dynamic, 1)
    for (int e = 0; e < N; ++e)
        for (int t = 0; t < T; ++t) {
            const double g = ds[(size_t)t * N + e];
            if (g == 0.0)
                continue;
            for (int i = 0; i < d; ++i)
                dWg[(size_t)e * d + i] += g * bf16_val(x[(size_t)t * d + i]);
        }
}

/* Gradients of the layer given the upstream gradient dy of y and weights
 * g_aux, g_z on the balance loss and the router z-loss (the training signal
 * the pages build around; [Infra] sec. 5). The TopK sets, the capacity drops
 * and the dispatch are the forward's: piecewise constant, so nothing flows
 * through the selection, the selection bias, the drops or the KL variant (a
 * function of the counts). With y_t = z_t + sum_k w_tk o_tk:
 *   dw_tk = <dy_t, o_tk> (0 when dropped), dO = w_tk dy_t into the expert;
 *   gate: ds_t[e] = w_te (dw_te - sum_k w_tk dw_tk) for e in the TopK set
 *         (softmax over the K kept logits, [Infra] sec. 2.1)
 *       + g_aux alpha N / T * p_te (f_e - sum_e' f_e' p_te')   (aux = alpha N sum f P,
 *         P_e = mean_t p_te with p_t = softmax over all N, f = demand / (T K) constant)
 *       + g_z 2 beta / T * lse_t p_te                          (z-loss, [Infra] sec. 5.3)
 *   dW_g = sum_t ds_t^T x_t,  dx_t += ds_t W_g;  the shared expert gets dO = dy.
 * s: the forward's logits [T, N]; idx, slot_of [T, K]; offsets [N + 1];
 * row_token [T K]; demand [N]; dy [T, d] bf16. Outputs (double, written, not
 * accumulated into): dx [T, d], dWg [N, d], dW1 [N, f, d], db1 [N, f],
 * dW2 [N, d, f], db2 [N, d], the shared expert's (when Ws1 != NULL) and
 * dw [T, K]. want (may be NULL = all): only tokens with want[t] != 0 get dx
 * and dw, and no weight or bias gradient is formed (those outputs may then be
 * NULL). */
void oracle_backward(int T, int d, int f, int N, int K, const uint16_t *x, const uint16_t *Wg,
                     const uint16_t *W1, const float *b1, const uint16_t *W2, const float *b2,
                     const uint16_t *Ws1, const float *bs1, const uint16_t *Ws2, const float *bs2,
                     const double *s, const int32_t *idx, const int32_t *slot_of, const int32_t *offsets,
                     const int32_t *row_token, const int32_t *demand, const uint16_t *dy, double alpha,
                     double beta, double g_aux, double g_z, int round_stored, const uint8_t *want, double *dx,
                     double *dWg, double *dW1, double *db1, double *dW2, double *db2, double *dWs1, double *dbs1,
                     double *dWs2, double *dbs2, double *dw_out)
{
    const int R = offsets[N];
    double *w = (double *)calloc((size_t)T * K, sizeof(double));
    double *dx_perm = (double *)calloc((size_t)(R > 0 ? R : 1) * d, sizeof(double));
    double *dx_shared = Ws1 ? (double *)calloc((size_t)T * d, sizeof(double)) : NULL;
    int *slot_k = (int *)malloc(sizeof(int) * (size_t)(R > 0 ? R : 1));

    routing_weights(T, N, K, s, idx, w);
    for (int t = 0; t < T; ++t) {
        for (int k = 0; k < K; ++k) {
            int r = slot_of[(size_t)t * K + k];
            if (r >= 0)
                slot_k[r] = k;
        }
    }
    const int weights = want == NULL;
    if (weights) {
        memset(dW1, 0, sizeof(double) * (size_t)N * f * d);
        memset(db1, 0, sizeof(double) * (size_t)N * f);
        memset(dW2, 0, sizeof(double) * (size_t)N * d * f);
        memset(db2, 0, sizeof(double) * (size_t)N * d);
    }
    for (size_t i = 0; i < (size_t)T * K; ++i)
        dw_out[i] = 0.0;

    /* routed experts: one thread per expert owns its weight gradients */
#pragma omp parallel
    {
        double *a = (double *)malloc(sizeof(double) * (size_t)f);
        double *h = (double *)malloc(sizeof(double) * (size_t)f);
        double *dO = (double *)malloc(sizeof(double) * (size_t)d);
        double *dh = (double *)malloc(sizeof(double) * (size_t)f);
#pragma omp for schedule(dynamic, 1)
        for (int e = 0; e < N; ++e) {
            for (int r = offsets[e]; r < offsets[e + 1]; ++r) {
                const int t = row_token[r], k = slot_k[r];
                if (want && !want[t])
                    continue;
                const double wgt = w[(size_t)t * K + k];
                dw_out[(size_t)t * K + k] = expert_row_backward(
                    d, f, x + (size_t)t * d, W1 + (size_t)e * f * d, b1 + (size_t)e * f, W2 + (size_t)e * d * f,
                    b2 + (size_t)e * d, dy + (size_t)t * d, wgt, round_stored, a, h, dO, dh,
                    weights ? dW1 + (size_t)e * f * d : NULL, weights ? db1 + (size_t)e * f : NULL,
                    weights ? dW2 + (size_t)e * d * f : NULL, weights ? db2 + (size_t)e * d : NULL,
                    dx_perm + (size_t)r * d);
            }
        }
        free(dh);
        free(dO);
        free(h);
        free(a);
    }

    /* shared expert: weight 1 on every token */
    if (Ws1) {
        if (weights) {
            memset(dWs1, 0, sizeof(double) * (size_t)f * d);
            memset(dbs1, 0, sizeof(double) * (size_t)f);
            memset(dWs2, 0, sizeof(double) * (size_t)d * f);
            memset(dbs2, 0, sizeof(double) * (size_t)d);
        }
        double *a = (double *)malloc(sizeof(double) * (size_t)f);
        double *h = (double *)malloc(sizeof(double) * (size_t)f);
        double *dO = (double *)malloc(sizeof(double) * (size_t)d);
        double *dh = (double *)malloc(sizeof(double) * (size_t)f);
        for (int t = 0; t < T; ++t)
            if (!want || want[t])
                (void)expert_row_backward(d, f, x + (size_t)t * d, Ws1, bs1, Ws2, bs2, dy + (size_t)t * d, 1.0,
                                          round_stored, a, h, dO, dh, weights ? dWs1 : NULL, weights ? dbs1 : NULL,
                                          weights ? dWs2 : NULL, weights ? dbs2 : NULL, dx_shared + (size_t)t * d);
        free(dh);
        free(dO);
        free(h);
        free(a);
    }

    /* gate and the token gradient */
    double *ds = (double *)calloc((size_t)T * N, sizeof(double));
    gate_logit_grads(T, N, K, s, idx, w, dw_out, demand, alpha, beta, g_aux, g_z, want, ds);
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        if (want && !want[t])
            continue;
        const double *dst = ds + (size_t)t * N;
        double *dxt = dx + (size_t)t * d;
        for (int i = 0; i < d; ++i) {
            double acc = dx_shared ? dx_shared[(size_t)t * d + i] : 0.0;
            for (int k = 0; k < K; ++k) {
                int r = slot_of[(size_t)t * K + k];
                if (r >= 0)
                    acc += dx_perm[(size_t)r * d + i];
            }
            for (int e = 0; e < N; ++e)
                acc += dst[e] * bf16_val(Wg[(size_t)e * d + i]);
            dxt[i] = acc;
        }
    }
    if (weights)
        gate_weight_grads(T, d, N, ds, x, dWg);
    free(ds);
    free(slot_k);
    free(dx_shared);
    free(dx_perm);
    free(w);
}

/* Pieces of the backward for full-size checks, each the same arithmetic as
 * oracle_backward (which calls the same helpers) restricted to one part. */

/* dw_tk = <dy_t, o_tk>: the combine's gradient with respect to the routing
 * weight of slot k ([Infra] sec. 3.2 combine equation), from the forward's
 * stored expert outputs y_perm [R, d] (bf16); 0 for a dropped slot. */
void oracle_combine_backward(int T, int d, int K, const uint16_t *dy, const uint16_t *y_perm,
                             const int32_t *slot_of, double *dw)
{
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t)
        for (int k = 0; k < K; ++k) {
            const int r = slot_of[(size_t)t * K + k];
            double dot = 0.0;
            if (r >= 0)
                for (int c = 0; c < d; ++c)
                    dot += bf16_val(dy[(size_t)t * d + c]) * bf16_val(y_perm[(size_t)r * d + c]);
            dw[(size_t)t * K + k] = dot;
        }
}

/* dW_g [N, d] from the slot gradients dw [T, K] (see gate_logit_grads). */
void oracle_gate_backward(int T, int d, int N, int K, const uint16_t *x, const double *s, const int32_t *idx,
                          const double *dw, const int32_t *demand, double alpha, double beta, double g_aux,
                          double g_z, double *dWg)
{
    double *w = (double *)malloc(sizeof(double) * (size_t)T * K);
    double *ds = (double *)calloc((size_t)T * N, sizeof(double));
    routing_weights(T, N, K, s, idx, w);
    gate_logit_grads(T, N, K, s, idx, w, dw, demand, alpha, beta, g_aux, g_z, NULL, ds);
    gate_weight_grads(T, d, N, ds, x, dWg);
    free(ds);
    free(w);
}

/* Weight and bias gradients of ONE expert: routed expert e >= 0 (its rows
 * [offsets[e], offsets[e+1]), token row_token[r], routing weight from the
 * logits), or the shared expert for e < 0 (every token, weight 1). W1e [f, d],
 * b1e [f], W2e [d, f], b2e [d] are that expert's. Every row is first taken
 * through expert_row_backward (the backward's own per-row step: h, dO, da),
 * then the sums over the rows are formed one output row at a time:
 *   dW2e[c, :] = sum_r dO[r, c] h[r, :],  db2e[c] = sum_r dO[r, c],
 *   dW1e[j, :] = sum_r da[r, j] x[t_r, :], db1e[j] = sum_r da[r, j]. */
void oracle_expert_backward(int T, int d, int f, int N, int K, int e, const double *s, const int32_t *idx,
                            const int32_t *slot_of, const int32_t *offsets, const int32_t *row_token,
                            const uint16_t *x, const uint16_t *W1e, const float *b1e, const uint16_t *W2e,
                            const float *b2e, const uint16_t *dy, int round_stored, double *dW1e, double *db1e,
                            double *dW2e, double *db2e)
{
    const int n = e >= 0 ? offsets[e + 1] - offsets[e] : T;
    int *tok = (int *)malloc(sizeof(int) * (size_t)(n > 0 ? n : 1));
    double *wgt = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    if (e >= 0) {
        double *w = (double *)malloc(sizeof(double) * (size_t)T * K);
        routing_weights(T, N, K, s, idx, w);
        for (int t = 0; t < T; ++t)
            for (int k = 0; k < K; ++k) {
                const int r = slot_of[(size_t)t * K + k];
                if (r >= offsets[e] && r < offsets[e + 1]) {
                    tok[r - offsets[e]] = t;
                    wgt[r - offsets[e]] = w[(size_t)t * K + k];
                }
            }
        free(w);
    } else {
        for (int t = 0; t < T; ++t) {
            tok[t] = t;
            wgt[t] = 1.0;
        }
    }
    (void)row_token;
    double *H = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * f);
    double *DO = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * d);
    double *DA = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * f);
#pragma omp parallel
    {
        double *a = (double *)malloc(sizeof(double) * (size_t)f);
        double *dxrow = (double *)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(dynamic, 1)
        for (int i = 0; i < n; ++i)
            (void)expert_row_backward(d, f, x + (size_t)tok[i] * d, W1e, b1e, W2e, b2e, dy + (size_t)tok[i] * d,
                                      wgt[i], round_stored, a, H + (size_t)i * f, DO + (size_t)i * d,
                                      DA + (size_t)i * f, NULL, NULL, NULL, NULL, dxrow);
        free(dxrow);
        free(a);
    }
#pragma omp parallel for schedule(static)
    for (int c = 0; c < d; ++c) {
        double *out = dW2e + (size_t)c * f;
        double bsum = 0.0;
        for (int j = 0; j < f; ++j)
            out[j] = 0.0;
        for (int i = 0; i < n; ++i) {
            const double g = DO[(size_t)i * d + c];
            const double *hi = H + (size_t)i * f;
            bsum += g;
            for (int j = 0; j < f; ++j)
                out[j] += g * hi[j];
        }
        db2e[c] = bsum;
    }
#pragma omp parallel for schedule(static)
    for (int j = 0; j < f; ++j) {
        double *out = dW1e + (size_t)j * d;
        double bsum = 0.0;
        for (int q = 0; q < d; ++q)
            out[q] = 0.0;
        for (int i = 0; i < n; ++i) {
            const double g = DA[(size_t)i * f + j];
            const uint16_t *xi = x + (size_t)tok[i] * d;
            bsum += g;
            for (int q = 0; q < d; ++q)
                out[q] += g * bf16_val(xi[q]);
        }
        db1e[j] = bsum;
    }
    free(DA);
    free(DO);
    free(H);
    free(wgt);
    free(tok);
}

/* ---------------------------------------------------------------- KL balance loss */

/* "MoE逐token路由与活跃参数率实战解析" sec. 3.1 and its MoELayer listing: the
 * per-expert frequency f_e = demand_e / (T K) is compared with the uniform
 * distribution, loss = coef * KL(U || f) = coef * sum_e (1/N) (log(1/N) -
 * log f_e) (what F.kl_div(f.log(), uniform, reduction='sum') evaluates).
 * An expert with no assignment makes the loss +infinity. */
double oracle_aux_kl(int T, int N, int K, double coef, const int32_t *demand)
{
    double acc = 0.0;
    const double u = 1.0 / (double)N;
    for (int e = 0; e < N; ++e) {
        double f = (double)demand[e] / ((double)T * (double)K);
        acc += u * (log(u) - log(f));
    }
    return coef * acc;
}

/* ---------------------------------------------------------------- router z-loss */

/* [Infra] sec. 5.3 (z-loss equation and its code): L_z = beta * (1/T) *
 * sum_t (log sum_i exp(s[t, i]))^2 over the unbiased logits. The log-sum-exp
 * is evaluated as m + log(sum exp(s - m)) with m the row maximum. */
double oracle_z_loss(int T, int N, const double *s, double beta)
{
    double acc = 0.0;
    for (int t = 0; t < T; ++t) {
        const double *st = s + (size_t)t * N;
        double m = -INFINITY;
        for (int e = 0; e < N; ++e)
            if (st[e] > m)
                m = st[e];
        double z = 0.0;
        for (int e = 0; e < N; ++e)
            z += exp(st[e] - m);
        double lse = m + log(z);
        acc += lse * lse;
    }
    return beta * acc / (double)T;
}

/* ---------------------------------------------------------------- balance loss */

/* [Infra] sec. 5.1-5.2: L = alpha * N * sum_i f_i P_i with
 * f_i = demand_i / (T K) and P_i the mean softmax probability of expert i. */
double oracle_aux_loss(int T, int N, int K, double alpha, const int32_t *demand, const double *P)
{
    double acc = 0.0;
    for (int e = 0; e < N; ++e)
        acc += ((double)demand[e] / ((double)T * (double)K)) * P[e];
    return alpha * (double)N * acc;
}
