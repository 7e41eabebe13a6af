/*
 * Float64 CPU oracle for the differential-attention head forward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may load, link or
 * call this file.  Its only users are the tests under tests/, the smoke()
 * check in __graft_entry__.py and the cpu_baseline / reference leg of
 * bench.py.  It shares no code, header, table or constant with the CUDA
 * library, and it includes nothing from it.
 *
 * What it computes (source: "Differential Transformer", Ultralytics glossary,
 * section "How differential attention works"; the Japanese, Portuguese and
 * Arabic editions of that page say the same thing):
 *
 *   map1 = softmax over keys of (Q1 K1^T / sqrt(d))
 *   map2 = softmax over keys of (Q2 K2^T / sqrt(d))
 *   out  = (map1 - lambda * map2) V            V has 2d columns
 *
 * followed, in the real model (same section, closing paragraph), by a
 * per-head normalisation of each head's output and a multiplication by
 * (1 - lambda_init), with lambda_init(l) = 0.8 - 0.6 exp(-0.3 (l - 1)).
 *
 * Readings of what the page leaves open (each is listed with its reason in
 * the design notes of this repository):
 *   - d in the 1/sqrt(d) scale is the width of one query/key half, as in the
 *     page's worked example (n = 6, d = 8, v of width 2d).
 *   - causal = 1 means key j is visible to query i iff j <= i (square,
 *     top-left aligned); the same mask is applied to both maps.  With fewer
 *     queries than keys (a key/value cache), the queries are the last
 *     positions of the sequence, so the mask is aligned bottom-right.
 *   - the per-head normalisation (headnorm = 1) is the RMS form over the 2d
 *     output channels of one (batch, head, token): y = o / sqrt(mean(o^2) +
 *     eps) * w[h, c], then times (1 - lambda_init).  No mean subtraction, no
 *     bias.  headnorm = 2 is the mean-subtracting form the page names
 *     (GroupNorm, one group per head), also without bias.
 *   - layers are numbered from 1 (the formula uses l - 1; l = 1 gives 0.2).
 *
 * The code is deliberately plain: one query row at a time, both maps
 * materialised in full for that row, max-subtracted softmax, no blocking, no
 * fusion, no reordering.  All arithmetic is IEEE float64.  Rows are
 * independent, so OpenMP spreads whole rows over host cores; that changes
 * nothing in any row's arithmetic.
 *
 * Tensor layout: q1, k1, q2, k2 are [B, H, N, d] and v, out are [B, H, N, 2d],
 * all contiguous row-major float64 (oracle_fwd_kv_rows: Nq query rows, Nkv
 * key and value rows).  lambda is [H]; w is [H, 2d] or NULL
 * (meaning all ones).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* lambda_init(l) = 0.8 - 0.6 * exp(-0.3 * (l - 1)); "Differential
 * Transformer", section "How differential attention works", last paragraph. */
double oracle_lambda_init(int layer)
{
    return 0.8 - 0.6 * exp(-0.3 * (double)(layer - 1));
}

/* Is key j visible to query i?  Causal reading: j <= i. */
static int visible(int64_t i, int64_t j, int causal)
{
    return causal ? (j <= i) : 1;
}

/* One softmax row over the visible keys: logits s[j] = (q . k_j) / sqrt(d),
 * p[j] = exp(s[j] - max) / sum.  Invisible keys get weight exactly 0. */
static void softmax_row(int64_t i, int64_t N, int d, const double *q_row,
                        const double *k, int causal, double *p)
{
    const double scale = 1.0 / sqrt((double)d);
    double mx = -INFINITY;
    for (int64_t j = 0; j < N; ++j) {
        if (!visible(i, j, causal)) {
            p[j] = -INFINITY;
            continue;
        }
        double s = 0.0;
        for (int c = 0; c < d; ++c)
            s += q_row[c] * k[j * d + c];
        p[j] = s * scale;
        if (p[j] > mx)
            mx = p[j];
    }
    double sum = 0.0;
    for (int64_t j = 0; j < N; ++j) {
        if (!visible(i, j, causal)) {
            p[j] = 0.0;
            continue;
        }
        p[j] = exp(p[j] - mx);
        sum += p[j];
    }
    for (int64_t j = 0; j < N; ++j)
        p[j] /= sum;
}

/* Row of the differential map for the query at position i (query vectors
 * q1_row, q2_row) against N keys: w[j] = map1[i][j] - lambda * map2[i][j].
 * Scratch p1, p2 hold N doubles each. */
static void diff_row(int64_t i, int64_t N, int d, const double *q1_row,
                     const double *k1, const double *q2_row, const double *k2,
                     double lam, int causal, double *p1, double *p2, double *w)
{
    softmax_row(i, N, d, q1_row, k1, causal, p1);
    softmax_row(i, N, d, q2_row, k2, causal, p2);
    for (int64_t j = 0; j < N; ++j)
        w[j] = p1[j] - lam * p2[j];
}

/* The page's own wording for the per-head normalisation is GroupNorm with one
 * group per head: subtract the row mean over the 2d channels, divide by the
 * square root of the (biased) variance plus eps, multiply by the per-channel
 * weight, then by (1 - lambda_init).  No bias (headnorm = 2). */
static void group_norm_row(double *o, int dv, const double *w_head, double eps,
                           double lambda_init)
{
    double mu = 0.0;
    for (int c = 0; c < dv; ++c)
        mu += o[c];
    mu /= (double)dv;
    double var = 0.0;
    for (int c = 0; c < dv; ++c)
        var += (o[c] - mu) * (o[c] - mu);
    var /= (double)dv;
    const double rg = 1.0 / sqrt(var + eps);
    for (int c = 0; c < dv; ++c) {
        const double g = w_head ? w_head[c] : 1.0;
        o[c] = (o[c] - mu) * rg * g * (1.0 - lambda_init);
    }
}

/* out_row = (map1 - lambda map2)[i, :] V for the query at position i with
 * vectors q1_row, q2_row against N keys, then optionally the per-head RMS
 * normalisation and the (1 - lambda_init) scale. */
static void out_row(int64_t i, int64_t N, int d, const double *q1_row,
                    const double *k1, const double *q2_row, const double *k2,
                    const double *v, double lam, int causal, int headnorm,
                    const double *w_head, double eps, double lambda_init,
                    double *scratch, double *o)
{
    double *p1 = scratch, *p2 = scratch + N, *wrow = scratch + 2 * N;
    const int dv = 2 * d;
    diff_row(i, N, d, q1_row, k1, q2_row, k2, lam, causal, p1, p2, wrow);
    for (int c = 0; c < dv; ++c)
        o[c] = 0.0;
    for (int64_t j = 0; j < N; ++j)
        for (int c = 0; c < dv; ++c)
            o[c] += wrow[j] * v[j * dv + c];
    if (!headnorm)
        return;
    if (headnorm == 2) {
        group_norm_row(o, dv, w_head, eps, lambda_init);
        return;
    }
    double ms = 0.0;
    for (int c = 0; c < dv; ++c)
        ms += o[c] * o[c];
    ms /= (double)dv;
    const double r = 1.0 / sqrt(ms + eps);
    for (int c = 0; c < dv; ++c) {
        const double g = w_head ? w_head[c] : 1.0;
        o[c] = o[c] * r * g * (1.0 - lambda_init);
    }
}

static void set_threads(int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

/* Number of host threads OpenMP will use for the next parallel region. */
int oracle_max_threads(int nthreads)
{
    set_threads(nthreads);
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Full forward: every (b, h, i).  Returns 0 on success, -1 on bad arguments,
 * -2 if scratch could not be allocated. */
int oracle_fwd(int B, int H, int64_t N, int d, const double *q1,
               const double *k1, const double *q2, const double *k2,
               const double *v, const double *lam, int causal, int headnorm,
               const double *w, double eps, double lambda_init, double *out,
               int nthreads)
{
    if (B < 0 || H < 0 || N < 0 || d <= 0)
        return -1;
    const int64_t BH = (int64_t)B * H;
    const int dv = 2 * d;
    int err = 0;
    set_threads(nthreads);
#pragma omp parallel
    {
        double *scratch = (double *)malloc(sizeof(double) * (size_t)(3 * N + 1));
        if (!scratch) {
#pragma omp atomic write
            err = -2;
        }
#pragma omp for schedule(dynamic, 16)
        for (int64_t r = 0; r < BH * N; ++r) {
            if (!scratch)
                continue;
            const int64_t bh = r / N, i = r % N;
            const int h = (int)(bh % H);
            const int64_t qk = bh * N * d, vo = bh * N * dv;
            out_row(i, N, d, q1 + qk + i * d, k1 + qk, q2 + qk + i * d, k2 + qk, v + vo,
                    lam[h], causal, headnorm, w ? w + (int64_t)h * dv : NULL,
                    eps, lambda_init, scratch, out + vo + i * dv);
        }
        free(scratch);
    }
    return err;
}

/* Selected rows only: for r in [0, nrows), compute the output row of head
 * bh_idx[r] (a flat b*H + h index) and query row_idx[r] into
 * out_rows[r * 2d .. r * 2d + 2d).  Same arithmetic as oracle_fwd. */
int oracle_fwd_rows(int B, int H, int64_t N, int d, const double *q1,
                    const double *k1, const double *q2, const double *k2,
                    const double *v, const double *lam, int causal,
                    int headnorm, const double *w, double eps,
                    double lambda_init, int64_t nrows, const int64_t *bh_idx,
                    const int64_t *row_idx, double *out_rows, int nthreads)
{
    if (B < 0 || H < 0 || N < 0 || d <= 0 || nrows < 0)
        return -1;
    const int64_t BH = (int64_t)B * H;
    for (int64_t r = 0; r < nrows; ++r)
        if (bh_idx[r] < 0 || bh_idx[r] >= BH || row_idx[r] < 0 || row_idx[r] >= N)
            return -1;
    const int dv = 2 * d;
    int err = 0;
    set_threads(nthreads);
#pragma omp parallel
    {
        double *scratch = (double *)malloc(sizeof(double) * (size_t)(3 * N + 1));
        if (!scratch) {
#pragma omp atomic write
            err = -2;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < nrows; ++r) {
            if (!scratch)
                continue;
            const int64_t bh = bh_idx[r], i = row_idx[r];
            const int h = (int)(bh % H);
            const int64_t qk = bh * N * d, vo = bh * N * dv;
            out_row(i, N, d, q1 + qk + i * d, k1 + qk, q2 + qk + i * d, k2 + qk, v + vo,
                    lam[h], causal, headnorm, w ? w + (int64_t)h * dv : NULL,
                    eps, lambda_init, scratch, out_rows + r * dv);
        }
        free(scratch);
    }
    return err;
}

/* KV-cache form: Nq queries attend to Nkv keys of the same head.  q1, q2 are
 * [B, H, Nq, d], k1, k2 are [B, H, Nkv, d], v is [B, H, Nkv, 2d] and out is
 * [B, H, Nq, 2d].  The queries are the last Nq positions of the sequence:
 * query i sits at position Nkv - Nq + i, so under the causal mask it sees keys
 * j <= Nkv - Nq + i (with Nq = Nkv this is oracle_fwd).  Rows are selected as
 * in oracle_fwd_rows (bh_idx[r], row_idx[r] < Nq); nrows < 0 means every row
 * in order, written to out_rows as a full [B, H, Nq, 2d] tensor. */
int oracle_fwd_kv_rows(int B, int H, int64_t Nq, int64_t Nkv, int d,
                       const double *q1, const double *k1, const double *q2,
                       const double *k2, const double *v, const double *lam,
                       int causal, int headnorm, const double *w, double eps,
                       double lambda_init, int64_t nrows, const int64_t *bh_idx,
                       const int64_t *row_idx, double *out_rows, int nthreads)
{
    if (B < 0 || H < 0 || Nq < 0 || Nkv < 0 || d <= 0)
        return -1;
    if (causal && Nq > Nkv)
        return -1;
    const int64_t BH = (int64_t)B * H;
    const int all = nrows < 0;
    const int64_t n = all ? BH * Nq : nrows;
    for (int64_t r = 0; !all && r < n; ++r)
        if (bh_idx[r] < 0 || bh_idx[r] >= BH || row_idx[r] < 0 || row_idx[r] >= Nq)
            return -1;
    const int dv = 2 * d;
    int err = 0;
    set_threads(nthreads);
#pragma omp parallel
    {
        double *scratch = (double *)malloc(sizeof(double) * (size_t)(3 * Nkv + 1));
        if (!scratch) {
#pragma omp atomic write
            err = -2;
        }
#pragma omp for schedule(dynamic, 4)
        for (int64_t r = 0; r < n; ++r) {
            if (!scratch)
                continue;
            const int64_t bh = all ? r / Nq : bh_idx[r];
            const int64_t i = all ? r % Nq : row_idx[r];
            const int h = (int)(bh % H);
            const int64_t pos = Nkv - Nq + i;
            const int64_t qo = bh * Nq * d, ko = bh * Nkv * d, vo = bh * Nkv * dv;
            out_row(pos, Nkv, d, q1 + qo + i * d, k1 + ko, q2 + qo + i * d, k2 + ko, v + vo,
                    lam[h], causal, headnorm, w ? w + (int64_t)h * dv : NULL, eps,
                    lambda_init, scratch, out_rows + r * dv);
        }
        free(scratch);
    }
    return err;
}

/* The whole differential map of one head, wmap[i * N + j] = map1 - lambda
 * map2 (0 where the key is masked).  This is the quantity the page's worked
 * example prints facts about (row sums, count of negative weights). */
int oracle_diff_map(int64_t N, int d, const double *q1, const double *k1,
                    const double *q2, const double *k2, double lam, int causal,
                    double *wmap)
{
    if (N < 0 || d <= 0)
        return -1;
    double *scratch = (double *)malloc(sizeof(double) * (size_t)(2 * N + 1));
    if (!scratch)
        return -2;
    for (int64_t i = 0; i < N; ++i)
        diff_row(i, N, d, q1 + i * d, k1, q2 + i * d, k2, lam, causal, scratch,
                 scratch + N, wmap + i * N);
    free(scratch);
    return 0;
}

/* Per-head group normalisation alone (the headnorm = 2 form), rows x[R, dv]
 * of head h_idx[r]; the same steps out_row takes for it. */
int oracle_groupnorm(int64_t R, int dv, int H, const double *x, const int64_t *h_idx,
                     const double *w, double eps, double lambda_init, double *y)
{
    if (R < 0 || dv <= 0 || H <= 0)
        return -1;
    for (int64_t r = 0; r < R; ++r) {
        if (h_idx[r] < 0 || h_idx[r] >= H)
            return -1;
        for (int c = 0; c < dv; ++c)
            y[r * dv + c] = x[r * dv + c];
        group_norm_row(y + r * dv, dv, w ? w + h_idx[r] * dv : NULL, eps, lambda_init);
    }
    return 0;
}

/* Per-head RMS normalisation alone, applied to given rows x[R, dv] of head
 * h_idx[r]: y = x / sqrt(mean(x^2) + eps) * w[h, c] * (1 - lambda_init).
 * The same steps out_row takes after the weighted value sum. */
int oracle_headnorm(int64_t R, int dv, int H, const double *x,
                    const int64_t *h_idx, const double *w, double eps,
                    double lambda_init, double *y)
{
    if (R < 0 || dv <= 0 || H <= 0)
        return -1;
    for (int64_t r = 0; r < R; ++r) {
        if (h_idx[r] < 0 || h_idx[r] >= H)
            return -1;
        const double *xr = x + r * dv;
        double ms = 0.0;
        for (int c = 0; c < dv; ++c)
            ms += xr[c] * xr[c];
        ms /= (double)dv;
        const double inv = 1.0 / sqrt(ms + eps);
        for (int c = 0; c < dv; ++c) {
            const double g = w ? w[h_idx[r] * dv + c] : 1.0;
            y[r * dv + c] = xr[c] * inv * g * (1.0 - lambda_init);
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------
 * Backward pass (gradients of the head forward above).
 *
 * The pages give the forward only; its gradient is the plain derivative of
 * that definition, written out here by the chain rule in float64, one query
 * row at a time, both maps materialised, nothing blocked or fused:
 *
 *   forward (row i):  p1 = softmax(s1), p2 = softmax(s2), s_k[j] = q_k.k_k[j] / sqrt(d)
 *                     o1 = p1 V, o2 = p2 V, o = o1 - lambda o2
 *                     y  = o r g,  r = 1 / sqrt(mean(o^2) + eps),  g = w (1 - lambda_init)
 *   given dy (row i):
 *     norm:    do = r g dy - (r^3 / 2d) o sum_c(dy_c g_c o_c);   dw += dy o r (1 - lambda_init)
 *              (without the norm: do = dy; with the group form, headnorm = 2,
 *              o above is the centred row o - mean(o), r is taken from it, and
 *              do then loses its mean: do -= mean_c(do))
 *     lambda:  dlambda += -(do . o2)
 *     values:  dV[j] += (p1[j] - lambda p2[j]) do
 *     maps:    dp1[j] = do . v_j,  dp2[j] = -lambda do . v_j
 *     softmax: ds_k[j] = p_k[j] (dp_k[j] - sum_j' p_k[j'] dp_k[j'])
 *     logits:  dq_k += ds_k[j] k_k[j] / sqrt(d),  dk_k[j] += ds_k[j] q_k / sqrt(d)
 *
 * Layouts as in oracle_fwd; gradients have the shapes of their tensors;
 * dlam is [H] and dw is [H, 2d] (dw is left untouched without the norm).
 * All outputs are overwritten.  Returns 0, -1 on bad arguments, -2 if
 * scratch could not be allocated.
 */
static void bwd_head(int64_t N, int d, const double *q1, const double *k1,
                     const double *q2, const double *k2, const double *v, double lam,
                     int causal, int headnorm, const double *w_head, double eps,
                     double lambda_init, const double *dy, double *dq1, double *dk1,
                     double *dq2, double *dk2, double *dv, double *dlam, double *dw,
                     double *scratch)
{
    const int dv_ = 2 * d;
    const double scale = 1.0 / sqrt((double)d);
    double *p1 = scratch, *p2 = scratch + N;
    double *o1 = scratch + 2 * N, *o2 = o1 + dv_, *o = o2 + dv_, *dout = o + dv_;
    for (int64_t i = 0; i < N; ++i) {
        const double *q1i = q1 + i * d, *q2i = q2 + i * d, *dyi = dy + i * dv_;
        softmax_row(i, N, d, q1i, k1, causal, p1);
        softmax_row(i, N, d, q2i, k2, causal, p2);
        for (int c = 0; c < dv_; ++c)
            o1[c] = o2[c] = 0.0;
        for (int64_t j = 0; j < N; ++j)
            for (int c = 0; c < dv_; ++c) {
                o1[c] += p1[j] * v[j * dv_ + c];
                o2[c] += p2[j] * v[j * dv_ + c];
            }
        for (int c = 0; c < dv_; ++c)
            o[c] = o1[c] - lam * o2[c];
        /* norm backward.  The group form normalises the centred row o - mean(o)
         * exactly as the RMS form normalises o, so the RMS formula applies to the
         * centred row; the derivative of the centring then removes the mean of
         * the result. */
        if (headnorm) {
            double mu = 0.0;
            if (headnorm == 2) {
                for (int c = 0; c < dv_; ++c)
                    mu += o[c];
                mu /= (double)dv_;
            }
            double ms = 0.0, t = 0.0;
            for (int c = 0; c < dv_; ++c)
                ms += (o[c] - mu) * (o[c] - mu);
            ms /= (double)dv_;
            const double r = 1.0 / sqrt(ms + eps);
            for (int c = 0; c < dv_; ++c) {
                const double g = (w_head ? w_head[c] : 1.0) * (1.0 - lambda_init);
                t += dyi[c] * g * (o[c] - mu);
            }
            for (int c = 0; c < dv_; ++c) {
                const double g = (w_head ? w_head[c] : 1.0) * (1.0 - lambda_init);
                dout[c] = r * g * dyi[c] - r * r * r / (double)dv_ * (o[c] - mu) * t;
                dw[c] += dyi[c] * (o[c] - mu) * r * (1.0 - lambda_init);
            }
            if (headnorm == 2) {
                double md = 0.0;
                for (int c = 0; c < dv_; ++c)
                    md += dout[c];
                md /= (double)dv_;
                for (int c = 0; c < dv_; ++c)
                    dout[c] -= md;
            }
        } else {
            for (int c = 0; c < dv_; ++c)
                dout[c] = dyi[c];
        }
        /* lambda */
        double do_o1 = 0.0, do_o2 = 0.0;
        for (int c = 0; c < dv_; ++c) {
            do_o1 += dout[c] * o1[c];
            do_o2 += dout[c] * o2[c];
        }
        *dlam -= do_o2;
        /* values, maps, softmax, logits */
        for (int64_t j = 0; j < N; ++j) {
            if (!visible(i, j, causal))
                continue;
            double dvj = 0.0; /* do . v_j */
            for (int c = 0; c < dv_; ++c) {
                dv[j * dv_ + c] += (p1[j] - lam * p2[j]) * dout[c];
                dvj += dout[c] * v[j * dv_ + c];
            }
            /* sum_j' p1 dp1 = do . o1 ; sum_j' p2 dp2 = -lambda do . o2 */
            const double ds1 = p1[j] * (dvj - do_o1);
            const double ds2 = p2[j] * (-lam * dvj + lam * do_o2);
            for (int c = 0; c < d; ++c) {
                dq1[i * d + c] += ds1 * k1[j * d + c] * scale;
                dk1[j * d + c] += ds1 * q1i[c] * scale;
                dq2[i * d + c] += ds2 * k2[j * d + c] * scale;
                dk2[j * d + c] += ds2 * q2i[c] * scale;
            }
        }
    }
}

int oracle_bwd(int B, int H, int64_t N, int d, const double *q1, const double *k1,
               const double *q2, const double *k2, const double *v, const double *lam,
               int causal, int headnorm, const double *w, double eps, double lambda_init,
               const double *dy, double *dq1, double *dk1, double *dq2, double *dk2,
               double *dv, double *dlam, double *dw, int nthreads)
{
    if (B < 0 || H <= 0 || N < 0 || d <= 0 || headnorm < 0 || headnorm > 2)
        return -1;
    const int64_t BH = (int64_t)B * H;
    const int dv_ = 2 * d;
    const size_t nqk = (size_t)(BH * N * d), nv = (size_t)(BH * N * dv_);
    memset(dq1, 0, nqk * sizeof(double));
    memset(dk1, 0, nqk * sizeof(double));
    memset(dq2, 0, nqk * sizeof(double));
    memset(dk2, 0, nqk * sizeof(double));
    memset(dv, 0, nv * sizeof(double));
    /* per-(b, h) partial sums of dlambda and dw, added up per head afterwards */
    double *plam = (double *)calloc((size_t)(BH > 0 ? BH : 1), sizeof(double));
    double *pw = (double *)calloc((size_t)(BH > 0 ? BH : 1) * dv_, sizeof(double));
    if (!plam || !pw) {
        free(plam);
        free(pw);
        return -2;
    }
    int err = 0;
    set_threads(nthreads);
#pragma omp parallel
    {
        double *scratch = (double *)malloc(sizeof(double) * (size_t)(2 * N + 4 * dv_ + 1));
        if (!scratch) {
#pragma omp atomic write
            err = -2;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t bh = 0; bh < BH; ++bh) {
            if (!scratch)
                continue;
            const int h = (int)(bh % H);
            const int64_t qk = bh * N * d, vo = bh * N * dv_;
            bwd_head(N, d, q1 + qk, k1 + qk, q2 + qk, k2 + qk, v + vo, lam[h], causal,
                     headnorm, w ? w + (int64_t)h * dv_ : NULL, eps, lambda_init, dy + vo,
                     dq1 + qk, dk1 + qk, dq2 + qk, dk2 + qk, dv + vo, plam + bh,
                     pw + bh * dv_, scratch);
        }
        free(scratch);
    }
    for (int h = 0; h < H; ++h) {
        dlam[h] = 0.0;
        if (headnorm)
            for (int c = 0; c < dv_; ++c)
                dw[(int64_t)h * dv_ + c] = 0.0;
    }
    for (int64_t bh = 0; bh < BH; ++bh) {
        const int h = (int)(bh % H);
        dlam[h] += plam[bh];
        if (headnorm)
            for (int c = 0; c < dv_; ++c)
                dw[(int64_t)h * dv_ + c] += pw[bh * dv_ + c];
    }
    free(plam);
    free(pw);
    return err;
}
