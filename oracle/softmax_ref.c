/*
 * Reference (oracle) implementation of row-wise numerically stable softmax.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or call
 * this file: only the tests, the smoke check and the CPU-baseline leg of the
 * benchmark use it.  It shares no code, header, table or constant with the CUDA
 * library; it is plain, slow C in double precision, written so that each step
 * can be checked against the pages by eye.
 *
 * Sources (page title, section):
 *  - "Softmax numerics architecture - max subtract, fp32 accumulate, fusion,
 *    online": the shift identity and the choice c = max x ("The max-subtraction
 *    identity, and why it is exact"); the per-block update of (m, d) ("Online
 *    softmax: one recurrence, one fewer pass"); log-sum-exp, log_softmax and
 *    cross-entropy ("Log-sum-exp: log-probabilities without probabilities");
 *    the vector-Jacobian product and the fused cross-entropy gradient ("The
 *    Jacobian, and the backward pass that never divides"); the fp16 worked
 *    example ("A worked example: naive fp16 versus the stable form").
 *  - "Kernel visualization: online softmax": the per-element recurrence with
 *    m_0 = -inf, d_0 = 0 ("Online softmax" and "Derivation"), and the tiled
 *    update m_new = max(m_old, max tile), d_new = d_old e^(m_old - m_new) +
 *    sum e^(tile - m_new) ("Tiled version").
 *  - "Online stable softmax": the two-block merge with the empty prefix
 *    (-inf, 0) ("Derive the update for two blocks"), the declared result for a
 *    fully masked row ("Masks, empty rows, and precision").
 *  - "Stable softmax: keep the normalizer consistent as tiles arrive": the
 *    exclusion value for masked lanes and the need for an explicit policy for
 *    +inf, NaN and empty rows.
 *
 * Declared policy (the pages ask for one but do not fix it; this is the reading
 * the library documents).  For a row x[0:cols] with valid prefix length L
 * (valid_len[r] clamped to [0, cols]; all of cols when no lengths are given):
 *   1. lanes j >= L are masked: output +0;
 *   2. L == 0: every output is +0; stats (m, d) = (-inf, 0), the merge identity;
 *   3. a NaN among x[0:L]: outputs 0..L-1 are NaN; stats (NaN, NaN);
 *   4. m = max x[0:L]; m == -inf (every valid lane is -inf): all outputs +0,
 *      stats (-inf, 0);
 *   5. m == +inf: outputs 0..L-1 are NaN (the stable formula evaluates
 *      inf - inf); stats (+inf, NaN);
 *   6. otherwise d = sum_{j<L} exp(x_j - m), p_j = exp(x_j - m) / d (a -inf
 *      lane contributes exp(-inf) = 0 and outputs +0).
 *
 * Everything is computed in double from inputs widened exactly from their
 * stored type.  Output conversion to fp16/bf16 is round-to-nearest-even straight
 * from double, written from the IEEE 754 definition of a binary format.
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_F32 = 0, ORC_F16 = 1, ORC_BF16 = 2 };

/* ---------------------------------------------------------------------------
 * Decoding stored values.  A binary format with w exponent bits and t trailing
 * significand bits has bias 2^(w-1) - 1; a zero exponent field means a
 * subnormal (or zero) with value frac * 2^(1 - bias - t); an all-ones field
 * means inf (frac == 0) or NaN.  Otherwise the value is (2^t + frac) *
 * 2^(E - bias - t).
 * ------------------------------------------------------------------------- */
static double decode_bits(uint32_t bits, int w, int t)
{
    uint32_t sign = (bits >> (w + t)) & 1u;
    uint32_t expf = (bits >> t) & ((1u << w) - 1u);
    uint32_t frac = bits & ((1u << t) - 1u);
    int bias = (1 << (w - 1)) - 1;
    double v;
    if (expf == 0) {
        v = ldexp((double)frac, 1 - bias - t);
    } else if (expf == (1u << w) - 1u) {
        v = frac ? NAN : INFINITY;
    } else {
        v = ldexp((double)((1u << t) + frac), (int)expf - bias - t);
    }
    return sign ? -v : v;
}

double orc_decode_f16(uint16_t h) { return decode_bits(h, 5, 10); }
double orc_decode_bf16(uint16_t b) { return decode_bits(b, 8, 7); }

static double load_elem(const void *x, int dtype, int64_t i)
{
    if (dtype == ORC_F32) {
        float f;
        memcpy(&f, (const char *)x + 4 * i, 4);
        return (double)f;
    }
    uint16_t h;
    memcpy(&h, (const char *)x + 2 * i, 2);
    return dtype == ORC_F16 ? orc_decode_f16(h) : orc_decode_bf16(h);
}

/* ---------------------------------------------------------------------------
 * Encoding: round a double to the nearest value of a binary format with p
 * significand bits (implicit bit included), minimum normal exponent emin and
 * maximum exponent emax, ties to even, subnormals kept.  The spacing of the
 * representable numbers around |v| is q = 2^(max(e, emin) - (p - 1)) where
 * 2^e <= |v| < 2^(e+1); |v|/q is then an exact double below 2^p and rounds to
 * an integer with nearbyint (ties to even in the default rounding mode).  A
 * result at or beyond 2^(emax+1) overflows to inf.
 * ------------------------------------------------------------------------- */
static uint32_t encode_bits(double v, int w, int t)
{
    int p = t + 1;
    int bias = (1 << (w - 1)) - 1;
    int emin = 1 - bias, emax = bias;
    uint32_t sign_bit = 1u << (w + t);
    uint32_t exp_all = ((1u << w) - 1u) << t;
    if (isnan(v)) return exp_all | (1u << (t - 1)); /* quiet NaN */
    uint32_t sign = signbit(v) ? sign_bit : 0u;
    double a = fabs(v);
    if (isinf(a)) return sign | exp_all;
    if (a == 0.0) return sign;
    int E;
    frexp(a, &E); /* a = f * 2^E, f in [0.5, 1): leading bit is 2^(E-1) */
    int e = E - 1;
    if (e < emin) e = emin;
    int qexp = e - (p - 1);
    double r = nearbyint(ldexp(a, -qexp)); /* integer in [0, 2^p] */
    double res = ldexp(r, qexp);
    if (res >= ldexp(1.0, emax + 1)) return sign | exp_all;
    if (r == 0.0) return sign;
    if (res < ldexp(1.0, emin)) /* subnormal: exponent field 0, frac = r */
        return sign | (uint32_t)r;
    frexp(res, &E);
    int er = E - 1;
    uint32_t frac = (uint32_t)(ldexp(res, -(er - t)) - ldexp(1.0, t));
    return sign | ((uint32_t)(er + bias) << t) | frac;
}

uint16_t orc_round_f16(double v) { return (uint16_t)encode_bits(v, 5, 10); }
uint16_t orc_round_bf16(double v) { return (uint16_t)encode_bits(v, 8, 7); }
uint32_t orc_round_f32_bits(double v) { return encode_bits(v, 8, 23); }

/* Round n doubles to the given storage type (raw little-endian bits out). */
void orc_round_array(const double *v, int64_t n, int dtype, void *out)
{
    for (int64_t i = 0; i < n; ++i) {
        if (dtype == ORC_F32) {
            uint32_t b = orc_round_f32_bits(v[i]);
            memcpy((char *)out + 4 * i, &b, 4);
        } else {
            uint16_t b = dtype == ORC_F16 ? orc_round_f16(v[i]) : orc_round_bf16(v[i]);
            memcpy((char *)out + 2 * i, &b, 2);
        }
    }
}

void orc_decode_array(const void *x, int64_t n, int dtype, double *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = load_elem(x, dtype, i);
}

/* ---------------------------------------------------------------------------
 * Row statistics by the plain three-pass definition ("safe softmax"):
 * pass 1 m = max x, pass 2 d = sum exp(x - m); the declared policy above
 * settles the special rows.  Returns the class of the row:
 *   0 normal, 1 empty or all -inf (zeros), 2 NaN row (NaN outputs).
 * ------------------------------------------------------------------------- */
static int row_stats_one(const void *x, int dtype, int64_t base, int64_t L,
                         double *m_out, double *d_out)
{
    if (L == 0) { *m_out = -INFINITY; *d_out = 0.0; return 1; }
    for (int64_t j = 0; j < L; ++j)
        if (isnan(load_elem(x, dtype, base + j))) { *m_out = NAN; *d_out = NAN; return 2; }
    double m = -INFINITY;
    for (int64_t j = 0; j < L; ++j) {
        double v = load_elem(x, dtype, base + j);
        if (v > m) m = v;
    }
    if (m == -INFINITY) { *m_out = -INFINITY; *d_out = 0.0; return 1; }
    if (m == INFINITY) { *m_out = INFINITY; *d_out = NAN; return 2; }
    double d = 0.0;
    for (int64_t j = 0; j < L; ++j) d += exp(load_elem(x, dtype, base + j) - m);
    *m_out = m;
    *d_out = d;
    return 0;
}

static int64_t row_len(const int32_t *valid_len, int64_t r, int64_t cols)
{
    if (!valid_len) return cols;
    int64_t L = valid_len[r];
    if (L < 0) L = 0;
    if (L > cols) L = cols;
    return L;
}

/* Softmax of the selected rows.  x is the whole [rows, cols] row-major input;
 * `sel` lists n_sel row indices (NULL: all rows 0..n_sel-1); p receives n_sel
 * output rows of cols doubles each. */
void orc_softmax_rows(const void *x, int dtype, int64_t cols, const int32_t *valid_len,
                      const int64_t *sel, int64_t n_sel, double *p)
{
    for (int64_t i = 0; i < n_sel; ++i) {
        int64_t r = sel ? sel[i] : i;
        int64_t L = row_len(valid_len, r, cols);
        int64_t base = r * cols;
        double *out = p + i * cols;
        double m, d;
        int cls = row_stats_one(x, dtype, base, L, &m, &d);
        for (int64_t j = 0; j < cols; ++j) out[j] = 0.0;
        if (cls == 1) continue;
        if (cls == 2) {
            for (int64_t j = 0; j < L; ++j) out[j] = NAN;
            continue;
        }
        /* pass 3: p_j = exp(x_j - m) / d */
        for (int64_t j = 0; j < L; ++j) out[j] = exp(load_elem(x, dtype, base + j) - m) / d;
    }
}

void orc_row_stats(const void *x, int dtype, int64_t cols, const int32_t *valid_len,
                   const int64_t *sel, int64_t n_sel, double *m_out, double *d_out)
{
    for (int64_t i = 0; i < n_sel; ++i) {
        int64_t r = sel ? sel[i] : i;
        row_stats_one(x, dtype, r * cols, row_len(valid_len, r, cols), &m_out[i], &d_out[i]);
    }
}

/* ---------------------------------------------------------------------------
 * Merge of two block summaries ("Derive the update for two blocks"):
 *   m' = max(m_a, m_b),  d' = d_a exp(m_a - m') + d_b exp(m_b - m').
 * (-inf, .) is the empty block and leaves the other operand unchanged; a NaN
 * maximum poisons the result; a +inf maximum gives (+inf, NaN), which is what
 * the row statistics of the concatenated blocks are under the policy above.
 * ------------------------------------------------------------------------- */
void orc_merge_stats(const double *m_a, const double *d_a, const double *m_b,
                     const double *d_b, double *m_out, double *d_out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) {
        double ma = m_a[i], da = d_a[i], mb = m_b[i], db = d_b[i];
        double m, d;
        if (isnan(ma) || isnan(mb)) { m = NAN; d = NAN; }
        else if (ma == -INFINITY) { m = mb; d = mb == -INFINITY ? 0.0 : db; }
        else if (mb == -INFINITY) { m = ma; d = da; }
        else {
            m = ma > mb ? ma : mb;
            if (m == INFINITY) d = NAN;
            else d = da * exp(ma - m) + db * exp(mb - m);
        }
        m_out[i] = m;
        d_out[i] = d;
    }
}

/* ---------------------------------------------------------------------------
 * The online recurrences as the pages state them, logging the state after
 * every step (used to pin the pages' traces).
 *
 * Per element: m_i = max(m_{i-1}, x_i), d_i = d_{i-1} e^(m_{i-1} - m_i) +
 * e^(x_i - m_i), from m_0 = -inf, d_0 = 0.  With rescale == 0 the correction
 * factor is left out: the deliberately wrong variant the exercise asks for.
 * The first step's factor e^(-inf - x_1) is taken as 0 (d_0 = 0 anyway).
 * ------------------------------------------------------------------------- */
void orc_online_elementwise(const double *x, int64_t n, int rescale, double *m_trace, double *d_trace)
{
    double m = -INFINITY, d = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        double m_new = x[i] > m ? x[i] : m;
        double factor = (m == -INFINITY) ? 0.0 : exp(m - m_new);
        if (!rescale) factor = 1.0;
        d = d * factor + exp(x[i] - m_new);
        m = m_new;
        m_trace[i] = m;
        d_trace[i] = d;
    }
}

/* Tiled: tiles of B consecutive elements (the last may be shorter).  For tile t
 * the log holds m after the tile, the corrected old sum d_old e^(m_old -
 * m_new) and d after adding the tile's own terms. */
void orc_online_tiled(const double *x, int64_t n, int64_t B, double *m_trace,
                      double *corrected_trace, double *d_trace)
{
    double m = -INFINITY, d = 0.0;
    int64_t t = 0;
    for (int64_t s = 0; s < n; s += B, ++t) {
        int64_t e = s + B < n ? s + B : n;
        double tile_max = -INFINITY;
        for (int64_t j = s; j < e; ++j) if (x[j] > tile_max) tile_max = x[j];
        double m_new = tile_max > m ? tile_max : m;
        double corrected = (m == -INFINITY) ? 0.0 : d * exp(m - m_new);
        double tile_sum = 0.0;
        for (int64_t j = s; j < e; ++j) tile_sum += exp(x[j] - m_new);
        d = corrected + tile_sum;
        m = m_new;
        m_trace[t] = m;
        corrected_trace[t] = corrected;
        d_trace[t] = d;
    }
}

/* ---------------------------------------------------------------------------
 * The naive, unshifted softmax evaluated in fp16 arithmetic: every
 * intermediate (each exp, each partial sum, each quotient) is rounded to fp16.
 * This is the negative control of the fp16 worked example; it is expected to
 * overflow.  Outputs are fp16 values widened to double.
 * ------------------------------------------------------------------------- */
static double f16(double v) { return orc_decode_f16(orc_round_f16(v)); }

void orc_naive_softmax_f16(const double *x, int64_t n, double *p)
{
    double s = 0.0;
    for (int64_t j = 0; j < n; ++j) s = f16(s + f16(exp(f16(x[j]))));
    for (int64_t j = 0; j < n; ++j) p[j] = f16(f16(exp(f16(x[j]))) / s);
}

/* The stable form evaluated in fp16 arithmetic (subtract the max, then as
 * above), for the same worked example. */
void orc_stable_softmax_f16(const double *x, int64_t n, double *shifted, double *e, double *p,
                            double *sum_out)
{
    double m = -INFINITY;
    for (int64_t j = 0; j < n; ++j) if (f16(x[j]) > m) m = f16(x[j]);
    double s = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        shifted[j] = f16(f16(x[j]) - m);
        e[j] = f16(exp(shifted[j]));
        s = f16(s + e[j]);
    }
    for (int64_t j = 0; j < n; ++j) p[j] = f16(e[j] / s);
    *sum_out = s;
}

/* ---------------------------------------------------------------------------
 * Log-space outputs ("Softmax numerics architecture...", section "Log-sum-exp:
 * log-probabilities without probabilities"):
 *   LSE(x) = m + log(sum_j exp(x_j - m)),  log_softmax(x)_i = x_i - LSE(x),
 *   CE(x, t) = LSE(x) - x_t.
 * Over the valid prefix with the same policy: an empty / all -inf row has
 * LSE = -inf and log_softmax outputs -inf in its valid lanes (log 0); a NaN row
 * NaN; a +inf row NaN.  Masked lanes output -inf (log of the +0 probability).
 * ------------------------------------------------------------------------- */
void orc_log_softmax_rows(const void *x, int dtype, int64_t cols, const int32_t *valid_len,
                          const int64_t *sel, int64_t n_sel, double *out, double *lse_out)
{
    for (int64_t i = 0; i < n_sel; ++i) {
        int64_t r = sel ? sel[i] : i;
        int64_t L = row_len(valid_len, r, cols);
        int64_t base = r * cols;
        double m, d;
        int cls = row_stats_one(x, dtype, base, L, &m, &d);
        double lse = cls == 0 ? m + log(d) : (cls == 1 ? -INFINITY : NAN);
        if (lse_out) lse_out[i] = lse;
        double *o = out ? out + i * cols : NULL;
        if (!o) continue;
        for (int64_t j = 0; j < cols; ++j) o[j] = -INFINITY;
        for (int64_t j = 0; j < L; ++j) {
            if (cls == 0) o[j] = load_elem(x, dtype, base + j) - lse;
            else if (cls == 2) o[j] = NAN;
        }
    }
}

/* Normalise rows with given statistics: y_j = exp(x_j - m) / d over the valid
 * prefix (+0 beyond), the step that completes a softmax whose statistics were
 * merged from blocks ("Online stable softmax": only m and l of the prefix are
 * needed).  m == -inf gives a zero row; a NaN m or d, or m == +inf, NaN lanes. */
void orc_apply_stats(const void *x, int dtype, int64_t cols, const int32_t *valid_len,
                     const double *m_in, const double *d_in, const int64_t *sel, int64_t n_sel,
                     double *p)
{
    for (int64_t i = 0; i < n_sel; ++i) {
        int64_t r = sel ? sel[i] : i;
        int64_t L = row_len(valid_len, r, cols);
        int64_t base = r * cols;
        double m = m_in[r], d = d_in[r];
        double *out = p + i * cols;
        for (int64_t j = 0; j < cols; ++j) out[j] = 0.0;
        if (m == -INFINITY || L == 0) continue;
        int bad = isnan(m) || isnan(d) || m == INFINITY;
        for (int64_t j = 0; j < L; ++j)
            out[j] = bad ? NAN : exp(load_elem(x, dtype, base + j) - m) / d;
    }
}

/* Softmax vector-Jacobian product ("The Jacobian, and the backward pass that
 * never divides"): the Jacobian diag(p) - p p^T is never formed; for the
 * upstream gradient g, dx_i = p_i (g_i - sum_j g_j p_j).  p is the softmax of
 * the row as the forward pass stored it and g the gradient, both in `dtype`;
 * the sum runs over the valid prefix, and masked lanes (where p is the constant
 * +0, so no input there affects the loss) give dx = 0.  Plain IEEE double
 * arithmetic otherwise: a NaN among the valid p or g makes every valid lane NaN. */
void orc_softmax_backward(const void *p, const void *g, int dtype, int64_t cols,
                          const int32_t *valid_len, const int64_t *sel, int64_t n_sel, double *dx)
{
    for (int64_t i = 0; i < n_sel; ++i) {
        int64_t r = sel ? sel[i] : i;
        int64_t L = row_len(valid_len, r, cols);
        int64_t base = r * cols;
        double *o = dx + i * cols;
        double gp = 0.0;
        for (int64_t j = 0; j < L; ++j) gp += load_elem(g, dtype, base + j) * load_elem(p, dtype, base + j);
        for (int64_t j = 0; j < cols; ++j) o[j] = 0.0;
        for (int64_t j = 0; j < L; ++j)
            o[j] = load_elem(p, dtype, base + j) * (load_elem(g, dtype, base + j) - gp);
    }
}

/* Cross-entropy with logits and its fused gradient ("Log-sum-exp..." and "The
 * Jacobian, and the backward pass that never divides"): loss_r = LSE(x_r) -
 * x_r[t_r], grad_rj = p_rj - [j == t_r].  A target outside [0, L) is ignored:
 * loss 0 and gradient 0 for the row (the convention of an ignored index). */
void orc_cross_entropy(const void *x, int dtype, int64_t cols, const int32_t *valid_len,
                       const int64_t *target, const int64_t *sel, int64_t n_sel, double *loss,
                       double *grad)
{
    for (int64_t i = 0; i < n_sel; ++i) {
        int64_t r = sel ? sel[i] : i;
        int64_t L = row_len(valid_len, r, cols);
        int64_t base = r * cols;
        int64_t t = target[r];
        double *gr = grad ? grad + i * cols : NULL;
        if (gr) for (int64_t j = 0; j < cols; ++j) gr[j] = 0.0;
        if (t < 0 || t >= L) { loss[i] = 0.0; continue; }
        double m, d;
        int cls = row_stats_one(x, dtype, base, L, &m, &d);
        if (cls != 0) {
            loss[i] = NAN;
            if (gr) for (int64_t j = 0; j < L; ++j) gr[j] = NAN;
            continue;
        }
        double lse = m + log(d);
        loss[i] = lse - load_elem(x, dtype, base + t);
        if (gr)
            for (int64_t j = 0; j < L; ++j)
                gr[j] = exp(load_elem(x, dtype, base + j) - m) / d - (j == t ? 1.0 : 0.0);
    }
}

/* ---------------------------------------------------------------------------
 * Attention with the weighted value numerator ("Online stable softmax",
 * "Carry a weighted value numerator for attention" and "Reference summary";
 * "Softmax numerics architecture...", "From online softmax to tiled
 * attention").  For query row i of head h, with scores s_j = scale * q_i . k_j
 * over the valid keys j (all Sk keys, or with the causal mask j <= i + Sk - Sq),
 *   m = max s_j,  l = sum exp(s_j - m),  o = sum exp(s_j - m) v_j / l,
 *   LSE = m + log l.
 * A row with no valid key is the declared empty row: o = 0, LSE = -inf.
 * q is [BH][Sq][D], k and v are [BH][Sk][D], all in `dtype`.  `sel` lists
 * n_sel (head, row) pairs as head * Sq + row (NULL: every row in order).
 * oabs receives sum p_j |v_j| per output element (the scale of the output's
 * rounding errors), smax the largest |s_j| computed from |q| . |k| (the scale of
 * the scores' rounding errors); either may be NULL.
 * ------------------------------------------------------------------------- */
void orc_attention_rows(const void *q, const void *k, const void *v, int dtype, int64_t Sq,
                        int64_t Sk, int64_t D, double scale, int causal, const int64_t *sel,
                        int64_t n_sel, double *o, double *lse, double *oabs, double *smax)
{
    double *s = (double *)malloc((size_t)(Sk > 0 ? Sk : 1) * sizeof(double));
    for (int64_t n = 0; n < n_sel; ++n) {
        int64_t idx = sel ? sel[n] : n;
        int64_t h = idx / Sq, i = idx % Sq;
        int64_t nk = Sk;
        if (causal) {
            nk = i + Sk - Sq + 1;
            if (nk < 0) nk = 0;
            if (nk > Sk) nk = Sk;
        }
        const int64_t qb = (h * Sq + i) * D, kb = h * Sk * D;
        double m = -INFINITY, amax = 0.0;
        for (int64_t j = 0; j < nk; ++j) {
            double acc = 0.0, aabs = 0.0;
            for (int64_t d = 0; d < D; ++d) {
                double qd = load_elem(q, dtype, qb + d), kd = load_elem(k, dtype, kb + j * D + d);
                acc += qd * kd;
                aabs += fabs(qd) * fabs(kd);
            }
            s[j] = scale * acc;
            if (s[j] > m) m = s[j];
            if (fabs(scale) * aabs > amax) amax = fabs(scale) * aabs;
        }
        if (smax) smax[n] = amax;
        for (int64_t d = 0; d < D; ++d) {
            o[n * D + d] = 0.0;
            if (oabs) oabs[n * D + d] = 0.0;
        }
        if (nk == 0 || m == -INFINITY || isnan(m)) {
            lse[n] = nk == 0 || m == -INFINITY ? -INFINITY : NAN;
            if (nk > 0 && isnan(m))
                for (int64_t d = 0; d < D; ++d) o[n * D + d] = NAN;
            continue;
        }
        double l = 0.0;
        for (int64_t j = 0; j < nk; ++j) l += exp(s[j] - m);
        for (int64_t j = 0; j < nk; ++j) {
            double p = exp(s[j] - m) / l;
            for (int64_t d = 0; d < D; ++d) {
                double vd = load_elem(v, dtype, kb + j * D + d);
                o[n * D + d] += p * vd;
                if (oabs) oabs[n * D + d] += p * fabs(vd);
            }
        }
        lse[n] = m + log(l);
    }
    free(s);
}

/* The running state (m, l, o) over blocks of B scores, as the pages state it
 * ("Reference summary"): from (-inf, 0, 0), each block with its own maximum
 * m2, sum l2 = sum exp(s - m2) and numerator o2 = sum exp(s - m2) v merges as
 *   m' = max(m, m2),  l' = exp(m - m') l + exp(m2 - m') l2,
 *   o' = exp(m - m') o + exp(m2 - m') o2,
 * and o / l at the end.  rescale_o == 0 is the pages' named error: the sum is
 * rescaled but the numerator is not.  s: n scores; v: [n][D] doubles. */
void orc_attention_online(const double *s, const double *v, int64_t n, int64_t D, int64_t B,
                          int rescale_o, double *o_out, double *m_out, double *l_out)
{
    double m = -INFINITY, l = 0.0;
    double *o = (double *)calloc((size_t)D, sizeof(double));
    double *o2 = (double *)calloc((size_t)D, sizeof(double));
    for (int64_t b0 = 0; b0 < n; b0 += B) {
        int64_t b1 = b0 + B < n ? b0 + B : n;
        double m2 = -INFINITY;
        for (int64_t j = b0; j < b1; ++j) if (s[j] > m2) m2 = s[j];
        double l2 = 0.0;
        for (int64_t d = 0; d < D; ++d) o2[d] = 0.0;
        for (int64_t j = b0; j < b1; ++j) {
            double e = exp(s[j] - m2);
            l2 += e;
            for (int64_t d = 0; d < D; ++d) o2[d] += e * v[j * D + d];
        }
        double mn = m > m2 ? m : m2;
        double fa = m == -INFINITY ? 0.0 : exp(m - mn);  /* the empty prefix: selected, not evaluated */
        double fb = exp(m2 - mn);
        l = fa * l + fb * l2;
        for (int64_t d = 0; d < D; ++d) o[d] = (rescale_o ? fa : 1.0) * o[d] + fb * o2[d];
        m = mn;
    }
    for (int64_t d = 0; d < D; ++d) o_out[d] = l > 0 ? o[d] / l : 0.0;
    *m_out = m;
    *l_out = l;
    free(o);
    free(o2);
}
