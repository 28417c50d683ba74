/*
 * spec_oracle.c -- plain fp64 CPU oracle for batched speculative-sampling
 * verification.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library may include, link
 * or call this file.  It exists so that tests, the smoke check and the
 * benchmark's CPU-baseline leg can check the CUDA path against an independent,
 * slow, obviously correct restatement of the method.  It shares no code,
 * header, constant or helper with the CUDA library.
 *
 * Source of the method: the tutorial page "5.1 投机解码核心原理" (core
 * principles of speculative decoding), infra-guide-du8.pages.dev:
 *   - section 2.1: q_i(.) = q(.|h, y_<i) proposes y_1..y_gamma; the target
 *     gives p_i for i = 1..gamma+1 from one forward pass; p and q are the
 *     distributions actually used for sampling (temperature already applied);
 *   - section 3.1: greedy rule (accept y_i iff it is the target argmax,
 *     otherwise emit the argmax and stop);
 *   - section 3.2: a_i(y_i) = min(1, p_i(y_i)/q_i(y_i)), accept iff u < a_i;
 *     on reject draw from r_i(x) = [p_i(x) - q_i(x)]_+ / sum_z [p_i(z)-q_i(z)]_+;
 *   - section 3.3: a draft that gives only tokens is a one-hot q; acceptance is
 *     p(y) and the residual is p with y removed, renormalised;
 *   - section 5.1: stop at the first reject, later candidates are void;
 *   - section 5.2: when all gamma are accepted draw one more token from
 *     p_{gamma+1}; every round commits between 1 and gamma+1 tokens.
 * and the SpecKV page (shdxiang-github-io.pages.dev, "草稿模型信号提取",
 * draft signal extraction): per draft step H(q_i) = -sum_v q_i(v) log2 q_i(v)
 * and max_v q_i(v); per request the mean and max entropy and the mean and min
 * confidence over the gamma steps.
 *
 * Everything is computed in fp64 with libm exp/log, sums in ascending token
 * order, one request at a time.  Requests are independent (the sequence-level
 * product in section 5 of the tutorial page), so an OpenMP loop over requests
 * changes no result.
 *
 * Readings where the pages leave a step open (each one is a choice of this
 * oracle, stated once here):
 *   - the same temperature T_b is applied to target and draft logits:
 *     p = softmax(x / T);
 *   - top-k / top-p are not applied;
 *   - the acceptance test is evaluated as  u * q(y) < p(y)  (strict), which is
 *     u < min(1, p/q) whenever q(y) > 0 and defines the q(y) = 0 case
 *     (accept iff p(y) > 0);
 *   - greedy ties: the lowest token index wins;
 *   - the draw is inverse-CDF in ascending token order: with W = sum_v w_v and
 *     t = u * W, the token is the smallest x with C(x) = sum_{v<=x} w_v > t;
 *     if rounding leaves no such x, the largest x with w_x > 0;
 *   - one-hot residual mass is summed (W = sum_{v != y} p(v)), not 1 - p(y);
 *   - zero residual mass (impossible in exact arithmetic, section 4.2) falls
 *     back to drawing from p, with an informational status bit;
 *   - uniforms are an input [B, G+1]: column i < gamma_b is the test at
 *     position i, column G is the final draw;
 *   - draft signals use q at the request's temperature, over all gamma_b
 *     draft rows (before verification);
 *   - a logit of -inf is a token of probability 0; NaN or +inf anywhere in a
 *     row that is read, or a row with no finite maximum, is an error;
 *   - rows are checked lazily in position order, so a bad row, token or
 *     uniform after the first reject is never looked at.
 *
 * Parity status of each output:
 *   - accept_len, tokens, status: pinned by the worked example of section 7,
 *     exact u-grid integrals, chi-square tests and closed forms (tests);
 *   - accept_prob: pinned through A = 1 - TV(p, q) (section 4.3);
 *   - signals: pinned by closed forms (uniform, two-way tie, near one-hot rows)
 *     and by scipy's entropy on random rows;
 *   - top-k / top-p filtering (oracle_filter): pinned by hand-computed rows
 *     (ties, the crossing value, top-k then top-p, temperature) and by a
 *     brute-force search over thresholds on random rows (tests);
 *   - gamma selection (oracle_gamma_select): pinned by scikit-learn's MLP
 *     regressor on the same weights, hand-built selectors with a known
 *     argmax, ties and non-finite features (tests);
 *   - divergence statistics (oracle_divergence): pinned by scipy's entropy
 *     and relative entropy on random rows, the identities A = 1 - TV and
 *     L1 = 2 TV, the acceptance probability of the verify path averaged over
 *     y ~ q, p = q and closed forms (tests);
 *   - the decision margins: accept_margin = |u_i - a_i| (the distance of the
 *     acceptance test of section 3.2 from its threshold), draw_margin (the
 *     distance of t = u W from the nearer edge of the drawn bucket, over W)
 *     and probe_distance (the distance of t from the bucket of a given token,
 *     over W) are pinned by hand-computed cases on rows whose probabilities
 *     are exact binary fractions (tests).
 *
 * Planted mistakes: compiling with -DORACLE_PLANT=n introduces one deliberate
 * error (see the ORACLE_PLANT switch below).  The tests build each planted
 * variant and check that the pin suite rejects it.  The default build
 * (ORACLE_PLANT undefined) has none.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifndef ORACLE_PLANT
#define ORACLE_PLANT 0
#endif

/* planted-mistake ids (test-only builds) */
#define PLANT_RESAMPLE_FROM_P 1      /* reject path draws from p, not [p-q]_+  */
#define PLANT_RATIO_INVERTED 2       /* accept iff u * p(y) < q(y)             */
#define PLANT_RESIDUAL_SIGN 3        /* residual [q-p]_+                       */
#define PLANT_BONUS_ROW 4            /* bonus drawn from row gamma-1           */
#define PLANT_NO_TEMPERATURE 5       /* temperature ignored                    */
#define PLANT_GREEDY_TIE_HIGH 6      /* greedy ties go to the highest index    */
#define PLANT_ENTROPY_NATS 7         /* entropy in nats                        */
#define PLANT_SIGNAL_MEAN_OVER_G 8   /* signal means divide by G, not gamma_b  */
#define PLANT_DRAW_NONSTRICT 9       /* smallest x with C(x) >= t              */
#define PLANT_ONEHOT_KEEP_Y 10       /* one-hot residual keeps y               */
#define PLANT_NO_STOP 11             /* keeps testing after a reject           */
#define PLANT_ACCEPT_NONSTRICT 12    /* accept iff u <= a                      */
#define PLANT_PROBE_NEXT_BUCKET 13   /* probe distance to the bucket after it  */
#define PLANT_MARGIN_ONE_SIDED 14    /* draw margin to the upper edge only     */
#define PLANT_ACCEPT_MARGIN_UNNORM 15 /* accept margin |u q(y) - p(y)|         */
#define PLANT_DIV_NATS 16            /* divergence KL and H in nats            */
#define PLANT_DIV_KL_SWAPPED 17      /* KL(p||q) slot holds KL(q||p)           */
#define PLANT_DIV_L1_HALF 18         /* L1 slot holds TV = L1 / 2              */
#define PLANT_DIV_A_MAX 19           /* A = sum max(p, q)                      */
#define PLANT_DIV_H_DRAFT 20         /* entropy of q instead of p              */
#define PLANT_GSEL_NO_RELU 21        /* gamma selector: hidden layer linear    */
#define PLANT_GSEL_NO_GAMMA_FACTOR 22 /* selector maximises f + 1, not f g + 1 */
#define PLANT_GSEL_TIE_HIGH 23       /* selector ties go to the larger gamma   */
#define PLANT_GSEL_FEATURE_ORDER 24  /* features in the library's signal order */
#define PLANT_FILT_TOPK_STRICT 25    /* top-k keeps x > k-th value, not >=     */
#define PLANT_FILT_TOPP_EXCLUSIVE 26 /* top-p stops before the crossing value  */
#define PLANT_FILT_TOPP_BEFORE_TOPK 27 /* top-p mass over the unfiltered row   */
#define PLANT_FILT_NO_TEMPERATURE 28 /* top-p mass at T = 1                     */

/* dtype codes of the input logits */
#define ORACLE_F32 0
#define ORACLE_BF16 1
#define ORACLE_F64 2

/* modes */
#define ORACLE_GREEDY 0
#define ORACLE_SAMPLE 1
#define ORACLE_ONEHOT 2
#define ORACLE_SIGNALS 3

/* per-request status bits */
#define OST_NONFINITE 1
#define OST_BAD_TOKEN 2
#define OST_BAD_GAMMA 4
#define OST_ZERO_RESIDUAL 8
#define OST_BAD_TEMPERATURE 64
#define OST_BAD_UNIFORM 128

/* ------------------------------------------------------------------------ */
/* input decoding                                                            */

/* bf16 is the top half of an IEEE binary32; widening to fp64 is exact. */
static double bf16_bits_to_double(uint16_t h)
{
    uint32_t w = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/* Copy logit row `row` (V entries) of a [*, V] array into fp64. */
static void load_row(const void* base, int dtype, size_t row, int V, double* out)
{
    size_t off = row * (size_t)V;
    if (dtype == ORACLE_BF16) {
        const uint16_t* p = (const uint16_t*)base + off;
        for (int v = 0; v < V; ++v) out[v] = bf16_bits_to_double(p[v]);
    } else if (dtype == ORACLE_F32) {
        const float* p = (const float*)base + off;
        for (int v = 0; v < V; ++v) out[v] = (double)p[v];
    } else {
        const double* p = (const double*)base + off;
        for (int v = 0; v < V; ++v) out[v] = p[v];
    }
}

/* ------------------------------------------------------------------------ */
/* the distributions                                                         */

/* Row is usable iff it holds no NaN, no +inf and has a finite maximum. */
static int row_max(const double* x, int V, double* m_out)
{
    double m = -INFINITY;
    for (int v = 0; v < V; ++v) {
        if (isnan(x[v])) return 0;
        if (x[v] > m) m = x[v];
    }
    if (!isfinite(m)) return 0;
    *m_out = m;
    return 1;
}

/* p(v) = exp((x_v - m)/T) / sum_z exp((x_z - m)/T): the temperature softmax
 * that the tutorial page (section 2.1) says p and q already include.
 * Returns 0 if the row is unusable. */
static int softmax_t(const double* x, int V, double T, double* p)
{
    double m;
    if (!row_max(x, V, &m)) return 0;
#if ORACLE_PLANT == PLANT_NO_TEMPERATURE
    T = 1.0;
#endif
    double S = 0.0;
    for (int v = 0; v < V; ++v) {
        p[v] = exp((x[v] - m) / T);
        S += p[v];
    }
    for (int v = 0; v < V; ++v) p[v] /= S;
    return 1;
}

/* Target argmax, lowest index among equal maxima (section 3.1 of the
 * tutorial page asks that tie handling agree; this is the reading). */
static int argmax_lowest(const double* x, int V, int* g)
{
    double m;
    if (!row_max(x, V, &m)) return 0;
    for (int v = 0; v < V; ++v) {
#if ORACLE_PLANT == PLANT_GREEDY_TIE_HIGH
        if (x[v] == m) *g = v;
#else
        if (x[v] == m) { *g = v; return 1; }
#endif
    }
    return 1;
}

/* Inverse-CDF draw from unnormalised non-negative weights w.
 * W = sum_v w_v (ascending), t = u W, token = smallest x with C(x) > t.
 * margin = distance from t to the nearer edge of the chosen bucket, over W.
 * If probe >= 0, *probe_dist = distance from t to the bucket
 * [C(probe-1), C(probe)) over W (0 when t lies inside it). */
static int draw_inverse_cdf(const double* w, int V, double u, double* margin,
                            int probe, double* probe_dist)
{
    double W = 0.0;
    for (int v = 0; v < V; ++v) W += w[v];
    double t = u * W;
    double C = 0.0, Cprev = 0.0;
    int z = -1;
    for (int v = 0; v < V; ++v) {
        Cprev = C;
        C += w[v];
#if ORACLE_PLANT == PLANT_PROBE_NEXT_BUCKET
        if (probe == v - 1 && probe_dist) {
#else
        if (probe == v && probe_dist) {
#endif
            double d = 0.0;
            if (t < Cprev) d = Cprev - t;
            else if (t >= C) d = t - C;
            *probe_dist = d / W;
        }
#if ORACLE_PLANT == PLANT_DRAW_NONSTRICT
        if (z < 0 && C >= t && w[v] >= 0.0) {
#else
        if (z < 0 && C > t) {
#endif
            z = v;
            double d0 = t - Cprev, d1 = C - t;
#if ORACLE_PLANT == PLANT_MARGIN_ONE_SIDED
            d0 = d1;
#endif
            *margin = (d0 < d1 ? d0 : d1) / W;
        }
    }
    if (z < 0) { /* rounding left t >= C(V-1): take the last positive weight */
        for (int v = V - 1; v >= 0; --v)
            if (w[v] > 0.0) { z = v; break; }
        *margin = 0.0;
    }
    return z;
}

/* Entropy in bits and max-probability of a normalised row (SpecKV page,
 * signal extraction); 0 log 0 = 0. */
static void entropy_conf(const double* q, int V, double* H, double* c)
{
    double h = 0.0, mx = 0.0;
    for (int v = 0; v < V; ++v) {
        if (q[v] > 0.0) {
#if ORACLE_PLANT == PLANT_ENTROPY_NATS
            h -= q[v] * log(q[v]);
#else
            h -= q[v] * log2(q[v]);
#endif
        }
        if (q[v] > mx) mx = q[v];
    }
    *H = h;
    *c = mx;
}

/* ------------------------------------------------------------------------ */
/* one request                                                               */

typedef struct {
    int mode;
    const void* target;
    const void* draft;
    int dtype, B, G, V;
    const int32_t* draft_tokens;
    const int32_t* gamma;
    const float* temperature;
    const float* uniforms;
    int32_t* accept_len;
    int32_t* tokens;
    int32_t* status;
    double* signals;
    double* row_signals;
    double* accept_prob;
    double* accept_margin;
    double* draw_margin;
    const int32_t* probe_token;
    double* probe_distance;
} job_t;

static int uniform_ok(double u) { return u >= 0.0 && u < 1.0; }

static void run_request(const job_t* J, int b, double* x, double* p, double* q, double* w)
{
    const int G = J->G, V = J->V, mode = J->mode;
    const int gam = J->gamma ? J->gamma[b] : G;
    int st = 0;
    const double NaN = NAN;

    /* outputs start as "nothing committed" */
    if (J->accept_len) J->accept_len[b] = 0;
    if (J->tokens) for (int i = 0; i <= G; ++i) J->tokens[(size_t)b * (G + 1) + i] = -1;
    if (J->accept_prob) for (int i = 0; i < G; ++i) J->accept_prob[(size_t)b * G + i] = NaN;
    if (J->accept_margin) for (int i = 0; i < G; ++i) J->accept_margin[(size_t)b * G + i] = NaN;
    if (J->draw_margin) J->draw_margin[b] = NaN;
    if (J->probe_distance) J->probe_distance[b] = NaN;
    if (J->signals) for (int j = 0; j < 4; ++j) J->signals[(size_t)b * 4 + j] = NaN;
    if (J->row_signals) for (int i = 0; i < 2 * G; ++i) J->row_signals[(size_t)b * 2 * G + i] = NaN;

    double T = 1.0;
    if (gam < 0 || gam > G) st |= OST_BAD_GAMMA;
    if (mode != ORACLE_GREEDY) {
        T = (double)J->temperature[b];
        if (!(T > 0.0) || !isfinite(T)) st |= OST_BAD_TEMPERATURE;
    }
    if (st) goto done;

    /* draft signals: every draft row i < gamma_b */
    if (J->signals || J->row_signals) {
        double Hsum = 0.0, Hmax = -INFINITY, csum = 0.0, cmin = INFINITY;
        for (int i = 0; i < gam; ++i) {
            load_row(J->draft, J->dtype, (size_t)b * G + i, V, x);
            if (!softmax_t(x, V, T, q)) { st |= OST_NONFINITE; goto done; }
            double H, c;
            entropy_conf(q, V, &H, &c);
            Hsum += H; csum += c;
            if (H > Hmax) Hmax = H;
            if (c < cmin) cmin = c;
            if (J->row_signals) {
                J->row_signals[((size_t)b * G + i) * 2 + 0] = H;
                J->row_signals[((size_t)b * G + i) * 2 + 1] = c;
            }
        }
        if (J->signals && gam > 0) {
#if ORACLE_PLANT == PLANT_SIGNAL_MEAN_OVER_G
            double n = (double)G;
#else
            double n = (double)gam;
#endif
            J->signals[(size_t)b * 4 + 0] = Hsum / n;
            J->signals[(size_t)b * 4 + 1] = Hmax;
            J->signals[(size_t)b * 4 + 2] = csum / n;
            J->signals[(size_t)b * 4 + 3] = cmin;
        }
    }
    if (mode == ORACLE_SIGNALS) goto done;

    const int32_t* y = J->draft_tokens ? J->draft_tokens + (size_t)b * G : NULL;
    const float* u = J->uniforms ? J->uniforms + (size_t)b * (G + 1) : NULL;
    int k = gam;          /* first reject (or gamma when all accepted) */
    int rejected = 0;

    if (mode == ORACLE_GREEDY) {
        /* section 3.1: accept y_i iff it equals argmax p_i, else emit argmax */
        int z = -1;
        for (int i = 0; i < gam; ++i) {
            load_row(J->target, J->dtype, (size_t)b * (G + 1) + i, V, x);
            int g;
            if (!argmax_lowest(x, V, &g)) { st |= OST_NONFINITE; goto done; }
            if (y[i] < 0 || y[i] >= V) { st |= OST_BAD_TOKEN; goto done; }
            if (y[i] != g) { k = i; z = g; break; }
        }
        if (z < 0) {
            load_row(J->target, J->dtype, (size_t)b * (G + 1) + gam, V, x);
            if (!argmax_lowest(x, V, &z)) { st |= OST_NONFINITE; goto done; }
        }
        if (J->accept_len) J->accept_len[b] = k;
        if (J->tokens) {
            for (int i = 0; i < k; ++i) J->tokens[(size_t)b * (G + 1) + i] = y[i];
            J->tokens[(size_t)b * (G + 1) + k] = z;
        }
        goto done;
    }

    /* stochastic modes: sections 3.2 / 3.3 of the tutorial page */
    for (int i = 0; i < gam; ++i) {
        load_row(J->target, J->dtype, (size_t)b * (G + 1) + i, V, x);
        if (!softmax_t(x, V, T, p)) { st |= OST_NONFINITE; goto done; }
        double qy;
        if (mode == ORACLE_SAMPLE) {
            load_row(J->draft, J->dtype, (size_t)b * G + i, V, x);
            if (!softmax_t(x, V, T, q)) { st |= OST_NONFINITE; goto done; }
        }
        if (y[i] < 0 || y[i] >= V) { st |= OST_BAD_TOKEN; goto done; }
        double ui = (double)u[i];
        if (!uniform_ok(ui)) { st |= OST_BAD_UNIFORM; goto done; }
        double py = p[y[i]];
        qy = (mode == ORACLE_SAMPLE) ? q[y[i]] : 1.0;   /* one-hot q: q(y) = 1 */
        double a;
        if (qy > 0.0) a = py / qy < 1.0 ? py / qy : 1.0;
        else a = py > 0.0 ? 1.0 : 0.0;
#if ORACLE_PLANT == PLANT_RATIO_INVERTED
        int accept = ui * py < qy;
#elif ORACLE_PLANT == PLANT_ACCEPT_NONSTRICT
        int accept = ui <= a;
#else
        int accept = ui * qy < py;
#endif
        if (J->accept_prob) J->accept_prob[(size_t)b * G + i] = a;
#if ORACLE_PLANT == PLANT_ACCEPT_MARGIN_UNNORM
        if (J->accept_margin) J->accept_margin[(size_t)b * G + i] = fabs(ui * qy - py);
#else
        if (J->accept_margin) J->accept_margin[(size_t)b * G + i] = fabs(ui - a);
#endif
        if (!accept) {
#if ORACLE_PLANT == PLANT_NO_STOP
            /* keeps going and remembers the residual of the last reject */
            k = i;
            rejected = 1;
            if (mode == ORACLE_SAMPLE) {
                for (int v = 0; v < V; ++v) w[v] = p[v] - q[v] > 0.0 ? p[v] - q[v] : 0.0;
            } else {
                for (int v = 0; v < V; ++v) w[v] = p[v];
                w[y[i]] = 0.0;
            }
            continue;
#else
            k = i;
            rejected = 1;
            break;
#endif
        }
    }
#if ORACLE_PLANT == PLANT_NO_STOP
    if (rejected) goto draw_ready;
#endif

    if (rejected) {
        /* residual of the rejected position; p, q still hold that row */
        if (mode == ORACLE_SAMPLE) {
            for (int v = 0; v < V; ++v) {
#if ORACLE_PLANT == PLANT_RESAMPLE_FROM_P
                w[v] = p[v];
#elif ORACLE_PLANT == PLANT_RESIDUAL_SIGN
                w[v] = q[v] - p[v] > 0.0 ? q[v] - p[v] : 0.0;
#else
                w[v] = p[v] - q[v] > 0.0 ? p[v] - q[v] : 0.0;
#endif
            }
        } else {
            for (int v = 0; v < V; ++v) w[v] = p[v];
#if ORACLE_PLANT != PLANT_ONEHOT_KEEP_Y
            w[y[k]] = 0.0;
#endif
        }
    } else {
        /* section 5.2: the bonus token from p_{gamma+1} (row gamma here) */
#if ORACLE_PLANT == PLANT_BONUS_ROW
        int brow = gam > 0 ? gam - 1 : 0;
#else
        int brow = gam;
#endif
        load_row(J->target, J->dtype, (size_t)b * (G + 1) + brow, V, x);
        if (!softmax_t(x, V, T, p)) { st |= OST_NONFINITE; goto done; }
        for (int v = 0; v < V; ++v) w[v] = p[v];
    }
#if ORACLE_PLANT == PLANT_NO_STOP
draw_ready:
#endif
    {
        double ud = (double)u[G];
        if (!uniform_ok(ud)) { st |= OST_BAD_UNIFORM; goto done; }
        double W = 0.0;
        for (int v = 0; v < V; ++v) W += w[v];
        if (!(W > 0.0)) {            /* fp fallback: draw from p itself */
            for (int v = 0; v < V; ++v) w[v] = p[v];
            st |= OST_ZERO_RESIDUAL;
        }
        double margin = 0.0, pd = NaN;
        int probe = J->probe_token ? J->probe_token[b] : -1;
        int z = draw_inverse_cdf(w, V, ud, &margin, probe, &pd);
        if (J->draw_margin) J->draw_margin[b] = margin;
        if (J->probe_distance) J->probe_distance[b] = pd;
        if (J->accept_len) J->accept_len[b] = k;
        if (J->tokens) {
            for (int i = 0; i < k; ++i) J->tokens[(size_t)b * (G + 1) + i] = y[i];
            J->tokens[(size_t)b * (G + 1) + k] = z;
        }
    }

done:
    if (st & ~OST_ZERO_RESIDUAL) {
        /* an error voids the request: nothing committed, no signals */
        if (J->accept_len) J->accept_len[b] = 0;
        if (J->tokens) for (int i = 0; i <= G; ++i) J->tokens[(size_t)b * (G + 1) + i] = -1;
        if (J->accept_prob) for (int i = 0; i < G; ++i) J->accept_prob[(size_t)b * G + i] = NaN;
        if (J->signals) for (int j = 0; j < 4; ++j) J->signals[(size_t)b * 4 + j] = NaN;
        if (J->row_signals) for (int i = 0; i < 2 * G; ++i) J->row_signals[(size_t)b * 2 * G + i] = NaN;
        if (J->draw_margin) J->draw_margin[b] = NaN;
    }
    if (J->status) J->status[b] = st;
}

/* ------------------------------------------------------------------------ */
/* entry point                                                               */

/* Run the oracle over B requests.  Layouts (row-major, contiguous):
 *   target [B, G+1, V], draft [B, G, V] (dtype: 0 f32, 1 bf16, 2 f64),
 *   draft_tokens [B, G], gamma [B] or NULL (= G), temperature [B],
 *   uniforms [B, G+1];
 * outputs, each optional (NULL = not wanted):
 *   accept_len [B], tokens [B, G+1], status [B], signals [B, 4]
 *   (mean H, max H, mean c, min c), row_signals [B, G, 2] (H_i, c_i),
 *   accept_prob [B, G], accept_margin [B, G] (|u_i - a_i|),
 *   draw_margin [B], probe_distance [B] (needs probe_token [B]).
 * Returns 0, or -1 on a bad argument or allocation failure. */
int oracle_run(int mode, const void* target, const void* draft, int dtype,
               int B, int G, int V,
               const int32_t* draft_tokens, const int32_t* gamma,
               const float* temperature, const float* uniforms,
               int32_t* accept_len, int32_t* tokens, int32_t* status,
               double* signals, double* row_signals, double* accept_prob,
               double* accept_margin, double* draw_margin,
               const int32_t* probe_token, double* probe_distance,
               int nthreads)
{
    if (B < 0 || G < 0 || V < 1 || dtype < 0 || dtype > 2 || mode < 0 || mode > 3) return -1;
    if (mode != ORACLE_SIGNALS && !target) return -1;
    if ((mode == ORACLE_SAMPLE || mode == ORACLE_SIGNALS) && G > 0 && !draft) return -1;
    if (mode != ORACLE_SIGNALS && G > 0 && !draft_tokens) return -1;
    if (mode != ORACLE_GREEDY && (!temperature)) return -1;
    if ((mode == ORACLE_SAMPLE || mode == ORACLE_ONEHOT) && !uniforms) return -1;
    if (mode != ORACLE_SAMPLE && mode != ORACLE_SIGNALS) { signals = NULL; row_signals = NULL; }
    job_t J = {mode, target, draft, dtype, B, G, V, draft_tokens, gamma, temperature, uniforms,
               accept_len, tokens, status, signals, row_signals, accept_prob,
               accept_margin, draw_margin, probe_token, probe_distance};
    int failed = 0;
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel num_threads(nthreads)
    {
        double* buf = (double*)malloc(sizeof(double) * (size_t)V * 4);
        if (!buf) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int b = 0; b < B; ++b) {
            if (buf) run_request(&J, b, buf, buf + V, buf + 2 * (size_t)V, buf + 3 * (size_t)V);
        }
        free(buf);
    }
    return failed ? -1 : 0;
}

/* ------------------------------------------------------------------------ */
/* per-position divergence statistics                                        */

/* The statistics of one position from its two normalised rows p (target)
 * and q (draft), sums in ascending token order:
 *   out[0] = A   = sum_v min(p(v), q(v))  (= 1 - TV(p, q), the expected
 *                acceptance of the position: tutorial page section 4.3);
 *   out[1] = L1  = sum_v |p(v) - q(v)|    (= 2 TV; the L1 distance of the
 *                DLite page's TV loss and of the DDTE page's selector inputs);
 *   out[2] = KL(p||q) = sum_{p(v)>0} p(v) log2(p(v)/q(v))  (forward KL of the
 *                DLite page; +inf if some q(v) = 0 < p(v));
 *   out[3] = KL(q||p), likewise (the DDTE page's "bidirectional KL");
 *   out[4] = H(p) = -sum_v p(v) log2 p(v)  (target entropy, DDTE page).
 * Reading: information quantities in bits, as the SpecKV signals. */
static void divergence_row(const double* p, const double* q, int V, double* out)
{
    double A = 0.0, L1 = 0.0, kpq = 0.0, kqp = 0.0, H = 0.0;
    for (int v = 0; v < V; ++v) {
        const double a = p[v], b = q[v];
#if ORACLE_PLANT == PLANT_DIV_A_MAX
        A += a > b ? a : b;
#else
        A += a < b ? a : b;
#endif
        L1 += fabs(a - b);
#if ORACLE_PLANT == PLANT_DIV_NATS
        if (a > 0.0) kpq += a * log(a / b);
        if (b > 0.0) kqp += b * log(b / a);
        if (a > 0.0) H -= a * log(a);
#else
        if (a > 0.0) kpq += a * log2(a / b);
        if (b > 0.0) kqp += b * log2(b / a);
#if ORACLE_PLANT == PLANT_DIV_H_DRAFT
        if (b > 0.0) H -= b * log2(b);
#else
        if (a > 0.0) H -= a * log2(a);
#endif
#endif
    }
#if ORACLE_PLANT == PLANT_DIV_L1_HALF
    L1 *= 0.5;
#endif
    out[0] = A;
    out[1] = L1;
#if ORACLE_PLANT == PLANT_DIV_KL_SWAPPED
    out[2] = kqp;
    out[3] = kpq;
#else
    out[2] = kpq;
    out[3] = kqp;
#endif
    out[4] = H;
}

/* Per-position divergence statistics (the five of divergence_row) of the
 * target row i and the draft row i of every request, for i < gamma_b, at the
 * request's temperature; stats [B, G, 5] (NaN past gamma_b, for a position
 * whose rows are not usable, and for every position of a request with a bad
 * gamma or temperature); status [B] or NULL: OST_BAD_GAMMA,
 * OST_BAD_TEMPERATURE, OST_NONFINITE (any position's row unusable).
 * Layouts as oracle_run.  Returns 0, or -1 on a bad argument or allocation
 * failure. */
int oracle_divergence(const void* target, const void* draft, int dtype, int B, int G, int V,
                      const int32_t* gamma, const float* temperature, double* stats,
                      int32_t* status, int nthreads)
{
    if (B < 0 || G < 0 || V < 1 || dtype < 0 || dtype > 2 || !stats || !temperature) return -1;
    if (G > 0 && (!target || !draft)) return -1;
    int failed = 0;
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel num_threads(nthreads)
    {
        double* buf = (double*)malloc(sizeof(double) * (size_t)V * 3);
        if (!buf) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int b = 0; b < B; ++b) {
            if (!buf) continue;
            double* x = buf;
            double* p = buf + V;
            double* q = buf + 2 * (size_t)V;
            int st = 0;
            const int gam = gamma ? gamma[b] : G;
            const double T = (double)temperature[b];
            if (gam < 0 || gam > G) st |= OST_BAD_GAMMA;
            if (!(T > 0.0 && isfinite(T))) st |= OST_BAD_TEMPERATURE;
            for (int i = 0; i < G; ++i) {
                double* o = stats + ((size_t)b * G + i) * 5;
                for (int k = 0; k < 5; ++k) o[k] = NAN;
                if ((st & (OST_BAD_GAMMA | OST_BAD_TEMPERATURE)) || i >= gam) continue;
                load_row(target, dtype, (size_t)b * (G + 1) + i, V, x);
                const int okp = softmax_t(x, V, T, p);
                load_row(draft, dtype, (size_t)b * G + i, V, x);
                const int okq = softmax_t(x, V, T, q);
                if (!okp || !okq) {
                    st |= OST_NONFINITE;
                    continue;
                }
                divergence_row(p, q, V, o);
            }
            if (st & (OST_BAD_GAMMA | OST_BAD_TEMPERATURE))
                for (int k = 0; k < G * 5; ++k) stats[(size_t)b * G * 5 + k] = NAN;
            if (status) status[b] = st;
        }
        free(buf);
    }
    return failed ? -1 : 0;
}

/* ------------------------------------------------------------------------ */
/* the SpecKV gamma selector                                                 */

/* The SpecKV page ("接受率预测与 gamma 选择", acceptance prediction and gamma
 * selection): with the context x = [mean H, mean c, max H, min c, comp] of a
 * request, a regressor f(x, gamma) predicts the acceptance rate; the expected
 * tokens of a step are f(x, gamma) gamma + 1, and the policy takes
 * gamma* = argmax over gamma in {2, 4, 6, 8}.  The regressor is an MLP with
 * 16 hidden units.  Readings: its inputs are [x, gamma], standardised as
 * (z - mu) / sd; one ReLU hidden layer; an identity output; ties go to the
 * smallest gamma.
 * Model layout (141 values): mu[6], sd[6], W1[16][6] (row h: the weights of
 * hidden unit h), b1[16], w2[16], b2.
 * signals [B, 4] in the library's order (mean H, max H, mean c, min c);
 * comp [B] or NULL (= 0).  Outputs: gamma_star [B] (-1 when a feature is not
 * finite), expected [B, 4] (f gamma + 1 for gamma = 2, 4, 6, 8). */
static double gsel_f(const double* model, const double* x5, double g)
{
    const double* mu = model;
    const double* sd = model + 6;
    const double* W1 = model + 12;
    const double* b1 = model + 108;
    const double* w2 = model + 124;
    const double b2 = model[140];
    double z[6];
    for (int k = 0; k < 5; ++k) z[k] = x5[k];
    z[5] = g;
    for (int k = 0; k < 6; ++k) z[k] = (z[k] - mu[k]) / sd[k];
    double f = b2;
    for (int h = 0; h < 16; ++h) {
        double a = b1[h];
        for (int k = 0; k < 6; ++k) a += W1[h * 6 + k] * z[k];
#if ORACLE_PLANT != PLANT_GSEL_NO_RELU
        if (a < 0.0) a = 0.0;
#endif
        f += w2[h] * a;
    }
    return f;
}

int oracle_gamma_select(const double* signals, const double* comp, const double* model, int B,
                        int32_t* gamma_star, double* expected)
{
    if (B < 0 || !signals || !model || !gamma_star) return -1;
    static const int cand[4] = {2, 4, 6, 8};
    for (int b = 0; b < B; ++b) {
        const double* s = signals + (size_t)b * 4;
#if ORACLE_PLANT == PLANT_GSEL_FEATURE_ORDER
        const double x5[5] = {s[0], s[1], s[2], s[3], comp ? comp[b] : 0.0};
#else
        const double x5[5] = {s[0], s[2], s[1], s[3], comp ? comp[b] : 0.0};   /* [mean H, mean c, max H, min c, comp] */
#endif
        int finite = 1;
        for (int k = 0; k < 5; ++k) finite &= isfinite(x5[k]);
        int best = -1;
        double bestE = -INFINITY;
        for (int j = 0; j < 4; ++j) {
            double E = NAN;
            if (finite) {
                const double f = gsel_f(model, x5, (double)cand[j]);
#if ORACLE_PLANT == PLANT_GSEL_NO_GAMMA_FACTOR
                E = f + 1.0;
#else
                E = f * cand[j] + 1.0;
#endif
#if ORACLE_PLANT == PLANT_GSEL_TIE_HIGH
                if (E >= bestE) { bestE = E; best = cand[j]; }
#else
                if (E > bestE) { bestE = E; best = cand[j]; }
#endif
            }
            if (expected) expected[(size_t)b * 4 + j] = E;
        }
        gamma_star[b] = finite ? best : -1;
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* top-k / top-p filtering before verification                               */

static int cmp_desc(const void* a, const void* b)
{
    const double x = *(const double*)a, y = *(const double*)b;
    return (x < y) - (x > y);
}

/* Filter one row of logits x[0..V) in place (tutorial page, section 2.1: p
 * and q are the distributions actually sampled from, "temperature / top-k /
 * top-p already applied, if used").  Readings (by value, so ties are kept
 * together):
 *   top-k (k >= 1 and k < V): keep x >= the k-th largest value;
 *   top-p (0 < top_p < 1), on the distribution left by top-k at temperature T:
 *     with the kept values in descending order, t* = the largest value v such
 *     that the mass of {x >= v} is >= top_p; keep x >= t*;
 *   a removed token becomes -inf.
 * margin (optional): for top-p, the distance of top_p from the nearer of the
 * masses of {x >= t*} and {x > t*} (a decision within rounding of its
 * threshold can come out either way in fp32).  Returns 0 if the row holds NaN
 * or +inf or has no finite maximum (left unchanged), else 1. */
static int filter_row(double* x, int V, int k, double top_p, double T, double* sorted, double* margin)
{
    double m;
    if (!row_max(x, V, &m)) return 0;
    if (margin) *margin = INFINITY;
    memcpy(sorted, x, sizeof(double) * (size_t)V);
    qsort(sorted, (size_t)V, sizeof(double), cmp_desc);
    double thr = -INFINITY;
    if (k >= 1 && k < V) {
        thr = sorted[k - 1];
#if ORACLE_PLANT == PLANT_FILT_TOPK_STRICT
        for (int v = 0; v < V; ++v) if (!(x[v] > thr)) x[v] = -INFINITY;
        thr = -INFINITY;
        memcpy(sorted, x, sizeof(double) * (size_t)V);
        qsort(sorted, (size_t)V, sizeof(double), cmp_desc);
#endif
    }
    if (top_p > 0.0 && top_p < 1.0) {
#if ORACLE_PLANT == PLANT_FILT_TOPP_BEFORE_TOPK
        const double lim = -INFINITY;
#else
        const double lim = thr;
#endif
#if ORACLE_PLANT == PLANT_FILT_NO_TEMPERATURE
        T = 1.0;
#endif
        double S = 0.0;
        for (int v = 0; v < V; ++v)
            if (sorted[v] >= lim) S += exp((sorted[v] - m) / T);
        double C = 0.0, Cprev = 0.0;
        double tstar = -INFINITY;
        for (int v = 0; v < V && sorted[v] >= lim;) {
            int w = v;
            double mass = 0.0;
            while (w < V && sorted[w] == sorted[v]) { mass += exp((sorted[w] - m) / T); ++w; }
            Cprev = C;
            C += mass;
            if (C / S >= top_p) {
#if ORACLE_PLANT == PLANT_FILT_TOPP_EXCLUSIVE
                tstar = v > 0 ? sorted[v - 1] : sorted[v];
#else
                tstar = sorted[v];
#endif
                if (margin) {
                    const double d1 = C / S - top_p, d0 = top_p - Cprev / S;
                    *margin = d0 < d1 ? d0 : d1;
                }
                break;
            }
            v = w;
        }
        if (tstar > thr) thr = tstar;
    }
    for (int v = 0; v < V; ++v)
        if (x[v] < thr) x[v] = -INFINITY;
    return 1;
}

/* Filter n rows [n, V] of logits (dtype 0 f32, 1 bf16 as uint16 bits, 2 f64)
 * into out [n, V] fp64 (a row with NaN, +inf or no finite maximum is copied
 * unchanged and gets status OST_NONFINITE).  top_k [n] int32 or NULL (no
 * top-k), top_p [n] or NULL (no top-p), temperature [n] or NULL (= 1; only
 * top-p uses it; an invalid temperature with top-p in use gives status
 * OST_BAD_TEMPERATURE and the row unchanged); margin [n] or NULL.
 * Returns 0, or -1 on a bad argument or allocation failure. */
int oracle_filter(const void* logits, int dtype, int n, int V, const int32_t* top_k, const float* top_p,
                  const float* temperature, double* out, int32_t* status, double* margin, int nthreads)
{
    if (n < 0 || V < 1 || dtype < 0 || dtype > 2 || !logits || !out) return -1;
    int failed = 0;
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel num_threads(nthreads)
    {
        double* buf = (double*)malloc(sizeof(double) * (size_t)V);
        if (!buf) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int r = 0; r < n; ++r) {
            if (!buf) continue;
            double* x = out + (size_t)r * V;
            load_row(logits, dtype, (size_t)r, V, x);
            const double pp = top_p ? (double)top_p[r] : 1.0;
            const double T = temperature ? (double)temperature[r] : 1.0;
            int st = 0;
            double mg = INFINITY;
            if (pp > 0.0 && pp < 1.0 && !(T > 0.0 && isfinite(T))) st = OST_BAD_TEMPERATURE;
            else if (!filter_row(x, V, top_k ? top_k[r] : 0, pp, T, buf, &mg)) st = OST_NONFINITE;
            if (st) load_row(logits, dtype, (size_t)r, V, x);
            if (status) status[r] = st;
            if (margin) margin[r] = mg;
        }
        free(buf);
    }
    return failed ? -1 : 0;
}

/* Which planted mistake this build carries (0 = none). */
int oracle_plant_id(void) { return ORACLE_PLANT; }
