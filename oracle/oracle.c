/*
 * oracle.c -- reference definition of batched speculative verification and of
 * the confidence-scheduled verify-length selector, written as plain,
 * single-threaded fp64 C.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, constant table or helper with the CUDA path, and it is never on the
 * product path.
 *
 * Sources (pages on speculative decoding):
 *   [AS]  "AngelSpec: Towards Real-World High Performance Inference with
 *         Speculative Decoding" -- §2.3 eqs. (4)-(5) (TV distance, overlap);
 *         §4.1 (keep depths n_i, budget K = sum (n_i + 1)); §4.2 eqs. (19)-(24)
 *         (prefix survival, estimated progress, top-K with shallow-first ties,
 *         budget selection against a profiled cost).
 *   [BL]  "breaking down dspark and its lineage" (blog) -- section
 *         "Preserving the target distribution during verification" (accept if
 *         p(x) >= q(x), else with probability p(x)/q(x); on rejection resample
 *         from the normalised residual max(p - q, 0)); section "Verify smarter,
 *         not longer" (prefix scheduler in prose).
 *   [US]  "UraionSpec: A Faithful Implementation of Confidence-Scheduled
 *         Speculative Decoding" -- §2.1 eq. (acceptance) and eq. (expected_tau);
 *         §3.5 Algorithm 1 (hardware-aware prefix scheduler).
 *
 * Readings taken where the pages are silent (each is also listed in the design
 * notes):
 *   - Temperature: p = softmax(z / T).  T == 0 is greedy: accept while the
 *     draft token equals the target argmax; the emitted token is the target
 *     argmax of the first rejected row (or of row ell_b).  Argmax ties go to
 *     the lowest index.
 *   - Accept test written without division: accept iff u * q(x) < p(x), which
 *     equals u < min(1, p(x)/q(x)) for u in [0, 1).
 *   - Uniform slots per request: [0, gamma) accept tests by position, gamma
 *     the residual draw, gamma + 1 the bonus draw.
 *   - Residual on rejection at n < ell_b; bonus from p of target row ell_b when
 *     every tested draft is accepted ([BL], [AS] §1); ell_b = 0 is a pure draw
 *     from p of target row 0.
 *   - Draw by inverse CDF: the smallest v with cumsum_{i<=v} w_i > u * sum(w),
 *     cumsum left to right in fp64.  If the residual sums to zero in floating
 *     point, draw from p of the same row instead.  If rounding leaves no v, take
 *     the last v with positive weight.
 *   - A needed row whose max is not finite (a NaN, +inf, or all -inf) makes the
 *     request invalid, as do a draft token outside [0, V) at a tested position,
 *     a uniform outside [0, 1) in a used slot, or ell_b outside [0, gamma].
 *     Invalid requests emit accept_len -1 and tokens -1.
 *   - Scheduler budget N = sum_b (ell_b + 1) (bonus positions count) and the
 *     objective is tau(N) / C(N), C a piecewise-linear cost table.
 *   - Progress sums are exact in fixed point: survivals rounded to multiples
 *     of 2^-46, summed as 64-bit integers (order-free).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Per-request status values (same numbers as the library's error codes). */
#define OR_OK 0
#define OR_ERR_SHAPE -2
#define OR_ERR_TEMPERATURE -4
#define OR_ERR_VERIFY_LEN -5
#define OR_ERR_TOKEN -6
#define OR_ERR_COST_TABLE -8
#define OR_ERR_NONFINITE -9
#define OR_ERR_UNIFORM -12
#define OR_ERR_CONFIDENCE -13

/* event bits reported per request */
#define EV_RESIDUAL_EMPTY 1 /* residual summed to zero: drew from p instead */
#define EV_NO_BIN 2         /* rounding left no bin above u*W: took last positive */

/* ------------------------------------------------------------------ inputs */

/* Widen one stored logit to fp64.  dtype 0 = fp32, 1 = bf16 (upper half of an
 * fp32 bit pattern), both exact. */
static double logit_at(const void* base, int dtype, int64_t idx) {
    if (dtype == 0) return (double)((const float*)base)[idx];
    uint32_t bits = (uint32_t)((const uint16_t*)base)[idx] << 16;
    float f;
    memcpy(&f, &bits, 4);
    return (double)f;
}

/* ------------------------------------------------- softmax of one row (T>0)
 * p_v = exp(y_v - m) / sum_u exp(y_u - m), y = z / T, m = max y.
 * The temperature-scaled softmax the acceptance rule is stated on
 * ([US] §2.1 eq. (acceptance); [AS] §2.5 names T = 0 and T = 0.9 settings).
 * Returns OR_ERR_NONFINITE when the row max is not finite. */
static int row_softmax(const void* base, int dtype, int64_t off, int V, double T, double* p) {
    double m = -INFINITY;
    for (int v = 0; v < V; ++v) {
        double y = logit_at(base, dtype, off + v) / T;
        if (isnan(y)) return OR_ERR_NONFINITE;
        p[v] = y;
        if (y > m) m = y;
    }
    if (!isfinite(m)) return OR_ERR_NONFINITE;
    double S = 0.0;
    for (int v = 0; v < V; ++v) {
        p[v] = exp(p[v] - m);
        S += p[v];
    }
    for (int v = 0; v < V; ++v) p[v] = p[v] / S;
    return OR_OK;
}

/* Greedy row: argmax of z with the lowest index on ties. */
static int row_argmax(const void* base, int dtype, int64_t off, int V, int32_t* arg) {
    double m = -INFINITY;
    int32_t a = 0;
    int have = 0;
    for (int v = 0; v < V; ++v) {
        double z = logit_at(base, dtype, off + v);
        if (isnan(z)) return OR_ERR_NONFINITE;
        if (!have || z > m) { m = z; a = v; have = 1; }
    }
    if (!isfinite(m)) return OR_ERR_NONFINITE;
    *arg = a;
    return OR_OK;
}

/* Inverse-CDF draw over nonnegative weights w[0..V-1]:
 * the smallest v with (w_0 + ... + w_v) > u * W, W the left-to-right sum.
 * Writes the normalised CDF edges of the chosen bin to *lo, *hi. */
static int32_t inverse_cdf(const double* w, int V, double u, double* lo, double* hi, int* ev) {
    double W = 0.0;
    for (int v = 0; v < V; ++v) W += w[v];
    double target = u * W;
    double cum = 0.0;
    for (int v = 0; v < V; ++v) {
        double before = cum;
        cum += w[v];
        if (cum > target) {
            *lo = before / W;
            *hi = cum / W;
            return v;
        }
    }
    /* rounding left no bin: the last bin with positive weight */
    *ev |= EV_NO_BIN;
    cum = 0.0;
    int32_t last = V - 1;
    double lo_last = 0.0, hi_last = 1.0;
    for (int v = 0; v < V; ++v) {
        double before = cum;
        cum += w[v];
        if (w[v] > 0.0) { last = v; lo_last = before / W; hi_last = cum / W; }
    }
    *lo = lo_last;
    *hi = hi_last;
    return last;
}

static int uniform_ok(float u) { return u >= 0.0f && u < 1.0f; }

/* The weights of the draw that emits the token at position n of request b
 * (n accepted drafts out of ell tested), T > 0:
 *   n < ell : [BL] residual w = max(p_n - q_n, 0), p_n from target row n and
 *             q_n from draft row n; if it sums to zero in floating point, w =
 *             p_n instead (EV_RESIDUAL_EMPTY);
 *   n == ell: the bonus draw, w = p of target row ell ([AS] §1, §4.1).
 * p, q: scratch of V doubles.  Returns the uniform slot of the draw (gamma for
 * the residual, gamma + 1 for the bonus). */
static int draw_weights(const void* target, const void* draft, int dtype, int b, int gamma, int V, int n,
                        int ell, double T, double* p, double* q, double* w, int* ev) {
    const int G1 = gamma + 1;
    row_softmax(target, dtype, ((int64_t)b * G1 + n) * V, V, T, p);
    if (n < ell) {
        row_softmax(draft, dtype, ((int64_t)b * gamma + n) * V, V, T, q);
        double W = 0.0;
        for (int v = 0; v < V; ++v) {
            double d = p[v] - q[v];
            w[v] = d > 0.0 ? d : 0.0;
            W += w[v];
        }
        if (!(W > 0.0)) {
            *ev |= EV_RESIDUAL_EMPTY;
            for (int v = 0; v < V; ++v) w[v] = p[v];
        }
        return gamma;
    }
    for (int v = 0; v < V; ++v) w[v] = p[v];
    return gamma + 1;
}

/* -------------------------------------------------------------- verification
 * Batched lossless verification, one request at a time.
 *
 * Layouts (row-major, contiguous):
 *   target   [B, gamma+1, V]  dtype 0 fp32 / 1 bf16
 *   draft    [B, gamma,   V]  (not read when T == 0)
 *   tokens   [B, gamma] int32, verify_len [B] int32 (NULL -> gamma)
 *   uniforms [B, gamma+2] fp32 (not read when T == 0)
 * Outputs: out_tokens [B, gamma+1] (-1 after the emitted token),
 *          out_accept_len [B] (-1 for an invalid request).
 * Diagnostics (each may be NULL):
 *   px, qx      [B, gamma]  p(x_j), q(x_j) for j < ell_b (NaN elsewhere / T == 0)
 *   margin      [B, gamma]  |u_j - p(x_j)/q(x_j)| at every tested position j
 *   resid_mass  [B]         sum of the draw's weights (residual or p)
 *   cdf_lo/hi   [B]         normalised CDF edges of the drawn bin
 *   u_draw      [B]         the uniform the draw used
 *   status      [B]         per-request status
 *   events      [B]         EV_* bits
 * Returns OR_OK, or a shape / temperature error for the whole call. */
int oracle_verify(const void* target, const void* draft, int dtype, int B, int gamma, int V,
                  const int32_t* tokens, const int32_t* verify_len, double T,
                  const float* uniforms, int32_t* out_tokens, int32_t* out_accept_len,
                  double* px, double* qx, double* margin, double* resid_mass, double* cdf_lo,
                  double* cdf_hi, double* u_draw, int32_t* status, int32_t* events) {
    if (B < 0 || gamma < 0 || gamma > 63 || V < 1 || (dtype != 0 && dtype != 1)) return OR_ERR_SHAPE;
    if (!(T >= 0.0) || !isfinite(T)) return OR_ERR_TEMPERATURE;
    const int G1 = gamma + 1, G2 = gamma + 2;
    double* p = (double*)malloc(sizeof(double) * (size_t)V);
    double* q = (double*)malloc(sizeof(double) * (size_t)V);
    double* w = (double*)malloc(sizeof(double) * (size_t)V);
    if (!p || !q || !w) { free(p); free(q); free(w); return OR_ERR_SHAPE; }

    for (int b = 0; b < B; ++b) {
        int32_t* ot = out_tokens + (int64_t)b * G1;
        for (int j = 0; j < G1; ++j) ot[j] = -1;
        out_accept_len[b] = -1;
        for (int j = 0; j < gamma; ++j) {
            if (px) px[(int64_t)b * gamma + j] = NAN;
            if (qx) qx[(int64_t)b * gamma + j] = NAN;
            if (margin) margin[(int64_t)b * gamma + j] = NAN;
        }
        if (resid_mass) resid_mass[b] = NAN;
        if (cdf_lo) cdf_lo[b] = NAN;
        if (cdf_hi) cdf_hi[b] = NAN;
        if (u_draw) u_draw[b] = NAN;
        if (events) events[b] = 0;
        int ev = 0;

        /* validate the request */
        int st = OR_OK;
        int ell = verify_len ? verify_len[b] : gamma;
        const int32_t* x = tokens + (int64_t)b * gamma;
        const float* u = uniforms ? uniforms + (int64_t)b * G2 : NULL;
        if (ell < 0 || ell > gamma) st = OR_ERR_VERIFY_LEN;
        if (st == OR_OK)
            for (int j = 0; j < ell; ++j)
                if (x[j] < 0 || x[j] >= V) { st = OR_ERR_TOKEN; break; }
        if (st == OR_OK && T > 0.0) {
            for (int j = 0; j < ell; ++j)
                if (!uniform_ok(u[j])) st = OR_ERR_UNIFORM;
            if (!uniform_ok(u[gamma]) || !uniform_ok(u[gamma + 1])) st = OR_ERR_UNIFORM;
        }

        if (st == OR_OK && T == 0.0) {
            /* Greedy: accept while x_j equals the target argmax of row j. */
            int32_t am[64];
            for (int j = 0; j <= ell && st == OR_OK; ++j)
                st = row_argmax(target, dtype, ((int64_t)b * G1 + j) * V, V, &am[j]);
            if (st == OR_OK) {
                int n = 0;
                while (n < ell && x[n] == am[n]) ++n;
                for (int j = 0; j < n; ++j) ot[j] = x[j];
                ot[n] = am[n];
                out_accept_len[b] = n;
            }
        } else if (st == OR_OK) {
            /* Every needed row must be valid: target 0..ell, draft 0..ell-1. */
            double pxv[64], qxv[64];
            for (int j = 0; j <= ell && st == OR_OK; ++j) {
                st = row_softmax(target, dtype, ((int64_t)b * G1 + j) * V, V, T, p);
                if (st == OR_OK && j < ell) {
                    pxv[j] = p[x[j]];
                    st = row_softmax(draft, dtype, ((int64_t)b * gamma + j) * V, V, T, q);
                    if (st == OR_OK) qxv[j] = q[x[j]];
                }
            }
            if (st == OR_OK) {
                for (int j = 0; j < ell; ++j) {
                    if (px) px[(int64_t)b * gamma + j] = pxv[j];
                    if (qx) qx[(int64_t)b * gamma + j] = qxv[j];
                }
                /* [US] eq. (acceptance): accept x_j with probability
                 * min(1, p/q); the first rejection ends the prefix. */
                int n = 0;
                while (n < ell) {
                    double uj = (double)u[n];
                    if (margin) margin[(int64_t)b * gamma + n] = fabs(uj - pxv[n] / qxv[n]);
                    if (uj * qxv[n] < pxv[n]) ++n;
                    else break;
                }
                for (int j = 0; j < n; ++j) ot[j] = x[j];

                /* The emitted token at position n. */
                const int slot = draw_weights(target, draft, dtype, b, gamma, V, n, ell, T, p, q, w, &ev);
                const double ud = (double)u[slot];
                double lo = NAN, hi = NAN, W = 0.0;
                for (int v = 0; v < V; ++v) W += w[v];
                int32_t tok = inverse_cdf(w, V, ud, &lo, &hi, &ev);
                ot[n] = tok;
                out_accept_len[b] = n;
                if (resid_mass) resid_mass[b] = W;
                if (cdf_lo) cdf_lo[b] = lo;
                if (cdf_hi) cdf_hi[b] = hi;
                if (u_draw) u_draw[b] = ud;
            }
        }
        if (st != OR_OK) {
            for (int j = 0; j < G1; ++j) ot[j] = -1;
            out_accept_len[b] = -1;
        }
        if (status) status[b] = st;
        if (events) events[b] = ev;
    }
    free(p);
    free(q);
    free(w);
    return OR_OK;
}

/* Normalised CDF edges of queried tokens in the oracle's own draw for request
 * b, given n accepted drafts out of the request's verify length: for token t,
 * lo = (w_0 + ... + w_{t-1}) / W and hi = (w_0 + ... + w_t) / W, with the
 * weights of draw_weights ([BL] residual or the bonus p) and the same
 * left-to-right fp64 sums as the draw itself, W their total.  A draw with
 * uniform u emits t exactly when lo <= u < hi (up to the last-positive-bin
 * rule), so the distance from u to [lo, hi] says how far u is from a value at
 * which t would be the correct token.  T > 0; inputs laid out as for
 * oracle_verify; request b must be valid.  Returns OR_OK or OR_ERR_SHAPE. */
int oracle_draw_cdf(const void* target, const void* draft, int dtype, int B, int gamma, int V,
                    const int32_t* verify_len, double T, int b, int n, const int32_t* query, int nq,
                    double* lo, double* hi) {
    if (b < 0 || b >= B || gamma < 0 || gamma > 63 || V < 1 || !(T > 0.0)) return OR_ERR_SHAPE;
    const int ell = verify_len ? verify_len[b] : gamma;
    if (ell < 0 || ell > gamma || n < 0 || n > ell) return OR_ERR_SHAPE;
    double* p = (double*)malloc(sizeof(double) * (size_t)V);
    double* q = (double*)malloc(sizeof(double) * (size_t)V);
    double* w = (double*)malloc(sizeof(double) * (size_t)V);
    double* cum = (double*)malloc(sizeof(double) * ((size_t)V + 1));
    if (!p || !q || !w || !cum) { free(p); free(q); free(w); free(cum); return OR_ERR_SHAPE; }
    int ev = 0;
    draw_weights(target, draft, dtype, b, gamma, V, n, ell, T, p, q, w, &ev);
    cum[0] = 0.0;
    for (int v = 0; v < V; ++v) cum[v + 1] = cum[v] + w[v];
    const double W = cum[V];
    for (int i = 0; i < nq; ++i) {
        const int t = query[i];
        if (t < 0 || t >= V) {
            lo[i] = hi[i] = NAN;
        } else {
            lo[i] = cum[t] / W;
            hi[i] = cum[t + 1] / W;
        }
    }
    free(p);
    free(q);
    free(w);
    free(cum);
    return OR_OK;
}

/* Oracle of the same verification step on probability vectors given directly
 * (fp64 [B, gamma+1, V] and [B, gamma, V]), used to pin the method on the
 * pages' worked example without a logit round trip.  Same slots and outputs as
 * oracle_verify (T > 0 path). */
int oracle_verify_probs(const double* P, const double* Q, int B, int gamma, int V,
                        const int32_t* tokens, const double* uniforms, int32_t* out_tokens,
                        int32_t* out_accept_len, double* resid_mass) {
    const int G1 = gamma + 1, G2 = gamma + 2;
    double* w = (double*)malloc(sizeof(double) * (size_t)V);
    if (!w) return OR_ERR_SHAPE;
    for (int b = 0; b < B; ++b) {
        const int32_t* x = tokens + (int64_t)b * gamma;
        const double* u = uniforms + (int64_t)b * G2;
        int32_t* ot = out_tokens + (int64_t)b * G1;
        for (int j = 0; j < G1; ++j) ot[j] = -1;
        int n = 0;
        while (n < gamma) {
            double pj = P[((int64_t)b * G1 + n) * V + x[n]];
            double qj = Q[((int64_t)b * gamma + n) * V + x[n]];
            if (u[n] * qj < pj) ++n;
            else break;
        }
        for (int j = 0; j < n; ++j) ot[j] = x[j];
        const double* pn = P + ((int64_t)b * G1 + n) * V;
        double ud, W = 0.0;
        if (n < gamma) {
            const double* qn = Q + ((int64_t)b * gamma + n) * V;
            for (int v = 0; v < V; ++v) {
                double d = pn[v] - qn[v];
                w[v] = d > 0.0 ? d : 0.0;
            }
            ud = u[gamma];
        } else {
            for (int v = 0; v < V; ++v) w[v] = pn[v];
            ud = u[gamma + 1];
        }
        for (int v = 0; v < V; ++v) W += w[v];
        double lo, hi;
        int ev = 0;
        ot[n] = inverse_cdf(w, V, ud, &lo, &hi, &ev);
        out_accept_len[b] = n;
        if (resid_mass) resid_mass[b] = W;
    }
    free(w);
    return OR_OK;
}

/* Dense packing of ragged prefixes ([AS] §4.2, "Packing and correctness": the
 * kept prefixes form one dense verification batch).  Request-major order:
 * request b's ell_b + 1 target rows follow those of requests 0..b-1, and so do
 * its ell_b draft rows; a verify length outside [0, gamma] contributes no rows.
 * Writes the first row of every request and the two row totals. */
int oracle_pack_rows(const int32_t* verify_len, int B, int gamma, int32_t* target_row, int32_t* draft_row,
                     int32_t* totals) {
    if (B < 0 || gamma < 0) return OR_ERR_SHAPE;
    int32_t t = 0, d = 0;
    for (int b = 0; b < B; ++b) {
        target_row[b] = t;
        draft_row[b] = d;
        const int ell = verify_len[b];
        if (ell >= 0 && ell <= gamma) {
            t += ell + 1;
            d += ell;
        }
    }
    totals[0] = t;
    totals[1] = d;
    return OR_OK;
}

/* ----------------------------------------------------------------- scheduler */

/* Piecewise-linear round cost C(N): knots (t_i, c_i) with strictly increasing
 * t, linear between knots, flat beyond both ends.  The evaluation order is
 * fixed: c_i + ((N - t_i) * (c_{i+1} - c_i)) / (t_{i+1} - t_i). */
static double cost_at(double N, const double* kt, const double* kc, int nk) {
    if (N <= kt[0]) return kc[0];
    if (N >= kt[nk - 1]) return kc[nk - 1];
    int i = 0;
    while (!(N < kt[i + 1])) ++i;
    return kc[i] + ((N - kt[i]) * (kc[i + 1] - kc[i])) / (kt[i + 1] - kt[i]);
}

int oracle_cost_at(double N, const double* kt, const double* kc, int nk, double* out) {
    *out = cost_at(N, kt, kc, nk);
    return OR_OK;
}

static int check_sched_args(const float* conf, int B, int gamma, const double* kt, const double* kc,
                            int nk, int min_len) {
    if (B < 0 || gamma < 0 || min_len < 0 || min_len > gamma) return OR_ERR_SHAPE;
    if (nk < 1 || nk > 32) return OR_ERR_COST_TABLE;
    for (int i = 0; i < nk; ++i) {
        if (!isfinite(kt[i]) || !isfinite(kc[i]) || !(kc[i] > 0.0)) return OR_ERR_COST_TABLE;
        if (i > 0 && !(kt[i] > kt[i - 1])) return OR_ERR_COST_TABLE;
    }
    for (int64_t i = 0; i < (int64_t)B * gamma; ++i)
        if (!(conf[i] >= 0.0f && conf[i] <= 1.0f)) return OR_ERR_CONFIDENCE;
    return OR_OK;
}

/* [US] §2.4 / §3.6 (STS): the calibrated confidence c^(1/T_k) of position k;
 * T == NULL leaves the confidence as it is. */
static double calibrated(float c, const double* T, int k) {
    return T ? pow((double)c, 1.0 / T[k - 1]) : (double)c;
}

/* [AS] eq. (20): s_{b,0} = 1, s_{b,k} = prod_{t<=k} c_{b,t}, products taken
 * left to right in fp64.  s has gamma + 1 entries per request. */
static const double* g_sts_T = NULL; /* calibration temperatures of the call in progress */

static void prefix_survival(const float* conf, int B, int gamma, double* s) {
    for (int b = 0; b < B; ++b) {
        double* sb = s + (int64_t)b * (gamma + 1);
        sb[0] = 1.0;
        for (int k = 1; k <= gamma; ++k)
            sb[k] = sb[k - 1] * calibrated(conf[(int64_t)b * gamma + k - 1], g_sts_T, k);
    }
}

/* Selects the calibration temperatures (or NULL) used by the scheduler
 * functions below until the next call. */
int oracle_set_sts(const double* T) {
    g_sts_T = T;
    return OR_OK;
}

/* Progress in fixed point.  [AS] eq. (21) defines the estimated progress as
 * the plain sum A_b(n) = sum_{k=0}^{n} s_{b,k}; the pages fix neither its
 * precision nor its order.  Reading: every survival is rounded (to nearest,
 * ties to even) to a multiple of 2^-46 and the sums are exact in 64-bit
 * integers, so a progress value depends only on the set of survivals summed,
 * never on the order.  Survivals lie in [0, 1] and at most B(gamma+1) <=
 * 4096 * 33 of them are summed, which stays below 2^64.  A progress enters an
 * objective as the double nearest to (integer) * 2^-46. */
#define PROG_FRAC_BITS 46
typedef uint64_t prog_t;

static prog_t prog_quant(double s) {
    return (prog_t)rint(ldexp(s, PROG_FRAC_BITS));
}

static double prog_value(prog_t t) {
    return ldexp((double)t, -PROG_FRAC_BITS);
}

static prog_t progress(const double* sb, int n) {
    prog_t a = 0;
    for (int k = 0; k <= n; ++k) a += prog_quant(sb[k]);
    return a;
}

typedef struct { prog_t q; int k; int b; } cand_t;

/* Candidate order: survival descending, then shallower position, then lower
 * request index ([AS] §4.2, top-K with ties broken toward shallower positions).
 * The survival compared is the fixed-point one, the value the progress sums
 * use. */
static int cand_cmp(const void* pa, const void* pb) {
    const cand_t* a = (const cand_t*)pa;
    const cand_t* c = (const cand_t*)pb;
    if (a->q > c->q) return -1;
    if (a->q < c->q) return 1;
    if (a->k != c->k) return a->k < c->k ? -1 : 1;
    if (a->b != c->b) return a->b < c->b ? -1 : 1;
    return 0;
}

/* Shared set-up of the exact and Algorithm-1 schedulers: survival products,
 * the base progress at min_len, and the sorted candidate list. */
static int sched_setup(const float* conf, int B, int gamma, int min_len, double** s_out,
                       cand_t** c_out, int64_t* nc_out, prog_t* base_out) {
    double* s = (double*)malloc(sizeof(double) * (size_t)B * (size_t)(gamma + 1) + 8);
    int64_t nc = (int64_t)B * (gamma - min_len);
    cand_t* c = (cand_t*)malloc(sizeof(cand_t) * (size_t)(nc > 0 ? nc : 1));
    if (!s || !c) { free(s); free(c); return OR_ERR_SHAPE; }
    prefix_survival(conf, B, gamma, s);
    prog_t base = 0;
    for (int b = 0; b < B; ++b) base += progress(s + (int64_t)b * (gamma + 1), min_len);
    int64_t i = 0;
    for (int b = 0; b < B; ++b)
        for (int k = min_len + 1; k <= gamma; ++k) {
            c[i].q = prog_quant(s[(int64_t)b * (gamma + 1) + k]);
            c[i].k = k;
            c[i].b = b;
            ++i;
        }
    qsort(c, (size_t)nc, sizeof(cand_t), cand_cmp);
    *s_out = s;
    *c_out = c;
    *nc_out = nc;
    *base_out = base;
    return OR_OK;
}

/* Exact scan: for every budget N from B(min_len+1) to B(gamma+1), the best
 * allocation keeps the top-(N - B(min_len+1)) candidates; tau(N) is the
 * fixed-point progress of the base and those candidates, and the selected N
 * is the first (smallest) strict maximum of tau(N) / C(N)
 * ([AS] eqs. (21), (23)-(24) with every budget a candidate).
 * out_gap: relative gap between the best objective and the best one at any
 * other N (for near-tie flags). */
int oracle_sched_exact(const float* conf, int B, int gamma, const double* kt, const double* kc,
                       int nk, int min_len, int32_t* out_len, double* out_obj, double* out_gap) {
    int st = check_sched_args(conf, B, gamma, kt, kc, nk, min_len);
    if (st != OR_OK) return st;
    if (B == 0) return OR_OK;
    double* s;
    cand_t* c;
    int64_t nc;
    prog_t tau;
    st = sched_setup(conf, B, gamma, min_len, &s, &c, &nc, &tau);
    if (st != OR_OK) return st;
    double N0 = (double)B * (double)(min_len + 1);
    double best = prog_value(tau) / cost_at(N0, kt, kc, nk);
    int64_t bestK = 0;
    double* objs = (double*)malloc(sizeof(double) * (size_t)(nc + 1));
    objs[0] = best;
    for (int64_t i = 0; i < nc; ++i) {
        tau += c[i].q;
        double obj = prog_value(tau) / cost_at(N0 + (double)(i + 1), kt, kc, nk);
        objs[i + 1] = obj;
        if (obj > best) { best = obj; bestK = i + 1; }
    }
    double second = -INFINITY;
    for (int64_t i = 0; i <= nc; ++i)
        if (i != bestK && objs[i] > second) second = objs[i];
    for (int b = 0; b < B; ++b) out_len[b] = min_len;
    for (int64_t i = 0; i < bestK; ++i) out_len[c[i].b] += 1;
    if (out_obj) *out_obj = best;
    if (out_gap) *out_gap = nc > 0 ? (best - second) / best : INFINITY;
    free(objs);
    free(s);
    free(c);
    return OR_OK;
}

/* [US] §3.5 Algorithm 1 as printed, generalised to a minimum length:
 * candidates with survival > eps (eps = 0), sorted descending; start with
 * ell_r = min_len, budget B = R(min_len+1) and tau = sum_r A_r(min_len); take
 * candidates in order while they extend a contiguous prefix, keeping each one
 * only while tau / C(budget) strictly improves, and stop at the first one that
 * does not (reverting it).  j is read as 0-based, so the candidate for depth k
 * extends ell_r = k - 1 to k. */
int oracle_sched_alg1(const float* conf, int B, int gamma, const double* kt, const double* kc,
                      int nk, int min_len, int32_t* out_len) {
    int st = check_sched_args(conf, B, gamma, kt, kc, nk, min_len);
    if (st != OR_OK) return st;
    if (B == 0) return OR_OK;
    double* s;
    cand_t* c;
    int64_t nc;
    prog_t tau;
    st = sched_setup(conf, B, gamma, min_len, &s, &c, &nc, &tau);
    if (st != OR_OK) return st;
    for (int b = 0; b < B; ++b) out_len[b] = min_len;
    double budget = (double)B * (double)(min_len + 1);
    double theta_star = prog_value(tau) / cost_at(budget, kt, kc, nk);
    const double eps = 0.0;
    for (int64_t i = 0; i < nc; ++i) {
        if (!(prog_value(c[i].q) > eps)) continue; /* not a valid candidate */
        int r = c[i].b;
        if (out_len[r] != c[i].k - 1) continue; /* non-contiguous prefix: skip */
        out_len[r] = c[i].k;
        budget += 1.0;
        tau += c[i].q;
        double theta = prog_value(tau) / cost_at(budget, kt, kc, nk);
        if (theta > theta_star) {
            theta_star = theta;
        } else {
            out_len[r] = c[i].k - 1; /* early stop: throughput saturated */
            break;
        }
    }
    free(s);
    free(c);
    return OR_OK;
}

/* Brute force over every allocation in [min_len, gamma]^B: tau = sum_b A_b(ell_b),
 * N = sum_b (ell_b + 1), objective tau / C(N).  Best = largest objective, ties
 * to the smaller N, then the first in odometer order (request 0 fastest).
 * out_gap: relative gap to the best objective of any other allocation.
 * Refuses more than 2^24 allocations. */
int oracle_sched_brute(const float* conf, int B, int gamma, const double* kt, const double* kc,
                       int nk, int min_len, int32_t* out_len, double* out_obj, double* out_gap) {
    int st = check_sched_args(conf, B, gamma, kt, kc, nk, min_len);
    if (st != OR_OK) return st;
    if (B == 0) return OR_OK;
    double count = pow((double)(gamma - min_len + 1), (double)B);
    if (count > 16777216.0) return OR_ERR_SHAPE;
    double* s = (double*)malloc(sizeof(double) * (size_t)B * (size_t)(gamma + 1));
    int32_t* cur = (int32_t*)malloc(sizeof(int32_t) * (size_t)B);
    prefix_survival(conf, B, gamma, s);
    for (int b = 0; b < B; ++b) cur[b] = min_len;
    double best = -INFINITY, second = -INFINITY;
    int64_t bestN = 0;
    for (;;) {
        prog_t tau = 0;
        int64_t N = 0;
        for (int b = 0; b < B; ++b) {
            tau += progress(s + (int64_t)b * (gamma + 1), cur[b]);
            N += cur[b] + 1;
        }
        double obj = prog_value(tau) / cost_at((double)N, kt, kc, nk);
        if (obj > best || (obj == best && N < bestN)) {
            if (best > second) second = best;
            best = obj;
            bestN = N;
            memcpy(out_len, cur, sizeof(int32_t) * (size_t)B);
        } else if (obj > second) {
            second = obj;
        }
        int b = 0;
        while (b < B && cur[b] == gamma) cur[b++] = min_len;
        if (b == B) break;
        cur[b] += 1;
    }
    if (out_obj) *out_obj = best;
    if (out_gap) *out_gap = (best - second) / best;
    free(s);
    free(cur);
    return OR_OK;
}

/* D-cut ([AS] §4.2, eqs. (22)-(24)): the budget is restricted to the ratios
 * rho_i of the full verification budget B(gamma+1): K_i = max(B(min_len+1),
 * ceil(rho_i * B(gamma+1))); top-K_i selection (the same candidate order as
 * the exact scan) gives the estimated progress U_i = tau(K_i) (fixed point,
 * as for the exact scan); the chosen ratio is the first maximum of U_i / C_i.
 * ratios strictly increasing in (0, 1], costs positive. */
int oracle_sched_dcut(const float* conf, int B, int gamma, const double* ratios, const double* costs, int nr,
                      int min_len, int32_t* out_len, int32_t* out_choice, double* out_obj) {
    if (nr < 1 || nr > 32) return OR_ERR_COST_TABLE;
    for (int i = 0; i < nr; ++i) {
        if (!(ratios[i] > 0.0 && ratios[i] <= 1.0) || !(costs[i] > 0.0) || !isfinite(costs[i]))
            return OR_ERR_COST_TABLE;
        if (i > 0 && !(ratios[i] > ratios[i - 1])) return OR_ERR_COST_TABLE;
    }
    int st = check_sched_args(conf, B, gamma, ratios, costs, nr, min_len);
    if (st != OR_OK) return st;
    if (B == 0) return OR_OK;
    double* s;
    cand_t* c;
    int64_t nc;
    prog_t base;
    st = sched_setup(conf, B, gamma, min_len, &s, &c, &nc, &base);
    if (st != OR_OK) return st;
    const double N0 = (double)B * (double)(min_len + 1);
    const double Nmax = (double)B * (double)(gamma + 1);
    double best = -INFINITY;
    int choice = -1;
    int64_t bestK = 0;
    for (int i = 0; i < nr; ++i) {
        double K = ceil(ratios[i] * Nmax);
        if (K < N0) K = N0;
        if (K > Nmax) K = Nmax;
        const int64_t take = (int64_t)(K - N0);
        prog_t tau = base;
        for (int64_t k = 0; k < take; ++k) tau += c[k].q;
        const double obj = prog_value(tau) / costs[i];
        if (out_obj) out_obj[i] = obj;
        if (obj > best) {
            best = obj;
            choice = i;
            bestK = take;
        }
    }
    for (int b = 0; b < B; ++b) out_len[b] = min_len;
    for (int64_t i = 0; i < bestK; ++i) out_len[c[i].b] += 1;
    if (out_choice) *out_choice = choice;
    free(s);
    free(c);
    return OR_OK;
}

/* Static threshold scheduler ([BL] "Verify smarter, not longer": a static
 * confidence threshold, zero recovering fixed-length verification; [US] §3.5
 * StaticScheduler with fixed-length and static-threshold modes): each request
 * keeps its leading positions whose confidence (calibrated if temperatures are
 * set) is at least the threshold, at most max_len and at least min_len of them;
 * threshold 0 with max_len L is fixed-length verification of L drafts. */
int oracle_sched_threshold(const float* conf, int B, int gamma, double threshold, int max_len, int min_len,
                           int32_t* out_len) {
    if (B < 0 || gamma < 0 || min_len < 0 || min_len > gamma || max_len < min_len || max_len > gamma)
        return OR_ERR_SHAPE;
    for (int64_t i = 0; i < (int64_t)B * gamma; ++i)
        if (!(conf[i] >= 0.0f && conf[i] <= 1.0f)) return OR_ERR_CONFIDENCE;
    for (int b = 0; b < B; ++b) {
        int n = 0;
        while (n < max_len && calibrated(conf[(int64_t)b * gamma + n], g_sts_T, n + 1) >= threshold) ++n;
        out_len[b] = n < min_len ? min_len : n;
    }
    return OR_OK;
}

/* ------------------------------------------------------------------- STS
 * Sequential Temperature Scaling ([US] §2.4 and §3.6): left to right over
 * positions k = 1..gamma, choose T_k on the grid T = (i+1)/10, i = 0..99 (the
 * 100 points of linspace(0.1, 10, 100)) minimising the expected calibration
 * error of the cumulative survival a_k = prod_{j<k} c_j^(1/T_j) * c_k^(1/T)
 * against the cumulative acceptance labels y_k = [accept_len >= k]; earlier
 * positions keep their chosen temperatures; ties go to the smaller T.
 * ECE with `bins` equal-width bins on [0, 1]: sum over bins of
 * |sum of a - sum of y| / n (equivalently the count-weighted gap of means). */
static double ece(const double* a, const int* y, int n, int bins, double* sa, double* sy) {
    for (int k = 0; k < bins; ++k) sa[k] = sy[k] = 0.0;
    for (int i = 0; i < n; ++i) {
        int k = (int)(a[i] * (double)bins);
        if (k >= bins) k = bins - 1;
        if (k < 0) k = 0;
        sa[k] += a[i];
        sy[k] += (double)y[i];
    }
    double e = 0.0;
    for (int k = 0; k < bins; ++k) e += fabs(sa[k] - sy[k]);
    return e / (double)n;
}

int oracle_sts_ece(const double* a, const int32_t* y, int n, int bins, double* out) {
    double* sa = (double*)malloc(sizeof(double) * (size_t)bins);
    double* sy = (double*)malloc(sizeof(double) * (size_t)bins);
    int* yy = (int*)malloc(sizeof(int) * (size_t)n);
    for (int i = 0; i < n; ++i) yy[i] = y[i];
    *out = ece(a, yy, n, bins, sa, sy);
    free(sa);
    free(sy);
    free(yy);
    return OR_OK;
}

int oracle_sts_fit(const float* conf, const int32_t* accept_len, int n, int gamma, int grid, int bins,
                   double* out_T, double* out_ece) {
    if (n < 1 || gamma < 1 || gamma > 63 || grid < 1 || bins < 1) return OR_ERR_SHAPE;
    double* prefix = (double*)malloc(sizeof(double) * (size_t)n); /* prod_{j<k} c_j^(1/T_j) */
    double* a = (double*)malloc(sizeof(double) * (size_t)n);
    int* y = (int*)malloc(sizeof(int) * (size_t)n);
    double* sa = (double*)malloc(sizeof(double) * (size_t)bins);
    double* sy = (double*)malloc(sizeof(double) * (size_t)bins);
    for (int i = 0; i < n; ++i) prefix[i] = 1.0;
    for (int k = 1; k <= gamma; ++k) {
        for (int i = 0; i < n; ++i) y[i] = accept_len[i] >= k ? 1 : 0;
        double best = INFINITY, bestT = 1.0;
        for (int g = 0; g < grid; ++g) {
            const double T = (double)(g + 1) / 10.0;
            for (int i = 0; i < n; ++i) a[i] = prefix[i] * pow((double)conf[(int64_t)i * gamma + k - 1], 1.0 / T);
            const double e = ece(a, y, n, bins, sa, sy);
            if (e < best) {
                best = e;
                bestT = T;
            }
        }
        out_T[k - 1] = bestT;
        if (out_ece) out_ece[k - 1] = best;
        for (int i = 0; i < n; ++i) prefix[i] *= pow((double)conf[(int64_t)i * gamma + k - 1], 1.0 / bestT);
    }
    free(prefix);
    free(a);
    free(y);
    free(sa);
    free(sy);
    return OR_OK;
}
