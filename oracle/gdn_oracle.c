/*
 * gdn_oracle.c -- plain fp64 CPU oracle for the GatedDeltaNet mixer.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference leg of bench.py may load or run this file.  The
 * product path (the CUDA library) shares no code, header or table with it.
 *
 * What it computes, and where each step is defined:
 *   - width-4 causal depthwise conv1d with explicit 3-token history, then SiLU
 *     over every projected channel: haskell-infer-demo README, "Architecture"
 *     (kernels/gdn_conv.cu, "causal-conv1d adapter (width 4)"); hyperflare
 *     core-design, prepared-model table ("GDN causal convolution ... raw
 *     projected QKV and explicit history") and the short-convolution
 *     paragraph (dilation 1, SiLU over the projection width; caller-owned
 *     history; inactive lanes write no state).
 *   - per-head L2 normalisation of q and k, the gates
 *     g = -exp(A_log) * softplus(u + dt_bias), a = exp(g), b = sigmoid(b_logit),
 *     and the gated delta rule
 *         S_t = a_t * S_{t-1} * (I - b_t k_t k_t^T) + b_t v_t k_t^T,  o_t = S_t q_t.
 *     The pages name these ("GatedDeltaNet layers (causal conv1d, gated delta
 *     rule, gated RMSNorm)", haskell-infer-demo README, "Highlights"; "FLA
 *     chunked/recurrent", Project Status phase 4) without printing the
 *     formulas; the formulas above are the standard statement of the rule.
 *   - gated RMSNorm y = o / sqrt(mean(o^2) + eps) * w * SiLU(z) per v-head:
 *     haskell-infer-demo README, "Highlights" and the kernels/gdn_norm.cu line
 *     ("model-specific gated norm").
 *   - FP32 recurrent state, chunks relative to each invocation, consumed
 *     endpoints as exact state-transfer boundaries: hyperflare core-design,
 *     serving-defaults table ("Main KV / GDN recurrence: BF16 / FP32") and the
 *     GDN numerics paragraph that follows the prepared short-conv interface.
 *
 * Everything here is evaluated in double precision, token by token, in the
 * order the definition states.  A second, independent restatement of the
 * recurrence in chunked (WY / UT) form is provided only so that tests can
 * check the chunk algebra against the sequential definition.
 *
 * Memory layout (shared with the library's ABI so that tests can compare
 * buffers directly):
 *   state  [n_slots][HV][dk][dv]: element (i, j) of head h holds S[j][i]
 *          (S of the recurrence is dv x dk; the buffer stores its transpose).
 *   conv   [n_slots][CH][3], oldest tap first.
 *   x      [T][CH] channels [q (HK*dk) | k (HK*dk) | v (HV*dv)], head-major.
 *   u, b   [T][HV]; z, o, y [T][HV*dv].
 * v-head h reads q/k head floor(h / (HV/HK)).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define S_AT(st, dv, j, i) ((st)[(size_t)(i) * (size_t)(dv) + (size_t)(j)])

static double silu(double x) { return x / (1.0 + exp(-x)); }
static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }
static double softplus(double x) { return x > 700.0 ? x : log1p(exp(x)); }

/* ------------------------------------------------------------------ conv */

/* Causal depthwise conv1d (width 4, dilation 1, no bias) followed by SiLU,
 * over a packed batch.  For channel c and in-sequence token t the output is
 *     sum_{j=0..3} w[c][j] * X[t-3+j][c],   X[-3..-1] = history (oldest first).
 * The new history is the last three raw inputs of the sequence (reaching back
 * into the old history when the sequence is shorter than 3).  A sequence
 * whose slot is negative reads zero history and writes none.
 * conv_state may be NULL: zero history, nothing written. */
void oracle_conv1d_silu(int CH, const double *x, const int32_t *cu_seqlens, int n_seqs,
                        const double *w, double *conv_state, const int32_t *slot_idx,
                        double *out)
{
    for (int n = 0; n < n_seqs; n++) {
        int t0 = cu_seqlens[n], L = cu_seqlens[n + 1] - cu_seqlens[n];
        int slot = slot_idx ? slot_idx[n] : n;
        double *hist = (conv_state && slot >= 0) ? conv_state + (size_t)slot * CH * 3 : NULL;
        for (int c = 0; c < CH; c++) {
            /* X[-3], X[-2], X[-1], X[0], ..., X[L-1] */
            double *X = malloc(sizeof(double) * (size_t)(L + 3));
            for (int j = 0; j < 3; j++) X[j] = hist ? hist[(size_t)c * 3 + j] : 0.0;
            for (int t = 0; t < L; t++) X[t + 3] = x[(size_t)(t0 + t) * CH + c];
            for (int t = 0; t < L; t++) {
                double acc = 0.0;
                for (int j = 0; j < 4; j++) acc += w[(size_t)c * 4 + j] * X[t + j];
                out[(size_t)(t0 + t) * CH + c] = silu(acc);
            }
            if (hist)
                for (int j = 0; j < 3; j++) hist[(size_t)c * 3 + j] = X[L + j];
            free(X);
        }
    }
}

/* ----------------------------------------------------------------- gates */

/* g = -exp(A_log[h]) * softplus(u + dt_bias[h]);  beta = sigmoid(b_logit). */
void oracle_gates(int T, int HV, const double *u, const double *b_logit, const double *A_log,
                  const double *dt_bias, double *g, double *beta)
{
    for (int t = 0; t < T; t++)
        for (int h = 0; h < HV; h++) {
            size_t e = (size_t)t * HV + h;
            g[e] = -exp(A_log[h]) * softplus(u[e] + dt_bias[h]);
            beta[e] = sigmoid(b_logit[e]);
        }
}

/* q <- q_scale * q / sqrt(sum q^2 + eps) over each head's dk channels, same for
 * k (without q_scale).  In place on the [T][CH] post-SiLU activations. */
void oracle_l2norm_qk(int T, int CH, int HK, int dk, double eps, double q_scale, double *xa)
{
    for (int t = 0; t < T; t++)
        for (int part = 0; part < 2; part++)
            for (int hh = 0; hh < HK; hh++) {
                double *p = xa + (size_t)t * CH + (size_t)part * HK * dk + (size_t)hh * dk;
                double ss = 0.0;
                for (int i = 0; i < dk; i++) ss += p[i] * p[i];
                double s = 1.0 / sqrt(ss + eps);
                if (part == 0) s *= q_scale;
                for (int i = 0; i < dk; i++) p[i] *= s;
            }
}

/* ------------------------------------------------------ sequential rule */

/* One (sequence, v-head) unit of the gated delta rule, token by token:
 *     S <- a_t * S * (I - b_t k_t k_t^T) + b_t v_t k_t^T ;  o_t = S q_t.
 * q/k/v point at the head's channels of token 0, rows strided by ld_x;
 * g/beta at token 0 of this head, strided by ld_g; o at token 0, strided by
 * ld_o.  st is this head's dk x dv buffer holding S^T, updated in place. */
static void delta_rule_unit(int L, int dk, int dv, const double *q, const double *k,
                            const double *v, size_t ld_x, const double *g, const double *beta,
                            size_t ld_g, double *st, double *o, size_t ld_o)
{
    double *p = malloc(sizeof(double) * (size_t)dv);
    for (int t = 0; t < L; t++) {
        const double *qt = q + (size_t)t * ld_x, *kt = k + (size_t)t * ld_x,
                     *vt = v + (size_t)t * ld_x;
        double a = exp(g[(size_t)t * ld_g]), b = beta[(size_t)t * ld_g];
        /* p = S k */
        for (int j = 0; j < dv; j++) {
            double acc = 0.0;
            for (int i = 0; i < dk; i++) acc += S_AT(st, dv, j, i) * kt[i];
            p[j] = acc;
        }
        /* S(I - b k k^T) = S - b (S k) k^T;  then scale by a and add b v k^T */
        for (int j = 0; j < dv; j++)
            for (int i = 0; i < dk; i++)
                S_AT(st, dv, j, i) = a * (S_AT(st, dv, j, i) - b * p[j] * kt[i]) + b * vt[j] * kt[i];
        /* o = S q */
        double *ot = o + (size_t)t * ld_o;
        for (int j = 0; j < dv; j++) {
            double acc = 0.0;
            for (int i = 0; i < dk; i++) acc += S_AT(st, dv, j, i) * qt[i];
            ot[j] = acc;
        }
    }
    free(p);
}

/* ---------------------------------------------------- chunked restatement */

/* The same unit in chunked form (chunks of C tokens restarting at the unit's
 * first token; the last chunk may be partial).  With M = S^T, G_r the
 * cumulative log-decay inside the chunk (r = 0..Lc-1), gamma_r = exp(G_r):
 *   A[r][i] = beta_r exp(G_r - G_i) k_r.k_i            (i < r)
 *   (I + A) U' = diag(beta) V - diag(beta gamma) K M    (forward substitution)
 *   O = diag(gamma) Q M + (Q K^T o Gamma) U',  Gamma[r][i] = exp(G_r - G_i), i <= r
 *   M <- gamma_last M + (diag(exp(G_last - G_r)) K)^T U'
 * Used only to check the chunk algebra against delta_rule_unit. */
static void delta_rule_unit_chunked(int L, int C, int dk, int dv, const double *q,
                                    const double *k, const double *v, size_t ld_x,
                                    const double *g, const double *beta, size_t ld_g, double *st,
                                    double *o, size_t ld_o)
{
    double *G = malloc(sizeof(double) * (size_t)C);
    double *Up = malloc(sizeof(double) * (size_t)C * dv);
    double *A = malloc(sizeof(double) * (size_t)C * C);
    double *M0 = malloc(sizeof(double) * (size_t)dk * dv);
    for (int c0 = 0; c0 < L; c0 += C) {
        int Lc = (L - c0 < C) ? (L - c0) : C;
        double acc = 0.0;
        for (int r = 0; r < Lc; r++) {
            acc += g[(size_t)(c0 + r) * ld_g];
            G[r] = acc;
        }
        memcpy(M0, st, sizeof(double) * (size_t)dk * dv);
        for (int r = 0; r < Lc; r++) {
            const double *kr = k + (size_t)(c0 + r) * ld_x;
            double br = beta[(size_t)(c0 + r) * ld_g];
            for (int i = 0; i < r; i++) {
                const double *ki = k + (size_t)(c0 + i) * ld_x;
                double d = 0.0;
                for (int e = 0; e < dk; e++) d += kr[e] * ki[e];
                A[(size_t)r * C + i] = br * exp(G[r] - G[i]) * d;
            }
        }
        for (int r = 0; r < Lc; r++) {
            const double *kr = k + (size_t)(c0 + r) * ld_x, *vr = v + (size_t)(c0 + r) * ld_x;
            double br = beta[(size_t)(c0 + r) * ld_g], gr = exp(G[r]);
            for (int j = 0; j < dv; j++) {
                double km = 0.0;
                for (int i = 0; i < dk; i++) km += kr[i] * M0[(size_t)i * dv + j];
                double rhs = br * vr[j] - br * gr * km;
                for (int i = 0; i < r; i++) rhs -= A[(size_t)r * C + i] * Up[(size_t)i * dv + j];
                Up[(size_t)r * dv + j] = rhs;
            }
        }
        for (int r = 0; r < Lc; r++) {
            const double *qr = q + (size_t)(c0 + r) * ld_x;
            double gr = exp(G[r]);
            double *orow = o + (size_t)(c0 + r) * ld_o;
            for (int j = 0; j < dv; j++) {
                double qm = 0.0;
                for (int i = 0; i < dk; i++) qm += qr[i] * M0[(size_t)i * dv + j];
                orow[j] = gr * qm;
            }
            for (int i = 0; i <= r; i++) {
                const double *ki = k + (size_t)(c0 + i) * ld_x;
                double d = 0.0;
                for (int e = 0; e < dk; e++) d += qr[e] * ki[e];
                double f = d * exp(G[r] - G[i]);
                for (int j = 0; j < dv; j++) orow[j] += f * Up[(size_t)i * dv + j];
            }
        }
        double glast = exp(G[Lc - 1]);
        for (int i = 0; i < dk; i++)
            for (int j = 0; j < dv; j++) {
                double m = glast * M0[(size_t)i * dv + j];
                for (int r = 0; r < Lc; r++)
                    m += exp(G[Lc - 1] - G[r]) * k[(size_t)(c0 + r) * ld_x + i] * Up[(size_t)r * dv + j];
                st[(size_t)i * dv + j] = m;
            }
    }
    free(G); free(Up); free(A); free(M0);
}

/* ----------------------------------------------------- threaded driver */

typedef struct {
    int n_seqs, HK, HV, dk, dv, CH, chunk; /* chunk == 0: sequential form */
    const int32_t *cu_seqlens, *slot_idx;
    const double *xa, *g, *beta;
    double *state; /* [slots][HV][dk][dv] or NULL */
    double *o;     /* [T][HV*dv] */
    int next;      /* work counter, guarded by mu */
    pthread_mutex_t mu;
} rule_job;

static void *rule_worker(void *arg)
{
    rule_job *J = arg;
    size_t hs = (size_t)J->dk * J->dv;
    double *scratch = malloc(sizeof(double) * hs);
    for (;;) {
        pthread_mutex_lock(&J->mu);
        int unit = J->next++;
        pthread_mutex_unlock(&J->mu);
        if (unit >= J->n_seqs * J->HV) break;
        int n = unit / J->HV, h = unit % J->HV, kh = h / (J->HV / J->HK);
        int t0 = J->cu_seqlens[n], L = J->cu_seqlens[n + 1] - t0;
        int slot = J->slot_idx ? J->slot_idx[n] : n;
        double *o = J->o + (size_t)t0 * J->HV * J->dv + (size_t)h * J->dv;
        size_t ld_o = (size_t)J->HV * J->dv;
        if (J->slot_idx && slot < 0) { /* padding lane: no state read or write, zero output */
            for (int t = 0; t < L; t++) memset(o + (size_t)t * ld_o, 0, sizeof(double) * J->dv);
            continue;
        }
        double *st = scratch;
        if (J->state && slot >= 0)
            memcpy(st, J->state + ((size_t)slot * J->HV + h) * hs, sizeof(double) * hs);
        else
            memset(st, 0, sizeof(double) * hs);
        const double *base = J->xa + (size_t)t0 * J->CH;
        const double *q = base + (size_t)kh * J->dk;
        const double *k = base + (size_t)J->HK * J->dk + (size_t)kh * J->dk;
        const double *v = base + (size_t)2 * J->HK * J->dk + (size_t)h * J->dv;
        const double *g = J->g + (size_t)t0 * J->HV + h, *b = J->beta + (size_t)t0 * J->HV + h;
        if (J->chunk > 0)
            delta_rule_unit_chunked(L, J->chunk, J->dk, J->dv, q, k, v, J->CH, g, b, J->HV, st, o, ld_o);
        else
            delta_rule_unit(L, J->dk, J->dv, q, k, v, J->CH, g, b, J->HV, st, o, ld_o);
        if (J->state && slot >= 0 && L > 0)
            memcpy(J->state + ((size_t)slot * J->HV + h) * hs, st, sizeof(double) * hs);
    }
    free(scratch);
    return NULL;
}

/* Gated delta rule over a packed batch, threaded over (sequence, v-head).
 * xa: post-SiLU, L2-normalised activations [T][CH].  state: [slots][HV][dk][dv]
 * in/out (NULL = zero initial state, final state discarded).  A sequence whose
 * slot is negative is a padding lane: its outputs are zero and no state is
 * read or written.  chunk = 0 runs
 * the token-by-token definition; chunk > 0 the chunked restatement. */
void oracle_delta_rule(int n_seqs, const int32_t *cu_seqlens, const int32_t *slot_idx, int HK,
                       int HV, int dk, int dv, const double *xa, const double *g,
                       const double *beta, double *state, double *o, int chunk, int n_threads)
{
    rule_job J;
    J.n_seqs = n_seqs; J.HK = HK; J.HV = HV; J.dk = dk; J.dv = dv;
    J.CH = 2 * HK * dk + HV * dv; J.chunk = chunk;
    J.cu_seqlens = cu_seqlens; J.slot_idx = slot_idx;
    J.xa = xa; J.g = g; J.beta = beta; J.state = state; J.o = o; J.next = 0;
    pthread_mutex_init(&J.mu, NULL);
    if (n_threads < 1) n_threads = 1;
    pthread_t *th = malloc(sizeof(pthread_t) * (size_t)n_threads);
    for (int i = 0; i < n_threads; i++) pthread_create(&th[i], NULL, rule_worker, &J);
    for (int i = 0; i < n_threads; i++) pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&J.mu);
}

/* ------------------------------------------------------------ gated norm */

/* y = o / sqrt(mean_j o_j^2 + eps) * w_j * SiLU(z_j), per token and v-head. */
void oracle_gated_rmsnorm(int T, int HV, int dv, const double *o, const double *z,
                          const double *w, double eps, double *y)
{
    for (int t = 0; t < T; t++)
        for (int h = 0; h < HV; h++) {
            size_t base = ((size_t)t * HV + h) * dv;
            double ss = 0.0;
            for (int j = 0; j < dv; j++) ss += o[base + j] * o[base + j];
            double r = 1.0 / sqrt(ss / dv + eps);
            for (int j = 0; j < dv; j++) y[base + j] = o[base + j] * r * w[j] * silu(z[base + j]);
        }
}

/* ------------------------------------------------------- the whole mixer */

/* Mixer over a packed batch (prefill) or one token per sequence (decode is
 * the case cu_seqlens = 0,1,2,...): conv+SiLU -> L2 -> gates -> delta rule ->
 * gated norm.  Optional dumps (NULL to skip): xa [T][CH] (post-SiLU, q/k
 * normalised) and o [T][HV*dv].  Returns 0, or -1 on allocation failure. */
int oracle_mixer(int n_seqs, const int32_t *cu_seqlens, const int32_t *slot_idx, int HK, int HV,
                 int dk, int dv, const double *x, const double *conv_w, double *conv_state,
                 const double *u, const double *b_logit, const double *A_log,
                 const double *dt_bias, const double *z, const double *norm_w, double q_scale,
                 double l2_eps, double norm_eps, double *state, double *y, double *xa_dump,
                 double *o_dump, int chunk, int n_threads)
{
    int CH = 2 * HK * dk + HV * dv;
    int T = cu_seqlens[n_seqs];
    size_t nt = (size_t)(T > 0 ? T : 1);
    double *xa = xa_dump ? xa_dump : malloc(sizeof(double) * nt * CH);
    double *o = o_dump ? o_dump : malloc(sizeof(double) * nt * HV * dv);
    double *g = malloc(sizeof(double) * nt * HV), *beta = malloc(sizeof(double) * nt * HV);
    if (!xa || !o || !g || !beta) return -1;
    oracle_conv1d_silu(CH, x, cu_seqlens, n_seqs, conv_w, conv_state, slot_idx, xa);
    oracle_l2norm_qk(T, CH, HK, dk, l2_eps, q_scale, xa);
    oracle_gates(T, HV, u, b_logit, A_log, dt_bias, g, beta);
    oracle_delta_rule(n_seqs, cu_seqlens, slot_idx, HK, HV, dk, dv, xa, g, beta, state, o, chunk,
                      n_threads);
    oracle_gated_rmsnorm(T, HV, dv, o, z, norm_w, norm_eps, y);
    if (!xa_dump) free(xa);
    if (!o_dump) free(o);
    free(g); free(beta);
    return 0;
}
