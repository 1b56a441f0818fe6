/*
 * CPU oracle of the gated delta-rule recurrent state update (test
 * infrastructure only: the product never links, loads or calls this file).
 *
 * Source of the definition: "Kestrel_VLLM - 24 · GDN linear attention to GPU"
 * (wsisp.com/helps/119760.html), section 4, the delta-recurrence kernel and
 * figure 1 step 5: per value head vi with a [kd][vd] fp32 state S and key head
 * hh = vi / (vh / kh),
 *     alpha  = exp(g[vi])
 *     S     *= alpha
 *     kv[dv] = sum_dk S[dk][dv] * k[hh][dk]            (the scaled S)
 *     tmp    = (v[vi][dv] - kv[dv]) * beta[vi]
 *     S[dk][dv] += k[hh][dk] * tmp[dv]
 *     o[vi][dv] = sum_dk S[dk][dv] * q[hh][dk]         (the updated S)
 * The same article fixes the head mapping (contiguous groups, hh = vi/rep)
 * and the storage of S as row-major [kd][vd].
 *
 * Precision: fp32, every product and every sum rounded separately (build with
 * -ffp-contract=off, no fast-math), each accumulator starting at 0.0f and
 * folding dk = 0, 1, ..., kd-1 left to right, matching the register-resident
 * kernel of "Kestrel_VLLM - 27 · register-resident & fused launch"
 * (juejin.cn/post/7703369445846777871), section 3.4, which states that order
 * and the separate rounding of every multiply and add.
 *
 * Multi-token calls apply the single step to tokens t = 0..T-1 in order, the
 * reading of "Kestrel_VLLM - 34 · batched M rows"
 * (juejin.cn/post/7704936491831377954), section 3.6: M tokens are M serial
 * state updates.  Checkpoint t holds the state after token t.
 *
 * Independent (b, vi) heads may run on several OpenMP threads; that changes
 * no arithmetic, since every head is computed by exactly one thread in the
 * order above.
 */
#include <math.h>
#include <stddef.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* One token of one head.  S: [kd][vd] in place.  k, q: [kd].  v, o: [vd].
 * work: 2*vd floats of scratch. */
static void head_step(float *S, const float *q, const float *k,
                      const float *v, float g, float beta, float *o,
                      int kd, int vd, float *work) {
    float *kv = work;        /* [vd] */
    float *oa = work + vd;   /* [vd] */
    const float alpha = expf(g);
    int dk, dv;
    for (dv = 0; dv < vd; dv++) kv[dv] = 0.0f;
    for (dk = 0; dk < kd; dk++) {
        float *row = S + (size_t)dk * (size_t)vd;
        const float kk = k[dk];
        for (dv = 0; dv < vd; dv++) {
            const float t = row[dv] * alpha;
            row[dv] = t;
            const float p = t * kk;
            kv[dv] = kv[dv] + p;
        }
    }
    /* kv now holds the scaled-state read-out; turn it into tmp in place */
    for (dv = 0; dv < vd; dv++) {
        const float d = v[dv] - kv[dv];
        kv[dv] = d * beta;
    }
    for (dv = 0; dv < vd; dv++) oa[dv] = 0.0f;
    for (dk = 0; dk < kd; dk++) {
        float *row = S + (size_t)dk * (size_t)vd;
        const float kk = k[dk];
        const float qq = q[dk];
        for (dv = 0; dv < vd; dv++) {
            const float u = kk * kv[dv];
            const float t = row[dv] + u;
            row[dv] = t;
            const float p = t * qq;
            oa[dv] = oa[dv] + p;
        }
    }
    for (dv = 0; dv < vd; dv++) o[dv] = oa[dv];
}

/* Advance every (b, vi) state over T tokens.
 *   S     [B][vh][kd][vd]   in: initial state, out: state after token T-1
 *   q, k  [B][T][kh][kd]
 *   v, o  [B][T][vh][vd]
 *   g, beta [B][T][vh]
 *   ckpt  [T][B][vh][kd][vd] or NULL: ckpt[t] = state after token t
 * Returns 0, or -1 on a bad shape, -2 when scratch cannot be allocated. */
int gdn_oracle_run(int B, int T, int kh, int vh, int kd, int vd, float *S,
                   const float *q, const float *k, const float *v,
                   const float *g, const float *beta, float *o, float *ckpt) {
    if (B < 0 || T < 0 || kh <= 0 || vh <= 0 || kd <= 0 || vd <= 0) return -1;
    if (vh % kh) return -1;
    const int rep = vh / kh;
    const long nheads = (long)B * vh;
    const size_t hsz = (size_t)kd * (size_t)vd;
    int bad = 0;
    long h;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (h = 0; h < nheads; h++) {
        float *work = (float *)malloc(sizeof(float) * 2 * (size_t)vd);
        if (!work) { bad |= 1; continue; }
        const int b = (int)(h / vh), vi = (int)(h % vh), hh = vi / rep;
        float *Sh = S + (size_t)h * hsz;
        int t;
        for (t = 0; t < T; t++) {
            const size_t bt = (size_t)b * (size_t)T + (size_t)t;
            const float *qt = q + (bt * (size_t)kh + (size_t)hh) * (size_t)kd;
            const float *kt = k + (bt * (size_t)kh + (size_t)hh) * (size_t)kd;
            const float *vt = v + (bt * (size_t)vh + (size_t)vi) * (size_t)vd;
            float *ot = o + (bt * (size_t)vh + (size_t)vi) * (size_t)vd;
            const size_t gi = bt * (size_t)vh + (size_t)vi;
            head_step(Sh, qt, kt, vt, g[gi], beta[gi], ot, kd, vd, work);
            if (ckpt)
                memcpy(ckpt + ((size_t)t * (size_t)nheads + (size_t)h) * hsz,
                       Sh, sizeof(float) * hsz);
        }
        free(work);
    }
    return bad ? -2 : 0;
}

/* Number of threads the parallel loop above would use. */
int gdn_oracle_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Set the thread count (no effect without OpenMP). */
void gdn_oracle_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ------------------------------------------------------------------------
 * The per-token layer steps around the recurrence ("Kestrel_VLLM - 24 · GDN
 * linear attention to GPU", section 3, figure 1 steps 2-5):
 *   conv:  for every channel ch of the mixed q|k|v projection (conv_dim =
 *          2*kh*kd + vh*vd channels, q first, then k, then v), a depthwise
 *          causal convolution of width ck over the last ck-1 inputs (the
 *          history, oldest first) and the current input, then SiLU; the
 *          history stores the convolution INPUTS and shifts by one per
 *          token;
 *   norm:  q and k scaled to unit L2 norm per key head, x / sqrt(sum x^2 +
 *          eps) (the article names the step but prints no formula; this is
 *          the plain reading, with eps a parameter);
 *   gates: xa = a + dt_bias;  softplus = xa (xa > 20), exp(xa) (xa < -20),
 *          log1p(exp(xa)) otherwise;  g = -exp(A_log) * softplus;
 *          beta = 1 / (1 + exp(-b));
 *   then the single-token update above with these q, k, v, g, beta.
 * fp32, separately rounded, left-to-right sums.
 */

/* The gate nonlinearity of the article's gate step: softplus, with the
 * input itself returned above 20 and e^x returned below -20 (where
 * log(1 + e^x) equals those to fp32 precision), log1p(e^x) in between. */
static float gate_softplus(float x) {
    if (x > 20.0f) return x;
    if (x < -20.0f) return expf(x);
    return log1pf(expf(x));
}

/* The logistic function 1 / (1 + e^-x). */
static float logistic(float x) {
    const float e = expf(-x);
    const float den = 1.0f + e;
    return 1.0f / den;
}

/* Advance the whole layer core over T tokens for every sequence.
 *   S      [B][vh][kd][vd]       in/out
 *   hist   [B][ck-1][conv_dim]   in/out (oldest row first)
 *   x      [B][T][conv_dim]      raw mixed projections
 *   conv_w [conv_dim][ck]
 *   a, b   [B][T][vh];  A_log, dt_bias [vh]
 *   o      [B][T][vh][vd]
 *   ckpt   [T][B][vh][kd][vd] or NULL
 * The convolution is read as a sliding window: per sequence, the rows
 * R = [hist rows 0..ck-2, x rows 0..T-1] (ck-1+T rows of conv_dim
 * channels, oldest first); token t sees rows t .. t+ck-1 of R, and channel
 * ch of its output is sum_j conv_w[ch][j] * R[t+j][ch] over j = 0..ck-1
 * (oldest row first, fp32, left to right).  The history after the call is
 * the last ck-1 rows of R.
 * Returns 0, -1 on a bad shape, -2 when scratch cannot be allocated. */
int gdn_oracle_layer(int B, int T, int kh, int vh, int kd, int vd, int ck,
                     float eps, float *S, float *hist, const float *x,
                     const float *conv_w, const float *a, const float *b,
                     const float *A_log, const float *dt_bias, float *o,
                     float *ckpt) {
    if (B < 0 || T < 0 || kh <= 0 || vh <= 0 || kd <= 0 || vd <= 0 ||
        ck < 1 || vh % kh)
        return -1;
    const size_t C = (size_t)(2 * kh * kd + vh * vd); /* conv channels */
    const size_t nh = (size_t)(ck - 1);               /* history rows   */
    const size_t hsz = (size_t)kd * (size_t)vd;
    const size_t qk_len = (size_t)kh * (size_t)kd;
    float *rows = (float *)malloc(sizeof(float) * (nh + (size_t)T) * C + 1);
    float *act = (float *)malloc(sizeof(float) * C);   /* conv + SiLU out */
    float *qu = (float *)malloc(sizeof(float) * qk_len);
    float *ku = (float *)malloc(sizeof(float) * qk_len);
    float *gv = (float *)malloc(sizeof(float) * (size_t)vh);
    float *bv = (float *)malloc(sizeof(float) * (size_t)vh);
    float *ob = (float *)malloc(sizeof(float) * (size_t)vh * vd);
    int rc = (rows && act && qu && ku && gv && bv && ob) ? 0 : -2;
    for (int s = 0; s < B && rc == 0; s++) {
        float *hs = hist + (size_t)s * nh * C;
        /* R: the stored rows, then this call's inputs */
        memcpy(rows, hs, sizeof(float) * nh * C);
        memcpy(rows + nh * C, x + (size_t)s * (size_t)T * C,
               sizeof(float) * (size_t)T * C);
        for (int t = 0; t < T && rc == 0; t++) {
            const float *win = rows + (size_t)t * C;  /* oldest window row */
            for (size_t ch = 0; ch < C; ch++) {
                float y = 0.0f;
                for (int j = 0; j < ck; j++) {
                    const float p = conv_w[ch * (size_t)ck + (size_t)j] *
                                    win[(size_t)j * C + ch];
                    y = y + p;
                }
                act[ch] = y * logistic(y);  /* SiLU */
            }
            /* unit L2 norm of every key head's q and k rows */
            for (size_t r = 0; r < 2 * (size_t)kh; r++) {
                const float *src = act + r * (size_t)kd;
                float ss = 0.0f;
                for (int d = 0; d < kd; d++) {
                    const float p = src[d] * src[d];
                    ss = ss + p;
                }
                const float nrm = sqrtf(ss + eps);
                float *dst = r < (size_t)kh ? qu + r * (size_t)kd
                                            : ku + (r - (size_t)kh) * (size_t)kd;
                for (int d = 0; d < kd; d++) dst[d] = src[d] / nrm;
            }
            /* decay and write strength of every value head */
            const size_t row = (size_t)s * (size_t)T + (size_t)t;
            for (int h = 0; h < vh; h++) {
                const float sp = gate_softplus(a[row * vh + h] + dt_bias[h]);
                gv[h] = -expf(A_log[h]) * sp;
                bv[h] = logistic(b[row * vh + h]);
            }
            /* the recurrence, one token, this sequence; v is the last block
             * of channels */
            float *Ss = S + (size_t)s * (size_t)vh * hsz;
            rc = gdn_oracle_run(1, 1, kh, vh, kd, vd, Ss, qu, ku,
                                act + 2 * qk_len, gv, bv, ob, NULL);
            memcpy(o + row * (size_t)vh * vd, ob, sizeof(float) * (size_t)vh * vd);
            if (ckpt)
                memcpy(ckpt + ((size_t)t * (size_t)B + (size_t)s) * vh * hsz,
                       Ss, sizeof(float) * (size_t)vh * hsz);
        }
        /* the history after the call: the last ck-1 rows of R */
        if (rc == 0)
            memcpy(hs, rows + (size_t)T * C, sizeof(float) * nh * C);
    }
    free(rows); free(act); free(qu); free(ku); free(gv); free(bv); free(ob);
    return rc;
}

/* ------------------------------------------------------------------------
 * Gated RMSNorm on the recurrence output ("Kestrel_VLLM - 24 · GDN linear
 * attention to GPU", figure 1 step 6, and section 4, which runs it one value
 * head at a time).  The article names the step without its formula; this is
 * the plain reading of an RMS normalisation with a per-channel weight and a
 * SiLU output gate:
 *   for every (sequence b, token t, value head h), over its vd channels c:
 *     ms   = (sum_c o[c]^2) / vd
 *     r    = 1 / sqrt(ms + eps)
 *     y[c] = ((o[c] * r) * w[c]) * (z[c] / (1 + exp(-z[c])))
 *   o, z, y [B][T][vh][vd];  w [vd] (shared by all heads);  eps >= 0.
 * fp32, separately rounded, left-to-right sum.  y may be o (in place).
 * Returns 0, or -1 on a bad shape.
 */
int gdn_oracle_gate_norm(int B, int T, int vh, int vd, float eps,
                         const float *o, const float *z, const float *w,
                         float *y) {
    if (B < 0 || T < 0 || vh <= 0 || vd <= 0 || !(eps >= 0.0f))
        return -1;
    const size_t rows = (size_t)B * (size_t)T * (size_t)vh;
    for (size_t r = 0; r < rows; r++) {
        const float *orow = o + r * (size_t)vd;
        const float *zrow = z + r * (size_t)vd;
        float *yrow = y + r * (size_t)vd;
        float ss = 0.0f;
        for (int c = 0; c < vd; c++) {
            const float p = orow[c] * orow[c];
            ss = ss + p;
        }
        const float ms = ss / (float)vd;
        const float rinv = 1.0f / sqrtf(ms + eps);
        for (int c = 0; c < vd; c++) {
            const float gate = zrow[c] / (1.0f + expf(-zrow[c]));
            const float n = orow[c] * rinv;
            const float nw = n * w[c];
            yrow[c] = nw * gate;
        }
    }
    return 0;
}
