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
