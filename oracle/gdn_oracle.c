/*
 * gdn_oracle.c -- plain fp64 CPU oracle for the Gated DeltaNet (GDN) layer hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or call this
 * file; only the tests, the package's smoke check and the benchmark's CPU-baseline leg
 * use it.  It shares no code, header, table or helper with the CUDA library.
 *
 * What it computes, token by token, in double precision:
 *
 *  1. Causal depthwise conv1d (width 4) + SiLU over packed variable-length sequences.
 *     Source: "[Feature] Add batch invariance support to GDN_ATTN backend - #45819"
 *     (vLLM PR), Birol's comment, part "3. The chunked delta-rule scan itself", fix (a):
 *     the conv input is the carried conv state concatenated in front of the new tokens,
 *     F.conv1d(..., padding=0, groups=conv_dim), then silu of the last seq_len outputs;
 *     the new conv state is the last state_len (= width-1 = 3) conv inputs.
 *     With x~ = [state(3 rows) ; x_seq], output t is
 *         y[t,c] = silu( b_c + sum_{j=0..3} w[c,j] * x~[t+j, c] ),  silu(z) = z/(1+e^-z).
 *
 *  2. Gated delta rule.  Source: "Qwen3.5-27B GPTQ Garbage Inference -- Root Cause
 *     Analysis" (FlexInfer docs), "Why abliteration failed on Qwen3.5", item 3
 *     (S = exp(g)*S + beta*dv (x) k), made precise as
 *         S_t = exp(g_t) S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,   o_t = S_t q_t.
 *     Read as: decay first, then the delta correction with dv = v - (decayed S) k,
 *     output after the update, optional output scale.  S is dv x dk; the stored state
 *     h has layout [dk][dv] with h[i][j] = S[j][i] (the recurrent-state shape
 *     (batch, v_heads, k_head_dim, v_head_dim) of the same PR, part "1. Recurrent
 *     state in fp32").  v-head h uses k-head floor(h / (Hv/Hk)).
 *     Optional per-head L2 normalisation of q and k (use_qk_l2norm_in_kernel=True in
 *     the same PR comment): x / sqrt(sum x^2 + eps).
 *
 * Work is split over (sequence, v-head) units with pthreads; every unit is computed
 * independently in a fixed order, so the result does not depend on the thread count.
 *
 * Parity pins (exercised by tests/test_oracle_pins.py): brute-force dense matrix form,
 * beta=0 closed form, store/retrieve with orthonormal keys, forget-all limit, an
 * independent chunked (WY/UT) fp64 form, split-and-carry invariance, the contraction
 * bound, and torch's fp64 conv1d for the conv.
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ conv1d */

int oracle_conv1d_varlen(int T, int C, const double *x, const double *w,
                         const double *bias, int N, const int *cu,
                         const double *state_in, double *y, double *state_out)
{
    if (T < 0 || C <= 0 || N < 0 || !x || !w || !cu || !y) return 1;
    if (cu[0] != 0 || cu[N] != T) return 2;
    for (int n = 0; n < N; ++n)
        if (cu[n + 1] < cu[n]) return 2;
    for (int n = 0; n < N; ++n) {
        const int start = cu[n];
        const int L = cu[n + 1] - cu[n];
        double *xt = (double *)malloc(sizeof(double) * (size_t)(L + 3));
        if (!xt) return 3;
        for (int c = 0; c < C; ++c) {
            for (int j = 0; j < 3; ++j)
                xt[j] = state_in ? state_in[((size_t)n * 3 + j) * C + c] : 0.0;
            for (int t = 0; t < L; ++t) xt[3 + t] = x[(size_t)(start + t) * C + c];
            for (int t = 0; t < L; ++t) {
                double z = bias ? bias[c] : 0.0;
                for (int j = 0; j < 4; ++j) z += w[(size_t)c * 4 + j] * xt[t + j];
                y[(size_t)(start + t) * C + c] = z / (1.0 + exp(-z));
            }
            if (state_out)
                for (int j = 0; j < 3; ++j)
                    state_out[((size_t)n * 3 + j) * C + c] = xt[L + j];
        }
        free(xt);
    }
    return 0;
}

/* ------------------------------------------------------- gated delta rule */

typedef struct {
    const double *q, *k, *v, *g, *beta, *h0;
    const int *cu;
    double *o, *hT;
    int N, Hk, Hv, dk, dv, l2norm;
    double scale, eps;
    int nthreads, tid;
    int status;
} gdr_job;

static void l2_normalise(const double *src, double *dst, int d, double eps)
{
    double ss = 0.0;
    for (int i = 0; i < d; ++i) ss += src[i] * src[i];
    const double inv = 1.0 / sqrt(ss + eps);
    for (int i = 0; i < d; ++i) dst[i] = src[i] * inv;
}

/* One (sequence n, v-head hv) unit: the literal token recurrence. */
static int gdr_unit(const gdr_job *J, int n, int hv)
{
    const int dk = J->dk, dv = J->dv;
    const int hk = hv / (J->Hv / J->Hk);
    double *h = (double *)calloc((size_t)dk * dv, sizeof(double));
    double *qn = (double *)malloc(sizeof(double) * dk);
    double *kn = (double *)malloc(sizeof(double) * dk);
    double *sk = (double *)malloc(sizeof(double) * dv);
    if (!h || !qn || !kn || !sk) {
        free(h); free(qn); free(kn); free(sk);
        return 3;
    }
    const size_t hoff = ((size_t)n * J->Hv + hv) * dk * dv;
    if (J->h0) memcpy(h, J->h0 + hoff, sizeof(double) * dk * dv);

    for (int t = J->cu[n]; t < J->cu[n + 1]; ++t) {
        const double *qt = J->q + ((size_t)t * J->Hk + hk) * dk;
        const double *kt = J->k + ((size_t)t * J->Hk + hk) * dk;
        const double *vt = J->v + ((size_t)t * J->Hv + hv) * dv;
        if (J->l2norm) {
            l2_normalise(qt, qn, dk, J->eps);
            l2_normalise(kt, kn, dk, J->eps);
        } else {
            memcpy(qn, qt, sizeof(double) * dk);
            memcpy(kn, kt, sizeof(double) * dk);
        }
        const double a = exp(J->g[(size_t)t * J->Hv + hv]);
        const double b = J->beta[(size_t)t * J->Hv + hv];

        /* S <- exp(g) S */
        for (int i = 0; i < dk * dv; ++i) h[i] *= a;
        /* (S k)[j] = sum_i S[j][i] k[i] = sum_i h[i][j] k[i] */
        for (int j = 0; j < dv; ++j) sk[j] = 0.0;
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dv; ++j) sk[j] += h[(size_t)i * dv + j] * kn[i];
        /* S <- S + beta (v - S k) k^T, i.e. h[i][j] += k[i] * beta (v[j] - (S k)[j]) */
        for (int j = 0; j < dv; ++j) sk[j] = b * (vt[j] - sk[j]);
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dv; ++j) h[(size_t)i * dv + j] += kn[i] * sk[j];
        /* o_t = scale * S_t q_t */
        double *ot = J->o + ((size_t)t * J->Hv + hv) * dv;
        for (int j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (int i = 0; i < dk; ++i) acc += h[(size_t)i * dv + j] * qn[i];
            ot[j] = J->scale * acc;
        }
    }
    if (J->hT) memcpy(J->hT + hoff, h, sizeof(double) * dk * dv);
    free(h); free(qn); free(kn); free(sk);
    return 0;
}

static void *gdr_worker(void *arg)
{
    gdr_job *J = (gdr_job *)arg;
    const int units = J->N * J->Hv;
    for (int u = J->tid; u < units; u += J->nthreads) {
        int rc = gdr_unit(J, u / J->Hv, u % J->Hv);
        if (rc) { J->status = rc; break; }
    }
    return NULL;
}

int oracle_gated_delta_rule(int N, const int *cu, int Hk, int Hv, int dk, int dv,
                            const double *q, const double *k, const double *v,
                            const double *g, const double *beta, double scale,
                            int l2norm, double eps, const double *h0, double *o,
                            double *hT, int nthreads)
{
    if (N < 0 || Hk <= 0 || Hv <= 0 || dk <= 0 || dv <= 0 || Hv % Hk) return 1;
    if (!cu || !q || !k || !v || !g || !beta || !o) return 1;
    if (cu[0] != 0) return 2;
    for (int n = 0; n < N; ++n)
        if (cu[n + 1] < cu[n]) return 2;
    if (nthreads <= 0) nthreads = 1;
    if (nthreads > N * Hv) nthreads = N * Hv > 0 ? N * Hv : 1;

    gdr_job *jobs = (gdr_job *)calloc((size_t)nthreads, sizeof(gdr_job));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) { free(jobs); free(th); return 3; }
    for (int t = 0; t < nthreads; ++t) {
        gdr_job J = {q, k, v, g, beta, h0, cu, o, hT, N, Hk, Hv, dk, dv, l2norm,
                     scale, eps, nthreads, t, 0};
        jobs[t] = J;
    }
    int status = 0;
    if (nthreads == 1) {
        gdr_worker(&jobs[0]);
    } else {
        int started = 0;
        for (int t = 0; t < nthreads; ++t) {
            if (pthread_create(&th[t], NULL, gdr_worker, &jobs[t]) != 0) break;
            ++started;
        }
        for (int t = started; t < nthreads; ++t) gdr_worker(&jobs[t]);
        for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
    }
    for (int t = 0; t < nthreads; ++t)
        if (jobs[t].status) status = jobs[t].status;
    free(jobs);
    free(th);
    return status;
}
