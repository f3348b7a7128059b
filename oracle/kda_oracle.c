/*
 * KDA CPU oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously-correct FP64 implementation of the Kimi Delta
 * Attention per-token recurrence.  Only the test-suite, the smoke check and
 * the benchmark's CPU-baseline leg may load this library; the GPU product
 * path never calls it and shares no source with it.
 *
 * Source of the arithmetic ("Kimi K3: KDA, attention residuals and Stable
 * LatentMoE", hs-black.github.io):
 *   Sec. 2.1, recurrence (single head, dk = dv):
 *       S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
 *       o~_t = S_t^T q_t
 *     with q, k passed through L2Norm and beta_t in (0, 1).
 *   Sec. 2.2, bounded decay gate:
 *       g_t = g_min * Sigmoid(exp(A_h) * z_t),  alpha_t = exp(g_t),  g_min = -5,
 *     and, with gate_mode = 1, the gate it replaces (Kimi Linear's, printed beside
 *     it in Sec. 2.2):  g_t = -exp(A_h) * Softplus(z_t), unbounded below.
 *   Sec. 2.3, full-rank output gate (the W_o projection and the W_g x
 *   product are outside this operator; g_in = W_g x is an input):
 *       y_t = Sigmoid(g_in_t) (.) RMSNorm(o~_t).
 *
 * Sec. 13.1, prefix cache: a cached prefix is reusable only where the
 * recurrent state can be restored at the same boundary.  With snap_interval > 0
 * the state of each sequence after every snap_interval of its tokens is copied
 * out (S_snap, rows of all sequences in order), so a later prefill can resume
 * from any of those boundaries through S0.
 *
 * The update is evaluated in the algebraically identical delta form
 *       S <- Diag(alpha) S;  u = beta (v - S^T k);  S <- S + k u^T
 * since (I - beta k k^T) X + beta k v^T = X + k (beta (v - X^T k))^T for
 * X = Diag(alpha) S.
 *
 * Readings where the page is silent (each is a parameter here):
 *   - readout scale: o = scale * S^T q (scale = 1 in every workload);
 *   - L2Norm: x / sqrt(sum x^2 + l2_eps), applied to q and k when qk_l2norm;
 *   - RMSNorm: per (token, head) over the dv channels,
 *       o / sqrt(mean(o^2) + norm_eps) * w, w = ones when norm_w is NULL.
 *
 * Layouts (row-major): q,k,z [tok][H][dk]; v,o,g_in,y [tok][H][dv];
 * beta [tok][H]; A [H]; S0,S_T [num_seqs][H][dk][dv]; cu_seqlens [num_seqs+1].
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

static void l2normalise(const double* x, double* out, int n, double eps) {
    double s = 0.0;
    for (int i = 0; i < n; ++i) s += x[i] * x[i];
    double r = 1.0 / sqrt(s + eps);
    for (int i = 0; i < n; ++i) out[i] = x[i] * r;
}

/* The decay gate of Sec. 2.2 for one channel: log-retention g. */
/* Softplus(x) = log(1 + e^x), written so that neither branch overflows */
static double softplus(double x) { return (x > 0.0 ? x : 0.0) + log1p(exp(-fabs(x))); }

/* Kimi Linear's gate (Sec. 2.2, the mapping K3 replaces): g = -exp(A_h) Softplus(z),
 * unbounded below */
double kda_oracle_log_decay_softplus(double z, double A_h) { return -exp(A_h) * softplus(z); }

double kda_oracle_log_decay(double z, double A_h, double g_min) {
    return g_min * sigmoid(exp(A_h) * z);
}

/* Output gate of Sec. 2.3 for one (token, head) row of dv values. */
void kda_oracle_gate_norm_row(const double* o, const double* g_in, const double* w,
                              double eps, double* y, int dv) {
    double ms = 0.0;
    for (int j = 0; j < dv; ++j) ms += o[j] * o[j];
    double r = 1.0 / sqrt(ms / dv + eps);
    for (int j = 0; j < dv; ++j)
        y[j] = sigmoid(g_in[j]) * (w ? w[j] : 1.0) * o[j] * r;
}

void kda_oracle_gate_norm(const double* o, const double* g_in, const double* w, double eps,
                          double* y, long rows, int dv) {
    for (long r = 0; r < rows; ++r)
        kda_oracle_gate_norm_row(o + r * dv, g_in + r * dv, w, eps, y + r * dv, dv);
}

/*
 * Per-token recurrence over packed sequences.  Each (sequence, head) pair is
 * independent; OpenMP (when compiled in) runs pairs in parallel.
 * S0 may be NULL (zero state).  S_T, g_in, y may be NULL.
 */
void kda_oracle_prefill(int num_seqs, const int32_t* cu_seqlens, int H, int dk, int dv,
                        const double* q, const double* k, const double* v,
                        const double* z, const double* beta, const double* A,
                        double g_min, double scale, int qk_l2norm, double l2_eps,
                        const double* S0, double* o, double* S_T,
                        const double* g_in, const double* norm_w, double norm_eps,
                        double* y, int snap_interval, double* S_snap, int gate_mode) {
    long pairs = (long)num_seqs * H;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (long p = 0; p < pairs; ++p) {
        int n = (int)(p / H), h = (int)(p % H);
        double* S = (double*)malloc(sizeof(double) * (size_t)dk * dv);
        double* qn = (double*)malloc(sizeof(double) * dk);
        double* kn = (double*)malloc(sizeof(double) * dk);
        double* u = (double*)malloc(sizeof(double) * dv);
        double* ot = (double*)malloc(sizeof(double) * dv);
        size_t sbase = ((size_t)n * H + h) * (size_t)dk * dv;
        if (S0) memcpy(S, S0 + sbase, sizeof(double) * (size_t)dk * dv);
        else memset(S, 0, sizeof(double) * (size_t)dk * dv);
        double eA = exp(A[h]);
        /* prefix-cache snapshots: rows of the sequences before this one come first */
        long snap_row = 0;
        if (S_snap)
            for (int m = 0; m < n; ++m) snap_row += (cu_seqlens[m + 1] - cu_seqlens[m]) / snap_interval;
        for (long t = cu_seqlens[n]; t < cu_seqlens[n + 1]; ++t) {
            const double* qt = q + ((size_t)t * H + h) * dk;
            const double* kt = k + ((size_t)t * H + h) * dk;
            const double* vt = v + ((size_t)t * H + h) * dv;
            const double* zt = z + ((size_t)t * H + h) * dk;
            double bt = beta[(size_t)t * H + h];
            if (qk_l2norm) { l2normalise(qt, qn, dk, l2_eps); l2normalise(kt, kn, dk, l2_eps); }
            else { memcpy(qn, qt, sizeof(double) * dk); memcpy(kn, kt, sizeof(double) * dk); }
            /* S <- Diag(alpha_t) S */
            for (int i = 0; i < dk; ++i) {
                double a = exp(gate_mode ? -eA * softplus(zt[i]) : g_min * sigmoid(eA * zt[i]));
                for (int j = 0; j < dv; ++j) S[(size_t)i * dv + j] *= a;
            }
            /* u = beta (v - S^T k) */
            for (int j = 0; j < dv; ++j) u[j] = 0.0;
            for (int i = 0; i < dk; ++i)
                for (int j = 0; j < dv; ++j) u[j] += S[(size_t)i * dv + j] * kn[i];
            for (int j = 0; j < dv; ++j) u[j] = bt * (vt[j] - u[j]);
            /* S <- S + k u^T */
            for (int i = 0; i < dk; ++i)
                for (int j = 0; j < dv; ++j) S[(size_t)i * dv + j] += kn[i] * u[j];
            /* o = scale S^T q */
            for (int j = 0; j < dv; ++j) ot[j] = 0.0;
            for (int i = 0; i < dk; ++i)
                for (int j = 0; j < dv; ++j) ot[j] += S[(size_t)i * dv + j] * qn[i];
            double* out = o + ((size_t)t * H + h) * dv;
            for (int j = 0; j < dv; ++j) out[j] = scale * ot[j];
            if (g_in && y)
                kda_oracle_gate_norm_row(out, g_in + ((size_t)t * H + h) * dv, norm_w, norm_eps,
                                         y + ((size_t)t * H + h) * dv, dv);
            /* S is now the state after token t; keep it when t closes an interval */
            if (S_snap && (t + 1 - cu_seqlens[n]) % snap_interval == 0) {
                memcpy(S_snap + ((size_t)snap_row * H + h) * (size_t)dk * dv, S,
                       sizeof(double) * (size_t)dk * dv);
                ++snap_row;
            }
        }
        if (S_T) memcpy(S_T + sbase, S, sizeof(double) * (size_t)dk * dv);
        free(S); free(qn); free(kn); free(u); free(ot);
    }
}

int kda_oracle_num_threads(void) {
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
