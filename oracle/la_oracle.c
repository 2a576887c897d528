/*
 * Float64 CPU oracle for the causal linear-attention operator with a fixed
 * matrix state. TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the
 * CPU-baseline leg of the benchmark call it. The CUDA library never links it.
 *
 * Each function runs the token-by-token recurrence exactly as the pages
 * write it, one (batch, head) sequence at a time, in double precision, with
 * no chunking, blocking or reordering. Inputs are the already-rounded values
 * the GPU also consumes, upcast to double. Independent sequences run in
 * parallel under OpenMP, and each sequence is a plain loop over t.
 *
 * Layouts (contiguous, row-major), with BH = batch*heads:
 *   q, k   [BH, T, dk]      v, o [BH, T, dv]
 *   norm:  state = S [dk, dv] followed by z [dk], per sequence
 *   norm with decay: gamma [BH]; state as norm
 *   gla:   gamma [BH, T, dk]; state = S [dk, dv] per sequence
 *   gdn:   g, beta [BH, T];   state = S [dv, dk] per sequence
 *   kda:   alpha [BH, T, dk], beta [BH, T]; state as gdn
 * A NULL state_in means a zero initial state; a NULL state_out skips the
 * write. Return value: 0 on success, 2 if a normalizer denominator was not
 * strictly positive (norm only), 1 on allocation failure.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* phi(x) = elu(x) + 1 with alpha = 1: x + 1 for x > 0, exp(x) otherwise.
 * "Linear attention and recurrent memory", The big idea (feature map);
 * "Linear attention and Hyena", section 11.2 (phi = elu + 1 > 0). */
static double phi(double x) { return x > 0.0 ? x + 1.0 : exp(x); }

static int set_threads(int nthreads) {
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
    return nthreads;
#else
    (void)nthreads;
    return 1;
#endif
}

int la_oracle_threads_available(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * (a) Normalized kernel linear attention, update first:
 *   S_t = S_{t-1} + phi(k_t) v_t^T,  z_t = z_{t-1} + phi(k_t),
 *   o_t = phi(q_t)^T S_t / phi(q_t)^T z_t.
 * "Linear Attention" concept page (normalized kernel formulation);
 * "Linear attention and recurrent memory", The big idea, and Pitfalls (the
 * update-first convention lets a token attend to itself). No epsilon is
 * added to the denominator, which phi > 0 keeps positive.
 */
int la_oracle_norm(int BH, int T, int dk, int dv,
                   const double* q, const double* k, const double* v,
                   const double* state_in, double* o, double* state_out,
                   double* den_out, int nthreads) {
    int bad = 0, oom = 0;
    int nt = set_threads(nthreads);
    (void)nt;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt) reduction(|:bad, oom)
#endif
    for (int bh = 0; bh < BH; ++bh) {
        double* S = (double*)malloc(sizeof(double) * ((size_t)dk * dv + dk + dk + dk + dv));
        if (!S) { oom = 1; continue; }
        double* z = S + (size_t)dk * dv;
        double* f = z + dk;
        double* p = f + dk;
        double* num = p + dk;
        const size_t sz = (size_t)dk * dv + dk;
        if (state_in) memcpy(S, state_in + bh * sz, sizeof(double) * sz);
        else memset(S, 0, sizeof(double) * sz);
        for (int t = 0; t < T; ++t) {
            const double* kt = k + ((size_t)bh * T + t) * dk;
            const double* qt = q + ((size_t)bh * T + t) * dk;
            const double* vt = v + ((size_t)bh * T + t) * dv;
            for (int i = 0; i < dk; ++i) f[i] = phi(kt[i]);
            for (int i = 0; i < dk; ++i) {
                for (int j = 0; j < dv; ++j) S[(size_t)i * dv + j] += f[i] * vt[j];
                z[i] += f[i];
            }
            for (int i = 0; i < dk; ++i) p[i] = phi(qt[i]);
            double d = 0.0;
            for (int i = 0; i < dk; ++i) d += p[i] * z[i];
            for (int j = 0; j < dv; ++j) num[j] = 0.0;
            for (int i = 0; i < dk; ++i)
                for (int j = 0; j < dv; ++j) num[j] += p[i] * S[(size_t)i * dv + j];
            if (!(d > 0.0)) bad = 1;
            double* ot = o + ((size_t)bh * T + t) * dv;
            for (int j = 0; j < dv; ++j) ot[j] = num[j] / d;
            if (den_out) den_out[(size_t)bh * T + t] = d;
        }
        if (state_out) memcpy(state_out + bh * sz, S, sizeof(double) * sz);
        free(S);
    }
    if (oom) return 1;
    return bad ? 2 : 0;
}

/*
 * (a') Normalized kernel linear attention with a fixed decay per sequence-head,
 * update first:
 *   S_t = gamma S_{t-1} + phi(k_t) v_t^T,  z_t = gamma z_{t-1} + phi(k_t),
 *   o_t = phi(q_t)^T S_t / phi(q_t)^T z_t.
 * "Linear attention and recurrent memory", Fixed decay versus an
 * input-dependent gate (one scalar per head decays both the matrix state and
 * the normalizer). gamma [BH]; gamma = 1 is variant (a).
 */
int la_oracle_norm_decay(int BH, int T, int dk, int dv,
                         const double* q, const double* k, const double* v, const double* gamma,
                         const double* state_in, double* o, double* state_out,
                         double* den_out, int nthreads) {
    int bad = 0, oom = 0;
    int nt = set_threads(nthreads);
    (void)nt;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt) reduction(|:bad, oom)
#endif
    for (int bh = 0; bh < BH; ++bh) {
        double* S = (double*)malloc(sizeof(double) * ((size_t)dk * dv + dk + dk + dk + dv));
        if (!S) { oom = 1; continue; }
        double* z = S + (size_t)dk * dv;
        double* f = z + dk;
        double* p = f + dk;
        double* num = p + dk;
        const size_t sz = (size_t)dk * dv + dk;
        const double g = gamma[bh];
        if (state_in) memcpy(S, state_in + bh * sz, sizeof(double) * sz);
        else memset(S, 0, sizeof(double) * sz);
        for (int t = 0; t < T; ++t) {
            const double* kt = k + ((size_t)bh * T + t) * dk;
            const double* qt = q + ((size_t)bh * T + t) * dk;
            const double* vt = v + ((size_t)bh * T + t) * dv;
            for (int i = 0; i < dk; ++i) f[i] = phi(kt[i]);
            for (int i = 0; i < dk; ++i) {
                for (int j = 0; j < dv; ++j) S[(size_t)i * dv + j] = g * S[(size_t)i * dv + j] + f[i] * vt[j];
                z[i] = g * z[i] + f[i];
            }
            for (int i = 0; i < dk; ++i) p[i] = phi(qt[i]);
            double d = 0.0;
            for (int i = 0; i < dk; ++i) d += p[i] * z[i];
            for (int j = 0; j < dv; ++j) num[j] = 0.0;
            for (int i = 0; i < dk; ++i)
                for (int j = 0; j < dv; ++j) num[j] += p[i] * S[(size_t)i * dv + j];
            if (!(d > 0.0)) bad = 1;
            double* ot = o + ((size_t)bh * T + t) * dv;
            for (int j = 0; j < dv; ++j) ot[j] = num[j] / d;
            if (den_out) den_out[(size_t)bh * T + t] = d;
        }
        if (state_out) memcpy(state_out + bh * sz, S, sizeof(double) * sz);
        free(S);
    }
    if (oom) return 1;
    return bad ? 2 : 0;
}

/*
 * (b) Per-channel gated linear attention (GLA / RetNet family):
 *   S_t = diag(gamma_t) S_{t-1} + phi(k_t) v_t^T,  o_t = S_t^T phi(q_t).
 * "Linear attention and Hyena", section 11.3: the gate gamma_t in (0,1)^{d_k}
 * attaches to the transition, and the unrolled solution in section 11.9
 * (Exercise 11.5) fixes its timing: token j is decayed by gamma_{j+1..t}.
 * With identity_phi != 0 the feature map is the identity.
 */
int la_oracle_gla(int BH, int T, int dk, int dv,
                  const double* q, const double* k, const double* v,
                  const double* gamma, const double* state_in,
                  double* o, double* state_out, int identity_phi, int nthreads) {
    int oom = 0;
    int nt = set_threads(nthreads);
    (void)nt;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt) reduction(|:oom)
#endif
    for (int bh = 0; bh < BH; ++bh) {
        double* S = (double*)malloc(sizeof(double) * ((size_t)dk * dv + dk + dk));
        if (!S) { oom = 1; continue; }
        double* f = S + (size_t)dk * dv;
        double* p = f + dk;
        const size_t sz = (size_t)dk * dv;
        if (state_in) memcpy(S, state_in + bh * sz, sizeof(double) * sz);
        else memset(S, 0, sizeof(double) * sz);
        for (int t = 0; t < T; ++t) {
            const size_t row = (size_t)bh * T + t;
            const double* kt = k + row * dk;
            const double* qt = q + row * dk;
            const double* vt = v + row * dv;
            const double* gt = gamma + row * dk;
            for (int i = 0; i < dk; ++i) {
                f[i] = identity_phi ? kt[i] : phi(kt[i]);
                p[i] = identity_phi ? qt[i] : phi(qt[i]);
            }
            for (int i = 0; i < dk; ++i)
                for (int j = 0; j < dv; ++j)
                    S[(size_t)i * dv + j] = gt[i] * S[(size_t)i * dv + j] + f[i] * vt[j];
            double* ot = o + row * dv;
            for (int j = 0; j < dv; ++j) ot[j] = 0.0;
            for (int i = 0; i < dk; ++i)
                for (int j = 0; j < dv; ++j) ot[j] += p[i] * S[(size_t)i * dv + j];
        }
        if (state_out) memcpy(state_out + bh * sz, S, sizeof(double) * sz);
        free(S);
    }
    return oom ? 1 : 0;
}

/*
 * (c) Gated delta rule, S in R^{dv x dk}, unit keys assumed (not enforced):
 *   S~_t = g_t S_{t-1},  S_t = S~_t + beta_t (v_t - S~_t k_t) k_t^T,
 *   o_t = S_t q_t.
 * "Linear Attention" concept page (gated delta rule form, error taken
 * against the decayed state S~); equal to g_t S_{t-1}(I - beta_t k_t k_t^T)
 * + beta_t v_t k_t^T of "Beyond attention", section 18.2.
 */
int la_oracle_gdn(int BH, int T, int dk, int dv,
                  const double* q, const double* k, const double* v,
                  const double* g, const double* beta, const double* state_in,
                  double* o, double* state_out, int nthreads) {
    int oom = 0;
    int nt = set_threads(nthreads);
    (void)nt;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt) reduction(|:oom)
#endif
    for (int bh = 0; bh < BH; ++bh) {
        double* S = (double*)malloc(sizeof(double) * ((size_t)dk * dv + dv));
        if (!S) { oom = 1; continue; }
        double* u = S + (size_t)dk * dv;
        const size_t sz = (size_t)dk * dv;
        if (state_in) memcpy(S, state_in + bh * sz, sizeof(double) * sz);
        else memset(S, 0, sizeof(double) * sz);
        for (int t = 0; t < T; ++t) {
            const size_t row = (size_t)bh * T + t;
            const double* kt = k + row * dk;
            const double* qt = q + row * dk;
            const double* vt = v + row * dv;
            const double gt = g[row], bt = beta[row];
            for (size_t e = 0; e < sz; ++e) S[e] *= gt;             /* S~ = g S */
            for (int i = 0; i < dv; ++i) {                           /* u = beta (v - S~ k) */
                double sk = 0.0;
                for (int c = 0; c < dk; ++c) sk += S[(size_t)i * dk + c] * kt[c];
                u[i] = bt * (vt[i] - sk);
            }
            for (int i = 0; i < dv; ++i)                             /* S = S~ + u k^T */
                for (int c = 0; c < dk; ++c) S[(size_t)i * dk + c] += u[i] * kt[c];
            double* ot = o + row * dv;                               /* o = S q */
            for (int i = 0; i < dv; ++i) {
                double acc = 0.0;
                for (int c = 0; c < dk; ++c) acc += S[(size_t)i * dk + c] * qt[c];
                ot[i] = acc;
            }
        }
        if (state_out) memcpy(state_out + bh * sz, S, sizeof(double) * sz);
        free(S);
    }
    return oom ? 1 : 0;
}

/*
 * (c') Gated delta rule with a per-channel (diagonal) decay, S in R^{dv x dk},
 * unit keys assumed (not enforced):
 *   S~_t = S_{t-1} Diag(alpha_t),  S_t = S~_t + beta_t (v_t - S~_t k_t) k_t^T,
 *   o_t = S_t q_t.
 * "Linear attention and recurrent memory", From fixed decay to KDA's gated
 * delta write: the decay gate of the corrective write acting per channel
 * (KDA's finer-grained diagonal decay), taken here on the d_k (key) channels
 * before the write, with the error against the decayed state as in (c).
 * alpha [BH, T, dk]; alpha_t = g_t 1 is variant (c).
 */
int la_oracle_kda(int BH, int T, int dk, int dv,
                  const double* q, const double* k, const double* v,
                  const double* alpha, const double* beta, const double* state_in,
                  double* o, double* state_out, int nthreads) {
    int oom = 0;
    int nt = set_threads(nthreads);
    (void)nt;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt) reduction(|:oom)
#endif
    for (int bh = 0; bh < BH; ++bh) {
        double* S = (double*)malloc(sizeof(double) * ((size_t)dk * dv + dv));
        if (!S) { oom = 1; continue; }
        double* u = S + (size_t)dk * dv;
        const size_t sz = (size_t)dk * dv;
        if (state_in) memcpy(S, state_in + bh * sz, sizeof(double) * sz);
        else memset(S, 0, sizeof(double) * sz);
        for (int t = 0; t < T; ++t) {
            const size_t row = (size_t)bh * T + t;
            const double* kt = k + row * dk;
            const double* qt = q + row * dk;
            const double* vt = v + row * dv;
            const double* at = alpha + row * dk;
            const double bt = beta[row];
            for (int i = 0; i < dv; ++i)                             /* S~ = S Diag(alpha) */
                for (int c = 0; c < dk; ++c) S[(size_t)i * dk + c] *= at[c];
            for (int i = 0; i < dv; ++i) {                           /* u = beta (v - S~ k) */
                double sk = 0.0;
                for (int c = 0; c < dk; ++c) sk += S[(size_t)i * dk + c] * kt[c];
                u[i] = bt * (vt[i] - sk);
            }
            for (int i = 0; i < dv; ++i)                             /* S = S~ + u k^T (after the decay) */
                for (int c = 0; c < dk; ++c) S[(size_t)i * dk + c] += u[i] * kt[c];
            double* ot = o + row * dv;                               /* o = S q, new state */
            for (int i = 0; i < dv; ++i) {
                double acc = 0.0;
                for (int c = 0; c < dk; ++c) acc += S[(size_t)i * dk + c] * qt[c];
                ot[i] = acc;
            }
        }
        if (state_out) memcpy(state_out + bh * sz, S, sizeof(double) * sz);
        free(S);
    }
    return oom ? 1 : 0;
}
