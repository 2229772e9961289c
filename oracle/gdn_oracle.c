/*
 * gdn_oracle.c -- float64 CPU oracle of the gated delta rule (TEST INFRASTRUCTURE).
 *
 * This file is test infrastructure.  Only the test-suite, the smoke check and the
 * benchmark's CPU-baseline / reference arm may load it.  It shares no code, header,
 * constant or helper with the CUDA library and is compiled on its own by gcc.
 *
 * What it computes (plain definition, written out token by token):
 *
 *   S_t = alpha_t * S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
 *   o_t = S_t q_t
 *
 * per (batch b, head h) stream, with S in [V, K] (value rows, key columns).
 *   - "Sparse Delta Memory: layer and kernels", section "What the layer computes":
 *     the per-token update (decay the touched rows, read r_t, write beta_t (v_t - r_t)
 *     along the key, then read y_t from the *updated* memory).  Its closing paragraph
 *     on the dense limit (one factor of width d_k, every slot selected, l2-normalised
 *     weights) states that this update then is exactly the Gated DeltaNet recurrence;
 *     the state here is the transpose of that memory, S = M^T.
 *   - "OpenGDN", section "Core operator reference": q, k [B,T,H,K], v [B,T,H,V],
 *     gates [B,T,H], recurrent state [B,H,V,K], and final_state passed back as the
 *     next call's state continues a stream exactly.
 *
 * Readings where the pages leave a choice open (each listed in the design notes):
 *   - no scale on q; the read o_t uses the state after the write;
 *   - alpha and beta are the linear gates (not log alpha); d alpha is w.r.t. alpha;
 *   - any alpha (also 0) and any beta are accepted here.
 *
 * The backward is the chain rule through the same token loop, walked in reverse.
 * With P_t = I - beta_t k_t k_t^T and dS = dL/dS_t accumulated from later tokens,
 * starting from dS = d_final_state (or 0), for t = T-1 .. 0:
 *   dS   += do_t q_t^T
 *   dq_t  = S_t^T do_t
 *   dv_t  = beta_t dS k_t
 *   dbeta_t  = (dS k_t) . (v_t - alpha_t S_{t-1} k_t)
 *   dalpha_t = <dS, S_{t-1} P_t>_F
 *   dk_t  = beta_t dS^T v_t - alpha_t beta_t (S_{t-1}^T dS k_t + dS^T S_{t-1} k_t)
 *   dS    = alpha_t dS P_t            (P_t is symmetric)
 * and d_initial_state = dS at the end.  S_{t-1} comes from a forward replay that keeps
 * a checkpoint every `seg` tokens and recomputes the states inside each segment; the
 * recurrence is never inverted.  The loss is L = sum <do, o> + <d_final_state, S_T>.
 *
 * Layout: every array is dense row-major float64 in the shapes above.
 * Streams are independent; they are spread over `nthreads` OpenMP threads
 * (nthreads <= 0 means the OpenMP default).
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define IDX_QK(b, t, h, j) ((((b) * T + (t)) * H + (h)) * K + (j))
#define IDX_V(b, t, h, j) ((((b) * T + (t)) * H + (h)) * V + (j))
#define IDX_G(b, t, h) (((b) * T + (t)) * H + (h))
#define IDX_S(b, h) (((b) * H + (h)) * V * K)

int oracle_version(void) { return 1; }

int oracle_threads(int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) return nthreads;
    return omp_get_max_threads();
#else
    (void)nthreads;
    return 1;
#endif
}

/* One token of the forward recurrence on a single stream's state S [V,K].
 * x is scratch of length V. */
static void token_step(int64_t K, int64_t V, double* S, const double* kt, const double* vt,
                       double a, double be, double* x) {
    for (int64_t r = 0; r < V; ++r) {
        double acc = 0.0;
        for (int64_t j = 0; j < K; ++j) acc += S[r * K + j] * kt[j];
        x[r] = acc; /* x = S_{t-1} k_t */
    }
    /* S_t = a S - a be x k^T + be v k^T  ==  a S (I - be k k^T) + be v k^T */
    for (int64_t r = 0; r < V; ++r) {
        double coef = be * (vt[r] - a * x[r]);
        for (int64_t j = 0; j < K; ++j) S[r * K + j] = a * S[r * K + j] + coef * kt[j];
    }
}

int oracle_gdn_fwd(int64_t B, int64_t T, int64_t H, int64_t K, int64_t V,
                   const double* q, const double* k, const double* v,
                   const double* alpha, const double* beta,
                   const double* s0, double* o, double* sT, int nthreads) {
    if (B < 0 || T < 0 || H < 0 || K <= 0 || V <= 0) return 1;
    int64_t nstreams = B * H;
    int nt = oracle_threads(nthreads);
    int failed = 0;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt) reduction(| : failed)
    for (int64_t s = 0; s < nstreams; ++s) {
        int64_t b = s / H, h = s % H;
        double* S = (double*)malloc(sizeof(double) * (size_t)(V * K));
        double* x = (double*)malloc(sizeof(double) * (size_t)V);
        if (!S || !x) { free(S); free(x); failed |= 1; continue; }
        if (s0) memcpy(S, s0 + IDX_S(b, h), sizeof(double) * (size_t)(V * K));
        else memset(S, 0, sizeof(double) * (size_t)(V * K));
        for (int64_t t = 0; t < T; ++t) {
            const double* kt = k + IDX_QK(b, t, h, 0);
            const double* qt = q + IDX_QK(b, t, h, 0);
            token_step(K, V, S, kt, v + IDX_V(b, t, h, 0), alpha[IDX_G(b, t, h)],
                       beta[IDX_G(b, t, h)], x);
            double* ot = o + IDX_V(b, t, h, 0);
            for (int64_t r = 0; r < V; ++r) {
                double acc = 0.0;
                for (int64_t j = 0; j < K; ++j) acc += S[r * K + j] * qt[j];
                ot[r] = acc; /* o_t = S_t q_t, read after the write */
            }
        }
        if (sT) memcpy(sT + IDX_S(b, h), S, sizeof(double) * (size_t)(V * K));
        free(S);
        free(x);
    }
    return failed ? 2 : 0;
}

int oracle_gdn_bwd(int64_t B, int64_t T, int64_t H, int64_t K, int64_t V,
                   const double* q, const double* k, const double* v,
                   const double* alpha, const double* beta, const double* s0,
                   const double* d_o, const double* dsT,
                   double* dq, double* dk, double* dv, double* dalpha, double* dbeta,
                   double* ds0, int64_t seg, int nthreads) {
    if (B < 0 || T < 0 || H < 0 || K <= 0 || V <= 0) return 1;
    if (seg <= 0) seg = 64;
    int64_t nstreams = B * H;
    int64_t nseg = (T + seg - 1) / seg;
    int nt = oracle_threads(nthreads);
    int failed = 0;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt) reduction(| : failed)
    for (int64_t s = 0; s < nstreams; ++s) {
        int64_t b = s / H, h = s % H;
        size_t VK = (size_t)(V * K);
        /* ckpt[i] = state before token i*seg; states[j] = state after token (a+j) */
        double* ckpt = (double*)malloc(sizeof(double) * VK * (size_t)(nseg > 0 ? nseg : 1));
        double* states = (double*)malloc(sizeof(double) * VK * (size_t)(seg + 1));
        double* dS = (double*)malloc(sizeof(double) * VK);
        double* x = (double*)malloc(sizeof(double) * (size_t)V);
        double* y = (double*)malloc(sizeof(double) * (size_t)V);
        if (!ckpt || !states || !dS || !x || !y) {
            free(ckpt); free(states); free(dS); free(x); free(y);
            failed |= 1;
            continue;
        }
        /* forward replay, keeping a checkpoint at the start of every segment */
        double* S = states; /* reuse the first slot as the running state */
        if (s0) memcpy(S, s0 + IDX_S(b, h), sizeof(double) * VK);
        else memset(S, 0, sizeof(double) * VK);
        for (int64_t t = 0; t < T; ++t) {
            if (t % seg == 0) memcpy(ckpt + (size_t)(t / seg) * VK, S, sizeof(double) * VK);
            token_step(K, V, S, k + IDX_QK(b, t, h, 0), v + IDX_V(b, t, h, 0),
                       alpha[IDX_G(b, t, h)], beta[IDX_G(b, t, h)], x);
        }
        if (dsT) memcpy(dS, dsT + IDX_S(b, h), sizeof(double) * VK);
        else memset(dS, 0, sizeof(double) * VK);

        for (int64_t sg = nseg - 1; sg >= 0; --sg) {
            int64_t t0 = sg * seg;
            int64_t t1 = t0 + seg < T ? t0 + seg : T;
            /* states[j] = S_{t0 + j - 1}, i.e. states[0] = state before token t0 */
            memcpy(states, ckpt + (size_t)sg * VK, sizeof(double) * VK);
            for (int64_t t = t0; t < t1; ++t) {
                double* nxt = states + (size_t)(t - t0 + 1) * VK;
                memcpy(nxt, states + (size_t)(t - t0) * VK, sizeof(double) * VK);
                token_step(K, V, nxt, k + IDX_QK(b, t, h, 0), v + IDX_V(b, t, h, 0),
                           alpha[IDX_G(b, t, h)], beta[IDX_G(b, t, h)], x);
            }
            for (int64_t t = t1 - 1; t >= t0; --t) {
                const double* Sp = states + (size_t)(t - t0) * VK;     /* S_{t-1} */
                const double* Sc = states + (size_t)(t - t0 + 1) * VK; /* S_t */
                const double* kt = k + IDX_QK(b, t, h, 0);
                const double* qt = q + IDX_QK(b, t, h, 0);
                const double* vt = v + IDX_V(b, t, h, 0);
                const double* dot = d_o + IDX_V(b, t, h, 0);
                double a = alpha[IDX_G(b, t, h)], be = beta[IDX_G(b, t, h)];
                /* dS += do_t q_t^T */
                for (int64_t r = 0; r < V; ++r)
                    for (int64_t j = 0; j < K; ++j) dS[r * K + j] += dot[r] * qt[j];
                /* dq_t = S_t^T do_t */
                double* dqt = dq + IDX_QK(b, t, h, 0);
                for (int64_t j = 0; j < K; ++j) {
                    double acc = 0.0;
                    for (int64_t r = 0; r < V; ++r) acc += Sc[r * K + j] * dot[r];
                    dqt[j] = acc;
                }
                /* x = S_{t-1} k_t ; y = dS k_t */
                for (int64_t r = 0; r < V; ++r) {
                    double ax = 0.0, ay = 0.0;
                    for (int64_t j = 0; j < K; ++j) {
                        ax += Sp[r * K + j] * kt[j];
                        ay += dS[r * K + j] * kt[j];
                    }
                    x[r] = ax;
                    y[r] = ay;
                }
                /* dv_t = beta dS k_t */
                double* dvt = dv + IDX_V(b, t, h, 0);
                for (int64_t r = 0; r < V; ++r) dvt[r] = be * y[r];
                /* dbeta_t = (dS k_t) . (v_t - alpha S_{t-1} k_t) */
                double db = 0.0;
                for (int64_t r = 0; r < V; ++r) db += y[r] * (vt[r] - a * x[r]);
                dbeta[IDX_G(b, t, h)] = db;
                /* dalpha_t = <dS, S_{t-1} P_t> = <dS, S_{t-1}> - beta <dS k_t, S_{t-1} k_t> */
                double ip = 0.0, yx = 0.0;
                for (size_t e = 0; e < VK; ++e) ip += dS[e] * Sp[e];
                for (int64_t r = 0; r < V; ++r) yx += y[r] * x[r];
                dalpha[IDX_G(b, t, h)] = ip - be * yx;
                /* dk_t = beta dS^T v_t - alpha beta (S_{t-1}^T (dS k_t) + dS^T (S_{t-1} k_t)) */
                double* dkt = dk + IDX_QK(b, t, h, 0);
                for (int64_t j = 0; j < K; ++j) {
                    double t1v = 0.0, t2 = 0.0, t3 = 0.0;
                    for (int64_t r = 0; r < V; ++r) {
                        t1v += dS[r * K + j] * vt[r];
                        t2 += Sp[r * K + j] * y[r];
                        t3 += dS[r * K + j] * x[r];
                    }
                    dkt[j] = be * t1v - a * be * (t2 + t3);
                }
                /* dS <- alpha dS P_t = alpha (dS - beta (dS k_t) k_t^T) */
                for (int64_t r = 0; r < V; ++r)
                    for (int64_t j = 0; j < K; ++j)
                        dS[r * K + j] = a * (dS[r * K + j] - be * y[r] * kt[j]);
            }
        }
        if (ds0) memcpy(ds0 + IDX_S(b, h), dS, sizeof(double) * VK);
        free(ckpt); free(states); free(dS); free(x); free(y);
    }
    return failed ? 2 : 0;
}
