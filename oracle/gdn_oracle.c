/*
 * gdn_oracle.c -- plain fp64 CPU oracle for the Gated DeltaNet recurrence.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file; only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header or constant with the CUDA
 * library: it is written from the definition of the method, not from the
 * kernels.
 *
 * What it computes (one (sequence n, value head h) at a time, k-head
 * hk = h / (HV/HK)):
 *
 *   S <- init_state[n,h]                    (zeros when absent)
 *   for every token t of sequence n, in order:
 *       q^ = q[t,hk] / sqrt(sum q^2 + eps),  k^ likewise  (when l2norm is on)
 *       a  = exp(g[t,h]),  b = beta[t,h]
 *       S  <- a * S (I - b k^ k^T) + b v[t,h] k^T
 *       o[t,h] = S q^
 *   final_state[n,h] = S
 *
 * Source: "Defending Against the Training-Inference Numeric Mismatch in RL
 * (Especially Linear Attention)", section 3.2 (the recurrent kernel walks
 * one sequence's tokens in order over that sequence's own state, fp32 state
 * cache in the section 4.2 setup tables).  The update equation, the gates
 * a = exp(g), b = sigmoid(.) applied by the caller, and the L2-normalised
 * q/k follow the standard Gated DeltaNet definition (Yang et al., "Gated
 * Delta Networks", ICLR 2025).  o is read from the UPDATED state, S_t q_t.
 *
 * The product S (I - b k k^T) is expanded by distributivity:
 *   [S (I - b k k^T)]_ij = S_ij - b (S k)_i k_j
 * which is the matrix product with a rank-one matrix written out, O(dv dk)
 * per token instead of forming the dense dk x dk projector.
 *
 * Backward: plain backpropagation through time in fp64 for the loss
 *   L = sum_t <dO_t, o_t> + <dS_T, S_T>,
 * with S_{t-1} recomputed from checkpoints every CKPT tokens.  For one step
 * with x = S_{t-1} k^, D = dL/dS_t (all later uses included), y = D k^:
 *   D     += dO_t q^^T               (o_t = S_t q^)
 *   dq^_t  = S_t^T dO_t
 *   dv_t   = b y
 *   db_t   = y . (v - a x)
 *   da_t   = <D, S_{t-1}> - b x . y   ( = <D, S_{t-1} (I - b k^ k^T)> )
 *   dg_t   = a da_t                   (a = exp(g))
 *   dk^_t  = b D^T (v - a x) - a b S_{t-1}^T y
 *   D     <- a (D - b y k^^T)         ( = a D (I - b k^ k^T) )
 * and d_init_state = D after the first token.  The L2-norm backward
 *   dx = (dx^ - x^ (x^ . dx^)) / sqrt(sum x^2 + eps)
 * is applied after the value heads sharing one k-head have been summed in
 * increasing head order (the GQA fold).
 *
 * All arrays are dense, row-major, float64:
 *   q, k   [T, HK, dk]     v, o, dO  [T, HV, dv]     g, beta  [T, HV]
 *   state  [N, HV, dv, dk] (dk fastest)              cu_seqlens int64 [N+1]
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define CKPT 64

/* q^ = x / sqrt(sum x^2 + eps) into out (or a plain copy when norm == 0);
 * returns the divisor (1 when norm == 0). */
static double normalise(const double* x, int n, int norm, double eps, double* out)
{
    if (!norm) {
        for (int j = 0; j < n; ++j) out[j] = x[j];
        return 1.0;
    }
    double ss = 0.0;
    for (int j = 0; j < n; ++j) ss += x[j] * x[j];
    double r = sqrt(ss + eps);
    for (int j = 0; j < n; ++j) out[j] = x[j] / r;
    return r;
}

/* One recurrence step on S (dv x dk): S <- a S (I - b k k^T) + b v k^T.
 * x is scratch of length dv and receives S_{t-1} k. */
static void step(double* S, int dv, int dk, const double* kh, const double* vv,
                 double a, double b, double* x)
{
    for (int i = 0; i < dv; ++i) {
        double s = 0.0;
        for (int j = 0; j < dk; ++j) s += S[(size_t)i * dk + j] * kh[j];
        x[i] = s;
    }
    for (int i = 0; i < dv; ++i)
        for (int j = 0; j < dk; ++j) {
            double* e = &S[(size_t)i * dk + j];
            *e = a * (*e - b * x[i] * kh[j]) + b * vv[i] * kh[j];
        }
}

static void matvec(const double* S, int dv, int dk, const double* xq, double* o)
{
    for (int i = 0; i < dv; ++i) {
        double s = 0.0;
        for (int j = 0; j < dk; ++j) s += S[(size_t)i * dk + j] * xq[j];
        o[i] = s;
    }
}

int gdn_oracle_fwd(int N, const long long* cu, int HK, int HV, int dk, int dv,
                   int l2norm, double eps,
                   const double* q, const double* k, const double* v,
                   const double* g, const double* beta,
                   const double* init_state, double* out, double* final_state,
                   int nthreads)
{
    if (N < 0 || HK <= 0 || HV <= 0 || HV % HK || dk <= 0 || dv <= 0) return -1;
    const int G = HV / HK;
    const size_t SS = (size_t)dv * dk;
    int bad = 0;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads) reduction(| : bad)
#endif
    for (long long unit = 0; unit < (long long)N * HV; ++unit) {
        const int n = (int)(unit / HV), h = (int)(unit % HV), hk = h / G;
        double* S = (double*)malloc(SS * sizeof(double));
        double* kh = (double*)malloc((size_t)dk * sizeof(double));
        double* qh = (double*)malloc((size_t)dk * sizeof(double));
        double* x = (double*)malloc((size_t)dv * sizeof(double));
        if (!S || !kh || !qh || !x) { bad = 1; free(S); free(kh); free(qh); free(x); continue; }
        if (init_state) memcpy(S, init_state + ((size_t)n * HV + h) * SS, SS * sizeof(double));
        else memset(S, 0, SS * sizeof(double));
        for (long long t = cu[n]; t < cu[n + 1]; ++t) {
            normalise(q + ((size_t)t * HK + hk) * dk, dk, l2norm, eps, qh);
            normalise(k + ((size_t)t * HK + hk) * dk, dk, l2norm, eps, kh);
            const double a = exp(g[(size_t)t * HV + h]);
            const double b = beta[(size_t)t * HV + h];
            step(S, dv, dk, kh, v + ((size_t)t * HV + h) * dv, a, b, x);
            matvec(S, dv, dk, qh, out + ((size_t)t * HV + h) * dv);
        }
        if (final_state) memcpy(final_state + ((size_t)n * HV + h) * SS, S, SS * sizeof(double));
        free(S); free(kh); free(qh); free(x);
    }
    return bad ? -2 : 0;
}

/*
 * Backward.  dq_hat / dk_hat are per value head ([T, HV, dk], caller-owned
 * scratch); the fold over the G value heads of one k-head and the L2-norm
 * backward run afterwards, serially, in increasing head order.
 * dq, dk: [T, HK, dk]; dv: [T, HV, dv]; dg, dbeta: [T, HV];
 * d_init_state: [N, HV, dv, dk] (may be NULL); d_final_state may be NULL.
 */
int gdn_oracle_bwd(int N, const long long* cu, int HK, int HV, int dk, int dv,
                   int l2norm, double eps,
                   const double* q, const double* k, const double* v,
                   const double* g, const double* beta, const double* init_state,
                   const double* dO, const double* d_final_state,
                   double* dq_hat, double* dk_hat,
                   double* dq, double* dkk, double* dvv, double* dg, double* dbeta,
                   double* d_init_state, int nthreads)
{
    if (N < 0 || HK <= 0 || HV <= 0 || HV % HK || dk <= 0 || dv <= 0) return -1;
    const int G = HV / HK;
    const size_t SS = (size_t)dv * dk;
    int bad = 0;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads) reduction(| : bad)
#endif
    for (long long unit = 0; unit < (long long)N * HV; ++unit) {
        const int n = (int)(unit / HV), h = (int)(unit % HV), hk = h / G;
        const long long bos = cu[n], L = cu[n + 1] - cu[n];
        const long long nck = (L + CKPT - 1) / CKPT;
        /* ckpt[c] = state before token bos + c*CKPT; blk[i] = state after token i of a block */
        double* ckpt = (double*)malloc((size_t)(nck > 0 ? nck : 1) * SS * sizeof(double));
        double* blk = (double*)malloc((size_t)(CKPT + 1) * SS * sizeof(double));
        double* D = (double*)malloc(SS * sizeof(double));
        double* kh = (double*)malloc((size_t)dk * sizeof(double));
        double* qh = (double*)malloc((size_t)dk * sizeof(double));
        double* x = (double*)malloc((size_t)dv * sizeof(double));
        double* y = (double*)malloc((size_t)dv * sizeof(double));
        double* r = (double*)malloc((size_t)dv * sizeof(double));
        if (!ckpt || !blk || !D || !kh || !qh || !x || !y || !r) {
            bad = 1;
            free(ckpt); free(blk); free(D); free(kh); free(qh); free(x); free(y); free(r);
            continue;
        }
        double* S = blk; /* running state during the checkpoint pass */
        if (init_state) memcpy(S, init_state + ((size_t)n * HV + h) * SS, SS * sizeof(double));
        else memset(S, 0, SS * sizeof(double));
        for (long long i = 0; i < L; ++i) {
            if (i % CKPT == 0) memcpy(ckpt + (size_t)(i / CKPT) * SS, S, SS * sizeof(double));
            const long long t = bos + i;
            normalise(k + ((size_t)t * HK + hk) * dk, dk, l2norm, eps, kh);
            step(S, dv, dk, kh, v + ((size_t)t * HV + h) * dv,
                 exp(g[(size_t)t * HV + h]), beta[(size_t)t * HV + h], x);
        }
        if (d_final_state) memcpy(D, d_final_state + ((size_t)n * HV + h) * SS, SS * sizeof(double));
        else memset(D, 0, SS * sizeof(double));

        for (long long c = nck - 1; c >= 0; --c) {
            const long long i0 = c * CKPT, i1 = (i0 + CKPT < L) ? i0 + CKPT : L;
            /* blk[0] = S_{i0-1} (state before token i0); blk[j+1] = state after token i0+j */
            memcpy(blk, ckpt + (size_t)c * SS, SS * sizeof(double));
            for (long long i = i0; i < i1; ++i) {
                const long long t = bos + i;
                double* Sn = blk + (size_t)(i - i0 + 1) * SS;
                memcpy(Sn, blk + (size_t)(i - i0) * SS, SS * sizeof(double));
                normalise(k + ((size_t)t * HK + hk) * dk, dk, l2norm, eps, kh);
                step(Sn, dv, dk, kh, v + ((size_t)t * HV + h) * dv,
                     exp(g[(size_t)t * HV + h]), beta[(size_t)t * HV + h], x);
            }
            for (long long i = i1 - 1; i >= i0; --i) {
                const long long t = bos + i;
                const double* Sprev = blk + (size_t)(i - i0) * SS;
                const double* Scur = blk + (size_t)(i - i0 + 1) * SS;
                const double* dOt = dO + ((size_t)t * HV + h) * dv;
                const double* vt = v + ((size_t)t * HV + h) * dv;
                const double a = exp(g[(size_t)t * HV + h]);
                const double b = beta[(size_t)t * HV + h];
                normalise(q + ((size_t)t * HK + hk) * dk, dk, l2norm, eps, qh);
                normalise(k + ((size_t)t * HK + hk) * dk, dk, l2norm, eps, kh);
                /* o_t = S_t q^  ->  D += dO q^^T,  dq^ = S_t^T dO */
                double* dqh = dq_hat + ((size_t)t * HV + h) * dk;
                for (int j = 0; j < dk; ++j) {
                    double s = 0.0;
                    for (int ii = 0; ii < dv; ++ii) s += Scur[(size_t)ii * dk + j] * dOt[ii];
                    dqh[j] = s;
                }
                for (int ii = 0; ii < dv; ++ii)
                    for (int j = 0; j < dk; ++j) D[(size_t)ii * dk + j] += dOt[ii] * qh[j];
                matvec(Sprev, dv, dk, kh, x); /* x = S_{t-1} k^ */
                matvec(D, dv, dk, kh, y);     /* y = D k^ */
                double dbt = 0.0, xy = 0.0, dS = 0.0;
                for (int ii = 0; ii < dv; ++ii) {
                    r[ii] = vt[ii] - a * x[ii];
                    dbt += y[ii] * r[ii];
                    xy += x[ii] * y[ii];
                    dvv[((size_t)t * HV + h) * dv + ii] = b * y[ii];
                }
                for (size_t e = 0; e < SS; ++e) dS += D[e] * Sprev[e];
                dbeta[(size_t)t * HV + h] = dbt;
                dg[(size_t)t * HV + h] = a * (dS - b * xy);
                double* dkh = dk_hat + ((size_t)t * HV + h) * dk;
                for (int j = 0; j < dk; ++j) {
                    double s1 = 0.0, s2 = 0.0;
                    for (int ii = 0; ii < dv; ++ii) {
                        s1 += D[(size_t)ii * dk + j] * r[ii];
                        s2 += Sprev[(size_t)ii * dk + j] * y[ii];
                    }
                    dkh[j] = b * s1 - a * b * s2;
                }
                for (int ii = 0; ii < dv; ++ii)
                    for (int j = 0; j < dk; ++j) {
                        double* e = &D[(size_t)ii * dk + j];
                        *e = a * (*e - b * y[ii] * kh[j]);
                    }
            }
        }
        if (d_init_state) memcpy(d_init_state + ((size_t)n * HV + h) * SS, D, SS * sizeof(double));
        free(ckpt); free(blk); free(D); free(kh); free(qh); free(x); free(y); free(r);
    }
    if (bad) return -2;

    /* GQA fold (increasing value head) then the L2-norm backward, per token and k-head. */
    const long long T = N > 0 ? cu[N] : 0;
    double* sq = (double*)malloc((size_t)dk * sizeof(double));
    double* sk = (double*)malloc((size_t)dk * sizeof(double));
    double* xh = (double*)malloc((size_t)dk * sizeof(double));
    if (!sq || !sk || !xh) { free(sq); free(sk); free(xh); return -2; }
    for (long long t = 0; t < T; ++t)
        for (int hk = 0; hk < HK; ++hk) {
            for (int j = 0; j < dk; ++j) { sq[j] = 0.0; sk[j] = 0.0; }
            for (int h = hk * G; h < (hk + 1) * G; ++h)
                for (int j = 0; j < dk; ++j) {
                    sq[j] += dq_hat[((size_t)t * HV + h) * dk + j];
                    sk[j] += dk_hat[((size_t)t * HV + h) * dk + j];
                }
            for (int which = 0; which < 2; ++which) {
                const double* xin = (which ? k : q) + ((size_t)t * HK + hk) * dk;
                const double* dxh = which ? sk : sq;
                double* dx = (which ? dkk : dq) + ((size_t)t * HK + hk) * dk;
                const double rr = normalise(xin, dk, l2norm, eps, xh);
                if (!l2norm) {
                    for (int j = 0; j < dk; ++j) dx[j] = dxh[j];
                    continue;
                }
                double dot = 0.0;
                for (int j = 0; j < dk; ++j) dot += xh[j] * dxh[j];
                for (int j = 0; j < dk; ++j) dx[j] = (dxh[j] - xh[j] * dot) / rr;
            }
        }
    free(sq); free(sk); free(xh);
    return 0;
}

int gdn_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
