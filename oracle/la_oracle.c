/*
 * la_oracle.c -- plain FP64 CPU oracle for the Lightning Attention prefill.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the checker, not the product: only
 * the test-suite, the smoke check and the CPU-baseline leg of the benchmark
 * may build, load or call it.  It shares no code, header, table or helper with
 * the CUDA path.
 *
 * What it computes (pages: "[Lightning Attention] Add Hopper SM90 CuTe DSL
 * prefill", Description and Reviewer notes; "[LA] Lightning Attention MTP
 * decode + KVBuffer parallel verify / commit", Description, closed form):
 *
 *   for every sequence n and value head hv, with q/k head hq = hv / (HV / H)
 *   and lambda = exp(-slope[hv]):
 *       S   = h0[slot][hv]            (or 0), S stored [V][K]
 *       for t = 0 .. L-1:
 *           S[v][k] = lambda * S[v][k] + v_t[v] * k_t[k]
 *           o_t[v]  = scale * sum_k S[v][k] * q_t[k]
 *       h_final[slot][hv] = S
 *
 * The state is updated before it is read, so o_t sees k_t v_t (same-token
 * causality), and h0 enters o_t with lambda^(t+1) ("exponent offset 1").
 *
 * Two independent evaluations are provided:
 *   la_oracle_tokenwise  -- the recurrence above, one token at a time.
 *   la_oracle_chunked    -- the chunkwise form the pages describe: per chunk
 *                           of C tokens an intra term (Q K^T masked by the
 *                           causal decay lambda^(s-j)) . V, an inter term
 *                           lambda^(s+1) * Q . S, and one state advance
 *                           S <- lambda^L S + sum_j lambda^(L-1-j) v_j k_j^T.
 *
 * Everything is double precision; q, k, v arrive as float32 (the BF16-rounded
 * values, upcast exactly) and h0 as double.  Build with -ffp-contract=off and no fast-math so
 * each multiply and add rounds in the order written.
 *
 * Storage note: inside a unit the state is kept transposed (St[k][v]) so the
 * two inner loops run over contiguous memory; every sum is still taken over k
 * (or j) in increasing order, exactly as the definition above reads.  The
 * public orientation [V][K] is used for h0 and h_final.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum {
    LAO_OK = 0,
    LAO_BAD_SHAPE = -1,
    LAO_BAD_SEQLENS = -2,
    LAO_BAD_INDEX = -3,
    LAO_NO_MEMORY = -4
};

typedef struct {
    const float *q, *k, *v, *slopes;
    const double *h0;
    const int32_t *state_indices, *cu_seqlens;
    double scale;
    int N, T, H, HV, D, V, pool_size;
    double *o, *h_final;
} lao_problem;

/* Sequence bounds: packed via cu_seqlens, else fixed length T. */
static void seq_bounds(const lao_problem *p, int n, int64_t *bos, int64_t *len)
{
    if (p->cu_seqlens) {
        *bos = p->cu_seqlens[n];
        *len = (int64_t)p->cu_seqlens[n + 1] - p->cu_seqlens[n];
    } else {
        *bos = (int64_t)n * p->T;
        *len = p->T;
    }
}

/* Host-side validation shared by both evaluations (argument checks only). */
static int validate(const lao_problem *p)
{
    if (p->N < 0 || p->H <= 0 || p->HV <= 0 || p->D <= 0 || p->V <= 0)
        return LAO_BAD_SHAPE;
    if (p->HV % p->H != 0)
        return LAO_BAD_SHAPE;
    if (!p->cu_seqlens && p->T < 0)
        return LAO_BAD_SHAPE;
    if (p->cu_seqlens) {
        if (p->cu_seqlens[0] != 0)
            return LAO_BAD_SEQLENS;
        for (int n = 0; n < p->N; ++n)
            if (p->cu_seqlens[n + 1] < p->cu_seqlens[n])
                return LAO_BAD_SEQLENS;
    }
    if (p->state_indices) {
        for (int n = 0; n < p->N; ++n)
            if (p->state_indices[n] >= p->pool_size)
                return LAO_BAD_INDEX;
    }
    return LAO_OK;
}

/* Which state slot a sequence reads and writes; -1 = padded (skipped). */
static int64_t slot_of(const lao_problem *p, int n)
{
    if (p->state_indices)
        return p->state_indices[n] < 0 ? -1 : p->state_indices[n];
    return n;
}

static void load_state(const lao_problem *p, int64_t slot, int hv, double *St)
{
    const int D = p->D, V = p->V;
    if (!p->h0) {
        memset(St, 0, sizeof(double) * (size_t)D * V);
        return;
    }
    const double *src = p->h0 + ((size_t)slot * p->HV + hv) * (size_t)V * D;
    for (int vv = 0; vv < V; ++vv)
        for (int kk = 0; kk < D; ++kk)
            St[(size_t)kk * V + vv] = src[(size_t)vv * D + kk];
}

static void store_state(const lao_problem *p, int64_t slot, int hv, const double *St)
{
    const int D = p->D, V = p->V;
    if (!p->h_final)
        return;
    double *dst = p->h_final + ((size_t)slot * p->HV + hv) * (size_t)V * D;
    for (int vv = 0; vv < V; ++vv)
        for (int kk = 0; kk < D; ++kk)
            dst[(size_t)vv * D + kk] = St[(size_t)kk * V + vv];
}

/* ---- tokenwise recurrence ------------------------------------------------ */

static void unit_tokenwise(const lao_problem *p, int n, int hv, double *St, double *acc)
{
    const int D = p->D, V = p->V, H = p->H, HV = p->HV;
    const int hq = hv / (HV / H);
    const double lam = exp(-(double)p->slopes[hv]);
    int64_t bos, len;
    seq_bounds(p, n, &bos, &len);
    const int64_t slot = slot_of(p, n);
    if (slot < 0)
        return; /* padded sequence: nothing read, nothing written */
    load_state(p, slot, hv, St);
    for (int64_t t = 0; t < len; ++t) {
        const float *qt = p->q + ((size_t)(bos + t) * H + hq) * D;
        const float *kt = p->k + ((size_t)(bos + t) * H + hq) * D;
        const float *vt = p->v + ((size_t)(bos + t) * HV + hv) * V;
        /* h_t = lambda h_{t-1} + k_t^T v_t */
        for (int kk = 0; kk < D; ++kk) {
            const double kv = (double)kt[kk];
            double *row = St + (size_t)kk * V;
            for (int vv = 0; vv < V; ++vv)
                row[vv] = lam * row[vv] + kv * (double)vt[vv];
        }
        /* o_t = scale * q_t h_t, summed over k in increasing order */
        for (int vv = 0; vv < V; ++vv)
            acc[vv] = 0.0;
        for (int kk = 0; kk < D; ++kk) {
            const double qk = (double)qt[kk];
            const double *row = St + (size_t)kk * V;
            for (int vv = 0; vv < V; ++vv)
                acc[vv] = acc[vv] + row[vv] * qk;
        }
        double *ot = p->o + ((size_t)(bos + t) * HV + hv) * V;
        for (int vv = 0; vv < V; ++vv)
            ot[vv] = p->scale * acc[vv];
    }
    store_state(p, slot, hv, St);
}

/* ---- chunkwise form -------------------------------------------------------- */

static void unit_chunked(const lao_problem *p, int n, int hv, int C, double *St,
                         double *acc, double *A, double *pw)
{
    const int D = p->D, V = p->V, H = p->H, HV = p->HV;
    const int hq = hv / (HV / H);
    const double lam = exp(-(double)p->slopes[hv]);
    int64_t bos, len;
    seq_bounds(p, n, &bos, &len);
    const int64_t slot = slot_of(p, n);
    if (slot < 0)
        return;
    /* pw[m] = lambda^m, with lambda^0 = 1 even when lambda underflows to 0 */
    for (int m = 0; m <= C; ++m)
        pw[m] = pow(lam, (double)m);
    load_state(p, slot, hv, St);
    for (int64_t c0 = 0; c0 < len; c0 += C) {
        const int L = (int)((len - c0) < C ? (len - c0) : C);
        const int64_t r0 = bos + c0;
        /* intra scores A[s][j] = q_s . k_j for j <= s */
        for (int s = 0; s < L; ++s) {
            const float *qs = p->q + ((size_t)(r0 + s) * H + hq) * D;
            for (int j = 0; j <= s; ++j) {
                const float *kj = p->k + ((size_t)(r0 + j) * H + hq) * D;
                double d = 0.0;
                for (int kk = 0; kk < D; ++kk)
                    d = d + (double)qs[kk] * (double)kj[kk];
                A[(size_t)s * C + j] = d;
            }
        }
        for (int s = 0; s < L; ++s) {
            const float *qs = p->q + ((size_t)(r0 + s) * H + hq) * D;
            /* inter term: lambda^(s+1) * (S q_s) with the chunk-entry state */
            for (int vv = 0; vv < V; ++vv)
                acc[vv] = 0.0;
            for (int kk = 0; kk < D; ++kk) {
                const double qk = (double)qs[kk];
                const double *row = St + (size_t)kk * V;
                for (int vv = 0; vv < V; ++vv)
                    acc[vv] = acc[vv] + row[vv] * qk;
            }
            double *ot = p->o + ((size_t)(r0 + s) * HV + hv) * V;
            for (int vv = 0; vv < V; ++vv)
                ot[vv] = pw[s + 1] * acc[vv];
            /* intra term: sum_{j<=s} lambda^(s-j) A[s][j] v_j */
            for (int vv = 0; vv < V; ++vv)
                acc[vv] = 0.0;
            for (int j = 0; j <= s; ++j) {
                const double w = pw[s - j] * A[(size_t)s * C + j];
                const float *vj = p->v + ((size_t)(r0 + j) * HV + hv) * V;
                for (int vv = 0; vv < V; ++vv)
                    acc[vv] = acc[vv] + w * (double)vj[vv];
            }
            for (int vv = 0; vv < V; ++vv)
                ot[vv] = p->scale * (ot[vv] + acc[vv]);
        }
        /* state advance: S <- lambda^L S + sum_j lambda^(L-1-j) v_j k_j^T */
        for (int kk = 0; kk < D; ++kk) {
            double *row = St + (size_t)kk * V;
            for (int vv = 0; vv < V; ++vv)
                row[vv] = pw[L] * row[vv];
        }
        for (int j = 0; j < L; ++j) {
            const float *kj = p->k + ((size_t)(r0 + j) * H + hq) * D;
            const float *vj = p->v + ((size_t)(r0 + j) * HV + hv) * V;
            const double w = pw[L - 1 - j];
            for (int kk = 0; kk < D; ++kk) {
                const double kt = w * (double)kj[kk];
                double *row = St + (size_t)kk * V;
                for (int vv = 0; vv < V; ++vv)
                    row[vv] = row[vv] + kt * (double)vj[vv];
            }
        }
    }
    store_state(p, slot, hv, St);
}

/* ---- drivers ------------------------------------------------------------- */

static int run(const lao_problem *p, int chunk, int nthreads)
{
    int rc = validate(p);
    if (rc != LAO_OK)
        return rc;
    const int64_t units = (int64_t)p->N * p->HV;
    const int D = p->D, V = p->V;
    const int C = chunk > 0 ? chunk : 1;
    int failed = 0;
#ifdef _OPENMP
    if (nthreads <= 0)
        nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads) reduction(| : failed)
#endif
    {
        double *St = (double *)malloc(sizeof(double) * (size_t)D * V);
        double *acc = (double *)malloc(sizeof(double) * (size_t)V);
        double *A = chunk > 0 ? (double *)malloc(sizeof(double) * (size_t)C * C) : NULL;
        double *pw = chunk > 0 ? (double *)malloc(sizeof(double) * (size_t)(C + 1)) : NULL;
        const int ok = St && acc && (chunk <= 0 || (A && pw));
        if (!ok)
            failed = 1;
        /* every thread reaches the work-sharing loop; one without buffers skips its share */
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int64_t u = 0; u < units; ++u) {
            if (!ok)
                continue;
            const int n = (int)(u / p->HV), hv = (int)(u % p->HV);
            if (chunk > 0)
                unit_chunked(p, n, hv, C, St, acc, A, pw);
            else
                unit_tokenwise(p, n, hv, St, acc);
        }
        free(St);
        free(acc);
        free(A);
        free(pw);
    }
    (void)nthreads;
    return failed ? LAO_NO_MEMORY : LAO_OK;
}

/*
 * Arguments (all host pointers, row-major, caller-owned):
 *   q, k       float [tokens, H, D]      (BF16 values upcast)
 *   v          float [tokens, HV, V]
 *   slopes     float [HV]                lambda = exp(-slope)
 *   h0         double [P, HV, V, D] or NULL (zero initial state; the FP32
 *              states of the GPU path upcast exactly)
 *   state_indices int32 [N] or NULL      slot per sequence, <0 = padded
 *   cu_seqlens int32 [N+1] or NULL       NULL = fixed length T
 *   o          double [tokens, HV, V]    rows of padded sequences untouched
 *   h_final    double [P, HV, V, D] or NULL; only the selected slots written
 * P is pool_size when state_indices is given, else N.
 */
int la_oracle_tokenwise(const float *q, const float *k, const float *v, const float *slopes,
                        double scale, const double *h0, const int32_t *state_indices,
                        const int32_t *cu_seqlens, int N, int T, int H, int HV, int D, int V,
                        int pool_size, double *o, double *h_final, int nthreads)
{
    lao_problem p = {q, k, v, slopes, h0, state_indices, cu_seqlens, scale,
                     N, T, H, HV, D, V, pool_size, o, h_final};
    return run(&p, 0, nthreads);
}

int la_oracle_chunked(const float *q, const float *k, const float *v, const float *slopes,
                      double scale, const double *h0, const int32_t *state_indices,
                      const int32_t *cu_seqlens, int N, int T, int H, int HV, int D, int V,
                      int pool_size, double *o, double *h_final, int chunk, int nthreads)
{
    lao_problem p = {q, k, v, slopes, h0, state_indices, cu_seqlens, scale,
                     N, T, H, HV, D, V, pool_size, o, h_final};
    if (chunk <= 0)
        return LAO_BAD_SHAPE;
    return run(&p, chunk, nthreads);
}

/* ---- backward: gradients of a scalar loss through the recurrence ----------
 *
 * The forward pass (tokens t = 0 .. L-1 of one sequence and value head, S_{-1} = h0):
 *     S_t = lambda S_{t-1} + v_t k_t^T        (S stored [V][K])
 *     o_t = scale S_t q_t                     h_final = S_{L-1}
 * Given dout_t = dL/do_t and dh_final = dL/dh_final (or 0), the chain rule gives
 *     dq_t = scale S_t^T dout_t
 *     G_t  = dL/dS_t = scale dout_t q_t^T + lambda G_{t+1},   G_L = dh_final
 *     dk_t = G_t^T v_t,    dv_t = G_t k_t,    dh0 = lambda G_0
 * (an empty sequence passes dh_final through: dh0 = dh_final).  With value heads sharing a
 * q/k head, dq and dk of that head are the sums over its value heads.  One forward sweep
 * per unit carries S and gives dq; one reverse sweep carries G and gives dk, dv, dh0.
 */
static void unit_backward(const lao_problem *p, const float *dout, const double *dh_final, double *dq, double *dk,
                          double *dv, double *dh0, int n, int hv, double *M, double *acc)
{
    const int D = p->D, V = p->V, H = p->H, HV = p->HV;
    const int hq = hv / (HV / H);
    const double lam = exp(-(double)p->slopes[hv]);
    int64_t bos, len;
    seq_bounds(p, n, &bos, &len);
    const int64_t slot = slot_of(p, n);
    /* forward sweep: M[v][k] = S_t, dq_t += scale S_t^T dout_t */
    if (p->h0) {
        const double *src = p->h0 + ((size_t)slot * HV + hv) * (size_t)V * D;
        memcpy(M, src, sizeof(double) * (size_t)V * D);
    } else {
        memset(M, 0, sizeof(double) * (size_t)V * D);
    }
    for (int64_t t = 0; t < len; ++t) {
        const float *kt = p->k + ((size_t)(bos + t) * H + hq) * D;
        const float *vt = p->v + ((size_t)(bos + t) * HV + hv) * V;
        const float *dot = dout + ((size_t)(bos + t) * HV + hv) * V;
        for (int vv = 0; vv < V; ++vv) {
            double *row = M + (size_t)vv * D;
            for (int kk = 0; kk < D; ++kk)
                row[kk] = lam * row[kk] + (double)vt[vv] * (double)kt[kk];
        }
        double *dqt = dq + ((size_t)(bos + t) * H + hq) * D;
        for (int kk = 0; kk < D; ++kk)
            acc[kk] = 0.0;
        for (int vv = 0; vv < V; ++vv) {
            const double g = (double)dot[vv];
            const double *row = M + (size_t)vv * D;
            for (int kk = 0; kk < D; ++kk)
                acc[kk] = acc[kk] + row[kk] * g;
        }
        for (int kk = 0; kk < D; ++kk)
            dqt[kk] = dqt[kk] + p->scale * acc[kk];
    }
    /* reverse sweep: M[v][k] = G_t */
    if (dh_final) {
        const double *src = dh_final + ((size_t)slot * HV + hv) * (size_t)V * D;
        memcpy(M, src, sizeof(double) * (size_t)V * D);
    } else {
        memset(M, 0, sizeof(double) * (size_t)V * D);
    }
    for (int64_t t = len - 1; t >= 0; --t) {
        const float *qt = p->q + ((size_t)(bos + t) * H + hq) * D;
        const float *kt = p->k + ((size_t)(bos + t) * H + hq) * D;
        const float *vt = p->v + ((size_t)(bos + t) * HV + hv) * V;
        const float *dot = dout + ((size_t)(bos + t) * HV + hv) * V;
        /* G_t = scale dout_t q_t^T + lambda G_{t+1} (M holds lambda-free G_{t+1} here) */
        for (int vv = 0; vv < V; ++vv) {
            const double g = p->scale * (double)dot[vv];
            double *row = M + (size_t)vv * D;
            for (int kk = 0; kk < D; ++kk)
                row[kk] = row[kk] + g * (double)qt[kk];
        }
        /* dk_t += G_t^T v_t, dv_t = G_t k_t */
        double *dkt = dk + ((size_t)(bos + t) * H + hq) * D;
        for (int kk = 0; kk < D; ++kk)
            acc[kk] = 0.0;
        for (int vv = 0; vv < V; ++vv) {
            const double x = (double)vt[vv];
            const double *row = M + (size_t)vv * D;
            for (int kk = 0; kk < D; ++kk)
                acc[kk] = acc[kk] + row[kk] * x;
        }
        for (int kk = 0; kk < D; ++kk)
            dkt[kk] = dkt[kk] + acc[kk];
        double *dvt = dv + ((size_t)(bos + t) * HV + hv) * V;
        for (int vv = 0; vv < V; ++vv) {
            const double *row = M + (size_t)vv * D;
            double d = 0.0;
            for (int kk = 0; kk < D; ++kk)
                d = d + row[kk] * (double)kt[kk];
            dvt[vv] = d;
        }
        /* carry lambda G_t to the previous token */
        for (size_t e = 0; e < (size_t)V * D; ++e)
            M[e] = lam * M[e];
    }
    if (dh0) {
        double *dst = dh0 + ((size_t)slot * HV + hv) * (size_t)V * D;
        memcpy(dst, M, sizeof(double) * (size_t)V * D);
    }
}

/*
 * Arguments as la_oracle_tokenwise, plus (host pointers, row-major, caller-owned):
 *   dout       float [tokens, HV, V]      dL/do (BF16 values upcast)
 *   dh_final   double [P, HV, V, D] or NULL   dL/dh_final (zero when NULL)
 *   dq, dk     double [tokens, H, D]      rows of padded sequences untouched
 *   dv         double [tokens, HV, V]     rows of padded sequences untouched
 *   dh0        double [P, HV, V, D] or NULL; only the selected slots written
 */
int la_oracle_backward(const float *q, const float *k, const float *v, const float *slopes, double scale,
                       const double *h0, const float *dout, const double *dh_final,
                       const int32_t *state_indices, const int32_t *cu_seqlens, int N, int T, int H, int HV,
                       int D, int V, int pool_size, double *dq, double *dk, double *dv, double *dh0, int nthreads)
{
    lao_problem p = {q, k, v, slopes, h0, state_indices, cu_seqlens, scale,
                     N, T, H, HV, D, V, pool_size, NULL, NULL};
    int rc = validate(&p);
    if (rc != LAO_OK)
        return rc;
    const int G = HV / H;
    const int64_t groups = (int64_t)N * H; /* one (sequence, q/k head) per task: no shared writes */
    int failed = 0;
#ifdef _OPENMP
    if (nthreads <= 0)
        nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads) reduction(| : failed)
#endif
    {
        double *M = (double *)malloc(sizeof(double) * (size_t)V * D);
        double *acc = (double *)malloc(sizeof(double) * (size_t)(D > V ? D : V));
        const int ok = M && acc;
        if (!ok)
            failed = 1;
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int64_t u = 0; u < groups; ++u) {
            if (!ok)
                continue;
            const int n = (int)(u / H), hq = (int)(u % H);
            if (slot_of(&p, n) < 0)
                continue; /* padded sequence: nothing read, nothing written */
            int64_t bos, len;
            seq_bounds(&p, n, &bos, &len);
            for (int64_t t = 0; t < len; ++t) {
                memset(dq + ((size_t)(bos + t) * H + hq) * D, 0, sizeof(double) * (size_t)D);
                memset(dk + ((size_t)(bos + t) * H + hq) * D, 0, sizeof(double) * (size_t)D);
            }
            for (int g = 0; g < G; ++g)
                unit_backward(&p, dout, dh_final, dq, dk, dv, dh0, n, hq * G + g, M, acc);
        }
        free(M);
        free(acc);
    }
    (void)nthreads;
    return failed ? LAO_NO_MEMORY : LAO_OK;
}

int la_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
