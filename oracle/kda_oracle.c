/*
 * kda_oracle.c -- float64 CPU oracle for the Kimi Delta Attention (KDA) forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * CPU-baseline leg of bench.py load this library.  The product library
 * (chunked_kda_gb300) never links, loads or calls it, and the two share no
 * code, header, table or helper.
 *
 * What it computes, per logical sequence n and head h, token by token, in
 * float64 (plain loops, no blocking, no reordering):
 *
 *     a_t[d] = per-token natural-log decay (gate activation, below)
 *     S      = Diag(exp(a_t)) S                    decay the key rows
 *     r      = S^T k_t                              read-out of the decayed state
 *     S     += beta_t k_t (v_t - r)^T               delta-rule update
 *     o_t    = S^T q_t / sqrt(K)                    read-out of the updated state
 *
 * This is the KDA recurrence: a delta rule whose K x V state decays per key
 * channel.  Where it comes from on the pages:
 *   - attention-gym PR #317 "Add fused recurrent_kda for decode and inference
 *     prefill", Agent note: the call contract (q, k, v, gate, beta,
 *     initial_state, cu_seqlens, output_final_state), FP32 recurrent states with
 *     one leading entry per logical sequence, int32 offsets where a repeated
 *     offset is an empty slot whose state passes through unchanged, a terminal
 *     offset below the physical capacity leaving the tail outside the contract,
 *     the recurrent gate given as a per-token log2 decay, and queries scaled by
 *     1/sqrt(K) inside the op.
 *   - FLA skill page "fla-kda", section "Gate modes": pre-gated mode (g already
 *     is the log-space decay) and the safe in-kernel activation
 *     lower_bound * sigmoid(exp(A_log) * (g + dt_bias)) with A_log required and
 *     dt_bias optional.
 *   - FLA skill page "fla-kda", section "Safe gate numerical note": the gate is
 *     in natural-log units before the RCP_LN2 (1/ln 2) conversion to base 2.
 *   - attention-gym PR #345 "Fuse q l2norm into the chunk_kda output kernel"
 *     (optional, q_eps >= 0): every query row is first normalised,
 *     q_t <- q_t / sqrt(sum_d q_t[d]^2 + q_eps), the l2norm of the inference
 *     callers (its eps floor).  The same normalisation of the key rows
 *     (k_eps >= 0) and beta given as logits (beta_t <- sigmoid(beta_t)) are the
 *     decode-side preprocessing of the recurrent path (attention-gym PR #317,
 *     "Test Plan"; FLA skill "fla-kda", "Correctness checklist": raw beta logits,
 *     qk l2norm in kernel).
 *
 * Layouts (all contiguous, row-major):
 *   q, k : [B, T, Hk, K]        g : [B, T, H, K]      v, o : [B, T, H, V]      beta : [B, T, H]
 *   Hk = H (multi-head) or a divisor of H: value head h reads query/key head h / (H / Hk)
 *   (grouped value heads, HV > H in FLA skill "fla-kda", "Correctness checklist"); gate,
 *   beta, values and states follow the value heads.
 *   A_log, dt_bias : [H, K]     S0, ST : [Nst, H, K, V]  (Nst = n_seqs or B)
 *   cu_seqlens : [n_seqs + 1] int32 (NULL = dense: B rows of length T each;
 *                otherwise B must be 1 and T is the physical capacity).
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* gate modes of the oracle (the last one is the recurrent entry point's input) */
#define ORC_GATE_PRE 0     /* g is the natural-log decay itself                   */
#define ORC_GATE_SAFE 1    /* a = lb * sigmoid(exp(A_log) * (g + dt_bias))        */
#define ORC_GATE_NONSAFE 2 /* a = -exp(A_log) * softplus(g + dt_bias)             */
#define ORC_GATE_LOG2 3    /* g is the per-token log2 decay: decay = 2^g            */

static const double ORC_LN2 = 0.693147180559945309417232121458176568;

/* softplus(x) = ln(1 + e^x), without overflow for large x */
static double softplus(double x)
{
    return x > 0.0 ? x + log1p(exp(-x)) : log1p(exp(x));
}

/*
 * Per-element gate activation, natural-log units.
 * FLA skill "fla-kda", "Gate modes": pre-gated mode passes g through; the safe
 * in-kernel mode is lower_bound * sigmoid(exp(A_log) * (g + dt_bias)); without
 * the safe gate the in-kernel activation is -exp(A_log) * softplus(g + dt_bias),
 * unbounded below.
 * attention-gym PR #317, Agent note: the recurrent gate is a log2 decay, so it
 * is converted back to natural-log units with a factor ln 2.
 */
double kda_oracle_gate_act(double g, double A_log, double dt_bias, int mode, double lb)
{
    if (mode == ORC_GATE_PRE) return g;
    if (mode == ORC_GATE_LOG2) return g * ORC_LN2;
    if (mode == ORC_GATE_NONSAFE) return -exp(A_log) * softplus(g + dt_bias);
    /* ORC_GATE_SAFE */
    double z = exp(A_log) * (g + dt_bias);
    double sig = 1.0 / (1.0 + exp(-z));
    return lb * sig;
}

/* [bos, eos) of logical sequence n; returns the state slot index */
static void seq_bounds(const int32_t* cu, int n, int T, long* bos, long* eos)
{
    if (cu) { *bos = cu[n]; *eos = cu[n + 1]; }
    else    { *bos = (long)n * T; *eos = (long)n * T + T; }
}

/*
 * Gate entry point: activation, then the chunk-local inclusive cumulative sum
 * converted to log2 units (multiply by 1/ln 2).  Chunks start at every
 * sequence start and every chunk_size tokens after it; chunk_size = 1 gives
 * the per-token log2 decay the recurrent entry point takes.
 * FLA skill "fla-kda", "Safe gate numerical note" (RCP_LN2 conversion before
 * exp2); attention-gym PR #317, Agent note (bounded_gate_cumsum with
 * chunk_size=1 is the recurrent gate) and Test Plan (chunk_size 1 vs 64).
 * Tokens outside every sequence (the capacity tail) are not written.
 */
int kda_oracle_gate(const double* g, const double* A_log, const double* dt_bias,
                    int mode, double lb, const int32_t* cu, int n_seqs,
                    int B, int T, int H, int K, int chunk_size, double* out)
{
    if (chunk_size < 1) return 1;
    int N = cu ? n_seqs : B;
    for (int n = 0; n < N; ++n) {
        long bos, eos;
        seq_bounds(cu, n, T, &bos, &eos);
        for (int h = 0; h < H; ++h) {
            for (int d = 0; d < K; ++d) {
                double acc = 0.0;
                for (long t = bos; t < eos; ++t) {
                    if ((t - bos) % chunk_size == 0) acc = 0.0;
                    size_t idx = ((size_t)t * H + h) * K + d;
                    double al = A_log ? A_log[(size_t)h * K + d] : 0.0;
                    double db = dt_bias ? dt_bias[(size_t)h * K + d] : 0.0;
                    acc += kda_oracle_gate_act(g[idx], al, db, mode, lb);
                    out[idx] = acc / ORC_LN2;
                }
            }
        }
    }
    return 0;
}

/*
 * The forward recurrence for one (sequence, head) unit.  S is K x V, row d is
 * key channel d.  Decay first, then the delta update against the decayed
 * state, then the read-out of the updated state (the read-out includes token t).
 */
static void run_unit(const double* q, const double* k, const double* v, const double* g,
                     const double* A_log, const double* dt_bias, int mode, double lb,
                     const double* beta, const double* S0, double* ST, double* o,
                     long bos, long eos, int n, int h, int H, int Hk, int K, int V, double q_eps,
                     double k_eps, int beta_logits, double* S, double* r, double* kn)
{
    size_t st_off = ((size_t)n * H + h) * (size_t)K * V;
    if (S0) memcpy(S, S0 + st_off, sizeof(double) * (size_t)K * V);
    else    memset(S, 0, sizeof(double) * (size_t)K * V);
    const double scale = 1.0 / sqrt((double)K);

    for (long t = bos; t < eos; ++t) {
        const int hk = h / (H / Hk); /* the query / key head of value head h */
        const double* qt = q + ((size_t)t * Hk + hk) * K;
        const double* kt = k + ((size_t)t * Hk + hk) * K;
        if (k_eps >= 0.0) {  /* k_t <- k_t / sqrt(|k_t|^2 + k_eps) */
            double ss = 0.0;
            for (int d = 0; d < K; ++d) ss += kt[d] * kt[d];
            const double ks = 1.0 / sqrt(ss + k_eps);
            for (int d = 0; d < K; ++d) kn[d] = kt[d] * ks;
            kt = kn;
        }
        const double* gt = g + ((size_t)t * H + h) * K;
        const double* vt = v + ((size_t)t * H + h) * V;
        const double braw = beta[(size_t)t * H + h];
        const double bt = beta_logits ? 1.0 / (1.0 + exp(-braw)) : braw;
        double* ot = o + ((size_t)t * H + h) * V;

        /* S = Diag(exp(a_t)) S */
        for (int d = 0; d < K; ++d) {
            double al = A_log ? A_log[(size_t)h * K + d] : 0.0;
            double db = dt_bias ? dt_bias[(size_t)h * K + d] : 0.0;
            double decay = exp(kda_oracle_gate_act(gt[d], al, db, mode, lb));
            for (int j = 0; j < V; ++j) S[(size_t)d * V + j] *= decay;
        }
        /* r = S^T k_t */
        for (int j = 0; j < V; ++j) r[j] = 0.0;
        for (int d = 0; d < K; ++d)
            for (int j = 0; j < V; ++j) r[j] += S[(size_t)d * V + j] * kt[d];
        /* S += beta_t k_t (v_t - r)^T */
        for (int d = 0; d < K; ++d)
            for (int j = 0; j < V; ++j) S[(size_t)d * V + j] += bt * kt[d] * (vt[j] - r[j]);
        /* o_t = S^T q_t / sqrt(K), q_t optionally l2-normalised first */
        double qs = 1.0;
        if (q_eps >= 0.0) {
            double ss = 0.0;
            for (int d = 0; d < K; ++d) ss += qt[d] * qt[d];
            qs = 1.0 / sqrt(ss + q_eps);
        }
        for (int j = 0; j < V; ++j) {
            double acc = 0.0;
            for (int d = 0; d < K; ++d) acc += S[(size_t)d * V + j] * (qt[d] * qs);
            ot[j] = acc * scale;
        }
    }
    /* an empty slot (eos == bos) passes its initial state through unchanged */
    if (ST) memcpy(ST + st_off, S, sizeof(double) * (size_t)K * V);
}

/*
 * Full forward over every unit, or over the listed units only.
 *   units / n_units : optional list of (n, h) pairs (2 * n_units ints); NULL = all.
 *   q_eps, k_eps    : < 0: q (k) as given; >= 0: each q (k) row l2-normalised with this
 *                     eps floor.
 *   beta_logits     : nonzero: beta holds logits, the forward uses sigmoid(beta).
 *   nthreads        : OpenMP threads over independent units (<= 0: library default).
 * Returns 0 on success, 1 on a bad argument, 2 on allocation failure.
 * Outputs of units not computed, and o rows outside every sequence, are not written.
 */
int kda_oracle_fwd(const double* q, const double* k, const double* v, const double* g,
                   const double* A_log, const double* dt_bias, int mode, double lb,
                   const double* beta, const double* S0, double* ST,
                   const int32_t* cu, int n_seqs, int B, int T, int H, int Hk, int K, int V,
                   double* o, double q_eps, double k_eps, int beta_logits,
                   const int32_t* units, int n_units, int nthreads)
{
    if (!q || !k || !v || !g || !beta || !o || H <= 0 || K <= 0 || V <= 0) return 1;
    if (Hk <= 0) Hk = H;
    if (H % Hk != 0) return 1;
    if ((mode == ORC_GATE_SAFE || mode == ORC_GATE_NONSAFE) && !A_log) return 1;
    if (cu && B != 1) return 1;
    int N = cu ? n_seqs : B;
    long total = units ? n_units : (long)N * H;
    int failed = 0;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads) reduction(| : failed)
#endif
    {
        double* S = (double*)malloc(sizeof(double) * (size_t)K * V);
        double* r = (double*)malloc(sizeof(double) * (size_t)V);
        double* kn = (double*)malloc(sizeof(double) * (size_t)K);
        if (!S || !r || !kn) {
            failed = 1;
        } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
            for (long u = 0; u < total; ++u) {
                int n = units ? units[2 * u] : (int)(u / H);
                int h = units ? units[2 * u + 1] : (int)(u % H);
                long bos, eos;
                seq_bounds(cu, n, T, &bos, &eos);
                run_unit(q, k, v, g, A_log, dt_bias, mode, lb, beta, S0, ST, o, bos, eos, n,
                         h, H, Hk, K, V, q_eps, k_eps, beta_logits, S, r, kn);
            }
        }
        free(S);
        free(r);
        free(kn);
    }
    return failed ? 2 : 0;
}

/* threads an OpenMP parallel region of the oracle would use (1 without OpenMP) */
int kda_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
