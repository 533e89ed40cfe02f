/*
 * gdn_oracle.c -- fp64 CPU oracle for the gated delta-rule (GDN) recurrence.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke check
 * of __graft_entry__ and the CPU-baseline leg of bench.py may load this file.
 * It shares no code, header, table or helper with the CUDA library; the two
 * meet only on the seeded input tensors.
 *
 * What it computes (plain definition, one token at a time, in fp64):
 *
 *   for every batch b and value head h, with query/key head hk = h / (Hv/Hk)
 *     ("GDN CTE Kernel API Reference", Notes: value head h reads key/query
 *      head h // (Hv//Hk)),
 *   starting from the supplied state S0 or from zeros
 *     ("GDN CTE Kernel API Reference", Parameters / recurrent_state:
 *      supplied -> incoming contents are the initial state; omitted -> zero),
 *   for t = 0 .. S-1 in order:
 *       a_t = exp(g_t)                         (g_log is a log-decay, Parameters / g_log)
 *       p   = S_{t-1}^T k_t                    (state S is [Dk, Dv], Parameters / recurrent_state)
 *       S_t = a_t S_{t-1} + beta_t k_t (v_t - a_t p)^T
 *       o_t = scale * S_t^T q_t                (scale applied to the query, Parameters / scale;
 *                                               output un-normalised, head-major, Returns)
 *
 * The update is the gated delta rule that the "Background" section of the
 * "GDN CTE Kernel API Reference" page names; the page does not print the
 * formula, so this file writes out the standard reading of it: decay inside the
 * error term, output read from the post-update state.  Layouts follow the
 * "Parameters" section of that page:
 *   q, k   [B, Hk, S, Dk]      v, out [B, Hv, S, Dv]
 *   g, beta [B, Hv, S]         state  [B, Hv, Dk, Dv]  (Dv contiguous)
 * All arrays are row-major fp64.
 *
 * Parallelism: the B*Hv sequences are independent, so an OpenMP loop runs over
 * them; each sequence is processed strictly in token order.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int gdn_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void gdn_oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* Returns 0 on success, 1 on inconsistent dims, 2 on allocation failure. */
int gdn_oracle_recurrence(const double* q, const double* k, const double* v,
                          const double* g_log, const double* beta, double scale,
                          const double* state_in, /* may be NULL: zero start */
                          long B, long Hk, long Hv, long S, long Dk, long Dv,
                          double* out, double* state_out)
{
    if (B < 0 || Hk <= 0 || Hv <= 0 || S < 0 || Dk <= 0 || Dv <= 0) return 1;
    if (Hv % Hk != 0) return 1;
    const long G = Hv / Hk;
    int failed = 0;

#pragma omp parallel for schedule(dynamic, 1)
    for (long bh = 0; bh < B * Hv; ++bh) {
        const long b = bh / Hv;
        const long h = bh % Hv;
        const long hk = h / G;
        double* St = state_out + bh * Dk * Dv;
        double* p = (double*)malloc((size_t)Dv * sizeof(double));
        double* d = (double*)malloc((size_t)Dv * sizeof(double));
        if (!p || !d) {
            free(p);
            free(d);
#pragma omp atomic write
            failed = 1;
            continue;
        }
        if (state_in)
            memcpy(St, state_in + bh * Dk * Dv, (size_t)(Dk * Dv) * sizeof(double));
        else
            memset(St, 0, (size_t)(Dk * Dv) * sizeof(double));

        for (long t = 0; t < S; ++t) {
            const double* kt = k + ((b * Hk + hk) * S + t) * Dk;
            const double* qt = q + ((b * Hk + hk) * S + t) * Dk;
            const double* vt = v + (bh * S + t) * Dv;
            const double a = exp(g_log[bh * S + t]);
            const double bt = beta[bh * S + t];
            double* ot = out + (bh * S + t) * Dv;

            /* p = S_{t-1}^T k_t */
            for (long j = 0; j < Dv; ++j) p[j] = 0.0;
            for (long i = 0; i < Dk; ++i) {
                const double ki = kt[i];
                const double* row = St + i * Dv;
                for (long j = 0; j < Dv; ++j) p[j] += row[j] * ki;
            }
            /* d = beta_t (v_t - a_t p) */
            for (long j = 0; j < Dv; ++j) d[j] = bt * (vt[j] - a * p[j]);
            /* S_t = a_t S_{t-1} + k_t d^T */
            for (long i = 0; i < Dk; ++i) {
                const double ki = kt[i];
                double* row = St + i * Dv;
                for (long j = 0; j < Dv; ++j) row[j] = a * row[j] + ki * d[j];
            }
            /* o_t = scale * S_t^T q_t */
            for (long j = 0; j < Dv; ++j) ot[j] = 0.0;
            for (long i = 0; i < Dk; ++i) {
                const double qi = qt[i];
                const double* row = St + i * Dv;
                for (long j = 0; j < Dv; ++j) ot[j] += row[j] * qi;
            }
            for (long j = 0; j < Dv; ++j) ot[j] *= scale;
        }
        free(p);
        free(d);
    }
    return failed ? 2 : 0;
}
