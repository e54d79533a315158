/*
 * liboracle -- float64 CPU oracle for the packed linear-attention pass.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the test-suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or helper with
 * the CUDA library.
 *
 * What it computes ("Serving 0.88M TPS from Two RTXs and Mac Minis",
 * section "The Workload" and section "Kernels"): unnormalised causal linear
 * attention, independently per head h, written as the plain recurrence
 *
 *     S_t = S_{t-1} + k_t v_t^T          (S is d_k x d_v, S[i][j] += k_t[i] v_t[j])
 *     o_t = S_t^T q_t                    (o_t[j] = sum_i S_t[i][j] q_t[i])
 *
 * The diagonal is inclusive: o_t already sees k_t v_t^T.  No feature map, no
 * normaliser, no decay and no 1/sqrt(d) scale.
 *
 * A packed pass holds views and branches (same page, section "The Workload":
 * one long view, many short branches; branches attend to the view but not to
 * each other).  Every view starts from S = 0; its state after its last row is
 * the view's final state.  Every branch starts from a copy of its parent
 * view's final state and runs the same recurrence over its own rows only, so
 * sibling branches never see one another (section "Long Requests": branches
 * only attend to their own view).
 *
 * Layout: q, k, v and out are row-major [T][H][D] float64; states are
 * [n][H][D][D] float64 with S[i][j] at i*D + j (row = key dim, col = value
 * dim).  Segments are given by non-decreasing absolute row offsets
 * (cu_seqlens).  Rows in no segment are not written.
 *
 * Work is split over (segment, head) with OpenMP; the arithmetic inside one
 * (segment, head) is strictly sequential in row order, so results do not
 * depend on the thread count.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Run the recurrence over rows [r0, r1) of head h, starting from S (updated in place). */
static void run_rows(const double *q, const double *k, const double *v,
                     int64_t H, int64_t D, int64_t h, int64_t r0, int64_t r1,
                     double *S, double *out)
{
    for (int64_t t = r0; t < r1; ++t) {
        const double *kt = k + (t * H + h) * D;
        const double *vt = v + (t * H + h) * D;
        const double *qt = q + (t * H + h) * D;
        double *ot = out + (t * H + h) * D;
        /* S_t = S_{t-1} + k_t v_t^T */
        for (int64_t i = 0; i < D; ++i) {
            const double ki = kt[i];
            double *Si = S + i * D;
            for (int64_t j = 0; j < D; ++j) Si[j] += ki * vt[j];
        }
        /* o_t = S_t^T q_t */
        for (int64_t j = 0; j < D; ++j) ot[j] = 0.0;
        for (int64_t i = 0; i < D; ++i) {
            const double qi = qt[i];
            const double *Si = S + i * D;
            for (int64_t j = 0; j < D; ++j) ot[j] += Si[j] * qi;
        }
    }
}

static int check_cu(const int32_t *cu, int32_t n, int64_t T)
{
    if (n < 0) return 1;
    if (n == 0) return 0;
    if (cu == NULL) return 1;
    for (int32_t s = 0; s < n; ++s) {
        if (cu[s] < 0 || cu[s + 1] < cu[s] || cu[s + 1] > T) return 1;
    }
    return 0;
}

/* Threads of one call: nthreads if positive, else the OpenMP default. */
static int threads_for(int nthreads)
{
#ifdef _OPENMP
    return nthreads > 0 ? nthreads : omp_get_max_threads();
#else
    (void)nthreads;
    return 1;
#endif
}

/*
 * Branches of one call: every branch b starts from init_states[parent[b]]
 * (copied, never modified) and runs over rows [branch_cu[b], branch_cu[b+1]).
 */
static int run_branches(const double *init_states, int32_t num_states,
                        const double *q, const double *k, const double *v,
                        int64_t H, int64_t D,
                        const int32_t *branch_cu, int32_t B, const int32_t *parent,
                        double *out, int nt)
{
    for (int32_t b = 0; b < B; ++b)
        if (parent[b] < 0 || parent[b] >= num_states) return 1;
    const int64_t items = (int64_t)B * H;
    int err = 0;
#pragma omp parallel num_threads(nt)
    {
        double *S = (double *)malloc(sizeof(double) * D * D);
        if (S == NULL) {
#pragma omp atomic write
            err = 2;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t it = 0; it < items; ++it) {
            if (S == NULL) continue;
            const int64_t b = it / H, h = it % H;
            const double *S0 = init_states + ((int64_t)parent[b] * H + h) * D * D;
            memcpy(S, S0, sizeof(double) * D * D);
            run_rows(q, k, v, H, D, h, branch_cu[b], branch_cu[b + 1], S, out);
        }
        free(S);
    }
    return err;
}

/*
 * One packed pass.  Views first (each from S = 0), writing each view's final
 * state to state_out[V][H][D][D]; then the branches, each from its parent
 * view's final state.  Returns 0 on success, 1 on bad metadata, 2 on
 * allocation failure.
 */
int oracle_pass(const double *q, const double *k, const double *v,
                int64_t T, int64_t H, int64_t D,
                const int32_t *view_cu, int32_t V,
                const int32_t *branch_cu, int32_t B, const int32_t *parent,
                double *out, double *state_out, int nthreads)
{
    if (H < 1 || D < 1 || T < 0) return 1;
    if (check_cu(view_cu, V, T) || check_cu(branch_cu, B, T)) return 1;
    if (B > 0 && (parent == NULL || V < 1)) return 1;
    const int nt = threads_for(nthreads);

    const int64_t items = (int64_t)V * H;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt)
    for (int64_t it = 0; it < items; ++it) {
        const int64_t vi = it / H, h = it % H;
        double *S = state_out + (vi * H + h) * D * D;
        memset(S, 0, sizeof(double) * D * D);
        run_rows(q, k, v, H, D, h, view_cu[vi], view_cu[vi + 1], S, out);
    }
    if (B == 0) return 0;
    return run_branches(state_out, V, q, k, v, H, D, branch_cu, B, parent, out, nt);
}

/*
 * Branches only, each from a caller-supplied state (the cached final state of
 * its view): states[P][H][D][D].
 */
int oracle_branches_from_state(const double *states, int32_t P,
                               const double *q, const double *k, const double *v,
                               int64_t T, int64_t H, int64_t D,
                               const int32_t *branch_cu, int32_t B, const int32_t *parent,
                               double *out, int nthreads)
{
    if (H < 1 || D < 1 || T < 0 || P < 0) return 1;
    if (check_cu(branch_cu, B, T)) return 1;
    if (B > 0 && (parent == NULL || states == NULL)) return 1;
    if (B == 0) return 0;
    return run_branches(states, P, q, k, v, H, D, branch_cu, B, parent, out, threads_for(nthreads));
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
