/*
 * Plain fp64 CPU attention: the oracle the CUDA path is checked against.
 *
 * TEST INFRASTRUCTURE ONLY. Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library. The product path never
 * calls it, links it or shares code with it.
 *
 * What it computes (FlashAttention-3 principles, section 1.2 "standard
 * attention" code and section 2.2 softmax definition): for one (sequence,
 * head) pair with Lq query rows and Lk key rows,
 *
 *     s_ij  = scale * sum_d q_id k_jd                (j visible from i)
 *     m_i   = max_j s_ij
 *     l_i   = sum_j exp(s_ij - m_i)
 *     O_id  = sum_j exp(s_ij - m_i) v_jd / l_i
 *     LSE_i = m_i + ln l_i
 *
 * Visibility: every key j < Lk, or with the causal mask (section 4.2 causal
 * rows; `causal=True` in the section 5.2 varlen call) only j <= i + Lk - Lq,
 * i.e. the mask is aligned to the bottom-right corner so that the last query
 * row sees every key. A row with no visible key gets O = 0 and LSE = -inf.
 *
 * Everything is fp64, straight loops, no blocking or reordering: the
 * materialised S row is built, reduced, exponentiated and contracted with V.
 * Rows are independent, so OpenMP splits them across host threads.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Number of host threads OpenMP will use (1 without OpenMP). */
int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/*
 * Attention for a set of query rows of ONE (sequence, head) pair.
 *
 *   q     [nq, D]   the query rows to evaluate (fp64, row-major)
 *   qpos  [nq]      position i of each of those rows inside the sequence
 *   k, v  [Lk, D]   every key / value row of the sequence for this head
 *   Lq            query length of the sequence (sets the causal offset)
 *   o     [nq, D]   output rows
 *   lse   [nq]      natural-log log-sum-exp of the scaled scores
 *
 * Returns 0, or -1 on an allocation failure or a bad argument.
 */
int oracle_attention_rows(const double *q, const int64_t *qpos, int64_t nq,
                          const double *k, const double *v, int64_t Lk,
                          int64_t Lq, int D, double scale, int causal,
                          double *o, double *lse) {
    if (nq < 0 || Lk < 0 || Lq < 0 || D <= 0) return -1;
    int status = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(Lk > 0 ? Lk : 1));
        if (!s) {
#pragma omp atomic write
            status = -1;
        }
#pragma omp for schedule(dynamic, 4)
        for (int64_t r = 0; r < nq; ++r) {
            if (!s) continue;
            const double *qr = q + (size_t)r * D;
            double *orow = o + (size_t)r * D;
            int64_t i = qpos[r];
            int64_t visible = Lk;
            if (causal) {
                int64_t lim = i + Lk - Lq + 1; /* keys j < lim are visible */
                if (lim < visible) visible = lim;
            }
            if (visible <= 0) {
                for (int d = 0; d < D; ++d) orow[d] = 0.0;
                lse[r] = -INFINITY;
                continue;
            }
            /* scores of the row */
            double m = -INFINITY;
            for (int64_t j = 0; j < visible; ++j) {
                const double *kj = k + (size_t)j * D;
                double acc = 0.0;
                for (int d = 0; d < D; ++d) acc += qr[d] * kj[d];
                s[j] = scale * acc;
                if (s[j] > m) m = s[j];
            }
            /* softmax numerator and normaliser */
            double l = 0.0;
            for (int64_t j = 0; j < visible; ++j) {
                s[j] = exp(s[j] - m);
                l += s[j];
            }
            for (int d = 0; d < D; ++d) orow[d] = 0.0;
            for (int64_t j = 0; j < visible; ++j) {
                const double *vj = v + (size_t)j * D;
                double p = s[j];
                for (int d = 0; d < D; ++d) orow[d] += p * vj[d];
            }
            for (int d = 0; d < D; ++d) orow[d] /= l;
            lse[r] = m + log(l);
        }
        free(s);
    }
    return status;
}

/*
 * Count of score entries (query row, visible key) for the given rows: the
 * number of exponentials the definition takes. Used to scale a timed sample
 * of rows to the whole problem.
 */
int64_t oracle_visible_pairs(const int64_t *qpos, int64_t nq, int64_t Lk,
                             int64_t Lq, int causal) {
    int64_t total = 0;
    for (int64_t r = 0; r < nq; ++r) {
        int64_t visible = Lk;
        if (causal) {
            int64_t lim = qpos[r] + Lk - Lq + 1;
            if (lim < visible) visible = lim;
        }
        if (visible > 0) total += visible;
    }
    return total;
}
