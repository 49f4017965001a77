/*
 * fp64 CPU oracle for the Mamba-2 SSD forward pass -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the package smoke check and the benchmark's CPU-baseline leg
 * may load this library.  It shares no code, header or constant with the CUDA
 * path.
 *
 * What it computes (the definition, not the chunked algorithm): the state-space
 * recurrence that "Jane Street ML Engineers Map Mamba-2 Recurrent State
 * Computation to Tensor Cores with cuTile" describes in its paragraph on the
 * fixed-size hidden state updated token by token (the RNN view of Mamba-2), with
 * the decay and input terms of the jump-formula paragraph:
 *
 *     h_t = exp(dt_t * A_h) * h_{t-1} + dt_t * x_t (outer) b_t      h in R^{P x N}
 *     y_t = h_t c_t + D_h * x_t
 *
 * for every batch b and head h, where head h reads group g = h / (H / G) of
 * Bm and Cm, h_{-1} is init_state (or zero) and final_state = h_{L-1}.
 * y_t sees the update of token t (inclusive state).
 *
 * Inputs are fp32 arrays (the exact values the GPU receives, bf16 workloads
 * already rounded); every product and sum is done in fp64.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Number of OpenMP threads a parallel region of this library would use. */
int ssd_oracle_threads(int requested) {
#ifdef _OPENMP
    if (requested > 0) return requested;
    return omp_get_max_threads();
#else
    (void)requested;
    return 1;
#endif
}

/*
 * Token-by-token recurrence for the (batch, head) pairs listed in `pairs`
 * (pairs[2k] = b, pairs[2k+1] = h); pairs == NULL means every pair.
 * Layouts (row-major, contiguous):
 *   x[B][L][H][P], dt[B][L][H], A[H], Bm/Cm[B][L][G][N], D[H],
 *   init_state[B][H][P][N] (may be NULL = zeros),
 *   y[B][L][H][P] (fp64, only the selected pairs are written),
 *   final_state[B][H][P][N] (fp64, may be NULL).
 * Returns the number of threads used, or -1 on a bad argument.
 */
int ssd_oracle_recurrence(int64_t B, int64_t L, int64_t H, int64_t P, int64_t G, int64_t N,
                          const float* x, const float* dt, const float* A,
                          const float* Bm, const float* Cm, const float* D,
                          const float* init_state, double* y, double* final_state,
                          const int64_t* pairs, int64_t npairs, int nthreads) {
    if (B < 0 || L < 0 || H <= 0 || P <= 0 || G <= 0 || N <= 0 || H % G != 0) return -1;
    if (!x || !dt || !A || !Bm || !Cm || !D || !y) return -1;
    const int64_t heads_per_group = H / G;
    const int64_t total = pairs ? npairs : B * H;
    int used = ssd_oracle_threads(nthreads);

#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(used)
#endif
    for (int64_t k = 0; k < total; ++k) {
        const int64_t b = pairs ? pairs[2 * k] : k / H;
        const int64_t h = pairs ? pairs[2 * k + 1] : k % H;
        const int64_t g = h / heads_per_group;
        double* state = (double*)malloc((size_t)(P * N) * sizeof(double));
        if (!state) continue;
        for (int64_t i = 0; i < P * N; ++i)
            state[i] = init_state ? (double)init_state[((b * H + h) * P) * N + i] : 0.0;
        const double a_h = (double)A[h];
        const double d_h = (double)D[h];
        for (int64_t t = 0; t < L; ++t) {
            const double dt_t = (double)dt[(b * L + t) * H + h];
            const double decay = exp(dt_t * a_h);
            const float* xt = x + ((b * L + t) * H + h) * P;
            const float* bt = Bm + ((b * L + t) * G + g) * N;
            const float* ct = Cm + ((b * L + t) * G + g) * N;
            double* yt = y + ((b * L + t) * H + h) * P;
            for (int64_t p = 0; p < P; ++p) {
                const double u = dt_t * (double)xt[p];
                double* row = state + p * N;
                double acc = 0.0;
                for (int64_t n = 0; n < N; ++n) {
                    row[n] = decay * row[n] + u * (double)bt[n];
                    acc += row[n] * (double)ct[n];
                }
                yt[p] = acc + d_h * (double)xt[p];
            }
        }
        if (final_state)
            memcpy(final_state + ((b * H + h) * P) * N, state, (size_t)(P * N) * sizeof(double));
        free(state);
    }
    return used;
}
