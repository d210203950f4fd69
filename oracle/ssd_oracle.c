/*
 * ssd_oracle.c -- fp64 CPU oracle for the selective state-space recurrence.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the correctness reference the CUDA
 * library is checked against.  Only the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark load it.  The product path never links,
 * loads or calls it, and it shares no code, header or constant with the CUDA
 * sources.
 *
 * What it computes (the definition, written out, not the chunked algorithm):
 *
 *   For every batch b, head h and head channel p, starting from
 *   h_{-1}[n] = init[b,h,p,n] (zero when no initial state is given):
 *
 *       a_t        = exp(dt[b,t,h] * A[h])
 *       h_t[n]     = a_t * h_{t-1}[n] + dt[b,t,h] * B[b,t,g,n] * x[b,t,h,p]
 *       y[b,t,h,p] = sum_n C[b,t,g,n] * h_t[n] + D[h] * x[b,t,h,p]
 *       final[b,h,p,n] = h_{L-1}[n]
 *
 *   with g = floor(h * G / H): heads are split into G contiguous groups that
 *   share B and C.
 *
 * Sources:
 *   - "Why SSM and linear-RNN FLOPs do not convert into GPU FLOPs: the
 *     sequential scan bypasses the tensor cores", paragraph 1: the selective
 *     SSM step h_t = a_t h_{t-1} + b_t x_t with an input-dependent decay, one
 *     scalar decay shared by all dimensions of a head (the Mamba-2 choice the
 *     HGRN2 quote there contrasts with per-dimension decay).
 *   - "Mamba-2 in NVIDIA cuTile: Faster Forward Kernels", section "Why Mamba-2
 *     is a useful kernel example": the forward pass whose result the chunked
 *     kernels reproduce.
 *   The pages never print the recurrence with indices.  Readings taken here:
 *   the decay of step t uses the same dt_t as its input term; y_t reads the
 *   state after the update of step t; the skip term D*x_t is added to the
 *   output and never enters the state; the state is stored with the head
 *   channel p outermost and the state index n innermost.
 *
 * Parity pins (tests/test_oracle_pins.py) tie this function to the quadratic
 * dual form, a closed form for a constant-decay scalar system, the impulse
 * response, chunked-versus-unchunked agreement, split/resume, linearity,
 * dt = 0, the A -> 0 limit (causal linear attention) and group replication.
 *
 * Build: gcc -O2 -fopenmp -shared -fPIC (no fast-math: IEEE fp64 throughout).
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* Returns the number of OpenMP threads a parallel region will use. */
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
 * Sequential recurrence, fp64.
 *
 * Layouts (all contiguous, row-major):
 *   x      [batch, L, H, P]      dt [batch, L, H]      A [H]
 *   B, C   [batch, L, G, N]      D  [H]     (may be NULL: no skip term)
 *   init   [batch, H, P, N]      (may be NULL: zero initial state)
 *   y      [batch, L, H, P]      (written)
 *   final  [batch, H, P, N]      (may be NULL; written)
 *   snap   [batch, nsnap, H, P, N] (may be NULL; written) where
 *          nsnap = ceil(L / snap_every): snap[b, k] is the state entering
 *          step k*snap_every, i.e. the state after step k*snap_every - 1
 *          (snap[b, 0] is the initial state).
 * Returns 0 on success, -1 on an invalid argument.
 */
int oracle_ssd_recurrence(int64_t batch, int64_t L, int64_t H, int64_t P,
                          int64_t N, int64_t G,
                          const double *x, const double *dt, const double *A,
                          const double *B, const double *C, const double *D,
                          const double *init, double *y, double *final_state,
                          double *snap, int64_t snap_every) {
    if (batch < 0 || L < 0 || H <= 0 || P <= 0 || N <= 0 || G <= 0) return -1;
    if (H % G != 0) return -1;
    if (!x || !dt || !A || !B || !C || !y) return -1;
    if (snap && snap_every <= 0) return -1;
    const int64_t nsnap = snap ? (L + snap_every - 1) / snap_every : 0;
    const int64_t nwork = batch * H * P;

#pragma omp parallel
    {
        double *h = (double *)malloc(sizeof(double) * (size_t)N);
#pragma omp for schedule(dynamic, 4)
        for (int64_t w = 0; w < nwork; ++w) {
            const int64_t b = w / (H * P);
            const int64_t hd = (w / P) % H;
            const int64_t p = w % P;
            const int64_t g = hd * G / H;
            const double a_h = A[hd];
            const double d_h = D ? D[hd] : 0.0;

            for (int64_t n = 0; n < N; ++n)
                h[n] = init ? init[((b * H + hd) * P + p) * N + n] : 0.0;

            for (int64_t t = 0; t < L; ++t) {
                if (snap && t % snap_every == 0) {
                    double *s = snap + (((b * nsnap + t / snap_every) * H + hd) * P + p) * N;
                    for (int64_t n = 0; n < N; ++n) s[n] = h[n];
                }
                const double dtv = dt[(b * L + t) * H + hd];
                const double xv = x[((b * L + t) * H + hd) * P + p];
                const double a = exp(dtv * a_h);
                const double u = dtv * xv;
                const double *Bt = B + ((b * L + t) * G + g) * N;
                const double *Ct = C + ((b * L + t) * G + g) * N;
                double acc = 0.0;
                for (int64_t n = 0; n < N; ++n) {
                    h[n] = a * h[n] + u * Bt[n];
                    acc += Ct[n] * h[n];
                }
                y[((b * L + t) * H + hd) * P + p] = acc + d_h * xv;
            }
            if (final_state) {
                double *f = final_state + ((b * H + hd) * P + p) * N;
                for (int64_t n = 0; n < N; ++n) f[n] = h[n];
            }
        }
        free(h);
    }
    return 0;
}
