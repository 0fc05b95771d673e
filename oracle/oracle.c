/*
 * CPU oracle for the frequency-sweep solver: TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may
 * load this file's library.  The CUDA library never links, calls or shares
 * code with it.
 *
 * What it computes is the plain definition of the method's answer:
 * x = Z(omega)^-1 b in complex128, where
 *     Z(omega) = j*omega*L - j*Psi/omega + Zs(omega)*G
 * (malusrfworks.com, "Solving Dense Matrices Fast in the Browser", section
 * "Fewer frequency points: adaptive frequency sampling", the formula for Z).
 * The page's mixed-precision refinement is designed to reach the answer of a
 * double-precision direct solve on the CPU to about 1e-11 relative (same page,
 * section "Double-precision answers from a GPU without double precision",
 * the paragraph after the four steps); the page's CPU direct solve falls back
 * to LU with partial pivoting (section "Measure first"), which is what this
 * file does, unblocked and in the textbook order:
 *   for each column k: pick the row with the largest |Re|+|Im| at or below k
 *   (first such row on ties), swap it into place, divide the column below
 *   the pivot by the pivot (Smith's complex division), subtract the rank-1
 *   product from the trailing block.
 * Forward substitution with the unit-lower factor and back substitution with
 * the upper factor follow, one right-hand side at a time.
 *
 * Storage: complex matrices are row-major, interleaved (re, im) doubles,
 * element (i, j) at index 2*(i*n + j).  Right-hand sides are nrhs rows of n
 * interleaved complex values.  Build with -ffp-contract=off so that no
 * multiply-add is fused: every expression rounds as it is written.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void orc_set_threads(int t) {
#ifdef _OPENMP
    if (t > 0) omp_set_num_threads(t);
#else
    (void)t;
#endif
}

/* Z_ij = Zs.re*G_ij + j*(omega*L_ij - Psi_ij/omega + Zs.im*G_ij), evaluated
 * left to right exactly as written (Z's formula on the page). */
void orc_assemble(int64_t n, const double *L, const double *Psi, const double *G,
                  double omega, double zs_re, double zs_im, double *Z) {
    int64_t total = n * n;
#pragma omp parallel for schedule(static)
    for (int64_t e = 0; e < total; e++) {
        double re = zs_re * G[e];
        double im = omega * L[e] - Psi[e] / omega + zs_im * G[e];
        Z[2 * e] = re;
        Z[2 * e + 1] = im;
    }
}

/* (a_re + j a_im) / (c_re + j c_im) by Smith's algorithm (R. L. Smith,
 * "Algorithm 116: Complex division", CACM 1962), which avoids overflow in the
 * intermediate c_re^2 + c_im^2. */
static void cdiv(double a_re, double a_im, double c_re, double c_im,
                 double *q_re, double *q_im) {
    if (fabs(c_re) >= fabs(c_im)) {
        double r = c_im / c_re;
        double den = c_re + c_im * r;
        *q_re = (a_re + a_im * r) / den;
        *q_im = (a_im - a_re * r) / den;
    } else {
        double r = c_re / c_im;
        double den = c_re * r + c_im;
        *q_re = (a_re * r + a_im) / den;
        *q_im = (a_im * r - a_re) / den;
    }
}

/* In-place LU with partial pivoting.  On return A holds the multipliers
 * below the diagonal (unit-lower L) and U on and above it; piv[k] is the row
 * swapped with row k at step k.  Returns 0, or k+1 if column k has no
 * non-zero entry at or below the diagonal (exactly singular). */
int orc_lu_pp(int64_t n, double *A, int64_t *piv) {
    for (int64_t k = 0; k < n; k++) {
        int64_t p = k;
        double best = fabs(A[2 * (k * n + k)]) + fabs(A[2 * (k * n + k) + 1]);
        for (int64_t i = k + 1; i < n; i++) {
            double m = fabs(A[2 * (i * n + k)]) + fabs(A[2 * (i * n + k) + 1]);
            if (m > best) {
                best = m;
                p = i;
            }
        }
        piv[k] = p;
        if (best == 0.0) return (int)(k + 1);
        if (p != k) {
            for (int64_t j = 0; j < n; j++) {
                double t0 = A[2 * (k * n + j)], t1 = A[2 * (k * n + j) + 1];
                A[2 * (k * n + j)] = A[2 * (p * n + j)];
                A[2 * (k * n + j) + 1] = A[2 * (p * n + j) + 1];
                A[2 * (p * n + j)] = t0;
                A[2 * (p * n + j) + 1] = t1;
            }
        }
        const double p_re = A[2 * (k * n + k)], p_im = A[2 * (k * n + k) + 1];
        const double *urow = A + 2 * (k * n);
#pragma omp parallel for schedule(static)
        for (int64_t i = k + 1; i < n; i++) {
            double *row = A + 2 * (i * n);
            double l_re, l_im;
            cdiv(row[2 * k], row[2 * k + 1], p_re, p_im, &l_re, &l_im);
            row[2 * k] = l_re;
            row[2 * k + 1] = l_im;
            for (int64_t j = k + 1; j < n; j++) {
                double u_re = urow[2 * j], u_im = urow[2 * j + 1];
                row[2 * j] -= l_re * u_re - l_im * u_im;
                row[2 * j + 1] -= l_re * u_im + l_im * u_re;
            }
        }
    }
    return 0;
}

/* LU without any row interchange (the factorisation the method itself
 * performs in low precision), in complex128, for checking factor kernels.
 * Returns 0, or k+1 if the pivot at step k is exactly zero. */
int orc_lu_nopiv(int64_t n, double *A) {
    for (int64_t k = 0; k < n; k++) {
        const double p_re = A[2 * (k * n + k)], p_im = A[2 * (k * n + k) + 1];
        if (p_re == 0.0 && p_im == 0.0) return (int)(k + 1);
        const double *urow = A + 2 * (k * n);
#pragma omp parallel for schedule(static)
        for (int64_t i = k + 1; i < n; i++) {
            double *row = A + 2 * (i * n);
            double l_re, l_im;
            cdiv(row[2 * k], row[2 * k + 1], p_re, p_im, &l_re, &l_im);
            row[2 * k] = l_re;
            row[2 * k + 1] = l_im;
            for (int64_t j = k + 1; j < n; j++) {
                double u_re = urow[2 * j], u_im = urow[2 * j + 1];
                row[2 * j] -= l_re * u_re - l_im * u_im;
                row[2 * j + 1] -= l_re * u_im + l_im * u_re;
            }
        }
    }
    return 0;
}

/* Solve A X = B given orc_lu_pp's output; B (nrhs x n) is overwritten by X.
 * piv may be NULL for factors without interchanges. */
void orc_lu_solve(int64_t n, const double *LU, const int64_t *piv, int64_t nrhs, double *B) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < nrhs; r++) {
        double *b = B + 2 * (r * n);
        if (piv) {
            for (int64_t k = 0; k < n; k++) {
                int64_t p = piv[k];
                if (p != k) {
                    double t0 = b[2 * k], t1 = b[2 * k + 1];
                    b[2 * k] = b[2 * p];
                    b[2 * k + 1] = b[2 * p + 1];
                    b[2 * p] = t0;
                    b[2 * p + 1] = t1;
                }
            }
        }
        for (int64_t i = 0; i < n; i++) { /* unit lower */
            double s_re = b[2 * i], s_im = b[2 * i + 1];
            const double *row = LU + 2 * (i * n);
            for (int64_t j = 0; j < i; j++) {
                s_re -= row[2 * j] * b[2 * j] - row[2 * j + 1] * b[2 * j + 1];
                s_im -= row[2 * j] * b[2 * j + 1] + row[2 * j + 1] * b[2 * j];
            }
            b[2 * i] = s_re;
            b[2 * i + 1] = s_im;
        }
        for (int64_t i = n - 1; i >= 0; i--) { /* upper */
            double s_re = b[2 * i], s_im = b[2 * i + 1];
            const double *row = LU + 2 * (i * n);
            for (int64_t j = i + 1; j < n; j++) {
                s_re -= row[2 * j] * b[2 * j] - row[2 * j + 1] * b[2 * j + 1];
                s_im -= row[2 * j] * b[2 * j + 1] + row[2 * j + 1] * b[2 * j];
            }
            cdiv(s_re, s_im, row[2 * i], row[2 * i + 1], &b[2 * i], &b[2 * i + 1]);
        }
    }
}

/* Conjugate-transpose solve A^H Y = C with A's LU factors (for the
 * condition estimate).  C (n) is overwritten by Y. */
static void lu_solve_ct(int64_t n, const double *LU, const int64_t *piv, double *c) {
    /* A = P^T L U, so A^H = U^H L^H P: solve U^H w = c, L^H v = w, y = P^T v */
    for (int64_t i = 0; i < n; i++) {
        double s_re = c[2 * i], s_im = c[2 * i + 1];
        for (int64_t j = 0; j < i; j++) { /* (U^H)_ij = conj(U_ji) */
            double u_re = LU[2 * (j * n + i)], u_im = -LU[2 * (j * n + i) + 1];
            s_re -= u_re * c[2 * j] - u_im * c[2 * j + 1];
            s_im -= u_re * c[2 * j + 1] + u_im * c[2 * j];
        }
        cdiv(s_re, s_im, LU[2 * (i * n + i)], -LU[2 * (i * n + i) + 1], &c[2 * i], &c[2 * i + 1]);
    }
    for (int64_t i = n - 1; i >= 0; i--) {
        double s_re = c[2 * i], s_im = c[2 * i + 1];
        for (int64_t j = i + 1; j < n; j++) { /* (L^H)_ij = conj(L_ji) */
            double l_re = LU[2 * (j * n + i)], l_im = -LU[2 * (j * n + i) + 1];
            s_re -= l_re * c[2 * j] - l_im * c[2 * j + 1];
            s_im -= l_re * c[2 * j + 1] + l_im * c[2 * j];
        }
        c[2 * i] = s_re;
        c[2 * i + 1] = s_im;
    }
    for (int64_t k = n - 1; k >= 0; k--) {
        int64_t p = piv[k];
        if (p != k) {
            double t0 = c[2 * k], t1 = c[2 * k + 1];
            c[2 * k] = c[2 * p];
            c[2 * k + 1] = c[2 * p + 1];
            c[2 * p] = t0;
            c[2 * p + 1] = t1;
        }
    }
}

/* Hager's estimate of ||A^-1||_1 (W. W. Hager, "Condition estimates",
 * SIAM J. Sci. Stat. Comput. 1984; complex form as in N. J. Higham,
 * "Accuracy and Stability of Numerical Algorithms", ch. 15), using the
 * factors from orc_lu_pp.  Multiply by ||A||_1 for the condition number. */
double orc_inv_norm1_est(int64_t n, const double *LU, const int64_t *piv) {
    double *x = (double *)malloc(sizeof(double) * 2 * n);
    double *y = (double *)malloc(sizeof(double) * 2 * n);
    for (int64_t i = 0; i < n; i++) {
        x[2 * i] = 1.0 / (double)n;
        x[2 * i + 1] = 0.0;
    }
    double est = 0.0;
    int64_t last_j = -1;
    for (int it = 0; it < 5; it++) {
        memcpy(y, x, sizeof(double) * 2 * n);
        orc_lu_solve(n, LU, piv, 1, y);
        double nrm = 0.0;
        for (int64_t i = 0; i < n; i++) nrm += hypot(y[2 * i], y[2 * i + 1]);
        if (it > 0 && nrm <= est) break; /* no further increase */
        est = nrm;
        for (int64_t i = 0; i < n; i++) { /* xi = sign(y) */
            double a = hypot(y[2 * i], y[2 * i + 1]);
            if (a > 0) {
                y[2 * i] /= a;
                y[2 * i + 1] /= a;
            } else {
                y[2 * i] = 1.0;
                y[2 * i + 1] = 0.0;
            }
        }
        lu_solve_ct(n, LU, piv, y); /* z = A^-H xi */
        int64_t j = 0;
        double zmax = -1.0, ztx = 0.0;
        for (int64_t i = 0; i < n; i++) {
            double a = hypot(y[2 * i], y[2 * i + 1]);
            if (a > zmax) {
                zmax = a;
                j = i;
            }
            ztx += y[2 * i] * x[2 * i] + y[2 * i + 1] * x[2 * i + 1]; /* Re(z^H x) */
        }
        if (zmax <= ztx || j == last_j) break;
        last_j = j;
        for (int64_t i = 0; i < n; i++) x[2 * i] = x[2 * i + 1] = 0.0;
        x[2 * j] = 1.0;
    }
    free(x);
    free(y);
    return est;
}

/* ||A||_1 = max column sum of |a_ij|. */
double orc_norm1(int64_t n, const double *A) {
    double best = 0.0;
    for (int64_t j = 0; j < n; j++) {
        double s = 0.0;
        for (int64_t i = 0; i < n; i++) s += hypot(A[2 * (i * n + j)], A[2 * (i * n + j) + 1]);
        if (s > best) best = s;
    }
    return best;
}

/* R = B - Z X (nrhs right-hand sides), plain double-precision sums taken in
 * column order. */
void orc_residual(int64_t n, const double *Z, int64_t nrhs, const double *X, const double *B,
                  double *R) {
    for (int64_t r = 0; r < nrhs; r++) {
        const double *x = X + 2 * (r * n);
#pragma omp parallel for schedule(static)
        for (int64_t i = 0; i < n; i++) {
            const double *row = Z + 2 * (i * n);
            double s_re = 0.0, s_im = 0.0;
            for (int64_t j = 0; j < n; j++) {
                s_re += row[2 * j] * x[2 * j] - row[2 * j + 1] * x[2 * j + 1];
                s_im += row[2 * j] * x[2 * j + 1] + row[2 * j + 1] * x[2 * j];
            }
            R[2 * (r * n + i)] = B[2 * (r * n + i)] - s_re;
            R[2 * (r * n + i) + 1] = B[2 * (r * n + i) + 1] - s_im;
        }
    }
}
