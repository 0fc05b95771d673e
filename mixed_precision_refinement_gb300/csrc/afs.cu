// Adaptive frequency sampling: a reduced-order model of the frequency sweep
// (malusrfworks.com, "Solving Dense Matrices Fast in the Browser", section
// "Fewer frequency points: adaptive frequency sampling").
//
// The library's mixed-precision solver runs at a few candidates; the real and
// imaginary parts of its solutions, made orthonormal, are the columns of a
// real basis V (n x q).  With L V, Psi V, G V the
// reduced matrix Z_r(omega) = j*omega*V^T L V - j*V^T Psi V/omega + Zs*V^T G V
// is q x q; its Galerkin solution y (Z_r y = V^T b) gives x ~ V y at every
// candidate, and the relative residual ||Z V y - b|| / ||b|| is estimated from
// small quantities only: with W = [L V | Psi V | G V] and
// c = [j*omega*y; -j*y/omega; Zs*y], Z V y = W c, so
// ||Z V y - b||^2 = c^H (W^T W) c - 2 Re(c^H W^T b) + ||b||^2.
// The next exact solve is at the largest estimate; the loop stops when every
// estimate is below the tolerance (the page uses 1e-4).
//
// Kernels (all float64; the FP64 pipe, not HBM, bounds each of them on this
// GPU except the projection's matrix reads at small basis growth):
//   k_afs_orth    two passes of classical Gram-Schmidt for each new real
//                 vector against the basis, drop test, normalisation (one
//                 cluster of 8 CTAs, rows split between them; the vectors are
//                 appended in order);
//   k_afs_project L, Psi, G times the new basis columns, one pass over the
//                 three matrices per group of 8 columns;
//   k_afs_gram    the new rows and columns of V^T L V, V^T Psi V, V^T G V and
//                 of W^T W, and W^T b, V^T b, ||b||^2 (one warp per entry);
//   k_afs_eval    one CTA per candidate: Z_r, complex LU with partial
//                 pivoting (largest |re|+|im|, lowest row on ties) on the
//                 system with V^T b appended, back substitution, the residual
//                 estimate (largest over the right-hand sides);
//   k_afs_expand  x = V y for every candidate and right-hand side.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <vector>

#include <cooperative_groups.h>

#include "common.cuh"
#include "zsolve.h"

namespace cg = cooperative_groups;

namespace {

constexpr int kMaxBasis = ZSOLVE_AFS_MAX_BASIS;
constexpr int kOrthCluster = 8;   // CTAs of the orthogonalisation cluster (portable size)
constexpr int kOrthThreads = 512;
constexpr int kProjThreads = 256;
constexpr int kProjCols = 8;
constexpr int kGramThreads = 256;
constexpr int kEvalThreads = 256;
constexpr int kExpandThreads = 256;
constexpr int kExpandGroup = 8;
constexpr int kMaxSmem = 227 * 1024;

// Sums on the FMA path: a + b = fma(a, 1, b) with 1 passed at run time (the
// FP64 pipe of this GPU retires DFMA at full rate, DADD more slowly).
__device__ __forceinline__ double add1(double a, double b, double one) { return __fma_rn(a, one, b); }

__device__ __forceinline__ double warp_sum(double v, double one) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v = add1(v, __shfl_xor_sync(0xffffffffu, v, o), one);
    return v;
}

// Sum over the block, in a fixed order; red holds 33 doubles.
__device__ double block_sum(double v, double *red, double one) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    v = warp_sum(v, one);
    __syncthreads();  // red may still be read from a previous call
    if (lane == 0) red[warp] = v;
    __syncthreads();
    if (warp == 0) {
        double s = lane < nw ? red[lane] : 0.0;
        s = warp_sum(s, one);
        if (lane == 0) red[32] = s;
    }
    __syncthreads();
    return red[32];
}

__device__ __forceinline__ double2 zmul(double2 a, double2 b) {
    return make_double2(fma(a.x, b.x, -a.y * b.y), fma(a.x, b.y, a.y * b.x));
}

// a - b*c
__device__ __forceinline__ double2 zfms(double2 a, double2 b, double2 c) {
    return make_double2(fma(-b.x, c.x, fma(b.y, c.y, a.x)), fma(-b.x, c.y, fma(-b.y, c.x, a.y)));
}

// 1/a by Smith's method (R. L. Smith, "Algorithm 116: Complex division",
// CACM 5(8), 1962): the ratio of the smaller to the larger part keeps the
// intermediate quantities in range.
__device__ __forceinline__ double2 zrecip(double2 a) {
    if (fabs(a.x) >= fabs(a.y)) {
        const double t = a.y / a.x, r = 1.0 / (a.x + a.y * t);
        return make_double2(r, -(t * r));
    }
    const double t = a.x / a.y, r = 1.0 / (a.y + a.x * t);
    return make_double2(t * r, -r);
}

// ------------------------------------------------------------------ basis

// Appends the real and imaginary parts of nsrc complex vectors (xs, n apart)
// to V, from column q0 on, in the order (vector, real part, imaginary part).
// Each is orthogonalised against the columns before it by two passes of
// h = V^T v, v -= V h; it is kept (normalised) if its norm after the passes
// exceeds drop times its norm before, else its column is reused.
// q_out[0] = columns after the call; q_out[1] = 1 if a vector was left out
// because V was full.
//
// One thread-block cluster of kOrthCluster CTAs; CTA r owns rows
// [r*slice, (r+1)*slice) of every column.  The sums over rows (the two norms
// and h) are formed per CTA, exchanged through distributed shared memory and
// added in rank order by every CTA, so all CTAs hold bit-identical sums and
// take the same keep/drop decision (the cluster barriers are reached by all).
// Four buffers, one per kind of sum, rotate: a buffer is rewritten only after
// the barrier that follows every CTA's reads of it.
__global__ void __cluster_dims__(kOrthCluster, 1, 1) __launch_bounds__(kOrthThreads)
k_afs_orth(double *__restrict__ V, int64_t n, int q0, int qmax, const double2 *__restrict__ xs, int nsrc,
           double drop, int *__restrict__ q_out, double one) {
    cg::cluster_group cl = cg::this_cluster();
    __shared__ double part[4][kMaxBasis];  // this CTA's sums: norm before, h pass 1, h pass 2, norm after
    __shared__ double h[kMaxBasis];        // the cluster's sums
    __shared__ double red[33];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t slice = (n + kOrthCluster - 1) / kOrthCluster;
    const int64_t r0 = min(n, (int64_t)cl.block_rank() * slice), r1 = min(n, r0 + slice);
    // h[0..count) = sum over the cluster's CTAs of part[buf][0..count), in rank order
    auto cluster_sum = [&](int buf, int count) {
        cl.sync();
        for (int j = tid; j < count; j += kOrthThreads) {
            double acc = 0.0;
            for (int rk = 0; rk < kOrthCluster; rk++) acc = add1(acc, cl.map_shared_rank(&part[buf][0], rk)[j], one);
            h[j] = acc;
        }
        __syncthreads();
    };
    int q = q0, full = 0;
    for (int s = 0; s < 2 * nsrc; s++) {
        if (q >= qmax) {
            full = 1;
            break;
        }
        const double2 *src = xs + (int64_t)(s >> 1) * n;
        const bool imag = (s & 1) != 0;
        double *col = V + (int64_t)q * n;
        double acc = 0.0;
        for (int64_t t = r0 + tid; t < r1; t += kOrthThreads) {
            const double2 z = src[t];
            const double v = imag ? z.y : z.x;
            col[t] = v;
            acc = fma(v, v, acc);
        }
        acc = block_sum(acc, red, one);
        if (tid == 0) part[0][0] = acc;
        cluster_sum(0, 1);
        const double n0 = sqrt(h[0]);
        for (int pass = 0; pass < 2; pass++) {
            for (int j = warp; j < q; j += kOrthThreads / 32) {
                const double *vj = V + (int64_t)j * n;
                double a = 0.0;
                for (int64_t t = r0 + lane; t < r1; t += 32) a = fma(vj[t], col[t], a);
                a = warp_sum(a, one);
                if (lane == 0) part[1 + pass][j] = a;
            }
            cluster_sum(1 + pass, q);
            for (int64_t t = r0 + tid; t < r1; t += kOrthThreads) {
                double c = col[t];
                const double *vt = V + t;
                for (int j = 0; j < q; j++, vt += n) c = fma(-h[j], *vt, c);
                col[t] = c;
            }
            __syncthreads();
        }
        acc = 0.0;
        for (int64_t t = r0 + tid; t < r1; t += kOrthThreads) acc = fma(col[t], col[t], acc);
        acc = block_sum(acc, red, one);
        if (tid == 0) part[3][0] = acc;
        cluster_sum(3, 1);
        const double n1 = sqrt(h[0]);
        if (n0 > 0.0 && isfinite(n0) && n1 > drop * n0) {
            for (int64_t t = r0 + tid; t < r1; t += kOrthThreads) col[t] = col[t] / n1;
            q++;
        }
        __syncthreads();
    }
    cl.sync();  // no CTA leaves while another may still read its buffers
    if (tid == 0 && cl.block_rank() == 0) {
        q_out[0] = q;
        q_out[1] = full;
    }
}

// W block k (k = 0: L, 1: Psi, 2: G), column j = that matrix times V column j,
// for the nc columns from c0 on.  One warp per row of the three matrices per
// group of kProjCols columns (blockIdx.y); a warp whose 32 entries of G are all
// zero skips the G products (exact zeros in every sum).
__global__ void __launch_bounds__(kProjThreads)
k_afs_project(const double *__restrict__ L, const double *__restrict__ Psi, const double *__restrict__ G, int64_t n,
              const double *__restrict__ V, int c0, int nc, double *__restrict__ W, int64_t wblk, double one) {
    const int lane = threadIdx.x & 31;
    const int64_t gw = ((int64_t)blockIdx.x * kProjThreads + threadIdx.x) >> 5;
    const int64_t nw = ((int64_t)gridDim.x * kProjThreads) >> 5;
    const int cb = c0 + (int)blockIdx.y * kProjCols;
    const int kc = min(kProjCols, c0 + nc - cb);
    const double *vb = V + (int64_t)cb * n;
    constexpr int U = 4;  // row chunks of 32 loaded ahead of their products
    for (int64_t i = gw; i < n; i += nw) {
        const double *Li = L + i * n, *Pi = Psi + i * n, *Gi = G + i * n;
        double aL[kProjCols], aP[kProjCols], aG[kProjCols];
#pragma unroll
        for (int c = 0; c < kProjCols; c++) aL[c] = aP[c] = aG[c] = 0.0;
        for (int64_t tw = 0; tw < n; tw += 32 * U) {
            double l[U], p[U], g[U];
            int64_t tc[U];
            bool valid[U];
            bool gnz = false;
#pragma unroll
            for (int u = 0; u < U; u++) {
                const int64_t t = tw + 32 * u + lane;
                valid[u] = t < n;
                tc[u] = valid[u] ? t : n - 1;  // in-bounds address for the tail lanes
                l[u] = Li[tc[u]];
                p[u] = Pi[tc[u]];
                g[u] = Gi[tc[u]];
                if (!valid[u]) l[u] = p[u] = g[u] = 0.0;
                gnz = gnz || !zs::is_zero(zs::bits_of(g[u]));
            }
            const bool gz = __all_sync(0xffffffffu, !gnz);
#pragma unroll
            for (int c = 0; c < kProjCols; c++) {
                if (c < kc) {
                    const double *vc = vb + (int64_t)c * n;
#pragma unroll
                    for (int u = 0; u < U; u++) {
                        const double v = valid[u] ? vc[tc[u]] : 0.0;
                        aL[c] = fma(l[u], v, aL[c]);
                        aP[c] = fma(p[u], v, aP[c]);
                        if (!gz) aG[c] = fma(g[u], v, aG[c]);
                    }
                }
            }
        }
#pragma unroll
        for (int c = 0; c < kProjCols; c++) {
            if (c < kc) {
                const double sl = warp_sum(aL[c], one), sp = warp_sum(aP[c], one), sg = warp_sum(aG[c], one);
                if (lane == 0) {
                    double *w = W + (int64_t)(cb + c) * n + i;
                    w[0] = sl;
                    w[wblk] = sp;
                    w[2 * wblk] = sg;
                }
            }
        }
    }
}

// Dot product of two strided float64 vectors by one warp.
__device__ __forceinline__ double wdot(const double *a, int64_t sa, const double *b, int64_t sb, int64_t n,
                                       int lane, double one) {
    double s = 0.0;
    for (int64_t t = lane; t < n; t += 32) s = fma(a[t * sa], b[t * sb], s);
    return warp_sum(s, one);
}

// New entries after the basis grew from P to Q columns (one warp per entry):
//   red[k][i][j] = V_i . W_kj           (k = L, Psi, G; i or j >= P)
//   M[c][d] = M[d][c] = W_c . W_d       (c, d over the 3 blocks; either column new)
//   wb[c][r] = W_c . b_r,  br[j][r] = V_j . b_r   (new columns)
//   bb[r] = ||b_r||^2                   (when P == 0)
// Column c = (k, i) of W sits at W + (k * qmax + i) * n; M has 3 qmax columns.
__global__ void __launch_bounds__(kGramThreads)
k_afs_gram(const double *__restrict__ V, const double *__restrict__ W, const double2 *__restrict__ b, int64_t n,
           int qmax, int P, int Q, int nrhs, double *__restrict__ red, double *__restrict__ M,
           double2 *__restrict__ wb, double2 *__restrict__ br, double *__restrict__ bb, double one) {
    int t = (int)(((int64_t)blockIdx.x * kGramThreads + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    const int tR = 3 * Q * Q, tM = 9 * Q * Q, tWB = 3 * Q * nrhs, tBR = Q * nrhs, tBB = P == 0 ? nrhs : 0;
    const int64_t q2 = (int64_t)qmax * qmax, m3 = 3 * (int64_t)qmax;
    const double *bre = (const double *)b, *bim = bre + 1;
    if (t < tR) {
        const int k = t / (Q * Q), rem = t - k * Q * Q, i = rem / Q, j = rem - (rem / Q) * Q;
        if (i < P && j < P) return;
        const double s = wdot(V + (int64_t)i * n, 1, W + ((int64_t)k * qmax + j) * n, 1, n, lane, one);
        if (lane == 0) red[k * q2 + (int64_t)i * qmax + j] = s;
        return;
    }
    t -= tR;
    if (t < tM) {
        const int c = t / (3 * Q), d = t - c * 3 * Q;
        if (c > d) return;
        const int kc = c / Q, ic = c - kc * Q, kd = d / Q, jd = d - kd * Q;
        if (ic < P && jd < P) return;
        const int64_t ca = (int64_t)kc * qmax + ic, da = (int64_t)kd * qmax + jd;
        const double s = wdot(W + ca * n, 1, W + da * n, 1, n, lane, one);
        if (lane == 0) {
            M[ca * m3 + da] = s;
            M[da * m3 + ca] = s;
        }
        return;
    }
    t -= tM;
    if (t < tWB) {
        const int c = t / nrhs, r = t - c * nrhs, k = c / Q, i = c - k * Q;
        if (i < P) return;
        const int64_t ca = (int64_t)k * qmax + i;
        const double *w = W + ca * n;
        const double sr = wdot(w, 1, bre + 2 * (int64_t)r * n, 2, n, lane, one);
        const double si = wdot(w, 1, bim + 2 * (int64_t)r * n, 2, n, lane, one);
        if (lane == 0) wb[ca * nrhs + r] = make_double2(sr, si);
        return;
    }
    t -= tWB;
    if (t < tBR) {
        const int j = t / nrhs, r = t - j * nrhs;
        if (j < P) return;
        const double *v = V + (int64_t)j * n;
        const double sr = wdot(v, 1, bre + 2 * (int64_t)r * n, 2, n, lane, one);
        const double si = wdot(v, 1, bim + 2 * (int64_t)r * n, 2, n, lane, one);
        if (lane == 0) br[(int64_t)j * nrhs + r] = make_double2(sr, si);
        return;
    }
    t -= tBR;
    if (t < tBB) {
        const int r = t;
        const double *re = bre + 2 * (int64_t)r * n, *im = bim + 2 * (int64_t)r * n;
        const double s = add1(wdot(re, 2, re, 2, n, lane, one), wdot(im, 2, im, 2, n, lane, one), one);
        if (lane == 0) bb[r] = s;
    }
}

// ------------------------------------------------------------------ evaluation

__host__ __device__ inline size_t eval_smem_bytes(int q, int nrhs) {
    return ((size_t)q * (q + nrhs) + 4 * (size_t)q) * sizeof(double2);
}

// One CTA per candidate: Z_r = Zs.re*Gr + j*((omega*Lr - Pr/omega) + Zs.im*Gr)
// with V^T b appended, eliminated with partial pivoting, solved, and the
// residual estimate for each right-hand side.  y goes to Y[cand][r][0..q);
// res[cand] = the largest relative estimate (+inf for an exactly singular or
// non-finite system, whose y is left zero).
__global__ void __launch_bounds__(kEvalThreads)
k_afs_eval(const ZsSlotParam *__restrict__ par, const double *__restrict__ red, const double *__restrict__ M,
           const double2 *__restrict__ wb, const double2 *__restrict__ br, const double *__restrict__ bb, int q,
           int qmax, int nrhs, double2 *__restrict__ Y, double *__restrict__ res, double one) {
    extern __shared__ double2 sm[];
    __shared__ double rsum[33];
    __shared__ int piv_s, bad_s;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int lda = q + nrhs;
    double2 *A = sm, *cv = sm + (size_t)q * lda, *rdiag = cv + 3 * q;  // rdiag[k] = 1 / pivot k
    const int64_t cand = blockIdx.x;
    const ZsSlotParam p = par[cand];
    const double w = p.omega;
    const int64_t q2 = (int64_t)qmax * qmax;
    for (int f = tid; f < q * q; f += kEvalThreads) {
        const int i = f / q, j = f - i * q;
        const int64_t e = (int64_t)i * qmax + j;
        const double l = red[e], ps = red[q2 + e], g = red[2 * q2 + e];
        // each operation rounded once, in the order the formula is written
        A[i * lda + j] = make_double2(__dmul_rn(p.zs_re, g),
                                      __dadd_rn(__dsub_rn(__dmul_rn(w, l), __ddiv_rn(ps, w)), __dmul_rn(p.zs_im, g)));
    }
    for (int f = tid; f < q * nrhs; f += kEvalThreads) {
        const int i = f / nrhs, r = f - i * nrhs;
        A[i * lda + q + r] = br[(int64_t)i * nrhs + r];
    }
    if (tid == 0) bad_s = 0;
    __syncthreads();
    for (int k = 0; k < q; k++) {
        if (warp == 0) {
            // |re| + |im| is >= 0 (or NaN, whose pattern is above every
            // number's), so its bit pattern orders like the value: the
            // comparisons are integer ones, off the FP64 pipe
            long long best = -1;
            int bi = q;
            for (int i = k + lane; i < q; i += 32) {
                const double2 a = A[i * lda + k];
                const long long v = __double_as_longlong(fabs(a.x) + fabs(a.y));
                if (v > best) {
                    best = v;
                    bi = i;
                }
            }
#pragma unroll
            for (int o = 16; o; o >>= 1) {
                const long long ob = __shfl_xor_sync(0xffffffffu, best, o);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
                if (ob > best || (ob == best && oi < bi)) {
                    best = ob;
                    bi = oi;
                }
            }
            if (lane == 0) {
                piv_s = bi;
                // zero pivot column, infinity or NaN: 0 < pattern < that of +inf
                if (best <= 0 || best >= 0x7FF0000000000000LL || bi >= q) bad_s = 1;
                else rdiag[k] = zrecip(A[bi * lda + k]);  // once per step, for the multipliers and the solve
            }
        }
        __syncthreads();
        if (bad_s) break;
        const int pr = piv_s;
        if (pr != k)
            for (int j = k + tid; j < lda; j += kEvalThreads) {
                const double2 a = A[k * lda + j];
                A[k * lda + j] = A[pr * lda + j];
                A[pr * lda + j] = a;
            }
        __syncthreads();
        const double2 inv = rdiag[k];
        for (int i = k + 1 + tid; i < q; i += kEvalThreads) A[i * lda + k] = zmul(A[i * lda + k], inv);
        __syncthreads();
        {
            const int rows = q - k - 1, cols = lda - k - 1;
            for (int f = tid; f < rows * cols; f += kEvalThreads) {
                const int i = k + 1 + f / cols, j = k + 1 + f % cols;
                A[i * lda + j] = zfms(A[i * lda + j], A[i * lda + k], A[k * lda + j]);
            }
        }
        __syncthreads();
    }
    const bool bad = bad_s != 0;
    if (!bad) {
        for (int i = q - 1; i >= 0; i--) {
            if (tid < nrhs) A[i * lda + q + tid] = zmul(A[i * lda + q + tid], rdiag[i]);
            __syncthreads();
            for (int e = tid; e < i * nrhs; e += kEvalThreads) {
                const int t = e / nrhs, r = e - t * nrhs;
                A[t * lda + q + r] = zfms(A[t * lda + q + r], A[t * lda + i], A[i * lda + q + r]);
            }
            __syncthreads();
        }
    }
    double worst = 0.0;
    const int64_t m3 = 3 * (int64_t)qmax;
    for (int r = 0; r < nrhs; r++) {
        double2 *yo = Y + (cand * nrhs + r) * qmax;
        for (int i = tid; i < q; i += kEvalThreads) {
            const double2 y = bad ? make_double2(0.0, 0.0) : A[i * lda + q + r];
            yo[i] = y;
            cv[i] = make_double2(-(w * y.y), w * y.x);                                  // j*omega*y
            cv[q + i] = make_double2(y.y / w, -(y.x / w));                              // -j*y/omega
            cv[2 * q + i] = make_double2(fma(p.zs_re, y.x, -(p.zs_im * y.y)), fma(p.zs_re, y.y, p.zs_im * y.x));  // Zs*y
        }
        __syncthreads();
        // sum over rows a of W^T W:  c_a^* (M c)_a (real part) - 2 Re(c_a^* wb_a),
        // a thread per row; M is symmetric (both halves hold the same dot
        // product), so row a is read as column a: consecutive threads read
        // consecutive addresses
        double part = 0.0;
        for (int a = tid; a < 3 * q; a += kEvalThreads) {
            const int ka = a / q, ia = a - ka * q;
            const double *Mcol = M + (int64_t)ka * qmax + ia;
            double ur = 0.0, ui = 0.0;
            for (int kb = 0; kb < 3; kb++) {
                const double *mc = Mcol + (int64_t)kb * qmax * m3;
                const double2 *cb = cv + kb * q;
                for (int ib = 0; ib < q; ib++, mc += m3) {
                    const double mv = *mc;
                    ur = fma(mv, cb[ib].x, ur);
                    ui = fma(mv, cb[ib].y, ui);
                }
            }
            const double2 ca = cv[a], wv = wb[((int64_t)ka * qmax + ia) * nrhs + r];
            part = add1(part, fma(ca.x, ur, ca.y * ui) - 2.0 * fma(ca.x, wv.x, ca.y * wv.y), one);
        }
        const double s = add1(block_sum(part, rsum, one), bb[r], one);
        const double b2 = bb[r];
        double rel = b2 > 0.0 ? sqrt(fmax(s, 0.0) / b2) : 0.0;
        if (!(rel == rel)) rel = INFINITY;
        worst = fmax(worst, rel);
        __syncthreads();  // cv is rewritten for the next right-hand side
    }
    if (tid == 0) res[cand] = bad ? INFINITY : worst;
}

// X[g][t] = sum_j V[j][t] * Y[g][j] for the nout = candidates x right-hand
// sides outputs, kExpandGroup outputs per CTA row (blockIdx.y).
__global__ void __launch_bounds__(kExpandThreads)
k_afs_expand(const double *__restrict__ V, int64_t n, int q, int qmax, const double2 *__restrict__ Y, int64_t g_first,
             int64_t nout, double2 *__restrict__ X) {
    __shared__ double2 ys[kExpandGroup][kMaxBasis];
    const int64_t g0 = g_first + (int64_t)blockIdx.y * kExpandGroup;
    const int ng = (int)min((int64_t)kExpandGroup, nout - g0);
    for (int e = threadIdx.x; e < kExpandGroup * kMaxBasis; e += kExpandThreads) {
        const int g = e / kMaxBasis, j = e - g * kMaxBasis;
        ys[g][j] = (g < ng && j < q) ? Y[(g0 + g) * qmax + j] : make_double2(0.0, 0.0);
    }
    __syncthreads();
    for (int64_t t = (int64_t)blockIdx.x * kExpandThreads + threadIdx.x; t < n; t += (int64_t)gridDim.x * kExpandThreads) {
        double2 acc[kExpandGroup];
#pragma unroll
        for (int g = 0; g < kExpandGroup; g++) acc[g] = make_double2(0.0, 0.0);
        const double *vt = V + t;
        for (int j = 0; j < q; j++, vt += n) {
            const double v = *vt;
#pragma unroll
            for (int g = 0; g < kExpandGroup; g++) {
                acc[g].x = fma(v, ys[g][j].x, acc[g].x);
                acc[g].y = fma(v, ys[g][j].y, acc[g].y);
            }
        }
#pragma unroll
        for (int g = 0; g < kExpandGroup; g++)
            if (g < ng) X[(g0 + g) * n + t] = acc[g];
    }
}

}  // namespace

// ------------------------------------------------------------------ host side

struct zsolve_afs {
    zsolve_ctx *ctx = nullptr;
    zsolve_afs_opts o{};
    int64_t n = 0;
    int nrhs_max = 0, qmax = 0, num_sms = 0;
    double *V = nullptr, *W = nullptr, *red = nullptr, *M = nullptr, *bb = nullptr;
    double2 *wb = nullptr, *br = nullptr, *xs = nullptr, *Y = nullptr;
    double *res = nullptr, *h_res = nullptr;
    int *d_q = nullptr, *h_q = nullptr;
    ZsSlotParam *d_par = nullptr, *h_par = nullptr;
    int64_t mcap = 0;
    cudaEvent_t ev[2] = {nullptr, nullptr};
    int64_t launches = 0;
    char err[512] = {0};
};

namespace {

int afs_fail(zsolve_afs *a, int code, const char *fmt, ...) {
    if (a) {
        va_list ap;
        va_start(ap, fmt);
        vsnprintf(a->err, sizeof(a->err), fmt, ap);
        va_end(ap);
    }
    return code;
}

#define AFS_CU(call)                                                                                          \
    do {                                                                                                      \
        cudaError_t e_ = (call);                                                                              \
        if (e_ != cudaSuccess)                                                                                \
            return afs_fail(a, ZSOLVE_ECUDA, "%s failed: %s (%s:%d)", #call, cudaGetErrorString(e_), __FILE__, \
                            __LINE__);                                                                        \
    } while (0)

void afs_free(zsolve_afs *a) {
    cudaFree(a->V);
    cudaFree(a->W);
    cudaFree(a->red);
    cudaFree(a->M);
    cudaFree(a->bb);
    cudaFree(a->wb);
    cudaFree(a->br);
    cudaFree(a->xs);
    cudaFree(a->Y);
    cudaFree(a->res);
    cudaFreeHost(a->h_res);
    cudaFree(a->d_q);
    cudaFreeHost(a->h_q);
    cudaFree(a->d_par);
    cudaFreeHost(a->h_par);
    for (auto e : a->ev)
        if (e) cudaEventDestroy(e);
}

int afs_reserve(zsolve_afs *a, int64_t m) {
    if (m <= a->mcap) return ZSOLVE_OK;
    cudaFree(a->Y);
    cudaFree(a->res);
    cudaFreeHost(a->h_res);
    cudaFree(a->d_par);
    cudaFreeHost(a->h_par);
    a->Y = nullptr;
    a->res = a->h_res = nullptr;
    a->d_par = a->h_par = nullptr;
    a->mcap = 0;
    if (cudaMalloc(&a->Y, (size_t)m * a->nrhs_max * a->qmax * sizeof(double2)) != cudaSuccess ||
        cudaMalloc(&a->res, (size_t)m * sizeof(double)) != cudaSuccess ||
        cudaMallocHost(&a->h_res, (size_t)m * sizeof(double)) != cudaSuccess ||
        cudaMalloc(&a->d_par, (size_t)m * sizeof(ZsSlotParam)) != cudaSuccess ||
        cudaMallocHost(&a->h_par, (size_t)m * sizeof(ZsSlotParam)) != cudaSuccess) {
        cudaGetLastError();
        return afs_fail(a, ZSOLVE_ENOMEM, "candidate buffers for %lld frequencies", (long long)m);
    }
    a->mcap = m;
    return ZSOLVE_OK;
}

// elapsed device time between the two events (both recorded on the stream)
float afs_span(zsolve_afs *a) {
    float ms = 0.f;
    if (cudaEventSynchronize(a->ev[1]) == cudaSuccess) cudaEventElapsedTime(&ms, a->ev[0], a->ev[1]);
    return ms;
}

}  // namespace

extern "C" {

int zsolve_afs_default_opts(zsolve_afs_opts *o) {
    if (!o) return ZSOLVE_EINVAL;
    o->tol = 1e-4;
    o->max_solves = 32;
    o->max_basis = kMaxBasis;
    o->drop = 1e-8;
    return ZSOLVE_OK;
}

int zsolve_afs_create(zsolve_afs **out, zsolve_ctx *ctx, const zsolve_afs_opts *opts) {
    if (!out || !ctx) return ZSOLVE_EINVAL;
    *out = nullptr;
    zsolve_afs *a = new (std::nothrow) zsolve_afs();
    if (!a) return ZSOLVE_ENOMEM;
    if (opts) a->o = *opts;
    else zsolve_afs_default_opts(&a->o);
    a->ctx = ctx;
    a->n = zs_ctx_n(ctx);
    a->nrhs_max = zs_ctx_nrhs_max(ctx);
    a->qmax = a->o.max_basis;
    if (!(a->o.tol > 0.0) || a->o.max_solves < 1 || a->o.max_basis < 1 || a->o.max_basis > kMaxBasis ||
        !(a->o.drop >= 0.0) || !(a->o.drop < 1.0) ||
        eval_smem_bytes(a->qmax, a->nrhs_max) > (size_t)kMaxSmem) {
        delete a;
        return ZSOLVE_EINVAL;
    }
    auto bail = [&](int code) {
        afs_free(a);
        delete a;
        return code;
    };
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return bail(ZSOLVE_ECUDA);
    cudaDeviceGetAttribute(&a->num_sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t n = a->n, qm = a->qmax, R = a->nrhs_max;
#define ALLOC(p, bytes) \
    if (cudaMalloc(&(p), (bytes)) != cudaSuccess) return bail(ZSOLVE_ENOMEM)
    ALLOC(a->V, (size_t)qm * n * sizeof(double));
    ALLOC(a->W, (size_t)3 * qm * n * sizeof(double));
    ALLOC(a->red, (size_t)3 * qm * qm * sizeof(double));
    ALLOC(a->M, (size_t)9 * qm * qm * sizeof(double));
    ALLOC(a->bb, (size_t)R * sizeof(double));
    ALLOC(a->wb, (size_t)3 * qm * R * sizeof(double2));
    ALLOC(a->br, (size_t)qm * R * sizeof(double2));
    ALLOC(a->xs, (size_t)2 * R * n * sizeof(double2));
    ALLOC(a->d_q, 2 * sizeof(int));
#undef ALLOC
    if (cudaMallocHost(&a->h_q, 2 * sizeof(int)) != cudaSuccess) return bail(ZSOLVE_ENOMEM);
    for (auto &e : a->ev)
        if (cudaEventCreate(&e) != cudaSuccess) return bail(ZSOLVE_ECUDA);
    *out = a;
    return ZSOLVE_OK;
}

int zsolve_afs_sweep(zsolve_afs *a, const double *L, const double *Psi, const double *G, const double *omega,
                     const double *zs, int m, const void *b, void *x, int nrhs, int *sampled, double *resid,
                     zsolve_afs_info *info) {
    if (!a) return ZSOLVE_EINVAL;
    if (!L || !Psi || !G || !omega || !zs || !b || m < 0)
        return afs_fail(a, ZSOLVE_EINVAL, "NULL argument or m < 0");
    if (nrhs < 1 || nrhs > a->nrhs_max)
        return afs_fail(a, ZSOLVE_EINVAL, "nrhs = %d outside 1..%d", nrhs, a->nrhs_max);
    for (int i = 0; i < m; i++)
        if (!(omega[i] > 0.0) || !std::isfinite(omega[i]) || !std::isfinite(zs[2 * i]) ||
            !std::isfinite(zs[2 * i + 1]))
            return afs_fail(a, ZSOLVE_EINVAL, "candidate %d: omega must be positive and finite, Zs finite", i);
    zsolve_afs_info inf{};
    if (m == 0) {
        inf.converged = 1;
        if (info) *info = inf;
        return ZSOLVE_OK;
    }
    int st = afs_reserve(a, m);
    if (st != ZSOLVE_OK) return st;
    cudaStream_t s = zs_ctx_stream(a->ctx);
    const int64_t n = a->n;
    const int qmax = a->qmax;
    const double one = 1.0;
    for (int i = 0; i < m; i++) a->h_par[i] = ZsSlotParam{omega[i], zs[2 * i], zs[2 * i + 1], 0.0};
    AFS_CU(cudaMemcpyAsync(a->d_par, a->h_par, (size_t)m * sizeof(ZsSlotParam), cudaMemcpyHostToDevice, s));
    std::vector<char> done(m, 0);
    std::vector<int> order;
    std::vector<int> pending;
    pending.push_back(0);
    if (m > 1 && a->o.max_solves > 1) pending.push_back(m - 1);
    int q = 0;
    bool full = false, converged = false;
    double worst = INFINITY;
    const size_t smem_cap = eval_smem_bytes(qmax, a->nrhs_max);
    // the limit is a property of the kernel, shared by every handle: set it
    // for this handle's largest reduced system on each call
    AFS_CU(cudaFuncSetAttribute(k_afs_eval, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_cap));
    bool first = true;
    while (true) {
        // step 1: exact solves at the pending candidates
        double om_sub[2], zs_sub[4];
        zsolve_info si[2];
        const int k = (int)pending.size();
        for (int i = 0; i < k; i++) {
            om_sub[i] = omega[pending[i]];
            zs_sub[2 * i] = zs[2 * pending[i]];
            zs_sub[2 * i + 1] = zs[2 * pending[i] + 1];
        }
        AFS_CU(cudaEventRecord(a->ev[0], s));
        st = zsolve_sweep(a->ctx, L, Psi, G, om_sub, zs_sub, k, b, a->xs, nrhs, si);
        if (st != ZSOLVE_OK)
            return afs_fail(a, st, "exact solve at candidate %d: %s", pending[0], zsolve_last_error(a->ctx));
        AFS_CU(cudaEventRecord(a->ev[1], s));
        inf.ms_exact += afs_span(a);
        for (int i = 0; i < k; i++) {
            done[pending[i]] = 1;
            order.push_back(pending[i]);
            inf.fallbacks += si[i].fallback ? 1 : 0;
        }
        inf.n_exact += k;
        // the real and imaginary parts into the basis, then the reduced terms
        AFS_CU(cudaEventRecord(a->ev[0], s));
        k_afs_orth<<<kOrthCluster, kOrthThreads, 0, s>>>(a->V, n, q, qmax, a->xs, k * nrhs, a->o.drop, a->d_q, one);
        AFS_CU(cudaGetLastError());
        AFS_CU(cudaMemcpyAsync(a->h_q, a->d_q, 2 * sizeof(int), cudaMemcpyDeviceToHost, s));
        AFS_CU(cudaStreamSynchronize(s));
        const int qn = a->h_q[0];
        full = full || a->h_q[1] != 0;
        a->launches++;
        if (qn > q) {
            const int nc = qn - q;
            const int64_t warps_needed = n;
            int gx = (int)std::min<int64_t>((warps_needed + kProjThreads / 32 - 1) / (kProjThreads / 32),
                                            (int64_t)a->num_sms * 4);
            dim3 grid(std::max(gx, 1), (nc + kProjCols - 1) / kProjCols);
            k_afs_project<<<grid, kProjThreads, 0, s>>>(L, Psi, G, n, a->V, q, nc, a->W, (int64_t)qmax * n, one);
            AFS_CU(cudaGetLastError());
            a->launches++;
        }
        if (qn > q || first) {  // the first launch also forms ||b||^2
            const int64_t tasks = 12LL * qn * qn + 4LL * qn * nrhs + (q == 0 ? nrhs : 0);
            const int64_t blocks = (tasks + kGramThreads / 32 - 1) / (kGramThreads / 32);
            k_afs_gram<<<(unsigned)std::max<int64_t>(blocks, 1), kGramThreads, 0, s>>>(
                a->V, a->W, (const double2 *)b, n, qmax, q, qn, nrhs, a->red, a->M, a->wb, a->br, a->bb, one);
            AFS_CU(cudaGetLastError());
            a->launches++;
        }
        q = qn;
        first = false;
        AFS_CU(cudaEventRecord(a->ev[1], s));
        inf.ms_basis += afs_span(a);
        // steps 2-3 at every candidate
        AFS_CU(cudaEventRecord(a->ev[0], s));
        const size_t smem = eval_smem_bytes(q, nrhs);
        if (smem > smem_cap) return afs_fail(a, ZSOLVE_EINVAL, "reduced system too large for shared memory");
        k_afs_eval<<<(unsigned)m, kEvalThreads, smem, s>>>(a->d_par, a->red, a->M, a->wb, a->br, a->bb, q, qmax,
                                                            nrhs, a->Y, a->res, one);
        AFS_CU(cudaGetLastError());
        a->launches++;
        AFS_CU(cudaMemcpyAsync(a->h_res, a->res, (size_t)m * sizeof(double), cudaMemcpyDeviceToHost, s));
        AFS_CU(cudaEventRecord(a->ev[1], s));
        inf.ms_eval += afs_span(a);
        inf.evals++;
        inf.eval_gflop += (double)m * (8.0 / 3.0 * q * (double)q * q + 44.0 * q * (double)q * nrhs) * 1e-9;
        // step 4: stop, or solve next at the largest estimate not yet solved
        worst = 0.0;
        for (int i = 0; i < m; i++) {
            const double v = std::isnan(a->h_res[i]) ? INFINITY : a->h_res[i];
            if (v > worst) worst = v;
        }
        if (worst < a->o.tol) {
            converged = true;
            break;
        }
        if ((int)order.size() >= std::min(a->o.max_solves, m) || full) break;
        int best = -1;
        double bv = -1.0;
        for (int i = 0; i < m; i++) {
            if (done[i]) continue;
            const double v = std::isnan(a->h_res[i]) ? INFINITY : a->h_res[i];
            if (v > bv) {
                bv = v;
                best = i;
            }
        }
        if (best < 0) break;
        pending.assign(1, best);
    }
    // x = V y at every candidate
    AFS_CU(cudaEventRecord(a->ev[0], s));
    if (x) {
        const int64_t nout = (int64_t)m * nrhs;
        const unsigned gx = (unsigned)std::max<int64_t>(1, (n + kExpandThreads - 1) / kExpandThreads);
        const int64_t ygroups = (nout + kExpandGroup - 1) / kExpandGroup;
        for (int64_t y0 = 0; y0 < ygroups; y0 += 65535) {
            const unsigned gy = (unsigned)std::min<int64_t>(65535, ygroups - y0);
            k_afs_expand<<<dim3(gx, gy), kExpandThreads, 0, s>>>(a->V, n, q, qmax, a->Y, y0 * kExpandGroup, nout,
                                                                 (double2 *)x);
            AFS_CU(cudaGetLastError());
            a->launches++;
        }
    }
    AFS_CU(cudaEventRecord(a->ev[1], s));
    inf.ms_expand = afs_span(a);
    AFS_CU(cudaStreamSynchronize(s));
    inf.q = q;
    inf.converged = converged ? 1 : 0;
    inf.basis_full = full ? 1 : 0;
    inf.max_resid = worst;
    if (sampled)
        for (size_t i = 0; i < order.size(); i++) sampled[i] = order[i];
    if (resid) std::memcpy(resid, a->h_res, (size_t)m * sizeof(double));
    if (info) *info = inf;
    return ZSOLVE_OK;
}

int64_t zsolve_afs_launches(const zsolve_afs *a) { return a ? a->launches : 0; }

const char *zsolve_afs_last_error(const zsolve_afs *a) { return a ? a->err : "NULL handle"; }

void zsolve_afs_destroy(zsolve_afs *a) {
    if (!a) return;
    afs_free(a);
    delete a;
}

}  // extern "C"
