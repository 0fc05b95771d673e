// Double-precision LU with partial pivoting on the GPU: the fallback for a
// frequency whose refinement does not converge (malusrfworks.com, "Solving
// Dense Matrices Fast in the Browser", section "Double-precision answers
// from a GPU without double precision": such a frequency alone switches to a
// direct solve; section "Measure first": the direct solve falls back to LU
// with partial pivoting).
//
// Right-looking, 32-column panels, complex float64, row-major with ld = n:
//   k_lu64_panel  one CTA factors the panel with partial pivoting (pivot =
//                 largest |Re|+|Im| in the column, lowest row on ties,
//                 multipliers by Smith's complex division);
//   k_lu64_swap   applies the panel's interchanges to the other columns;
//   k_lu64_trsm   U12 = L11^-1 A12;
//   k_lu64_gemm   A22 -= L21 U12 (DFMA).
// Substitution: interchanges on the right-hand sides, then forward (unit
// lower) and back (upper) substitution in 32-row blocks (a diagonal solve in
// one CTA, then an update of the remaining rows).  Runs only for stalled
// frequencies; bound by the FP64 pipe.
#include "common.cuh"

namespace {

constexpr int W = 32;  // panel width
constexpr int kPanelThreads = 1024;

__device__ __forceinline__ double2 zmul(double2 a, double2 b) {
    return make_double2(a.x * b.x - a.y * b.y, a.x * b.y + a.y * b.x);
}

// a - b*c
__device__ __forceinline__ double2 zfms(double2 a, double2 b, double2 c) {
    return make_double2(a.x - (b.x * c.x - b.y * c.y), a.y - (b.x * c.y + b.y * c.x));
}

// Smith's complex division a / c
__device__ __forceinline__ double2 zdiv(double2 a, double2 c) {
    if (fabs(c.x) >= fabs(c.y)) {
        const double r = c.y / c.x, den = c.x + c.y * r;
        return make_double2((a.x + a.y * r) / den, (a.y - a.x * r) / den);
    }
    const double r = c.x / c.y, den = c.x * r + c.y;
    return make_double2((a.x * r + a.y) / den, (a.y * r - a.x) / den);
}

__global__ void __launch_bounds__(kPanelThreads)
k_lu64_panel(double2 *__restrict__ a, int64_t n, int64_t k0, int w, int64_t *__restrict__ piv,
             int *__restrict__ info) {
    __shared__ double s_val[kPanelThreads / 32];
    __shared__ int64_t s_idx[kPanelThreads / 32];
    __shared__ double2 s_prow[W];
    __shared__ int64_t s_p;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (*(volatile int *)info) return;
    for (int kk = 0; kk < w; kk++) {
        const int64_t k = k0 + kk;
        // argmax of |Re|+|Im| over rows k..n-1, lowest index on ties
        double best = -1.0;
        int64_t bi = n;
        for (int64_t i = k + tid; i < n; i += kPanelThreads) {
            const double2 v = a[i * n + k];
            const double m = fabs(v.x) + fabs(v.y);
            if (m > best) {  // rows visited in increasing order: first max kept
                best = m;
                bi = i;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const double ob = __shfl_xor_sync(0xffffffffu, best, o);
            const int64_t oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ob > best || (ob == best && oi < bi)) {
                best = ob;
                bi = oi;
            }
        }
        if (lane == 0) {
            s_val[warp] = best;
            s_idx[warp] = bi;
        }
        __syncthreads();
        if (tid == 0) {
            double b = s_val[0];
            int64_t ix = s_idx[0];
            for (int q = 1; q < kPanelThreads / 32; q++)
                if (s_val[q] > b || (s_val[q] == b && s_idx[q] < ix)) {
                    b = s_val[q];
                    ix = s_idx[q];
                }
            if (!(b > 0.0)) {  // zero column (or NaN): singular
                *info = (int)(k + 1);
                ix = -1;
            }
            s_p = ix;
            piv[k] = ix < 0 ? k : ix;
        }
        __syncthreads();
        const int64_t p = s_p;
        if (p < 0) return;
        // swap rows k and p inside the panel columns, stage the pivot row
        if (tid < w) {
            const int64_t c = k0 + tid;
            double2 t = a[k * n + c];
            if (p != k) {
                const double2 u = a[p * n + c];
                a[p * n + c] = t;
                a[k * n + c] = u;
                t = u;
            }
            s_prow[tid] = t;
        }
        __syncthreads();
        const double2 pv = s_prow[kk];
        for (int64_t i = k + 1 + tid; i < n; i += kPanelThreads) {
            double2 *row = a + i * n + k0;
            const double2 l = zdiv(row[kk], pv);
            row[kk] = l;
            for (int j = kk + 1; j < w; j++) row[j] = zfms(row[j], l, s_prow[j]);
        }
        __syncthreads();
    }
}

__global__ void k_lu64_swap(double2 *__restrict__ a, int64_t n, int64_t k0, int w,
                            const int64_t *__restrict__ piv, const int *__restrict__ info) {
    if (*info) return;
    const int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= n || (j >= k0 && j < k0 + w)) return;
    for (int kk = 0; kk < w; kk++) {
        const int64_t k = k0 + kk, p = piv[k];
        if (p != k) {
            const double2 t = a[k * n + j];
            a[k * n + j] = a[p * n + j];
            a[p * n + j] = t;
        }
    }
}

__global__ void k_lu64_trsm(double2 *__restrict__ a, int64_t n, int64_t k0, int w, const int *__restrict__ info) {
    __shared__ double2 sl[W][W + 1];
    if (*info) return;
    for (int idx = threadIdx.x; idx < w * w; idx += blockDim.x) {
        const int i = idx / w, c = idx - i * w;
        sl[i][c] = a[(k0 + i) * n + k0 + c];
    }
    __syncthreads();
    const int64_t j = k0 + w + (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= n) return;
    double2 u[W];
#pragma unroll
    for (int i = 0; i < W; i++) {
        if (i < w) {
            double2 s = a[(k0 + i) * n + j];
#pragma unroll
            for (int m = 0; m < W; m++)
                if (m < i) s = zfms(s, sl[i][m], u[m]);
            u[i] = s;
            a[(k0 + i) * n + j] = s;
        }
    }
}

constexpr int kGT = 32;  // output tile of the trailing update

__global__ void __launch_bounds__(256)
k_lu64_gemm(double2 *__restrict__ a, int64_t n, int64_t k0, int w, const int *__restrict__ info) {
    __shared__ double2 sL[kGT][W + 1];
    __shared__ double2 sU[W][kGT + 1];
    if (*info) return;
    const int64_t base = k0 + w;
    const int64_t i0 = base + (int64_t)blockIdx.y * kGT, j0 = base + (int64_t)blockIdx.x * kGT;
    for (int idx = threadIdx.x; idx < kGT * w; idx += blockDim.x) {
        const int r = idx / w, c = idx - r * w;
        sL[r][c] = (i0 + r < n) ? a[(i0 + r) * n + k0 + c] : make_double2(0.0, 0.0);
        const int kr = idx / kGT, jc = idx - kr * kGT;
        sU[kr][jc] = (j0 + jc < n) ? a[(k0 + kr) * n + j0 + jc] : make_double2(0.0, 0.0);
    }
    __syncthreads();
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 8 rows of warps, 4 rows each
#pragma unroll
    for (int q = 0; q < 4; q++) {
        const int r = ty * 4 + q;
        const int64_t i = i0 + r, j = j0 + tx;
        if (i < n && j < n) {
            double2 acc = a[i * n + j];
            for (int k = 0; k < w; k++) acc = zfms(acc, sL[r][k], sU[k][tx]);
            a[i * n + j] = acc;
        }
    }
}

__global__ void k_lu64_apply_piv(double2 *__restrict__ x, int64_t n, const int64_t *__restrict__ piv) {
    double2 *xs = x + (int64_t)blockIdx.x * n;
    if (threadIdx.x != 0) return;
    for (int64_t k = 0; k < n; k++) {
        const int64_t p = piv[k];
        if (p != k) {
            const double2 t = xs[k];
            xs[k] = xs[p];
            xs[p] = t;
        }
    }
}

// diagonal block solve: one CTA, one thread per right-hand side
__global__ void k_lu64_trsv_diag(const double2 *__restrict__ lu, int64_t n, double2 *__restrict__ x, int nrhs,
                                 int64_t r0, int bw, int upper) {
    __shared__ double2 sd[W][W + 1];
    for (int idx = threadIdx.x; idx < bw * bw; idx += blockDim.x) {
        const int i = idx / bw, c = idx - i * bw;
        sd[i][c] = lu[(r0 + i) * n + r0 + c];
    }
    __syncthreads();
    const int r = threadIdx.x;
    if (r >= nrhs) return;
    double2 *xs = x + (int64_t)r * n + r0;
    double2 v[W];
    for (int i = 0; i < bw; i++) v[i] = xs[i];
    if (!upper) {
        for (int i = 0; i < bw; i++)
            for (int c = 0; c < i; c++) v[i] = zfms(v[i], sd[i][c], v[c]);
    } else {
        for (int i = bw - 1; i >= 0; i--) {
            for (int c = i + 1; c < bw; c++) v[i] = zfms(v[i], sd[i][c], v[c]);
            v[i] = zdiv(v[i], sd[i][i]);
        }
    }
    for (int i = 0; i < bw; i++) xs[i] = v[i];
}

// rows on the far side of the block: x[i] -= LU[i, block] . x[block]; a warp per row
__global__ void k_lu64_trsv_update(const double2 *__restrict__ lu, int64_t n, double2 *__restrict__ x, int nrhs,
                                   int64_t r0, int bw, int upper) {
    const int lane = threadIdx.x & 31;
    const int64_t w = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    const int64_t i = upper ? w : r0 + bw + w;
    if (upper ? (i >= r0) : (i >= n)) return;
    const double2 l = lane < bw ? lu[i * n + r0 + lane] : make_double2(0.0, 0.0);
    for (int r = 0; r < nrhs; r++) {
        const double2 xv = lane < bw ? x[(int64_t)r * n + r0 + lane] : make_double2(0.0, 0.0);
        double2 p = zmul(l, xv);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            p.x += __shfl_xor_sync(0xffffffffu, p.x, o);
            p.y += __shfl_xor_sync(0xffffffffu, p.y, o);
        }
        if (lane == 0) {
            double2 *t = x + (int64_t)r * n + i;
            *t = make_double2(t->x - p.x, t->y - p.y);
        }
    }
}

}  // namespace

cudaError_t zs_lu64_factor(double2 *a, int64_t n, int64_t *piv, int *info, cudaStream_t st, int64_t *launches) {
    int64_t cnt = 0;
    cudaError_t e = cudaMemsetAsync(info, 0, sizeof(int), st);
    if (e != cudaSuccess) return e;
    for (int64_t k0 = 0; k0 < n; k0 += W) {
        const int w = (int)((n - k0) < W ? (n - k0) : W);
        k_lu64_panel<<<1, kPanelThreads, 0, st>>>(a, n, k0, w, piv, info);
        k_lu64_swap<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(a, n, k0, w, piv, info);
        cnt += 2;
        const int64_t m = n - k0 - w;
        if (m > 0) {
            k_lu64_trsm<<<(unsigned)((m + 127) / 128), 128, 0, st>>>(a, n, k0, w, info);
            const unsigned t = (unsigned)((m + kGT - 1) / kGT);
            k_lu64_gemm<<<dim3(t, t), 256, 0, st>>>(a, n, k0, w, info);
            cnt += 2;
        }
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (launches) *launches += cnt;
    return cudaSuccess;
}

cudaError_t zs_lu64_solve(const double2 *lu, int64_t n, const int64_t *piv, double2 *x, int nrhs,
                          cudaStream_t st, int64_t *launches) {
    if (nrhs > 32) return cudaErrorInvalidValue;
    int64_t cnt = 1;
    k_lu64_apply_piv<<<nrhs, 32, 0, st>>>(x, n, piv);
    for (int64_t r0 = 0; r0 < n; r0 += W) {  // forward, unit lower
        const int bw = (int)((n - r0) < W ? (n - r0) : W);
        k_lu64_trsv_diag<<<1, 32, 0, st>>>(lu, n, x, nrhs, r0, bw, 0);
        const int64_t rows = n - r0 - bw;
        cnt += 1 + (rows > 0);
        if (rows > 0) k_lu64_trsv_update<<<(unsigned)((rows + 7) / 8), 256, 0, st>>>(lu, n, x, nrhs, r0, bw, 0);
    }
    const int64_t last = ((n - 1) / W) * W;
    for (int64_t r0 = last; r0 >= 0; r0 -= W) {  // backward, upper
        const int bw = (int)((n - r0) < W ? (n - r0) : W);
        k_lu64_trsv_diag<<<1, 32, 0, st>>>(lu, n, x, nrhs, r0, bw, 1);
        cnt += 1 + (r0 > 0);
        if (r0 > 0) k_lu64_trsv_update<<<(unsigned)((r0 + 7) / 8), 256, 0, st>>>(lu, n, x, nrhs, r0, bw, 1);
    }
    if (launches) *launches += cnt;
    return cudaGetLastError();
}
