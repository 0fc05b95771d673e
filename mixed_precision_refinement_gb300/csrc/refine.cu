// Double-precision steps of the refinement (malusrfworks.com, "Solving Dense
// Matrices Fast in the Browser", section "Double-precision answers from a GPU
// without double precision": step 3, r = b - Z x in double precision; step 4,
// x += d; the stopping test on the size of the correction).
//
// k_residual: one warp per row of the float64 matrix, lanes stride the row
// with 16-byte loads (coalesced), warp-shuffle reduction; the result is
// written rounded to complex float32 (the input of the next low-precision
// solve) or, for the stage-level call, in float64.  A complex entry costs
// four DFMA per right-hand side; a warp step of 128 entries whose real parts
// are all exact zeros (Re Z_ij = Zs.re G_ij vanishes wherever G_ij = 0) takes
// a branch with two.  The skipped products are exact zeros added to the
// running sums, so the float64 result is the one the four-DFMA sequence in
// the same order gives (finite x).  The final sums are fma(a, 1, b), the same
// rounding as an add: the FP64 pipe here retires DFMA several times faster
// than DADD.  Bound: HBM or the FP64 pipe, whichever is lower -- the kernel
// moves 16 n^2 bytes per frequency.
//
// k_update / k_relcorr: x (float64) += d (float32), and per (frequency, RHS)
// ||d||_2 / ||x||_2 from per-block partial sums reduced in a fixed order, so
// the stopping test is deterministic.
#include "common.cuh"

namespace {

constexpr int kResThreads = 256;  // 8 warps, one row each

template <int R>
__global__ void __launch_bounds__(kResThreads)
k_residual(const double2 *__restrict__ z64, int64_t z64_stride, int64_t n, const double2 *__restrict__ b,
           const double2 *__restrict__ x, int64_t x_stride, float2 *__restrict__ out64,
           int64_t out64_stride, double2 *__restrict__ out128, int64_t out128_stride,
           const int *__restrict__ slots, double one) {
    const int slot = slots[blockIdx.y];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t row = (int64_t)blockIdx.x * (kResThreads / 32) + warp;
    if (row >= n) return;
    const double2 *zr = z64 + (int64_t)slot * z64_stride + row * n;
    const double2 *xs = x + (int64_t)slot * x_stride;
    // NA independent accumulator pairs per right-hand side (sub-step u uses
    // u % NA): the FP64 unit's latency is long, so each warp needs about eight
    // independent chains; with several right-hand sides they come from R
    constexpr int NA = R >= 4 ? 1 : 4 / R;
    double ar[NA][R], ai[NA][R];
#pragma unroll
    for (int u = 0; u < NA; u++)
#pragma unroll
        for (int r = 0; r < R; r++) ar[u][r] = ai[u][r] = 0.0;
    // full 128-entry steps first: the bound is the same for every lane, so the
    // warp vote below always sees the whole warp.  Loop counts are 32-bit and
    // addresses advance by pointer steps: 64-bit integer tests and products
    // can be issued to the FP64 pipe on this part, the bound of this kernel.
    const int nn = (int)n, nfull = nn >> 7;
    const double2 *zp = zr + lane;
    const double2 *xp[R];
#pragma unroll
    for (int r = 0; r < R; r++) xp[r] = xs + r * n + lane;
#pragma unroll 1
    for (int s = 0; s < nfull; s++) {
        double2 z[4];
#pragma unroll
        for (int u = 0; u < 4; u++) z[u] = __ldcs(zp + 32 * u);
        // warp-uniform test: every real part in these 128 entries an exact zero
        bool re0 = true;
#pragma unroll
        for (int u = 0; u < 4; u++) re0 = re0 && zs::is_zero(zs::bits_of(z[u].x));
        if (__all_sync(0xffffffffu, re0)) {
#pragma unroll
            for (int u = 0; u < 4; u++)
#pragma unroll
                for (int r = 0; r < R; r++) {
                    const double2 xv = __ldg(xp[r] + 32 * u);
                    ar[u % NA][r] = fma(zs::neg_bits(z[u].y), xv.y, ar[u % NA][r]);
                    ai[u % NA][r] = fma(z[u].y, xv.x, ai[u % NA][r]);
                }
        } else {
#pragma unroll
            for (int u = 0; u < 4; u++)
#pragma unroll
                for (int r = 0; r < R; r++) {
                    const double2 xv = __ldg(xp[r] + 32 * u);
                    ar[u % NA][r] = fma(z[u].x, xv.x, ar[u % NA][r]);
                    ai[u % NA][r] = fma(z[u].x, xv.y, ai[u % NA][r]);
                    ar[u % NA][r] = fma(zs::neg_bits(z[u].y), xv.y, ar[u % NA][r]);
                    ai[u % NA][r] = fma(z[u].y, xv.x, ai[u % NA][r]);
                }
        }
        zp += 128;
#pragma unroll
        for (int r = 0; r < R; r++) xp[r] += 128;
    }
    for (int j = (nfull << 7) + lane; j < nn; j += 32) {
        const double2 z = __ldcs(zp);
#pragma unroll
        for (int r = 0; r < R; r++) {
            const double2 xv = __ldg(xp[r]);
            ar[0][r] = fma(z.x, xv.x, ar[0][r]);
            ai[0][r] = fma(z.x, xv.y, ai[0][r]);
            ar[0][r] = fma(zs::neg_bits(z.y), xv.y, ar[0][r]);
            ai[0][r] = fma(z.y, xv.x, ai[0][r]);
            xp[r] += 32;
        }
        zp += 32;
    }
#pragma unroll
    for (int r = 0; r < R; r++) {
        // sums as fma(a, 1, b): the same rounding as an add, on the full-rate DFMA path
#pragma unroll
        for (int u = 1; u < NA; u++) {
            ar[0][r] = fma(ar[u][r], one, ar[0][r]);
            ai[0][r] = fma(ai[u][r], one, ai[0][r]);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            ar[0][r] = fma(__shfl_xor_sync(0xffffffffu, ar[0][r], o), one, ar[0][r]);
            ai[0][r] = fma(__shfl_xor_sync(0xffffffffu, ai[0][r], o), one, ai[0][r]);
        }
    }
    if (lane < R) {
        double vr = 0.0, vi = 0.0;
#pragma unroll
        for (int r = 0; r < R; r++)
            if (r == lane) {
                vr = ar[0][r];
                vi = ai[0][r];
            }
        const double2 bv = b[(int64_t)lane * n + row];
        const double rr = bv.x - vr, ri = bv.y - vi;
        if (out64)
            out64[(int64_t)slot * out64_stride + (int64_t)lane * n + row] =
                make_float2(__double2float_rn(rr), __double2float_rn(ri));
        else
            out128[(int64_t)slot * out128_stride + (int64_t)lane * n + row] = make_double2(rr, ri);
    }
}

__global__ void k_cast_rhs(const double2 *__restrict__ b, int64_t n, int nrhs, float2 *__restrict__ v,
                           int64_t v_stride, const int *__restrict__ slots) {
    const int slot = slots[blockIdx.y];
    const int64_t total = (int64_t)nrhs * n;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x) {
        const double2 t = b[e];
        v[(int64_t)slot * v_stride + e] = make_float2(__double2float_rn(t.x), __double2float_rn(t.y));
    }
}

constexpr int kUpdThreads = 256;
constexpr int kUpdPer = 4;
constexpr int kUpdChunk = kUpdThreads * kUpdPer;

// grid: (chunks, nslot * nrhs)
__global__ void __launch_bounds__(kUpdThreads)
k_update(double2 *__restrict__ x, int64_t x_stride, const float2 *__restrict__ d, int64_t d_stride,
         int64_t n, int nrhs, int assign, double *__restrict__ partials, int nchunks,
         const int *__restrict__ slots) {
    const int si = blockIdx.y / nrhs, r = blockIdx.y - si * nrhs;
    const int slot = slots[si];
    double2 *xs = x + (int64_t)slot * x_stride + (int64_t)r * n;
    const float2 *ds = d + (int64_t)slot * d_stride + (int64_t)r * n;
    double dd = 0.0, xx = 0.0;
    const int64_t base = (int64_t)blockIdx.x * kUpdChunk;
#pragma unroll
    for (int u = 0; u < kUpdPer; u++) {
        const int64_t i = base + u * kUpdThreads + threadIdx.x;
        if (i < n) {
            const float2 dv = ds[i];
            const double dr = (double)dv.x, di = (double)dv.y;
            double2 xv = assign ? make_double2(0.0, 0.0) : xs[i];
            xv.x += dr;
            xv.y += di;
            xs[i] = xv;
            dd = fma(dr, dr, fma(di, di, dd));
            xx = fma(xv.x, xv.x, fma(xv.y, xv.y, xx));
        }
    }
    __shared__ double sd[kUpdThreads / 32], sx[kUpdThreads / 32];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        dd += __shfl_xor_sync(0xffffffffu, dd, o);
        xx += __shfl_xor_sync(0xffffffffu, xx, o);
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) {
        sd[warp] = dd;
        sx[warp] = xx;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        double a = 0.0, c = 0.0;
        for (int w = 0; w < kUpdThreads / 32; w++) {
            a += sd[w];
            c += sx[w];
        }
        double *p = partials + (((int64_t)slot * nrhs + r) * nchunks + blockIdx.x) * 2;
        p[0] = a;
        p[1] = c;
    }
}

__global__ void k_relcorr(const double *__restrict__ partials, int nchunks, int nrhs,
                          double *__restrict__ relcorr, const int *__restrict__ slots, int nslot) {
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= nslot * nrhs) return;
    const int si = t / nrhs, r = t - si * nrhs;
    const int slot = slots[si];
    const double *p = partials + ((int64_t)slot * nrhs + r) * nchunks * 2;
    double dd = 0.0, xx = 0.0;
    for (int c = 0; c < nchunks; c++) {
        dd += p[2 * c];
        xx += p[2 * c + 1];
    }
    double rc;
    if (!isfinite(dd) || !isfinite(xx)) rc = nan("");
    else if (xx == 0.0) rc = (dd == 0.0) ? 0.0 : INFINITY;
    else rc = sqrt(dd / xx);
    relcorr[(int64_t)slot * nrhs + r] = rc;
}

__global__ void k_widen(const float2 *__restrict__ v, double2 *__restrict__ d, int64_t count) {
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < count; e += (int64_t)gridDim.x * blockDim.x)
        d[e] = make_double2((double)v[e].x, (double)v[e].y);
}

__global__ void k_narrow(const double2 *__restrict__ d, float2 *__restrict__ v, int64_t count) {
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < count; e += (int64_t)gridDim.x * blockDim.x)
        v[e] = make_float2(__double2float_rn(d[e].x), __double2float_rn(d[e].y));
}

__global__ void k_copy_z32_out(const float *__restrict__ z32, int64_t ld, int64_t plane, int64_t n,
                               float *__restrict__ ore, float *__restrict__ oim) {
    for (int64_t i = blockIdx.x; i < n; i += gridDim.x)
        for (int64_t j = threadIdx.x; j < n; j += blockDim.x) {
            ore[i * n + j] = z32[i * ld + j];
            oim[i * n + j] = z32[plane + i * ld + j];
        }
}

unsigned grid1d(int64_t count, int threads) {
    int64_t g = (count + threads - 1) / threads;
    if (g > 65535) g = 65535;
    if (g < 1) g = 1;
    return (unsigned)g;
}

template <int R>
void launch_res(const double2 *z64, int64_t z64_stride, int64_t n, const double2 *b, const double2 *x,
                int64_t x_stride, float2 *o64, int64_t o64s, double2 *o128, int64_t o128s, const int *slots,
                int nslot, cudaStream_t st) {
    dim3 grid((unsigned)((n + 7) / 8), nslot);
    k_residual<R><<<grid, kResThreads, 0, st>>>(z64, z64_stride, n, b, x, x_stride, o64, o64s, o128, o128s,
                                                slots, 1.0);
}

}  // namespace

cudaError_t zs_launch_residual(const double2 *z64, int64_t z64_stride, int64_t n, const double2 *b,
                               const double2 *x, int64_t x_stride, int nrhs, float2 *out_c64,
                               int64_t out64_stride, double2 *out_c128, int64_t out128_stride,
                               const int *slots, int nslot, cudaStream_t st) {
    // right-hand sides in chunks of 8, 4, 2, 1
    int r0 = 0;
    while (r0 < nrhs) {
        const int left = nrhs - r0;
        const int R = left >= 8 ? 8 : left >= 4 ? 4 : left >= 2 ? 2 : 1;
        const double2 *bb = b + (int64_t)r0 * n;
        const double2 *xx = x + (int64_t)r0 * n;
        float2 *o64 = out_c64 ? out_c64 + (int64_t)r0 * n : nullptr;
        double2 *o128 = out_c128 ? out_c128 + (int64_t)r0 * n : nullptr;
        switch (R) {
            case 8: launch_res<8>(z64, z64_stride, n, bb, xx, x_stride, o64, out64_stride, o128, out128_stride, slots, nslot, st); break;
            case 4: launch_res<4>(z64, z64_stride, n, bb, xx, x_stride, o64, out64_stride, o128, out128_stride, slots, nslot, st); break;
            case 2: launch_res<2>(z64, z64_stride, n, bb, xx, x_stride, o64, out64_stride, o128, out128_stride, slots, nslot, st); break;
            default: launch_res<1>(z64, z64_stride, n, bb, xx, x_stride, o64, out64_stride, o128, out128_stride, slots, nslot, st); break;
        }
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        r0 += R;
    }
    return cudaSuccess;
}

cudaError_t zs_launch_cast_rhs(const double2 *b, int64_t n, int nrhs, float2 *v, int64_t v_stride,
                               const int *slots, int nslot, cudaStream_t st) {
    dim3 grid(grid1d((int64_t)nrhs * n, 256), nslot);
    k_cast_rhs<<<grid, 256, 0, st>>>(b, n, nrhs, v, v_stride, slots);
    return cudaGetLastError();
}

int zs_update_chunks(int64_t n) { return (int)((n + kUpdChunk - 1) / kUpdChunk); }

cudaError_t zs_launch_update(double2 *x, int64_t x_stride, const float2 *d, int64_t d_stride, int64_t n,
                             int nrhs, int assign, double *partials, int nchunks, const int *slots, int nslot,
                             cudaStream_t st) {
    dim3 grid(nchunks, nslot * nrhs);
    k_update<<<grid, kUpdThreads, 0, st>>>(x, x_stride, d, d_stride, n, nrhs, assign, partials, nchunks, slots);
    return cudaGetLastError();
}

cudaError_t zs_launch_relcorr(const double *partials, int nchunks, int nrhs, double *relcorr, const int *slots,
                              int nslot, cudaStream_t st) {
    const int t = nslot * nrhs;
    k_relcorr<<<(t + 127) / 128, 128, 0, st>>>(partials, nchunks, nrhs, relcorr, slots, nslot);
    return cudaGetLastError();
}

cudaError_t zs_launch_widen(const float2 *v, double2 *d, int64_t count, cudaStream_t st) {
    k_widen<<<grid1d(count, 256), 256, 0, st>>>(v, d, count);
    return cudaGetLastError();
}

cudaError_t zs_launch_narrow(const double2 *d, float2 *v, int64_t count, cudaStream_t st) {
    k_narrow<<<grid1d(count, 256), 256, 0, st>>>(d, v, count);
    return cudaGetLastError();
}

cudaError_t zs_launch_copy_z32_out(const float *z32, int64_t ld, int64_t plane, int64_t n, float *re, float *im,
                                   cudaStream_t st) {
    unsigned g = (unsigned)(n < 4096 ? n : 4096);
    if (g < 1) g = 1;
    k_copy_z32_out<<<g, 256, 0, st>>>(z32, ld, plane, n, re, im);
    return cudaGetLastError();
}
