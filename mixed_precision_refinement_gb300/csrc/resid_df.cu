// Double-float residual: r = b - Z x with the float64 Z and x represented as
// unevaluated sums of two float32 values and multiplied on the FP32 pipes
// (malusrfworks.com, "Solving Dense Matrices Fast in the Browser", section
// "The shader compiler was erasing the error": the GPU residual there is
// computed in double-float, two single-precision numbers giving about 48
// bits, with an error-free addition at its heart; the same section's last
// paragraph adds a start-up check of the GPU residual against the CPU's).
//
// On GB300 the FP64 unit is 64 times slower than the FP32 pipes, so the
// float64 residual is bound by FP64 arithmetic, not by HBM.  Here every
// float64 operand is split exactly from its bit pattern (hi = its top 24
// significand bits, lo = the remaining 29 rounded to 24), products are formed
// as p = hi*hi exactly (TwoProd by FMA) plus the cross terms, and each warp
// lane accumulates them in a float pair with an error-free TwoSum (Knuth's
// two-sum: s = a + b, e = (a - (s - (s - a))) + (b - (s - a))); the pairs are
// turned into float64 only for the final warp reduction.  Accuracy: about
// 2^-46 relative to sum |z||x| (no FP64 units involved except the reduction).
// No compiler reassociation: CUDA does not reorder float additions, and
// every operation of the error-free steps is written out.
//
// x is split once per refinement step by k_split_x (float4 per element:
// Re hi, Re lo, Im hi, Im lo).
#include "common.cuh"

namespace {

constexpr int kResThreads = 256;  // 8 warps, one row each

// z = hi + lo exactly up to the rounding of lo (relative 2^-47 of z).
__device__ __forceinline__ void split_f64(double z, float &hi, float &lo) {
    const zs::Bits64 b = zs::bits_of(z);
    const unsigned hw = b.hi, lw = b.lo;
    const unsigned e = (hw >> 20) & 0x7FFu;
    if (e >= 950u && e <= 1150u) {
        const unsigned sign = hw & 0x80000000u;
        hi = __uint_as_float(sign | ((e - 896u) << 23) | ((hw & 0xFFFFFu) << 3) | (lw >> 29));
        // remaining 29 significand bits, value rem * 2^(e - 1075)
        const float rem = __uint2float_rn(lw & 0x1FFFFFFFu);
        const float scale = __uint_as_float(sign | ((e - 1075u + 127u) << 23));
        lo = rem * scale;
    } else if (zs::is_zero(b)) {
        hi = __uint_as_float(hw & 0x80000000u);
        lo = 0.f;
    } else {  // outside the fast range: exact split with float64 arithmetic
        hi = __double2float_rn(z);
        lo = __double2float_rn(z - (double)hi);
    }
}

// acc (S, C) += a * b for double-float a, b
__device__ __forceinline__ void df_mac(float &S, float &C, float ah, float al, float bh, float bl) {
    const float p = ah * bh;
    float e = fmaf(ah, bh, -p);  // exact low part of ah*bh
    e = fmaf(ah, bl, e);
    e = fmaf(al, bh, e);
    const float s = S + p;
    const float bp = s - S;
    const float ap = s - bp;
    const float err = (S - ap) + (p - bp);
    C = C + (err + e);
    S = s;
}

__global__ void k_split_x(const double2 *__restrict__ x, int64_t x_stride, int64_t n, int nrhs,
                          float4 *__restrict__ xs, int64_t xs_stride, const int *__restrict__ slots) {
    const int slot = slots[blockIdx.y];
    const int64_t total = (int64_t)nrhs * n;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x) {
        const double2 v = x[(int64_t)slot * x_stride + e];
        float4 o;
        split_f64(v.x, o.x, o.y);
        split_f64(v.y, o.z, o.w);
        xs[(int64_t)slot * xs_stride + e] = o;
    }
}

// Two rows per warp: every split-x load serves both rows.
constexpr int kRowsPerWarp = 2;

template <int R>
__global__ void __launch_bounds__(kResThreads)
k_residual_df(const double2 *__restrict__ z64, int64_t z64_stride, int64_t n, const double2 *__restrict__ b,
              const float4 *__restrict__ xs, int64_t xs_stride, float2 *__restrict__ out64, int64_t out64_stride,
              double2 *__restrict__ out128, int64_t out128_stride, const int *__restrict__ slots) {
    const int slot = slots[blockIdx.y];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t row0 = ((int64_t)blockIdx.x * (kResThreads / 32) + warp) * kRowsPerWarp;
    if (row0 >= n) return;  // whole warp
    const int nrow = (int)zs::min64(kRowsPerWarp, n - row0);
    const double2 *zr[kRowsPerWarp];
#pragma unroll
    for (int q = 0; q < kRowsPerWarp; q++)
        zr[q] = z64 + (int64_t)slot * z64_stride + (row0 + (q < nrow ? q : 0)) * n;
    const float4 *xsl = xs + (int64_t)slot * xs_stride;
    float Sr[kRowsPerWarp][R], Cr[kRowsPerWarp][R], Si[kRowsPerWarp][R], Ci[kRowsPerWarp][R];
#pragma unroll
    for (int q = 0; q < kRowsPerWarp; q++)
#pragma unroll
        for (int r = 0; r < R; r++) Sr[q][r] = Cr[q][r] = Si[q][r] = Ci[q][r] = 0.f;
    int64_t base = 0;
    for (; base + 128 <= n; base += 128) {  // bound uniform across the warp
        const int64_t j = base + lane;
        double2 z[kRowsPerWarp][4];
#pragma unroll
        for (int q = 0; q < kRowsPerWarp; q++)
#pragma unroll
            for (int u = 0; u < 4; u++) z[q][u] = __ldcs(zr[q] + j + 32 * u);
        bool re0 = true;
#pragma unroll
        for (int q = 0; q < kRowsPerWarp; q++)
#pragma unroll
            for (int u = 0; u < 4; u++) re0 = re0 && zs::is_zero(zs::bits_of(z[q][u].x));
        const bool skip = __all_sync(0xffffffffu, re0);
#pragma unroll
        for (int u = 0; u < 4; u++) {
            float4 xv[R];
#pragma unroll
            for (int r = 0; r < R; r++) xv[r] = __ldg(xsl + r * n + j + 32 * u);
#pragma unroll
            for (int q = 0; q < kRowsPerWarp; q++) {
                float yh, yl, xh = 0.f, xl = 0.f;
                split_f64(z[q][u].y, yh, yl);
                if (!skip) split_f64(z[q][u].x, xh, xl);
#pragma unroll
                for (int r = 0; r < R; r++) {
                    // re += Re z Re x - Im z Im x ; im += Re z Im x + Im z Re x
                    df_mac(Sr[q][r], Cr[q][r], -yh, -yl, xv[r].z, xv[r].w);
                    df_mac(Si[q][r], Ci[q][r], yh, yl, xv[r].x, xv[r].y);
                    if (!skip) {
                        df_mac(Sr[q][r], Cr[q][r], xh, xl, xv[r].x, xv[r].y);
                        df_mac(Si[q][r], Ci[q][r], xh, xl, xv[r].z, xv[r].w);
                    }
                }
            }
        }
    }
    for (int64_t j = base + lane; j < n; j += 32) {
#pragma unroll
        for (int q = 0; q < kRowsPerWarp; q++) {
            const double2 z = __ldcs(zr[q] + j);
            float yh, yl, xh, xl;
            split_f64(z.y, yh, yl);
            split_f64(z.x, xh, xl);
#pragma unroll
            for (int r = 0; r < R; r++) {
                const float4 xv = __ldg(xsl + r * n + j);
                df_mac(Sr[q][r], Cr[q][r], -yh, -yl, xv.z, xv.w);
                df_mac(Si[q][r], Ci[q][r], yh, yl, xv.x, xv.y);
                df_mac(Sr[q][r], Cr[q][r], xh, xl, xv.x, xv.y);
                df_mac(Si[q][r], Ci[q][r], xh, xl, xv.z, xv.w);
            }
        }
    }
#pragma unroll
    for (int q = 0; q < kRowsPerWarp; q++) {
        double ar[R], ai[R];
#pragma unroll
        for (int r = 0; r < R; r++) {
            ar[r] = (double)Sr[q][r] + (double)Cr[q][r];
            ai[r] = (double)Si[q][r] + (double)Ci[q][r];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                ar[r] += __shfl_xor_sync(0xffffffffu, ar[r], o);
                ai[r] += __shfl_xor_sync(0xffffffffu, ai[r], o);
            }
        }
        const int64_t row = row0 + q;
        if (lane < R && q < nrow) {
            double vr = 0.0, vi = 0.0;
#pragma unroll
            for (int r = 0; r < R; r++)
                if (r == lane) {
                    vr = ar[r];
                    vi = ai[r];
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
}

template <int R>
void launch_df(const double2 *z64, int64_t z64_stride, int64_t n, const double2 *b, const float4 *xs, int64_t xs_stride,
               float2 *o64, int64_t o64s, double2 *o128, int64_t o128s, const int *slots, int nslot, cudaStream_t st) {
    const int64_t rows_per_cta = (kResThreads / 32) * kRowsPerWarp;
    dim3 grid((unsigned)((n + rows_per_cta - 1) / rows_per_cta), nslot);
    k_residual_df<R><<<grid, kResThreads, 0, st>>>(z64, z64_stride, n, b, xs, xs_stride, o64, o64s, o128, o128s,
                                                   slots);
}

// synthetic self-test system: entries (1 + u) 2^k with k in [-20, 20], positive,
// so that |Z x| = sum |z||x| and the comparison has no cancellation
__device__ __forceinline__ double hash_val(uint64_t i, uint32_t salt) {
    uint64_t h = i * 0x9E3779B97F4A7C15ull + salt;
    h ^= h >> 31;
    h *= 0xBF58476D1CE4E5B9ull;
    h ^= h >> 29;
    const double u = (double)(h >> 11) * (1.0 / 9007199254740992.0);
    const int k = (int)((h >> 3) % 41) - 20;
    return ldexp(1.0 + u, k);
}

__global__ void k_selftest_fill(double2 *__restrict__ z, double2 *__restrict__ x, int64_t n, int zero_re) {
    const int64_t total = n * n;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += (int64_t)gridDim.x * blockDim.x) {
        z[e] = make_double2(zero_re ? 0.0 : hash_val(e, 1u), hash_val(e, 2u));
        if (e < n) x[e] = make_double2(hash_val(e, 3u), 0.0);
    }
}

}  // namespace

cudaError_t zs_launch_split_x(const double2 *x, int64_t x_stride, int64_t n, int nrhs, float4 *xs, int64_t xs_stride,
                              const int *slots, int nslot, cudaStream_t st) {
    int64_t g = ((int64_t)nrhs * n + 255) / 256;
    if (g > 4096) g = 4096;
    k_split_x<<<dim3((unsigned)g, nslot), 256, 0, st>>>(x, x_stride, n, nrhs, xs, xs_stride, slots);
    return cudaGetLastError();
}

cudaError_t zs_launch_residual_df(const double2 *z64, int64_t z64_stride, int64_t n, const double2 *b, const float4 *xs,
                                  int64_t xs_stride, int nrhs, float2 *out_c64, int64_t out64_stride,
                                  double2 *out_c128, int64_t out128_stride, const int *slots, int nslot,
                                  cudaStream_t st) {
    int r0 = 0;
    while (r0 < nrhs) {
        const int left = nrhs - r0;
        const int R = left >= 4 ? 4 : left >= 2 ? 2 : 1;
        const double2 *bb = b + (int64_t)r0 * n;
        const float4 *xx = xs + (int64_t)r0 * n;
        float2 *o64 = out_c64 ? out_c64 + (int64_t)r0 * n : nullptr;
        double2 *o128 = out_c128 ? out_c128 + (int64_t)r0 * n : nullptr;
        switch (R) {
            case 4: launch_df<4>(z64, z64_stride, n, bb, xx, xs_stride, o64, out64_stride, o128, out128_stride, slots, nslot, st); break;
            case 2: launch_df<2>(z64, z64_stride, n, bb, xx, xs_stride, o64, out64_stride, o128, out128_stride, slots, nslot, st); break;
            default: launch_df<1>(z64, z64_stride, n, bb, xx, xs_stride, o64, out64_stride, o128, out128_stride, slots, nslot, st); break;
        }
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        r0 += R;
    }
    return cudaSuccess;
}

cudaError_t zs_launch_selftest_fill(double2 *z, double2 *x, int64_t n, int zero_re, cudaStream_t st) {
    int64_t g = (n * n + 255) / 256;
    if (g > 4096) g = 4096;
    k_selftest_fill<<<(unsigned)g, 256, 0, st>>>(z, x, n, zero_re);
    return cudaGetLastError();
}
