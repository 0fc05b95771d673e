// Fused assembly of Z(omega) = j*omega*L - j*Psi/omega + Zs(omega)*G
// (malusrfworks.com, "Solving Dense Matrices Fast in the Browser", section
// "Fewer frequency points: adaptive frequency sampling": the form of Z, with
// L, Psi, G independent of frequency).
//
// One pass reads L, Psi, G once and, for every frequency of the batch, writes
// the float64 matrix (interleaved complex, kept for the double-precision
// residual) and its round-to-nearest complex float32 copy (two planes, padded
// rows, to be factorised).  The float64 matrix is the correctly rounded
// evaluation of the formula in the order it is written -- Zs.re*G for the
// real part, (omega*L - Psi/omega) + Zs.im*G for the imaginary part, each
// operation rounded once -- computed with few FP64-pipe instructions, since
// that pipe, not HBM, bounds this kernel on GB300:
//  - Psi/omega: q0 = Psi*r with r = RN(1/omega) from the host, then one
//    correction q = RN(q0 + (Psi - omega*q0)*r) with the remainder exact by
//    FMA; this gives the correctly rounded quotient (P. Markstein, "Computation
//    of elementary functions on the IBM RISC System/6000 processor", IBM J.
//    Res. Dev. 1990, the division theorem); a zero q0 is returned as is, so a
//    -0 dividend keeps its sign;
//  - where G_ij = 0 for all 32 entries of a warp (all but three diagonals
//    in the generated workloads) Zs*G is an exact zero, so the products are
//    skipped and only the sign of zero they would produce is reproduced
//    (integer ops);
//  - zero tests and signs of zero are done on the 32-bit halves of the bit
//    pattern (see zs::bits_of), so no FP64 compare is issued;
//  - float64 -> float32 round-to-nearest-even is done on the integer bit
//    pattern; the hardware conversion (an FP64-pipe instruction) is kept for
//    subnormal results, overflow and NaN, in a function of its own so that it
//    is not evaluated for every entry;
//  - every remaining product and sum is issued as a fused multiply-add with
//    an exact second operand: RN(a*b) = fma(a, b, -0) and RN(a+b) =
//    fma(a, 1, b), identical to IEEE multiply and add including the signs of
//    zero.  The FP64 pipe of this GPU retires DFMA at its full rate (2 per SM
//    per clock) but DMUL and DADD several times more slowly.  The constants
//    -0 and 1 arrive as kernel arguments so that the compiler cannot fold
//    the fma back into a plain multiply or add.
//
// When asked (zexp != NULL), the kernel also records for every row and
// frequency the largest biased exponent of the row's float64 entries (real
// and imaginary parts): the scale of the fixed-point residual (resid_fx.cu).
//
// Bound: FP64 pipe (then HBM).  Algorithmic bytes per launch = 24 n^2 (read)
// + 24 n^2 per frequency (16 written as float64 complex, 8 as float32 complex).
//
// k_assemble32 forms the float32 planes alone, for sweeps whose residual
// never reads the float64 matrix (the tensor-core residual works from L, Psi
// and G; so does the grouped one).  It issues no float64 arithmetic per
// frequency: every input is split once into a pair of floats, hi = RN32(x)
// and lo = RN32(x - hi) (one DFMA for the exact difference, the roundings on
// the bit pattern), and per frequency the entry is formed in double-float
// arithmetic (products with their exact FMA errors, Knuth's TwoSum for the
// sums; T. J. Dekker, "A floating-point technique for extending the available
// precision", Numer. Math. 1971) and rounded once.  The pair carries about 44
// bits, so the result is RN32 of the float64 entry except where that entry
// lies within about 2^-20 of its float32 ulp from a rounding midpoint (or
// where omega L and Psi/omega cancel to that degree), where it may be one
// float32 ulp away: the factorisation of either matrix serves the
// refinement alike.  Bound: HBM, 24 n^2 read + 8 n^2 per frequency written.
#include "common.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kMaxSlots = 64;

__device__ __noinline__ float d2f_slow(double x) { return __double2float_rn(x); }

// round-to-nearest-even float64 -> float32 from the bit pattern
__device__ __forceinline__ float d2f_rn(double x) {
    const zs::Bits64 b = zs::bits_of(x);
    const unsigned hi = b.hi, lo = b.lo;
    if (zs::is_zero(b)) return __uint_as_float(hi & 0x80000000u);  // signed zero
    const unsigned e = (hi >> 20) & 0x7FFu;
    if (e < 897u || e > 1150u) return d2f_slow(x);  // subnormal result, overflow, inf/nan
    const unsigned fm = ((hi & 0xFFFFFu) << 3) | (lo >> 29);  // top 23 mantissa bits
    const unsigned rest = lo & 0x1FFFFFFFu;                    // 29 bits rounded away
    unsigned f = ((e - 896u) << 23) | fm;
    f += (rest > 0x10000000u || (rest == 0x10000000u && (fm & 1u))) ? 1u : 0u;  // carry may bump the exponent
    return __uint_as_float(f | (hi & 0x80000000u));
}

// Exact-as-IEEE product and sum on the FMA path (mz = -0.0, one = 1.0 at run time)
struct Fp64Ops {
    double mz, one;
    __device__ __forceinline__ double mul(double a, double b) const { return __fma_rn(a, b, mz); }
    __device__ __forceinline__ double add(double a, double b) const { return __fma_rn(a, one, b); }
    __device__ __forceinline__ double sub(double a, double b) const { return __fma_rn(zs::neg_bits(b), one, a); }
};

// Z64[e] and both float32 planes for one frequency.  warp_gzero: every
// entry this warp handles has G = +-0 (warp-uniform), so the Zs*G products
// are exact zeros and only their signs of zero are reproduced (integer ops);
// otherwise the whole warp multiplies, which gives the same result for the
// entries whose G is zero.  A per-entry choice would be if-converted and the
// FP64 pipe would issue the products for every warp with most lanes off.
__device__ __forceinline__ int one_entry(const ZsSlotParam &sp, double l, double p, double g, bool warp_gzero,
                                         bool valid, double2 *__restrict__ z64e, float *__restrict__ z32e,
                                         int64_t plane, const Fp64Ops &op) {
    const double w = sp.omega, r = sp.pad;  // pad holds RN(1/omega)
    const double q0 = op.mul(p, r);
    // RN(p / w); a zero first quotient is already exact (and keeps its sign)
    const double q = zs::sel_bits(zs::is_zero(zs::bits_of(q0)), q0, __fma_rn(__fma_rn(zs::neg_bits(w), q0, p), r, q0));
    const double t = op.sub(op.mul(w, l), q);
    double re, im;
    if (warp_gzero) {
        // Zs.re * (+-0) and t + Zs.im * (+-0): exact zeros; only signs of zero to reproduce
        const unsigned gs = zs::bits_of(g).hi & 0x80000000u;
        const unsigned zr = (zs::bits_of(sp.zs_re).hi & 0x80000000u) ^ gs;
        const unsigned zi = (zs::bits_of(sp.zs_im).hi & 0x80000000u) ^ gs;
        re = zs::double_of(0u, zr);
        const zs::Bits64 tb = zs::bits_of(t);
        // t + z: equals t unless t is a zero; (-0) + (-0) = -0, any other pair of zeros = +0
        im = zs::sel_bits(zs::is_zero(tb), zs::double_of(0u, tb.hi & zi), t);
    } else {
        re = op.mul(sp.zs_re, g);
        im = op.add(t, op.mul(sp.zs_im, g));
    }
    if (valid) {
        __stcs(z64e, make_double2(re, im));
        if (plane >= 0) {  // plane < 0: the float64 matrix only
            __stcs(z32e, d2f_rn(re));
            __stcs(z32e + plane, d2f_rn(im));
        }
    }
    // the larger biased exponent of the two parts (0 for an entry not stored)
    const int er = (int)((zs::bits_of(re).hi >> 20) & 0x7FFu), ei = (int)((zs::bits_of(im).hi >> 20) & 0x7FFu);
    return valid ? max(er, ei) : 0;
}

// per-slot exponent maxima of the current row: the warp's maximum, then one
// shared-memory atomic per warp
__device__ __forceinline__ void row_max(int *s_exp, int s, int e, int lane) {
    const int m = __reduce_max_sync(0xffffffffu, e);
    if (lane == 0) atomicMax(s_exp + s, m);
}

__global__ void __launch_bounds__(kThreads)
k_assemble(const double *__restrict__ L, const double *__restrict__ Psi, const double *__restrict__ G, int64_t n,
           int64_t r0, int64_t r1, const ZsSlotParam *__restrict__ params, int nslot, double2 *__restrict__ z64,
           int64_t z64_stride, float *__restrict__ z32, int64_t ld, int64_t plane, int64_t z32_stride,
           int *__restrict__ zexp, double mz, double one) {
    __shared__ ZsSlotParam sp[kMaxSlots];
    __shared__ int s_exp[kMaxSlots];
    const Fp64Ops op{mz, one};
    const int lane = threadIdx.x & 31;
    for (int s = threadIdx.x; s < nslot; s += blockDim.x) sp[s] = params[s];
    for (int s = threadIdx.x; s < kMaxSlots; s += blockDim.x) s_exp[s] = 0;
    __syncthreads();
    for (int64_t i = r0 + blockIdx.x; i < r1; i += gridDim.x) {
        const int64_t row = i * n, row32 = i * ld;
        // warp-uniform column walk (the tail lanes compute on a clamped index
        // and do not store), so the warp vote below always sees the full warp
        for (int64_t jw = threadIdx.x - lane; jw < n; jw += blockDim.x) {
            const int64_t jv = jw + lane;
            const bool valid = jv < n;
            const int64_t j = valid ? jv : n - 1;
            const int64_t e = row + j, o32 = row32 + j;
            const double l = __ldcs(L + e), p = __ldcs(Psi + e), g = __ldcs(G + e);
            const bool warp_gzero = __all_sync(0xffffffffu, zs::is_zero(zs::bits_of(g)));
            // four frequencies at a time: independent FP64 chains to cover the
            // unit's latency.  The per-frequency addresses advance by adding
            // the strides: 64-bit integer products would go to the FP64 pipe.
            double2 *zp = z64 + e;
            float *zq = z32 + o32;
            int s = 0;
#pragma unroll 1
            for (; s + 4 <= nslot; s += 4) {
                double2 *zp1 = zp + z64_stride, *zp2 = zp1 + z64_stride, *zp3 = zp2 + z64_stride;
                float *zq1 = zq + z32_stride, *zq2 = zq1 + z32_stride, *zq3 = zq2 + z32_stride;
                const int e0 = one_entry(sp[s], l, p, g, warp_gzero, valid, zp, zq, plane, op);
                const int e1 = one_entry(sp[s + 1], l, p, g, warp_gzero, valid, zp1, zq1, plane, op);
                const int e2 = one_entry(sp[s + 2], l, p, g, warp_gzero, valid, zp2, zq2, plane, op);
                const int e3 = one_entry(sp[s + 3], l, p, g, warp_gzero, valid, zp3, zq3, plane, op);
                if (zexp) {
                    row_max(s_exp, s, e0, lane);
                    row_max(s_exp, s + 1, e1, lane);
                    row_max(s_exp, s + 2, e2, lane);
                    row_max(s_exp, s + 3, e3, lane);
                }
                zp = zp3 + z64_stride;
                zq = zq3 + z32_stride;
            }
#pragma unroll 1
            for (; s < nslot; s++) {
                const int e = one_entry(sp[s], l, p, g, warp_gzero, valid, zp, zq, plane, op);
                if (zexp) row_max(s_exp, s, e, lane);
                zp += z64_stride;
                zq += z32_stride;
            }
        }
        if (zexp) {  // the row's maxima out, and reset for the next row
            __syncthreads();
            for (int s = threadIdx.x; s < nslot; s += blockDim.x) {
                zexp[(int64_t)s * n + i] = s_exp[s];
                s_exp[s] = 0;
            }
            __syncthreads();
        }
    }
}

// ---------------------------------------------------------------- float32 planes only

__device__ __noinline__ double f2d_slow(float x) { return (double)x; }

// float32 -> float64 from the bit pattern (the hardware conversion for
// subnormals, infinities and NaN)
__device__ __forceinline__ double f2d_bits(float x) {
    const unsigned u = __float_as_uint(x), e = (u >> 23) & 0xFFu;
    if ((u & 0x7FFFFFFFu) == 0u) return zs::double_of(0u, u);  // signed zero
    if (e == 0u || e == 0xFFu) return f2d_slow(x);
    return zs::double_of(u << 29, (u & 0x80000000u) | ((e + 896u) << 20) | ((u & 0x7FFFFFu) >> 3));
}

// x = hi + lo + O(2^-48 |x|): hi = RN32(x), lo = RN32(x - hi) (mone = -1 at run time)
struct F2 {
    float h, l;
};
__device__ __forceinline__ F2 split2(double x, double mone) {
    const float h = d2f_rn(x);
    return {h, d2f_rn(__fma_rn(f2d_bits(h), mone, x))};
}

// a * b for pairs, as a pair (h, l) with h = RN(ah bh)
__device__ __forceinline__ F2 mul2(F2 a, F2 b) {
    const float h = __fmul_rn(a.h, b.h);
    return {h, __fmaf_rn(a.h, b.l, __fmaf_rn(a.l, b.h, __fmaf_rn(a.h, b.h, -h)))};
}

// a + b for pairs (TwoSum of the high parts; the low parts added to its error)
__device__ __forceinline__ F2 add2(F2 a, F2 b) {
    const float s = __fadd_rn(a.h, b.h);
    const float v = __fsub_rn(s, a.h);
    const float e = __fadd_rn(__fsub_rn(a.h, __fsub_rn(s, v)), __fsub_rn(b.h, v));
    return {s, __fadd_rn(e, __fadd_rn(a.l, b.l))};
}
__device__ __forceinline__ F2 neg2(F2 a) { return {-a.h, -a.l}; }
// RN32 of the pair; a zero low part leaves the high part, sign of zero included
__device__ __forceinline__ float round2(F2 a) { return a.l == 0.f ? a.h : __fadd_rn(a.h, a.l); }

struct SlotF {  // a frequency's constants as pairs: omega, RN(1/omega), Zs
    F2 w, r, zr, zi;
};

// both float32 parts of one entry at one frequency; warp_gzero as in one_entry
__device__ __forceinline__ void one_entry32(const SlotF &sf, F2 l, F2 p, F2 g, bool warp_gzero, bool valid,
                                            float *__restrict__ z32e, int64_t plane) {
    const F2 t = add2(mul2(sf.w, l), neg2(mul2(sf.r, p)));  // omega L - Psi / omega
    float re, im;
    if (warp_gzero) {
        // Zs.re * (+-0) and t + Zs.im * (+-0): zeros, with the signs the
        // float64 formula gives them
        const unsigned gs = __float_as_uint(g.h) & 0x80000000u;
        const unsigned zr = (__float_as_uint(sf.zr.h) & 0x80000000u) ^ gs;
        const unsigned zi = (__float_as_uint(sf.zi.h) & 0x80000000u) ^ gs;
        re = __uint_as_float(zr);
        const float tv = round2(t);
        const unsigned tb = __float_as_uint(tv);
        im = (tb & 0x7FFFFFFFu) == 0u ? __uint_as_float(tb & zi) : tv;
    } else {
        re = round2(mul2(sf.zr, g));
        im = round2(add2(t, mul2(sf.zi, g)));
    }
    if (valid) {
        __stcs(z32e, re);
        __stcs(z32e + plane, im);
    }
}

__global__ void __launch_bounds__(kThreads)
k_assemble32(const double *__restrict__ L, const double *__restrict__ Psi, const double *__restrict__ G, int64_t n,
             int64_t r0, int64_t r1, const ZsSlotParam *__restrict__ params, int nslot, float *__restrict__ z32,
             int64_t ld, int64_t plane, int64_t z32_stride, double mone) {
    __shared__ SlotF sf[kMaxSlots];
    const int lane = threadIdx.x & 31;
    for (int s = threadIdx.x; s < nslot; s += blockDim.x) {
        const ZsSlotParam q = params[s];
        sf[s] = SlotF{split2(q.omega, mone), split2(q.pad, mone), split2(q.zs_re, mone), split2(q.zs_im, mone)};
    }
    __syncthreads();
    for (int64_t i = r0 + blockIdx.x; i < r1; i += gridDim.x) {
        const int64_t row = i * n, row32 = i * ld;
        for (int64_t jw = threadIdx.x - lane; jw < n; jw += blockDim.x) {
            const int64_t jv = jw + lane;
            const bool valid = jv < n;
            const int64_t j = valid ? jv : n - 1;
            const int64_t e = row + j;
            const double gd = __ldcs(G + e);
            const F2 l = split2(__ldcs(L + e), mone), p = split2(__ldcs(Psi + e), mone);
            const bool warp_gzero = __all_sync(0xffffffffu, zs::is_zero(zs::bits_of(gd)));
            const F2 g = warp_gzero ? F2{__uint_as_float(zs::bits_of(gd).hi & 0x80000000u), 0.f} : split2(gd, mone);
            float *zq = z32 + row32 + j;
            int s = 0;
#pragma unroll 1
            for (; s + 4 <= nslot; s += 4) {
                float *zq1 = zq + z32_stride, *zq2 = zq1 + z32_stride, *zq3 = zq2 + z32_stride;
                one_entry32(sf[s], l, p, g, warp_gzero, valid, zq, plane);
                one_entry32(sf[s + 1], l, p, g, warp_gzero, valid, zq1, plane);
                one_entry32(sf[s + 2], l, p, g, warp_gzero, valid, zq2, plane);
                one_entry32(sf[s + 3], l, p, g, warp_gzero, valid, zq3, plane);
                zq = zq3 + z32_stride;
            }
#pragma unroll 1
            for (; s < nslot; s++) {
                one_entry32(sf[s], l, p, g, warp_gzero, valid, zq, plane);
                zq += z32_stride;
            }
        }
    }
}

}  // namespace

cudaError_t zs_launch_assemble(const double *L, const double *Psi, const double *G, int64_t n, int64_t r0, int64_t r1,
                               const ZsSlotParam *params, int nslot, double2 *z64, int64_t z64_stride,
                               float *z32, int64_t ld, int64_t plane, int64_t z32_stride,
                               cudaStream_t st, int *zexp) {
    if (nslot > kMaxSlots || r0 < 0 || r1 > n || r0 > r1) return cudaErrorInvalidValue;
    if (r0 == r1) return cudaSuccess;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int64_t blocks = r1 - r0;
    int64_t cap = (int64_t)sms * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    k_assemble<<<(unsigned)blocks, kThreads, 0, st>>>(L, Psi, G, n, r0, r1, params, nslot, z64, z64_stride, z32, ld,
                                                      z32 ? plane : -1, z32_stride, zexp, -0.0, 1.0);
    return cudaGetLastError();
}

cudaError_t zs_launch_assemble32(const double *L, const double *Psi, const double *G, int64_t n, int64_t r0,
                                 int64_t r1, const ZsSlotParam *params, int nslot, float *z32, int64_t ld,
                                 int64_t plane, int64_t z32_stride, cudaStream_t st) {
    if (nslot > kMaxSlots || r0 < 0 || r1 > n || r0 > r1 || !z32) return cudaErrorInvalidValue;
    if (r0 == r1) return cudaSuccess;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int64_t blocks = r1 - r0;
    int64_t cap = (int64_t)sms * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    k_assemble32<<<(unsigned)blocks, kThreads, 0, st>>>(L, Psi, G, n, r0, r1, params, nslot, z32, ld, plane,
                                                        z32_stride, -1.0);
    return cudaGetLastError();
}
