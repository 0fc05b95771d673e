// Float64-accurate residual r = b - Z x on the integer and FP32 pipes
// (malusrfworks.com, "Solving Dense Matrices Fast in the Browser", section
// "Double-precision answers from a GPU without double precision", step 3: the
// residual in double precision; the page's own GPU residual is double-float,
// section "The shader compiler was erasing the error").
//
// On GB300 the FP64 unit retires 2 DFMA per SM per clock, so a float64 GEMV
// at one right-hand side cannot read Z faster than about 0.7 of HBM, and a
// double-float one keeps only about 48 bits.  Here the float64 operands are
// turned exactly into fixed point and the products summed in integers:
//  - an entry a of row i (real or imaginary part, 53-bit significand m,
//    biased exponent e) becomes A = a * 2^(1094 - E), 72-bit fixed point
//    relative to the row's scale 2^(E - 1022) > |a| (E = the largest exponent
//    in the row, recorded by the assembly), as three signed 24-bit limbs
//    A = a0 2^48 + a1 2^24 + a2, cut out of m with 32-bit funnel shifts;
//  - x is split the same way once per refinement step, relative to the
//    largest exponent of the vector (k_split_fx);
//  - a x = A X 2^(E + Ex - 2188) and
//      A X = a0 x0 2^96 + (a0 x1 + a1 x0) 2^72 + (a0 x2 + a1 x1 + a2 x0) 2^48 + ...
//    The first two levels are summed exactly: each limb product is formed by
//    a 32-bit mul.lo and mul.hi pair and added into a 64-bit integer by an
//    add-with-carry chain (a 64-bit integer multiply would run on the FP64
//    pipe of this GPU).  The third level, 2^-48 of the scale, needs only a
//    few correct bits: it is summed in float32 from float copies of the limbs
//    (the entry's by an exact integer-to-float bit trick, after dropping two
//    low bits).  The terms below 2^48 are left out.
//  - each lane's sums become one float64 value, rounded once, at the end of
//    the row (and every kFlushSteps steps, so that no sum can overflow); the
//    32 lanes' values are added in float64 by a shuffle tree.
// Error: Z and x are truncated at 2^-72 of their scales, the dropped terms
// and the third level's float32 rounding stay below about 2^-62 of the
// product of the scales per entry, and the roundings to float64 add a few
// units of 2^-53 of the partial sums.  That is well inside the float64
// GEMV's bound n u (|Z| |x| + |b|) unless a row's products are spread over
// more than about 2^19 n in magnitude.
// Entries of Z equal to zero (or subnormal, below 2^-1022) contribute
// nothing; an infinite or NaN entry of Z or x makes the row's result NaN.
// In a warp step of 128 columns whose real parts are all exact zeros (Re Z =
// Zs.re G vanishes where G does) the real-part products are skipped.
//
// Hybrid: of every four 32-column sub-steps, the first NDF take float64
// products (DFMA) instead, so that the FP64 pipe and the integer pipes work
// side by side; the float64 partial sums join the fixed-point ones at the end.
//
// Bound: HBM (16 n^2 bytes per frequency).
#include "common.cuh"

namespace {

constexpr int kThreads = 256;  // 8 warps
constexpr unsigned kM24 = 0xFFFFFFu;
constexpr int kFlushSteps = 512;  // 128-column steps between flushes (2048 entries per lane)

struct Limbs {
    int a0, a1, a2;
};

// 32 bits of the 53-bit significand (mh:ml) starting at bit s >= 0 (zero from bit 53 on)
__device__ __forceinline__ unsigned sig_window(unsigned ml, unsigned mh, int s) {
    const unsigned lo = __funnelshift_rc(ml, mh, (unsigned)s);       // s < 32
    const unsigned hi = s < 64 ? (mh >> (unsigned)(s - 32)) : 0u;   // s >= 32
    return s < 32 ? lo : hi;
}

// Limbs of the float64 with bits (hi, lo) and biased exponent e (1 <= e <=
// E) relative to 2^(E - 1022): A = m * 2^(48 - t), t = E - e + 29 >= 29,
// truncated toward zero, with the sign of the value.
__device__ __forceinline__ Limbs fx_limbs(unsigned hi, unsigned lo, int e, int E) {
    const unsigned mh = (hi & 0xFFFFFu) | 0x100000u;
    const int t = E - e + 29;
    const unsigned a0 = sig_window(lo, mh, t);              // < 2^24 since t >= 29
    const unsigned a1 = sig_window(lo, mh, t - 24) & kM24;  // t - 24 >= 5
    const unsigned a2 = (t >= 48 ? sig_window(lo, mh, t - 48) : (lo << (unsigned)(48 - t))) & kM24;
    const int sg = (int)hi >> 31;  // 0 or -1: v ^ sg - sg is v or -v
    Limbs l;
    l.a0 = ((int)a0 ^ sg) - sg;
    l.a1 = ((int)a1 ^ sg) - sg;
    l.a2 = ((int)a2 ^ sg) - sg;
    return l;
}

// float(v / 4) for |v| < 2^24, truncating two bits: 1.5 * 2^23 + w is exact
// for |w| < 2^22, and subtracting 1.5 * 2^23 leaves w exactly
__device__ __forceinline__ float quarter_f(int v) { return __int_as_float(0x4B400000 + (v >> 2)) - 12582912.0f; }

struct LimbsF {  // the limbs / 4 as floats (third level only)
    float a0, a1, a2;
};

__device__ __forceinline__ LimbsF limbs_f(const Limbs &l) {
    return LimbsF{quarter_f(l.a0), quarter_f(l.a1), quarter_f(l.a2)};
}

// Sums of one output: S0 = sum a0 x0 and S1 = sum (a0 x1 + a1 x0), exact
// 64-bit integers as (hi:lo); S2 = sum (a0 x2 + a1 x1 + a2 x0) / 4 in float32.
// Value: S0 2^48 + S1 2^24 + 4 S2 (units 2^(E + Ex - 2188)).
struct FxAcc {
    unsigned l0, l1;
    int h0, h1;
    float s2;
};

// (hi:lo) += a * b exactly, |a|, |b| < 2^24
__device__ __forceinline__ void mac64(unsigned &lo, int &hi, int a, int b) {
    const unsigned pl = (unsigned)a * (unsigned)b;
    const int ph = __mulhi(a, b);
    asm("add.cc.u32 %0, %0, %2;\n\taddc.u32 %1, %1, %3;" : "+r"(lo), "+r"(hi) : "r"(pl), "r"(ph));
}

// x limbs of one part: ints x0, x1 (levels 0, 1) and floats x0, x1, x2 (level 2)
__device__ __forceinline__ void fx_mac(FxAcc &c, const Limbs &a, const LimbsF &af, int x0, int x1, float f0, float f1,
                                       float f2) {
    mac64(c.l0, c.h0, a.a0, x0);
    mac64(c.l1, c.h1, a.a0, x1);
    mac64(c.l1, c.h1, a.a1, x0);
    c.s2 = __fmaf_rn(af.a0, f2, c.s2);
    c.s2 = __fmaf_rn(af.a1, f1, c.s2);
    c.s2 = __fmaf_rn(af.a2, f0, c.s2);
}

__device__ __forceinline__ long long as64(unsigned lo, int hi) {
    return (long long)(((unsigned long long)(unsigned)hi << 32) | lo);
}

// The value of the sums, rounded to float64.  Ex == 2047 marks a non-finite
// x (the value is then NaN).
__device__ __forceinline__ double fx_value(const FxAcc &c, int E, int Ex) {
    if (Ex == 2047) return __longlong_as_double(0x7FF8000000000000ll);
    const double t = __fma_rn((double)as64(c.l0, c.h0), 281474976710656.0 /* 2^48 */,
                              __fma_rn((double)as64(c.l1, c.h1), 16777216.0 /* 2^24 */, 4.0 * (double)c.s2));
    return ldexp(t, E + Ex - 2140);
}

// x limbs in blocks of 128 columns (kXBlock bytes each): for the block's 128
// columns an int4 {re x0, re x1, im x0, im x1} each (the exact levels), then
// a float4 {re x0, re x1, re x2, im x0} and a float2 {im x1, im x2} each (the
// limbs as floats, exact, for the third level).
constexpr int kXBlock = 128 * 40;
__host__ __device__ inline int64_t fx_x_bytes(int64_t n) { return ((n + 127) / 128) * kXBlock; }

// x (c128, nrhs x n per slot) -> fixed-point limbs relative to the largest
// exponent of each right-hand side (layout above; xl_stride bytes per slot,
// fx_x_bytes(n) per right-hand side); xe[slot * nrhs_max + r] = that
// exponent (biased; 2047 if an entry is not finite).  One CTA per
// (right-hand side, slot).
__global__ void __launch_bounds__(kThreads)
k_split_fx(const double2 *__restrict__ x, int64_t x_stride, int64_t n, unsigned char *__restrict__ xl,
           int64_t xl_stride, int *__restrict__ xe, int nrhs_max, const int *__restrict__ slots) {
    __shared__ int s_e;
    const int r = blockIdx.x, slot = slots[blockIdx.y];
    const double2 *xv = x + (int64_t)slot * x_stride + (int64_t)r * n;
    int emax = 0;
    for (int64_t j = threadIdx.x; j < n; j += kThreads) {
        const double2 v = xv[j];
        const int er = (int)((zs::bits_of(v.x).hi >> 20) & 0x7FFu), ei = (int)((zs::bits_of(v.y).hi >> 20) & 0x7FFu);
        emax = max(emax, max(er, ei));
    }
    emax = __reduce_max_sync(0xffffffffu, emax);
    if (threadIdx.x == 0) s_e = 0;
    __syncthreads();
    if ((threadIdx.x & 31) == 0) atomicMax(&s_e, emax);
    __syncthreads();
    const int E = s_e;
    if (threadIdx.x == 0) xe[slot * nrhs_max + r] = E;
    unsigned char *o = xl + (int64_t)slot * xl_stride + (int64_t)r * fx_x_bytes(n);
    for (int64_t j = threadIdx.x; j < n; j += kThreads) {
        const double2 v = xv[j];
        const zs::Bits64 br = zs::bits_of(v.x), bi = zs::bits_of(v.y);
        const int er = (int)((br.hi >> 20) & 0x7FFu), ei = (int)((bi.hi >> 20) & 0x7FFu);
        Limbs lr{0, 0, 0}, li{0, 0, 0};
        if (E != 2047) {
            if (er != 0) lr = fx_limbs(br.hi, br.lo, er, E);
            if (ei != 0) li = fx_limbs(bi.hi, bi.lo, ei, E);
        }
        unsigned char *blk = o + (j >> 7) * kXBlock;
        const int c = (int)(j & 127);
        reinterpret_cast<int4 *>(blk)[c] = make_int4(lr.a0, lr.a1, li.a0, li.a1);
        reinterpret_cast<float4 *>(blk + 128 * 16)[c] = make_float4((float)lr.a0, (float)lr.a1, (float)lr.a2, (float)li.a0);
        reinterpret_cast<float2 *>(blk + 128 * 32)[c] = make_float2((float)li.a1, (float)li.a2);
    }
}

// One row of Z64 per warp (R right-hand sides) against x, 8 rows of one
// frequency per CTA.  The rows stream through a ring of kStages slots per
// warp, 128 columns each, and the matching block of x's limbs (and, when
// NDF > 0, of x itself) through a ring shared by the CTA; cp.async fills both
// kStages - 1 steps ahead.  One barrier per step makes every thread's copies
// of the step visible and frees the slot the next copy goes to.
// Of the four 32-column sub-steps of a step, the first NDF are multiplied in
// float64 (DFMA) and the others in fixed point.
constexpr int kStages = 3;
constexpr int kZSlot = 128 * (int)sizeof(double2);  // one warp's slot: 2 KB
template <int R, int NDF>
struct FxSmem {
    static constexpr int kXSlot = R * (kXBlock + (NDF > 0 ? kZSlot : 0));  // x blocks of one step
    static constexpr size_t bytes = (size_t)kStages * ((kThreads / 32) * kZSlot + kXSlot);
};

template <int R, int NDF>
__global__ void __launch_bounds__(kThreads, R == 1 ? 3 : (R == 2 ? 2 : 1))
k_residual_fx(const double2 *__restrict__ z64, int64_t z64_stride, const int *__restrict__ zexp, int64_t n,
              const double2 *__restrict__ b, const double2 *__restrict__ x, int64_t x_stride,
              const unsigned char *__restrict__ xl, int64_t xl_stride, const int *__restrict__ xe, int nrhs_max,
              float2 *__restrict__ out64, int64_t out64_stride, double2 *__restrict__ out128, int64_t out128_stride,
              const int *__restrict__ slots, double one) {
    constexpr int kXSlot = FxSmem<R, NDF>::kXSlot;
    extern __shared__ __align__(16) unsigned char sm[];
    unsigned char *const zring = sm;                                        // [stage][warp][128] double2
    unsigned char *const xring = sm + kStages * (kThreads / 32) * kZSlot;   // [stage][kXSlot]
    const uint32_t zring_a = (uint32_t)__cvta_generic_to_shared(zring), xring_a = (uint32_t)__cvta_generic_to_shared(xring);
    const int slot = slots[blockIdx.y];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t row = (int64_t)blockIdx.x * (kThreads / 32) + warp;
    const bool live = row < n;                // rows past the end take part in the copies and barriers only
    const int64_t rowc = live ? row : n - 1;
    const double2 *zr = z64 + (int64_t)slot * z64_stride + rowc * n;
    const int E = zexp[(int64_t)slot * n + rowc];
    const unsigned char *xs = xl + (int64_t)slot * xl_stride;
    const double2 *xd = x + (int64_t)slot * x_stride;
    const int64_t xrb = fx_x_bytes(n);
    int Ex[R];
#pragma unroll
    for (int r = 0; r < R; r++) Ex[r] = xe[slot * nrhs_max + r];
    // are: sum Re z Re x; aii: sum Im z Im x (subtracted at the flush); aim: the imaginary part
    FxAcc are[R], aii[R], aim[R];
    double dre[R], dim[R];
#pragma unroll
    for (int r = 0; r < R; r++) {
        are[r] = aii[r] = aim[r] = FxAcc{0u, 0u, 0, 0, 0.f};
        dre[r] = dim[r] = 0.0;
    }
    auto flush = [&]() {
#pragma unroll
        for (int r = 0; r < R; r++) {
            dre[r] = __fma_rn(fx_value(are[r], E, Ex[r]), one, dre[r]);
            dre[r] = __fma_rn(zs::neg_bits(fx_value(aii[r], E, Ex[r])), one, dre[r]);
            dim[r] = __fma_rn(fx_value(aim[r], E, Ex[r]), one, dim[r]);
            are[r] = aii[r] = aim[r] = FxAcc{0u, 0u, 0, 0, 0.f};
        }
    };
    // one entry z in fixed point; xb[r] = the x limb block of right-hand side r, c = column in it
    auto entry = [&](double2 z, const unsigned char *const (&xb)[R], int c, bool with_re) {
        const zs::Bits64 bi = zs::bits_of(z.y), br = zs::bits_of(z.x);
        const int ei = (int)((bi.hi >> 20) & 0x7FFu);
        const int er = with_re ? (int)((br.hi >> 20) & 0x7FFu) : 0;
        if (ei == 0 && er == 0) return;
        int4 xi[R];
        float4 f4[R];
        float2 f2[R];
#pragma unroll
        for (int r = 0; r < R; r++) {
            xi[r] = reinterpret_cast<const int4 *>(xb[r])[c];
            f4[r] = reinterpret_cast<const float4 *>(xb[r] + 128 * 16)[c];
            f2[r] = reinterpret_cast<const float2 *>(xb[r] + 128 * 32)[c];
        }
        if (ei != 0) {
            const Limbs l = fx_limbs(bi.hi, bi.lo, ei, E);
            const LimbsF lf = limbs_f(l);
#pragma unroll
            for (int r = 0; r < R; r++) {
                fx_mac(aii[r], l, lf, xi[r].z, xi[r].w, f4[r].w, f2[r].x, f2[r].y);  // Im z Im x (re -=)
                fx_mac(aim[r], l, lf, xi[r].x, xi[r].y, f4[r].x, f4[r].y, f4[r].z);  // im += Im z Re x
            }
        }
        if (er != 0) {
            const Limbs l = fx_limbs(br.hi, br.lo, er, E);
            const LimbsF lf = limbs_f(l);
#pragma unroll
            for (int r = 0; r < R; r++) {
                fx_mac(are[r], l, lf, xi[r].x, xi[r].y, f4[r].x, f4[r].y, f4[r].z);    // re += Re z Re x
                fx_mac(aim[r], l, lf, xi[r].z, xi[r].w, f4[r].w, f2[r].x, f2[r].y);    // im += Re z Im x
            }
        }
    };
    const int nn = (int)n, nfull = nn >> 7;
    // copies of step st into stage st % kStages: the warp's 128 entries of its
    // row (each lane its own four), and the CTA's x blocks (all threads)
    auto issue = [&](int st) {
        if (st < nfull) {
            const int stage = st % kStages;
            const uint32_t zdst = zring_a + (uint32_t)((stage * (kThreads / 32) + warp) * kZSlot + lane * 16);
            const double2 *zsrc = zr + ((int64_t)st << 7) + lane;
#pragma unroll
            for (int u = 0; u < 4; u++)
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(zdst + u * 512), "l"(zsrc + 32 * u)
                             : "memory");
            const uint32_t xdst = xring_a + (uint32_t)(stage * kXSlot);
            constexpr int kChunksPerRhs = (kXBlock + (NDF > 0 ? kZSlot : 0)) / 16;
            for (int q = tid; q < R * kChunksPerRhs; q += kThreads) {
                const int r = q / kChunksPerRhs, k = q - r * kChunksPerRhs;
                const unsigned char *src = k < kXBlock / 16
                    ? xs + r * xrb + (int64_t)st * kXBlock + 16 * k
                    : reinterpret_cast<const unsigned char *>(xd + (int64_t)r * n + ((int64_t)st << 7)) +
                          16 * (k - kXBlock / 16);
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(xdst + (uint32_t)(r * (kXSlot / R) + 16 * k)),
                             "l"(src)
                             : "memory");
            }
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };
#pragma unroll
    for (int st = 0; st < kStages - 1; st++) issue(st);
    int since = 0;
#pragma unroll 1
    for (int s = 0; s < nfull; s++) {
        asm volatile("cp.async.wait_group %0;" ::"n"(kStages - 2) : "memory");
        __syncthreads();
        issue(s + kStages - 1);
        const int stage = s % kStages;
        const double2 *cur = reinterpret_cast<const double2 *>(zring + (stage * (kThreads / 32) + warp) * kZSlot) + lane;
        const unsigned char *xb[R];
#pragma unroll
        for (int r = 0; r < R; r++) xb[r] = xring + stage * kXSlot + r * (kXSlot / R);
        double2 z[4];
#pragma unroll
        for (int u = 0; u < 4; u++) z[u] = cur[32 * u];
        bool re0 = true;
#pragma unroll
        for (int u = 0; u < 4; u++) re0 = re0 && zs::is_zero(zs::bits_of(z[u].x));
        const bool with_re = !__all_sync(0xffffffffu, re0);
#pragma unroll
        for (int u = 0; u < 4; u++) {
            if (u < NDF) {  // float64 products, x from the staged copy
#pragma unroll
                for (int r = 0; r < R; r++) {
                    const double2 xv = reinterpret_cast<const double2 *>(xb[r] + kXBlock)[lane + 32 * u];
                    dre[r] = __fma_rn(zs::neg_bits(z[u].y), xv.y, dre[r]);
                    dim[r] = __fma_rn(z[u].y, xv.x, dim[r]);
                    if (with_re) {
                        dre[r] = __fma_rn(z[u].x, xv.x, dre[r]);
                        dim[r] = __fma_rn(z[u].x, xv.y, dim[r]);
                    }
                }
            } else {
                entry(z[u], xb, lane + 32 * u, with_re);
            }
        }
        if (++since == kFlushSteps) {
            since = 0;
            flush();
        }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    if (!live) return;  // no barrier follows
    {  // the last (partial) block of columns, straight from global memory
        const unsigned char *xb[R];
#pragma unroll
        for (int r = 0; r < R; r++) xb[r] = xs + r * xrb + (int64_t)nfull * kXBlock;
        for (int j = (nfull << 7) + lane; j < nn; j += 32) entry(__ldcs(zr + j), xb, j & 127, true);
    }
    flush();
    const double nan = __longlong_as_double(0x7FF8000000000000ll);
    const bool bad = E == 2047;  // an infinite or NaN entry in the row
    double vr[R], vi[R];
#pragma unroll
    for (int r = 0; r < R; r++) {
        vr[r] = bad ? nan : dre[r];
        vi[r] = bad ? nan : dim[r];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            vr[r] = __fma_rn(__shfl_xor_sync(0xffffffffu, vr[r], o), one, vr[r]);
            vi[r] = __fma_rn(__shfl_xor_sync(0xffffffffu, vi[r], o), one, vi[r]);
        }
    }
    if (lane < R) {
        double sr = 0.0, si = 0.0;
#pragma unroll
        for (int r = 0; r < R; r++)
            if (r == lane) {
                sr = vr[r];
                si = vi[r];
            }
        const double2 bv = b[(int64_t)lane * n + row];
        // b - s as fma(-s, 1, b): the same rounding as the subtraction
        const double rr = __fma_rn(zs::neg_bits(sr), one, bv.x), ri = __fma_rn(zs::neg_bits(si), one, bv.y);
        if (out64)
            out64[(int64_t)slot * out64_stride + (int64_t)lane * n + row] =
                make_float2(__double2float_rn(rr), __double2float_rn(ri));
        else
            out128[(int64_t)slot * out128_stride + (int64_t)lane * n + row] = make_double2(rr, ri);
    }
}

template <int R, int NDF>
cudaError_t launch_fx_ndf(dim3 grid, cudaStream_t st, const double2 *z64, int64_t z64_stride, const int *zexp,
                          int64_t n, const double2 *b, const double2 *x, int64_t x_stride, const unsigned char *xl,
                          int64_t xl_stride, const int *xe, int nrhs_max, float2 *o64, int64_t o64s, double2 *o128,
                          int64_t o128s, const int *slots) {
    constexpr size_t kBytes = FxSmem<R, NDF>::bytes;
    // once per process and instance (thread-safe initialisation of a local static)
    static const cudaError_t attr =
        cudaFuncSetAttribute(k_residual_fx<R, NDF>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kBytes);
    if (attr != cudaSuccess) return attr;
    k_residual_fx<R, NDF><<<grid, kThreads, kBytes, st>>>(z64, z64_stride, zexp, n, b, x, x_stride, xl, xl_stride, xe,
                                                          nrhs_max, o64, o64s, o128, o128s, slots, 1.0);
    return cudaGetLastError();
}

template <int R>
cudaError_t launch_fx(const double2 *z64, int64_t z64_stride, const int *zexp, int64_t n, const double2 *b,
                      const double2 *x, int64_t x_stride, const unsigned char *xl, int64_t xl_stride, const int *xe,
                      int nrhs_max, float2 *o64, int64_t o64s, double2 *o128, int64_t o128s, const int *slots,
                      int nslot, int ndf, cudaStream_t st) {
    const dim3 grid((unsigned)((n + kThreads / 32 - 1) / (kThreads / 32)), nslot);
    switch (ndf) {
        case 0: return launch_fx_ndf<R, 0>(grid, st, z64, z64_stride, zexp, n, b, x, x_stride, xl, xl_stride, xe, nrhs_max, o64, o64s, o128, o128s, slots);
        case 1: return launch_fx_ndf<R, 1>(grid, st, z64, z64_stride, zexp, n, b, x, x_stride, xl, xl_stride, xe, nrhs_max, o64, o64s, o128, o128s, slots);
        case 2: return launch_fx_ndf<R, 2>(grid, st, z64, z64_stride, zexp, n, b, x, x_stride, xl, xl_stride, xe, nrhs_max, o64, o64s, o128, o128s, slots);
        default: return launch_fx_ndf<R, 3>(grid, st, z64, z64_stride, zexp, n, b, x, x_stride, xl, xl_stride, xe, nrhs_max, o64, o64s, o128, o128s, slots);
    }
}

}  // namespace

int64_t zs_fx_x_bytes(int64_t n) { return fx_x_bytes(n); }

cudaError_t zs_launch_split_fx(const double2 *x, int64_t x_stride, int64_t n, int nrhs, unsigned char *xl,
                               int64_t xl_stride, int *xe, int nrhs_max, const int *slots, int nslot, cudaStream_t st) {
    if (nrhs < 1 || nrhs > nrhs_max || nslot < 1) return cudaErrorInvalidValue;
    k_split_fx<<<dim3((unsigned)nrhs, (unsigned)nslot), kThreads, 0, st>>>(x, x_stride, n, xl, xl_stride, xe, nrhs_max,
                                                                            slots);
    return cudaGetLastError();
}

cudaError_t zs_launch_residual_fx(const double2 *z64, int64_t z64_stride, const int *zexp, int64_t n, const double2 *b,
                                  const double2 *x, int64_t x_stride, const unsigned char *xl, int64_t xl_stride,
                                  const int *xe, int nrhs_max, int nrhs, float2 *out_c64, int64_t out64_stride,
                                  double2 *out_c128, int64_t out128_stride, const int *slots, int nslot, int ndf,
                                  cudaStream_t st) {
    if (ndf < 0 || ndf > 3 || !zexp) return cudaErrorInvalidValue;
    int r0 = 0;
    while (r0 < nrhs) {
        const int left = nrhs - r0;
        const int R = left >= 4 ? 4 : left >= 2 ? 2 : 1;
        const double2 *bb = b + (int64_t)r0 * n;
        const unsigned char *xx = xl + (int64_t)r0 * fx_x_bytes(n);
        const double2 *xr = x + (int64_t)r0 * n;
        const int *ee = xe + r0;
        float2 *o64 = out_c64 ? out_c64 + (int64_t)r0 * n : nullptr;
        double2 *o128 = out_c128 ? out_c128 + (int64_t)r0 * n : nullptr;
        cudaError_t e;
        switch (R) {
            case 4: e = launch_fx<4>(z64, z64_stride, zexp, n, bb, xr, x_stride, xx, xl_stride, ee, nrhs_max, o64, out64_stride, o128, out128_stride, slots, nslot, ndf, st); break;
            case 2: e = launch_fx<2>(z64, z64_stride, zexp, n, bb, xr, x_stride, xx, xl_stride, ee, nrhs_max, o64, out64_stride, o128, out128_stride, slots, nslot, ndf, st); break;
            default: e = launch_fx<1>(z64, z64_stride, zexp, n, bb, xr, x_stride, xx, xl_stride, ee, nrhs_max, o64, out64_stride, o128, out128_stride, slots, nslot, ndf, st); break;
        }
        if (e != cudaSuccess) return e;
        r0 += R;
    }
    return cudaSuccess;
}
