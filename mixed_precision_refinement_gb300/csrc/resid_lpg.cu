// Residual computed directly from L, Psi and G for several frequencies in one
// pass (malusrfworks.com, "Solving Dense Matrices Fast in the Browser":
// section "Double-precision answers from a GPU without double precision",
// step 3, r = b - Z x in double precision, with Z in the form of section
// "Fewer frequency points: adaptive frequency sampling",
// Z(omega) = j*omega*L - j*Psi/omega + Zs(omega)*G, L, Psi, G independent of
// frequency):
//
//   r_f = b - ( j w_f (L x_f) - j (Psi x_f) / w_f + Zs_f (G x_f) )
//
// for the frequencies f of a batch, whose solutions x_f differ.  A warp takes
// one row of L, Psi and G and a group of up to kGroup frequencies: it streams
// the row once for the group and forms the three real-matrix-times-complex
// products of every frequency in float64 (DFMA), then combines them.  Where
// G is zero in all 128 entries of a warp step (all but three diagonals in the
// generated workloads) its products are skipped.  Compared with the float64
// GEMV over the assembled Z, this reads 24 n^2 bytes per group of kGroup
// frequencies instead of 16 n^2 per frequency, and does not need Z in float64
// at all; it makes 4-6 DFMA per entry and frequency instead of 2-4.
//
// Rounding: each of the three sums carries float64 rounding errors relative
// to its own terms (|L||x|, |Psi||x|, |G||x|), so the result is float64
// accurate relative to w|L||x| + |Psi||x|/w + |Zs||G||x| (which exceeds
// |Z||x| where the terms of Z cancel, near a resonance).  The quotient by w
// is a product with RN(1/w).
//
// Bound: the FP64 pipe at one right-hand side.
#include "common.cuh"

namespace {

constexpr int kThreads = 256;  // 8 warps, one row each
constexpr int kGroup = 4;      // frequencies per pass over a row

template <int NF>
__global__ void __launch_bounds__(kThreads)
k_residual_lpg(const double *__restrict__ Lm, const double *__restrict__ Pm, const double *__restrict__ Gm, int64_t n,
               const ZsSlotParam *__restrict__ params, const double2 *__restrict__ b, const double2 *__restrict__ x,
               int64_t x_stride, int rhs, float2 *__restrict__ out64, int64_t out64_stride,
               double2 *__restrict__ out128, int64_t out128_stride, const int *__restrict__ slots, int nslot,
               double one) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t row = (int64_t)blockIdx.x * (kThreads / 32) + warp;
    if (row >= n) return;  // whole warp
    const int g0 = blockIdx.y * NF;
    const int nf = min(NF, nslot - g0);
    int slot[NF];
    const double2 *xp[NF];
#pragma unroll
    for (int k = 0; k < NF; k++) {
        slot[k] = slots[g0 + (k < nf ? k : 0)];
        xp[k] = x + (int64_t)slot[k] * x_stride + (int64_t)rhs * n + lane;
    }
    // per frequency: L x, Psi x, G x (re, im)
    double yr[NF], yi[NF], pr[NF], pi[NF], qr[NF], qi[NF];
#pragma unroll
    for (int k = 0; k < NF; k++) yr[k] = yi[k] = pr[k] = pi[k] = qr[k] = qi[k] = 0.0;
    const double *lp = Lm + row * n + lane, *pp = Pm + row * n + lane, *gp = Gm + row * n + lane;
    const int nn = (int)n, nfull = nn >> 7;
#pragma unroll 1
    for (int s = 0; s < nfull; s++) {
        double l[4], p[4], g[4];
#pragma unroll
        for (int u = 0; u < 4; u++) {
            l[u] = __ldg(lp + 32 * u);
            p[u] = __ldg(pp + 32 * u);
            g[u] = __ldg(gp + 32 * u);
        }
        bool g0z = true;
#pragma unroll
        for (int u = 0; u < 4; u++) g0z = g0z && zs::is_zero(zs::bits_of(g[u]));
        const bool skip_g = __all_sync(0xffffffffu, g0z);
#pragma unroll
        for (int u = 0; u < 4; u++)
#pragma unroll
            for (int k = 0; k < NF; k++) {
                const double2 xv = __ldg(xp[k] + 32 * u);
                yr[k] = __fma_rn(l[u], xv.x, yr[k]);
                yi[k] = __fma_rn(l[u], xv.y, yi[k]);
                pr[k] = __fma_rn(p[u], xv.x, pr[k]);
                pi[k] = __fma_rn(p[u], xv.y, pi[k]);
                if (!skip_g) {
                    qr[k] = __fma_rn(g[u], xv.x, qr[k]);
                    qi[k] = __fma_rn(g[u], xv.y, qi[k]);
                }
            }
        lp += 128;
        pp += 128;
        gp += 128;
#pragma unroll
        for (int k = 0; k < NF; k++) xp[k] += 128;
    }
    for (int j = (nfull << 7) + lane; j < nn; j += 32) {
        const double l = __ldg(lp), p = __ldg(pp), g = __ldg(gp);
#pragma unroll
        for (int k = 0; k < NF; k++) {
            const double2 xv = __ldg(xp[k]);
            yr[k] = __fma_rn(l, xv.x, yr[k]);
            yi[k] = __fma_rn(l, xv.y, yi[k]);
            pr[k] = __fma_rn(p, xv.x, pr[k]);
            pi[k] = __fma_rn(p, xv.y, pi[k]);
            qr[k] = __fma_rn(g, xv.x, qr[k]);
            qi[k] = __fma_rn(g, xv.y, qi[k]);
            xp[k] += 32;
        }
        lp += 32;
        pp += 32;
        gp += 32;
    }
#pragma unroll
    for (int k = 0; k < NF; k++)
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            yr[k] = __fma_rn(__shfl_xor_sync(0xffffffffu, yr[k], o), one, yr[k]);
            yi[k] = __fma_rn(__shfl_xor_sync(0xffffffffu, yi[k], o), one, yi[k]);
            pr[k] = __fma_rn(__shfl_xor_sync(0xffffffffu, pr[k], o), one, pr[k]);
            pi[k] = __fma_rn(__shfl_xor_sync(0xffffffffu, pi[k], o), one, pi[k]);
            qr[k] = __fma_rn(__shfl_xor_sync(0xffffffffu, qr[k], o), one, qr[k]);
            qi[k] = __fma_rn(__shfl_xor_sync(0xffffffffu, qi[k], o), one, qi[k]);
        }
    // lane k writes frequency k: Z x = j w Y - j P / w + Zs Q
#pragma unroll
    for (int k = 0; k < NF; k++) {
        if (lane != k || k >= nf) continue;
        const ZsSlotParam sp = params[slot[k]];
        const double w = sp.omega, rw = sp.pad;  // pad = RN(1/omega)
        const double sre = -w * yi[k] + pi[k] * rw + (sp.zs_re * qr[k] - sp.zs_im * qi[k]);
        const double sim = w * yr[k] - pr[k] * rw + (sp.zs_re * qi[k] + sp.zs_im * qr[k]);
        const double2 bv = b[(int64_t)rhs * n + row];
        const double rr = bv.x - sre, ri = bv.y - sim;
        if (out64)
            out64[(int64_t)slot[k] * out64_stride + (int64_t)rhs * n + row] =
                make_float2(__double2float_rn(rr), __double2float_rn(ri));
        else
            out128[(int64_t)slot[k] * out128_stride + (int64_t)rhs * n + row] = make_double2(rr, ri);
    }
}

}  // namespace

cudaError_t zs_launch_residual_lpg(const double *L, const double *Psi, const double *G, int64_t n,
                                   const ZsSlotParam *params, const double2 *b, const double2 *x, int64_t x_stride,
                                   int nrhs, float2 *out_c64, int64_t out64_stride, double2 *out_c128,
                                   int64_t out128_stride, const int *slots, int nslot, cudaStream_t st) {
    if (nslot < 1 || nrhs < 1) return cudaErrorInvalidValue;
    const dim3 grid((unsigned)((n + kThreads / 32 - 1) / (kThreads / 32)), (unsigned)((nslot + kGroup - 1) / kGroup));
    for (int r = 0; r < nrhs; r++) {
        k_residual_lpg<kGroup><<<grid, kThreads, 0, st>>>(L, Psi, G, n, params, b, x, x_stride, r, out_c64,
                                                          out64_stride, out_c128, out128_stride, slots, nslot, 1.0);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}
