// Fused assembly of Z(omega) = j*omega*L - j*Psi/omega + Zs(omega)*G
// (malusrfworks.com, "Solving Dense Matrices Fast in the Browser", section
// "Fewer frequency points: adaptive frequency sampling": the form of Z, with
// L, Psi, G independent of frequency).
//
// One pass reads L, Psi, G once and, for every frequency of the batch, writes
// the float64 matrix (interleaved complex, kept for the double-precision
// residual) and its round-to-nearest complex float32 copy (two planes, padded
// rows, to be factorised).  Every float64 operation is rounded separately and
// in the order the formula is written -- Zs.re*G for the real part,
// (omega*L - Psi/omega) + Zs.im*G for the imaginary part -- so the float64
// matrix is the correctly rounded evaluation of that expression.
//
// Bound: HBM.  Algorithmic bytes per launch = 24 n^2 (read) + 24 n^2 per
// frequency (16 written as float64 complex, 8 as float32 complex).
#include "common.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kMaxSlots = 64;

__global__ void __launch_bounds__(kThreads)
k_assemble(const double *__restrict__ L, const double *__restrict__ Psi,
           const double *__restrict__ G, int64_t n, const ZsSlotParam *__restrict__ params,
           int nslot, double2 *__restrict__ z64, int64_t z64_stride, float *__restrict__ z32,
           int64_t ld, int64_t plane, int64_t z32_stride) {
    __shared__ ZsSlotParam sp[kMaxSlots];
    for (int s = threadIdx.x; s < nslot; s += blockDim.x) sp[s] = params[s];
    __syncthreads();
    for (int64_t i = blockIdx.x; i < n; i += gridDim.x) {
        const int64_t row = i * n, row32 = i * ld;
        for (int64_t j = threadIdx.x; j < n; j += blockDim.x) {
            const int64_t e = row + j, o32 = row32 + j;
            const double l = __ldcs(L + e), p = __ldcs(Psi + e), g = __ldcs(G + e);
#pragma unroll 1
            for (int s = 0; s < nslot; s++) {
                const double w = sp[s].omega;
                const double re = __dmul_rn(sp[s].zs_re, g);
                const double im = __dadd_rn(__dsub_rn(__dmul_rn(w, l), __ddiv_rn(p, w)),
                                            __dmul_rn(sp[s].zs_im, g));
                __stcs(z64 + s * z64_stride + e, make_double2(re, im));
                float *zr = z32 + s * z32_stride;
                __stcs(zr + o32, __double2float_rn(re));
                __stcs(zr + plane + o32, __double2float_rn(im));
            }
        }
    }
}

}  // namespace

cudaError_t zs_launch_assemble(const double *L, const double *Psi, const double *G, int64_t n,
                               const ZsSlotParam *params, int nslot, double2 *z64, int64_t z64_stride,
                               float *z32, int64_t ld, int64_t plane, int64_t z32_stride,
                               cudaStream_t st) {
    if (nslot > kMaxSlots) return cudaErrorInvalidValue;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int64_t blocks = n;
    int64_t cap = (int64_t)sms * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    k_assemble<<<(unsigned)blocks, kThreads, 0, st>>>(L, Psi, G, n, params, nslot, z64, z64_stride,
                                                      z32, ld, plane, z32_stride);
    return cudaGetLastError();
}
