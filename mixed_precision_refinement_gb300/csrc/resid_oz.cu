// Residual r = b - Z x in float64-class accuracy on the bf16 tensor cores
// (malusrfworks.com, "Solving Dense Matrices Fast in the Browser": section
// "Double-precision answers from a GPU without double precision", step 3,
// the residual in double precision, with Z in the form of section "Fewer
// frequency points: adaptive frequency sampling",
// Z(omega) = j*omega*L - j*Psi/omega + Zs(omega)*G, L, Psi, G real and
// independent of frequency).
//
// The products L x_f, Psi x_f, G x_f of all the batch's frequencies f (and
// right-hand sides) are one real matrix product
//     Y = A' X,   A' = [L; Psi; G] (3n x n),   X = [Re x_f, Im x_f, ...] (n x ncol),
// a dense contraction, which the 5th-generation tensor cores run at
// thousands of times the rate of this GPU's FP64 pipe.  Float64 accuracy
// comes from error-free splitting (the Ozaki scheme: K. Ozaki, T. Ogita,
// S. Oishi, S. M. Rump, "Error-free transformations of matrix multiplication
// by using fast routines of matrix multiplication and its applications",
// Numer. Algorithms 59, 2012; on tensor cores: D. Mukunoki, K. Ozaki,
// T. Ogita, T. Imamura, "DGEMM using Tensor Cores, and Its Accurate and
// Reproducible Versions", ISC 2020):
//
//  - every row i of A' (scale 2^Ea_i from its largest exponent) and every
//    column c of X (scale 2^Ex_c) is written as 8 balanced base-2^7 digits,
//    a = 2^Ea sum_k d_k 2^(7(7-k)), |d_k| <= 64 -- 56 bits, the float64
//    significand of the row's (column's) largest entries and those within
//    2^-3 of it exactly, smaller ones to 2^-55 of the largest; digits are
//    small integers, exact in bf16;
//  - a digit product is exact in the MMA; the products of level
//    l = k_a + k_x (l < 8; higher levels weigh below 2^-56) are summed by the
//    MMA into one fp32 accumulator block.  At most 8 digit pairs per level and
//    128 K per flush give |sum| <= 8 * 128 * 64^2 = 2^22: every partial sum is
//    an integer below 2^24, exact in fp32 whatever the summation order;
//  - every 128 K the eight level blocks are read out of TMEM, turned into
//    integers and gathered exactly into two 64-bit integers per output
//    (levels 0-3 and 4-7, 7 bits apart), which accumulate over the whole K
//    range without rounding; at the end each output is rounded once to
//    float64 and scaled by 2^(Ea + Ex).
//
// Per level, one tcgen05.mma covers every digit pair at once: the MMA of A
// digit k_a has B = [X digit 0 | X digit 1 | ... | X digit 7-k_a] (N = 32 per
// digit) and writes from TMEM column 32 k_a on, so X digit k_x lands in level
// block k_a + k_x.  Eight MMAs (N = 256, 224, ..., 32) per 16 K.
//
// The combination r_f = b - (j w Lx_f - j (Psi x_f) / w + Zs_f G x_f) is that
// of the L, Psi, G residual: accurate relative to
// w|L||x| + |Psi||x|/w + |Zs||G||x|; on top, the splitting's representation
// error is below 2^-54 of each row's and column's largest entry.
//
// Bound: HBM (the 16 bytes of digits per entry of L, Psi, G, read once per
// evaluation for all frequencies of the batch); the digits of A' are formed
// once per sweep, those of X per evaluation.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <algorithm>

#include "common.cuh"

namespace {

constexpr int kDig = 8;         // digits per value
constexpr int TM = 128;         // rows of A' per tile (TMEM lanes)
constexpr int W = 32;           // X columns per group (N of one digit block)
constexpr int KS = 32;          // K per stage: one 64-byte swizzle row of bf16 (two MMA K steps)
constexpr int KCH = 128;        // K per accumulator flush
constexpr int kStepsPerCh = KCH / KS;
constexpr int A_SLICE = TM * KS * 2;        // 8 KB: one digit plane of the A tile
constexpr int X_SLICE = W * KS * 2;         // 2 KB
constexpr int A_STAGE = kDig * A_SLICE;     // 64 KB
constexpr int STAGE = A_STAGE + kDig * X_SLICE;  // 80 KB
constexpr int STAGES = 2;
constexpr int SMEM = STAGES * STAGE + 1024;  // + alignment slack
constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + 32 * kEpiWarps;  // warp 0 TMA, warp 1 MMA and TMEM, warps 2-9 epilogue
constexpr uint32_t TMEM_COLS = 512;          // two accumulators of 8 level blocks x 32 columns
constexpr uint32_t kWaitLimit = 1u << 19;    // try_wait polls before a wait gives up (about a second)
constexpr unsigned kSite = 0x60u;            // wait-site code of this kernel (bits 8-15 of the status word)

// ------------------------------------------------------------------ digits

// Largest biased exponent of a float64 (1 for subnormals and zero), and
// whether it is finite.
__device__ __forceinline__ int exp_of(double a, bool &finite) {
    const zs::Bits64 b = zs::bits_of(a);
    const int e = (int)((b.hi >> 20) & 0x7FFu);
    finite = e != 0x7FF;
    return e == 0 ? 1 : e;
}

// Balanced base-2^7 digits of a at scale q (q >= the biased exponent of a):
// a = 2^(q - 1077) sum_k d[k] 2^(7 (7 - k)) + e, |e| <= 2^(q - 1078),
// |d[k]| <= 64.  Integer operations only.
__device__ __forceinline__ void digits_of(double a, int q, int (&d)[kDig]) {
    const zs::Bits64 b = zs::bits_of(a);
    const int ef = (int)((b.hi >> 20) & 0x7FFu);
    uint64_t m = ((uint64_t)(b.hi & 0xFFFFFu) << 32) | b.lo;
    int e = ef;
    if (ef) m |= 1ull << 52;
    else e = 1;
    // v = round(m 2^(e - q + 2)), an integer below 2^55
    const int sh = q - e - 2;
    uint64_t v;
    if (sh <= 0) v = m << (-sh);
    else if (sh < 60) v = (m + (1ull << (sh - 1))) >> sh;
    else v = 0;
#pragma unroll
    for (int k = kDig - 1; k > 0; k--) {
        int t = (int)(v & 127u);
        v >>= 7;
        if (t >= 64) {
            t -= 128;
            v += 1;
        }
        d[k] = t;
    }
    d[0] = (int)v;  // <= 64
    if (b.hi >> 31) {
#pragma unroll
        for (int k = 0; k < kDig; k++) d[k] = -d[k];
    }
}

__device__ __forceinline__ uint32_t pack_bf16(int lo, int hi) {
    const __nv_bfloat16 a = __float2bfloat16_rn((float)lo), b = __float2bfloat16_rn((float)hi);
    return (uint32_t)__bfloat16_as_ushort(a) | ((uint32_t)__bfloat16_as_ushort(b) << 16);
}

// Eight consecutive values (entries j0..j0+7 of a row or column; those at
// j >= n are zero) as digit planes: plane k gets 8 bf16 (16 bytes) at dst + k * plane.
__device__ __forceinline__ void write_digits8(const double (&a)[8], int q, __nv_bfloat16 *dst, int64_t plane) {
    int d[8][kDig];
#pragma unroll
    for (int u = 0; u < 8; u++) digits_of(a[u], q, d[u]);
#pragma unroll
    for (int k = 0; k < kDig; k++) {
        uint4 w;
        w.x = pack_bf16(d[0][k], d[1][k]);
        w.y = pack_bf16(d[2][k], d[3][k]);
        w.z = pack_bf16(d[4][k], d[5][k]);
        w.w = pack_bf16(d[6][k], d[7][k]);
        *reinterpret_cast<uint4 *>(dst + (int64_t)k * plane) = w;
    }
}

// Tile-major layout of A's digits: unit (row tile t, K chunk c) holds the 8
// planes of 128 rows x 128 K, 256 KB contiguous, so that the product streams
// whole units from HBM: element (row, j) of plane p sits at
// ((((t nch + c) 8 + p) 128 + row % 128) 128 + j % 128).  Rows past 3n and
// K past n are zero.
__host__ __device__ __forceinline__ int64_t oz_a_offset(int64_t row, int64_t j, int p, int64_t nch) {
    return ((((row / TM) * nch + j / KCH) * kDig + p) * TM + row % TM) * KCH + j % KCH;
}

// Digits of A' = [L; Psi; G], rows r0..r1-1 of each matrix: one warp per
// row; ea[row] = the row's largest biased exponent, or -1 if the row holds a
// non-finite value.
__global__ void __launch_bounds__(256) k_oz_split_a(const double *__restrict__ L, const double *__restrict__ Psi,
                                                    const double *__restrict__ G, int64_t n, int64_t nch,
                                                    int64_t r0, int64_t r1, __nv_bfloat16 *__restrict__ dig,
                                                    int *__restrict__ ea) {
    const int lane = threadIdx.x & 31;
    const int64_t t = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5), band = r1 - r0;
    if (t >= 3 * band) return;  // whole warp
    const int m = (int)(t / band);
    const int64_t i = r0 + (t - m * band), row = m * n + i;
    const double *src = (m == 0 ? L : m == 1 ? Psi : G) + i * n;
    int q = 1;
    bool fin = true;
    for (int64_t j = lane; j < n; j += 32) {
        bool f;
        q = max(q, exp_of(__ldg(src + j), f));
        fin = fin && f;
    }
    q = __reduce_max_sync(0xffffffffu, q);
    fin = __all_sync(0xffffffffu, fin);
    if (lane == 0) ea[row] = fin ? q : -1;
    for (int64_t j0 = 8 * lane; j0 < nch * KCH; j0 += 256) {
        double a[8];
#pragma unroll
        for (int u = 0; u < 8; u++) a[u] = (j0 + u < n && fin) ? __ldg(src + j0 + u) : 0.0;
        write_digits8(a, q, dig + oz_a_offset(row, j0, 0, nch), (int64_t)TM * KCH);
    }
}

// Digits of X: one CTA per column c = (slot index k, right-hand side r, part p):
// x_{slots[k]}[r][j].(re, im).  ex[c] as ea above.
__global__ void __launch_bounds__(256) k_oz_split_x(const double2 *__restrict__ x, int64_t x_stride, int64_t n,
                                                    int64_t n_pad, int nrhs, const int *__restrict__ slots,
                                                    int ncol, int ncol_alloc, __nv_bfloat16 *__restrict__ dig,
                                                    int *__restrict__ ex) {
    __shared__ int s_q[8], s_f[8];
    const int c = blockIdx.x, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int k = c / (2 * nrhs), r = (c >> 1) % nrhs, p = c & 1;
    const double *src = reinterpret_cast<const double *>(x + (int64_t)slots[k] * x_stride + (int64_t)r * n) + p;
    int q = 1;
    bool fin = true;
    for (int64_t j = threadIdx.x; j < n; j += blockDim.x) {
        bool f;
        q = max(q, exp_of(src[2 * j], f));
        fin = fin && f;
    }
    q = __reduce_max_sync(0xffffffffu, q);
    fin = __all_sync(0xffffffffu, fin);
    if (lane == 0) {
        s_q[warp] = q;
        s_f[warp] = fin;
    }
    __syncthreads();
    for (int w = 0; w < (int)(blockDim.x >> 5); w++) {
        q = max(q, s_q[w]);
        fin = fin && s_f[w];
    }
    if (threadIdx.x == 0) ex[c] = fin ? q : -1;
    const int64_t plane = (int64_t)ncol_alloc * n_pad;
    for (int64_t j0 = 8 * (int64_t)threadIdx.x; j0 < n_pad; j0 += 8 * blockDim.x) {
        double a[8];
#pragma unroll
        for (int u = 0; u < 8; u++) a[u] = (j0 + u < n && fin) ? src[2 * (j0 + u)] : 0.0;
        write_digits8(a, q, dig + (int64_t)c * n_pad + j0, plane);
    }
}

// ------------------------------------------------------------------ tcgen05 product

__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait: gives up if another role already did (abort flag) or after
// kWaitLimit polls, raising the status bit with the wait site in bits 8-15.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag, unsigned *status,
                                          unsigned site) {
    uint32_t it = 0;
    while (!mbar_try_wait(bar, parity)) {
        if (*abort_flag) return false;
        if (++it > kWaitLimit) {
            *abort_flag = 1;
            atomicOr(status, ZS_DEV_TIMEOUT | (site << 8));
            return false;
        }
    }
    return true;
}
__device__ __forceinline__ void tma_load_5d(uint32_t dst, const CUtensorMap *map, int c0, int c1, int c2, int c3,
                                            int c4, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
        "l"((uint64_t)map), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int c0, int c1, int c2,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"((uint64_t)map), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// K-major operand, 64-byte swizzle: rows of 64 bytes (32 bf16), 8-row groups
// 512 bytes apart; an MMA K step of 16 (32 bytes) inside the row advances the
// start address.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr) {
    uint64_t d = 0;
    d |= (uint64_t)((addr >> 4) & 0x3FFF);  // start address
    d |= (uint64_t)1 << 16;                 // leading byte offset (unused for this layout)
    d |= (uint64_t)(512 >> 4) << 32;        // stride byte offset
    d |= (uint64_t)1 << 46;                 // descriptor version
    d |= (uint64_t)4 << 61;                 // SWIZZLE_64B
    return d;
}

// Instruction descriptor, kind::f16: D fp32, A and B bf16, both K-major, M = 128, N = 32 (8 - k).
__host__ __device__ constexpr uint32_t idesc_for(int k) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)((W * (kDig - k)) >> 3) << 17) |
           ((uint32_t)(TM >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

// 32 lanes x 16 consecutive fp32 columns of the accumulator, asynchronously:
// the registers hold the values after the next tmem_wait()
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// An integer-valued float with |v| <= 2^22 as an int: v + 1.5 * 2^23 lies in
// [2^23, 2^24] with unit spacing, so its low bits are v (two FP32/INT ops).
__device__ __forceinline__ int int_of(float v) {
    return (int)(__float_as_uint(v + 12582912.0f) - 0x4B400000u);
}

// Work units: (column group g, row tile t of A', K chunk c of 128), in the
// order u = (g * tiles + t) * nch + c.  CTA k of the G takes the units
// [k U / G, (k + 1) U / G) (U units in all): a contiguous run, so every SM
// has work whatever the number of row tiles, and a tile's K range is split
// among at most a few consecutive CTAs.  CTA k writes its part of tile
// q = g * tiles + t as segment k - first_cta(q) of part:
// part[segment][3n][ncol_alloc] float64.
__host__ __device__ __forceinline__ int64_t oz_cta_of(int64_t u, int64_t U, int64_t G) {
    return ((u + 1) * G - 1) / U;  // the CTA whose run holds unit u
}

__global__ void __launch_bounds__(kThreads, 1)
k_oz_gemm(const __grid_constant__ CUtensorMap amap, const __grid_constant__ CUtensorMap xmap,
          const int *__restrict__ ea, const int *__restrict__ ex, int64_t rows, int ncol, int ncol_alloc, int nch,
          int tiles, int64_t units, double *__restrict__ part, unsigned *__restrict__ status) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bar_full[STAGES], bar_empty[STAGES], bar_accf[2], bar_acce[2], bar_drain;
    __shared__ uint32_t s_tmem;
    __shared__ volatile int s_abort;
    const uint32_t base_addr = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t G = gridDim.x, k = blockIdx.x;
    const int64_t u_begin = k * units / G, u_end = (k + 1) * units / G;  // at least one unit (G <= units)
    const int nchunk = (int)(u_end - u_begin);

    if (threadIdx.x == 0) {
        s_abort = 0;
        for (int s = 0; s < STAGES; s++) {
            mbar_init(smem_u32(&bar_full[s]), 1);
            mbar_init(smem_u32(&bar_empty[s]), 1);
        }
        for (int b = 0; b < 2; b++) {
            mbar_init(smem_u32(&bar_accf[b]), 1);
            mbar_init(smem_u32(&bar_acce[b]), kEpiWarps);
        }
        mbar_init(smem_u32(&bar_drain), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    const int nsteps = nchunk * kStepsPerCh;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&amap) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&xmap) : "memory");
            uint32_t g = 0;
            for (; g < (uint32_t)nsteps; g++) {
                const uint32_t st = g % STAGES, ph = (g / STAGES) & 1u;
                if (!mbar_wait(smem_u32(&bar_empty[st]), ph ^ 1u, &s_abort, status, kSite | 1u)) break;
                const uint32_t fb = smem_u32(&bar_full[st]);
                mbar_expect_tx(fb, STAGE);
                const uint32_t sa = base_addr + st * STAGE;
                const int64_t u = u_begin + g / kStepsPerCh, q = u / nch;
                const int c = (int)(u - q * nch), kin = (int)(g % kStepsPerCh) * KS;
                tma_load_5d(sa, &amap, kin, 0, 0, c, (int)(q % tiles), fb);
                tma_load_3d(sa + A_STAGE, &xmap, c * KCH + kin, (int)(q / tiles) * W, 0, fb);
            }
            // our own copies in flight: wait (bounded) for the last stages to land
            for (uint32_t q = g > (uint32_t)STAGES ? g - STAGES : 0; q < g; q++) {
                uint32_t it = 0;
                while (!mbar_try_wait(smem_u32(&bar_full[q % STAGES]), (q / STAGES) & 1u) && ++it < kWaitLimit) {
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            uint32_t g = 0;
            bool ok = true;
            for (int c = 0; c < nchunk && ok; c++) {
                const uint32_t buf = (uint32_t)c & 1u, aph = ((uint32_t)c >> 1) & 1u;
                if (!mbar_wait(smem_u32(&bar_acce[buf]), aph ^ 1u, &s_abort, status, kSite | 2u)) break;
                tc_fence_after();
                const uint32_t d = tmem + buf * 256u;
                for (int s = 0; s < kStepsPerCh; s++, g++) {
                    const uint32_t st = g % STAGES, ph = (g / STAGES) & 1u;
                    if (!mbar_wait(smem_u32(&bar_full[st]), ph, &s_abort, status, kSite | 3u)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = base_addr + st * STAGE;
#pragma unroll
                    for (int ks = 0; ks < KS / 16; ks++) {
                        const uint64_t bd = smem_desc(sa + A_STAGE + 32 * ks);
#pragma unroll
                        for (int k = 0; k < kDig; k++)  // A digit k against X digits 0 .. 7-k: level blocks k .. 7
                            mma_bf16(d + (uint32_t)(W * k), smem_desc(sa + k * A_SLICE + 32 * ks), bd, idesc_for(k),
                                     (s > 0 || ks > 0 || k > 0) ? 1u : 0u);
                    }
                    mma_commit(smem_u32(&bar_empty[st]));  // stage free once these MMAs finish
                }
                if (ok) mma_commit(smem_u32(&bar_accf[buf]));  // chunk's level sums ready
            }
            // drain: every MMA issued so far completes before TMEM is freed
            mma_commit(smem_u32(&bar_drain));
            uint32_t w = 0;
            while (!mbar_try_wait(smem_u32(&bar_drain), 0) && ++w < kWaitLimit) {
            }
        }
    } else {
        // ------------------------------------------------ epilogue (warps 2-9)
        const int quad = warp & 3;              // TMEM lanes 32 quad .. 32 quad + 31
        const int half = (warp - 2) >> 2;       // columns 16 half .. 16 half + 15 of each level block
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        long long ga[16], gb[16];               // levels 0-3 and 4-7 (7 bits apart within each)
#pragma unroll
        for (int i = 0; i < 16; i++) ga[i] = gb[i] = 0;
        for (int c = 0; c < nchunk; c++) {
            const uint32_t buf = (uint32_t)c & 1u, aph = ((uint32_t)c >> 1) & 1u;
            const bool ok = mbar_wait(smem_u32(&bar_accf[buf]), aph, &s_abort, status, kSite | 4u);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc_fence_after();
            const uint32_t t0 = tmem + buf * 256u + (uint32_t)(16 * half) + lane_base;
#pragma unroll
            for (int grp = 0; grp < 2; grp++) {
                // the group's four level blocks in flight together, one wait
                uint32_t v[4][16];
#pragma unroll
                for (int l = 0; l < 4; l++) tmem_ld16(t0 + (uint32_t)(W * (4 * grp + l)), v[l]);
                tmem_wait();
#pragma unroll
                for (int i = 0; i < 16; i++) {
                    // level pairs 7 bits apart (< 2^30), then the pairs 14 bits apart
                    const int p0 = int_of(__uint_as_float(v[0][i])) * 128 + int_of(__uint_as_float(v[1][i]));
                    const int p1 = int_of(__uint_as_float(v[2][i])) * 128 + int_of(__uint_as_float(v[3][i]));
                    const long long t = ((long long)p0 << 14) + p1;
                    if (grp == 0) ga[i] += t;
                    else gb[i] += t;
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bar_acce[buf]));  // accumulator free for chunk c + 2
            // the end of this CTA's part of a tile: Y = 2^(Ea + Ex + 77) (ga +
            // 2^-28 gb), rounded once, as the tile's segment k - first CTA; a
            // non-finite row or column gives NaN
            const int64_t u = u_begin + c, q = u / nch;
            if (u + 1 < u_end && (u + 1) / nch == q) continue;
            const int64_t seg = k - oz_cta_of(q * nch, units, G);
            const int64_t row = (q % tiles) * TM + quad * 32 + lane;
            const int col0 = (int)(q / tiles) * W + 16 * half;
            if (row < rows) {
                const int qa = ea[row];
                double *dst = part + (seg * rows + row) * ncol_alloc + col0;
                const double two_m28 = 3.7252902984619141e-09;  // 2^-28
#pragma unroll
                for (int i = 0; i < 16; i++) {
                    const int cx = col0 + i;
                    if (cx >= ncol) break;
                    const int qx = ex[cx];
                    // 2^(Ea + Ex + 98 - 21) = 2^(qa + qx - 2077); ga, gb are exact integers below 2^53
                    dst[i] = (qa < 0 || qx < 0)
                                 ? __longlong_as_double(0x7FF8000000000000ll)
                                 : ldexp(__fma_rn((double)gb[i], two_m28, (double)ga[i]), qa + qx - 2077);
                }
            }
#pragma unroll
            for (int i = 0; i < 16; i++) ga[i] = gb[i] = 0;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
    }
}

// r_f = b - (j w (L x_f) - j (Psi x_f) / w + Zs_f (G x_f)) from the partial
// products, one thread per (row, slot index, right-hand side): the segments of
// each tile are summed in a fixed order.
__global__ void k_oz_combine(const double *__restrict__ part, int64_t n, int ncol_alloc, int nch, int tiles,
                             int64_t units, int64_t grid, const ZsSlotParam *__restrict__ params,
                             const double2 *__restrict__ b, int nrhs, const int *__restrict__ slots, int nslot,
                             float2 *__restrict__ out64, int64_t out64_stride, double2 *__restrict__ out128,
                             int64_t out128_stride) {
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= n * nslot * nrhs) return;
    const int64_t i = t % n;
    const int kr = (int)(t / n);  // k * nrhs + r
    const int k = kr / nrhs, r = kr - k * nrhs;
    const int c = 2 * kr;         // columns (re, im) of x_{slots[k]}[r], in one column group
    const int64_t rows = 3 * n;
    double y[3][2] = {{0.0, 0.0}, {0.0, 0.0}, {0.0, 0.0}};
#pragma unroll
    for (int m = 0; m < 3; m++) {
        const int64_t row = m * n + i;
        const int64_t q = (int64_t)(c / W) * tiles + row / TM, u0 = q * nch;
        const int64_t k0 = oz_cta_of(u0, units, grid), k1 = oz_cta_of(u0 + nch - 1, units, grid);
        for (int64_t sg = 0; sg <= k1 - k0; sg++) {
            const double2 v = *reinterpret_cast<const double2 *>(part + (sg * rows + row) * ncol_alloc + c);
            y[m][0] += v.x;
            y[m][1] += v.y;
        }
    }
    const int slot = slots[k];
    const ZsSlotParam sp = params[slot];
    const double w = sp.omega, rw = sp.pad;  // pad = RN(1/omega)
    const double sre = -w * y[0][1] + y[1][1] * rw + (sp.zs_re * y[2][0] - sp.zs_im * y[2][1]);
    const double sim = w * y[0][0] - y[1][0] * rw + (sp.zs_re * y[2][1] + sp.zs_im * y[2][0]);
    const double2 bv = b[(int64_t)r * n + i];
    const double rr = bv.x - sre, ri = bv.y - sim;
    if (out64)
        out64[(int64_t)slot * out64_stride + (int64_t)r * n + i] = make_float2(__double2float_rn(rr), __double2float_rn(ri));
    else
        out128[(int64_t)slot * out128_stride + (int64_t)r * n + i] = make_double2(rr, ri);
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void *p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
    }
    return fn;
}

// dims (K = n, rows, digit plane = 8); boxes of 32 K x box_rows rows x 8 planes, 64-byte swizzle
cudaError_t encode_digits(void *map_out, const __nv_bfloat16 *base, int64_t n, int64_t n_pad, int64_t rows,
                          int64_t rows_alloc, int box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = get_encode();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[3] = {(cuuint64_t)n, (cuuint64_t)rows, (cuuint64_t)kDig};
    const cuuint64_t strides[2] = {(cuuint64_t)n_pad * 2, (cuuint64_t)(rows_alloc * n_pad * 2)};
    const cuuint32_t box[3] = {(cuuint32_t)KS, (cuuint32_t)box_rows, (cuuint32_t)kDig};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(reinterpret_cast<CUtensorMap *>(map_out), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, (void *)base,
                     dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

int64_t zs_oz_n_pad(int64_t n) { return (n + 7) / 8 * 8; }
int64_t zs_oz_a_bytes(int64_t n) {
    const int64_t tiles = (3 * n + TM - 1) / TM, nch = (n + KCH - 1) / KCH;
    return tiles * nch * kDig * TM * KCH * 2;
}
int zs_oz_ncol_alloc(int ncol) { return (ncol + W - 1) / W * W; }

cudaError_t zs_launch_oz_split_a(const double *L, const double *Psi, const double *G, int64_t n, int64_t r0,
                                 int64_t r1, void *dig, int *ea, cudaStream_t st) {
    if (n < 1 || r0 < 0 || r1 > n || r0 > r1) return cudaErrorInvalidValue;
    if (r1 == r0) return cudaSuccess;
    const int64_t warps = 3 * (r1 - r0);
    k_oz_split_a<<<(unsigned)((warps + 7) / 8), 256, 0, st>>>(L, Psi, G, n, (n + KCH - 1) / KCH, r0, r1,
                                                               static_cast<__nv_bfloat16 *>(dig), ea);
    return cudaGetLastError();
}

// dims (K in chunk = 128, row in tile = 128, plane = 8, chunk = nch, tile);
// boxes of KS K x 128 rows x 8 planes of one unit, 64-byte swizzle
cudaError_t zs_oz_a_map(const void *dig, int64_t n, void *map_out) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = get_encode();
    if (!enc) return cudaErrorNotSupported;
    const int64_t tiles = (3 * n + TM - 1) / TM, nch = (n + KCH - 1) / KCH;
    const cuuint64_t dims[5] = {(cuuint64_t)KCH, (cuuint64_t)TM, (cuuint64_t)kDig, (cuuint64_t)nch,
                                (cuuint64_t)tiles};
    const cuuint64_t unit = (cuuint64_t)kDig * TM * KCH * 2;
    const cuuint64_t strides[4] = {(cuuint64_t)KCH * 2, (cuuint64_t)TM * KCH * 2, unit, unit * nch};
    const cuuint32_t box[5] = {(cuuint32_t)KS, (cuuint32_t)TM, (cuuint32_t)kDig, 1, 1};
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = enc(reinterpret_cast<CUtensorMap *>(map_out), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, (void *)dig, dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t zs_launch_residual_oz(const void *amap, const int *ea, int64_t n, const ZsSlotParam *params,
                                  const double2 *b, const double2 *x, int64_t x_stride, int nrhs, float2 *out_c64,
                                  int64_t out64_stride, double2 *out_c128, int64_t out128_stride, const int *slots,
                                  int nslot, void *xdig, int *ex, int ncol_cap, double *part, int64_t part_cap,
                                  unsigned *status, int num_sms, cudaStream_t st) {
    if (nslot < 1 || nrhs < 1) return cudaErrorInvalidValue;
    const int ncol = 2 * nslot * nrhs;
    const int ncol_alloc = zs_oz_ncol_alloc(ncol);
    if (ncol_alloc > ncol_cap) return cudaErrorInvalidValue;
    static const cudaError_t attr =
        cudaFuncSetAttribute(k_oz_gemm, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (attr != cudaSuccess) return attr;
    const int64_t n_pad = zs_oz_n_pad(n), rows = 3 * n;
    __nv_bfloat16 *xd = static_cast<__nv_bfloat16 *>(xdig);
    k_oz_split_x<<<(unsigned)ncol, 256, 0, st>>>(x, x_stride, n, n_pad, nrhs, slots, ncol, ncol_alloc, xd, ex);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    alignas(64) CUtensorMap xmap;
    e = encode_digits(&xmap, xd, n, n_pad, ncol, ncol_alloc, W);
    if (e != cudaSuccess) return e;
    // the units over one CTA per SM (fewer if there are fewer units, or if the
    // segments of the most split tile would not fit the partial buffer)
    const int tiles = (int)((rows + TM - 1) / TM), col_groups = ncol_alloc / W;
    const int nch = (int)((n + KCH - 1) / KCH);
    const int64_t units = (int64_t)col_groups * tiles * nch;
    int64_t grid = std::min<int64_t>(num_sms, units);
    auto max_segments = [&](int64_t G) {
        int64_t most = 0;
        for (int64_t q = 0; q < (int64_t)col_groups * tiles; q++)
            most = std::max(most, oz_cta_of(q * nch + nch - 1, units, G) - oz_cta_of(q * nch, units, G) + 1);
        return most;
    };
    while (grid > 1 && max_segments(grid) * rows * ncol_alloc > part_cap) grid--;
    if (max_segments(grid) * rows * ncol_alloc > part_cap) return cudaErrorInvalidValue;
    const CUtensorMap &am = *reinterpret_cast<const CUtensorMap *>(amap);
    k_oz_gemm<<<(unsigned)grid, kThreads, SMEM, st>>>(am, xmap, ea, ex, rows, ncol, ncol_alloc, nch, tiles, units, part,
                                                     status);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int64_t threads = n * nslot * nrhs;
    k_oz_combine<<<(unsigned)((threads + 255) / 256), 256, 0, st>>>(part, n, ncol_alloc, nch, tiles, units, grid,
                                                                   params, b, nrhs, slots, nslot, out_c64,
                                                                   out64_stride, out_c128, out128_stride);
    return cudaGetLastError();
}
