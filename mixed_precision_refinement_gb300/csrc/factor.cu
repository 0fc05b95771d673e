// Low-precision unpivoted blocked LU of the complex float32 matrix
// (malusrfworks.com, "Solving Dense Matrices Fast in the Browser", section
// "Double-precision answers from a GPU without double precision", step 1:
// single-precision factorisation on the GPU, LU in blocks of 32; the same
// paragraph states that it does not pivot).
//
// The host walks the matrix in outer blocks of ZS_NB = 128 columns.  At
// outer column J the diagonal block is factored by k_diag_block
// (diag_block.cu), which also leaves the inverses of its 32 x 32 diagonal
// sub-blocks behind.  This file holds the FP32 (FFMA) kernels of the rest of
// the step and the operand packing of the tensor-core path:
//   k_trsm_l    L21 = A21 U11^-1, one row per warp (row-oriented solve);
//   k_trsm_u    U12 = L11^-1 A12, one column per warp;
//   k_schur_simt  A22 -= L21 U12 (FP32 FFMA; schur_tc.cu: tcgen05);
//   k_pack_trsm A21 and A12^T as tf32 operand packs for the tensor-core
//               block solves (schur_tc.cu).
// k_trsm_l / k_trsm_u also write L21 and U12 as K-major operand packs for
// the trailing update: A = [Re L21 | Im L21], Br = [Re U12^T | -Im U12^T],
// Bi = [Im U12^T | Re U12^T], so that Re(L21 U12) = A Br^T and
// Im(L21 U12) = A Bi^T are plain real products with K = 2*128.
#include "common.cuh"

namespace {

using zs::cf;

constexpr int NB = ZS_NB;
constexpr int P = ZS_PANEL;
constexpr int LDS = NB + 1;  // padded shared row

__device__ __forceinline__ float tf32_rna(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}

// Write one float of an operand pack in the requested arithmetic mode.
__device__ __forceinline__ void pack_put(float *hi, float *lo, int64_t off, float v, int mode) {
    if (mode == 0) {
        hi[off] = v;
    } else if (mode == 1) {
        hi[off] = tf32_rna(v);
    } else {
        float h = tf32_rna(v);
        hi[off] = h;
        lo[off] = tf32_rna(v - h);
    }
}

// Four consecutive floats of an operand pack (16-byte aligned offset).
__device__ __forceinline__ void pack_put4(float *hi, float *lo, int64_t off, float4 v, int mode) {
    if (mode == 0) {
        *reinterpret_cast<float4 *>(hi + off) = v;
        return;
    }
    const float4 h = make_float4(tf32_rna(v.x), tf32_rna(v.y), tf32_rna(v.z), tf32_rna(v.w));
    *reinterpret_cast<float4 *>(hi + off) = h;
    if (mode == 2)
        *reinterpret_cast<float4 *>(lo + off) =
            make_float4(tf32_rna(v.x - h.x), tf32_rna(v.y - h.y), tf32_rna(v.z - h.z), tf32_rna(v.w - h.w));
}

// ---------------------------------------------------------------- L21 = A21 U11^-1

// Both block solves run in four 32-column steps with the inverted 32x32
// diagonal sub-blocks from k_diag_block: for step kb, x_kb = r_kb . inv(U_kb,kb)
// (resp. inv(L_kb,kb) . r_kb), then the later sub-blocks are updated with the
// off-diagonal blocks of U11 (resp. L11).  Every product is a register-tiled
// multiply-add with operands broadcast from shared memory; no step is a
// sequential substitution.

constexpr int kTrsmThreads = 512;  // 16 warps
constexpr int kTLRows = 128;       // L21 rows per CTA (8 per warp)

__global__ void __launch_bounds__(kTrsmThreads, 1)
k_trsm_l(float *__restrict__ z32, int64_t ld, int64_t plane, int64_t z32_stride, int64_t n, int64_t J,
         const float *__restrict__ inv32, int64_t inv32_stride, float *__restrict__ pack, int64_t pack_stride,
         int mode, const int *__restrict__ slots) {
    extern __shared__ float sm[];
    float *ure = sm;                 // [NB][NB]: U11 above the diagonal blocks, inv(U_kb,kb) on them
    float *uim = sm + NB * NB;
    cf *xs = reinterpret_cast<cf *>(sm + 2 * NB * NB);  // [16 warps][8 rows][32] broadcast buffer
    const int slot = slots[blockIdx.y];
    float *re = z32 + (int64_t)slot * z32_stride;
    float *im = re + plane;
    const float *inv = inv32 + (int64_t)slot * inv32_stride + (J / NB) * ZS_INV32_STRIDE;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int idx = tid; idx < NB * NB; idx += kTrsmThreads) {
        const int i = idx >> 7, j = idx & (NB - 1);
        float a = 0.f, b = 0.f;
        if ((i >> 5) == (j >> 5)) {
            const float *u = inv + ((i >> 5) * 2 + 0) * 2 * P * P;
            a = u[(i & 31) * P + (j & 31)];
            b = u[P * P + (i & 31) * P + (j & 31)];
        } else if (j > i) {
            const int64_t g = (J + i) * ld + J + j;
            a = re[g];
            b = im[g];
        }
        ure[idx] = a;
        uim[idx] = b;
    }
    __syncthreads();
    cf *xw = xs + warp * 8 * 32;
    const int64_t r0 = J + NB + (int64_t)blockIdx.x * kTLRows + warp * 8;
    cf v[8][4];
#pragma unroll
    for (int t = 0; t < 8; t++) {
        const int64_t r = r0 + t;
#pragma unroll
        for (int h = 0; h < 4; h++) {
            const int64_t g = r * ld + J + 32 * h + lane;
            v[t][h] = (r < n) ? cf{re[g], im[g]} : cf{0.f, 0.f};
        }
    }
#pragma unroll
    for (int kb = 0; kb < 4; kb++) {
        // x_kb = r_kb . inv(U_kb,kb): lane = output column
#pragma unroll
        for (int t = 0; t < 8; t++) xw[t * 32 + lane] = v[t][kb];
        __syncwarp();
        cf acc[8];
#pragma unroll
        for (int t = 0; t < 8; t++) acc[t] = cf{0.f, 0.f};
#pragma unroll 4
        for (int k = 0; k < 32; k++) {
            const cf w = cf{ure[(kb * 32 + k) * NB + kb * 32 + lane], uim[(kb * 32 + k) * NB + kb * 32 + lane]};
#pragma unroll
            for (int t = 0; t < 8; t++) {
                const cf rk = xw[t * 32 + k];
                acc[t].re = fmaf(rk.re, w.re, fmaf(-rk.im, w.im, acc[t].re));
                acc[t].im = fmaf(rk.re, w.im, fmaf(rk.im, w.re, acc[t].im));
            }
        }
        __syncwarp();
#pragma unroll
        for (int t = 0; t < 8; t++) {
            v[t][kb] = acc[t];
            xw[t * 32 + lane] = acc[t];
        }
        __syncwarp();
        // later sub-blocks: r_h -= x_kb . U(kb, h)
        if (kb < 3) {
#pragma unroll 4
            for (int k = 0; k < 32; k++) {
                cf xk[8];
#pragma unroll
                for (int t = 0; t < 8; t++) xk[t] = xw[t * 32 + k];
#pragma unroll
                for (int h = kb + 1; h < 4; h++) {
                    const cf u = cf{ure[(kb * 32 + k) * NB + h * 32 + lane], uim[(kb * 32 + k) * NB + h * 32 + lane]};
#pragma unroll
                    for (int t = 0; t < 8; t++) v[t][h] = zs::cfms(v[t][h], xk[t], u);
                }
            }
        }
        __syncwarp();
    }
    float *pA_hi = pack + (int64_t)slot * pack_stride;
    float *pA_lo = pA_hi + zs_pack_plane(n);
#pragma unroll
    for (int t = 0; t < 8; t++) {
        const int64_t r = r0 + t;
        if (r >= n) break;
        float *ah = pA_hi + r * ZS_PACK_K, *al = pA_lo + r * ZS_PACK_K;
#pragma unroll
        for (int h = 0; h < 4; h++) {
            const int c = 32 * h + lane;
            re[r * ld + J + c] = v[t][h].re;
            im[r * ld + J + c] = v[t][h].im;
            pack_put(ah, al, c, v[t][h].re, mode);
            pack_put(ah, al, NB + c, v[t][h].im, mode);
        }
    }
}

// ---------------------------------------------------------------- U12 = L11^-1 A12

constexpr int kTUCols = 64;  // U12 columns per CTA (4 per warp)
constexpr int kTUPad = kTUCols + 1;

__global__ void __launch_bounds__(kTrsmThreads, 1)
k_trsm_u(float *__restrict__ z32, int64_t ld, int64_t plane, int64_t z32_stride, int64_t n, int64_t J,
         const float *__restrict__ inv32, int64_t inv32_stride, float *__restrict__ pack, int64_t pack_stride,
         int mode, const int *__restrict__ slots) {
    extern __shared__ float sm[];
    float *lre = sm;                 // [NB][LDS]: L11 below the diagonal blocks, inv(L_kb,kb) on them
    float *lim = sm + NB * LDS;
    float *tre = sm + 2 * NB * LDS;  // [NB][kTUPad] tile of A12 / U12
    float *tim = tre + NB * kTUPad;
    cf *xs = reinterpret_cast<cf *>(tim + NB * kTUPad);  // [16 warps][4 cols][32]
    const int slot = slots[blockIdx.y];
    float *re = z32 + (int64_t)slot * z32_stride;
    float *im = re + plane;
    const float *inv = inv32 + (int64_t)slot * inv32_stride + (J / NB) * ZS_INV32_STRIDE;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t c0 = J + NB + (int64_t)blockIdx.x * kTUCols;
    const int ncol = (int)zs::min64(kTUCols, n - c0);
    for (int idx = tid; idx < NB * NB; idx += kTrsmThreads) {
        const int i = idx >> 7, j = idx & (NB - 1);
        float a = 0.f, b = 0.f;
        if ((i >> 5) == (j >> 5)) {
            const float *l = inv + ((i >> 5) * 2 + 1) * 2 * P * P;
            a = l[(i & 31) * P + (j & 31)];
            b = l[P * P + (i & 31) * P + (j & 31)];
        } else if (i > j) {
            const int64_t g = (J + i) * ld + J + j;
            a = re[g];
            b = im[g];
        }
        lre[i * LDS + j] = a;
        lim[i * LDS + j] = b;
    }
    for (int idx = tid; idx < NB * kTUCols; idx += kTrsmThreads) {
        const int i = idx >> 6, c = idx & (kTUCols - 1);
        float a = 0.f, b = 0.f;
        if (c < ncol) {
            const int64_t g = (J + i) * ld + c0 + c;
            a = re[g];
            b = im[g];
        }
        tre[i * kTUPad + c] = a;
        tim[i * kTUPad + c] = b;
    }
    __syncthreads();
    cf *xw = xs + warp * 4 * 32;
    // warp w: columns 4w..4w+3; lane holds rows 32h + lane
    cf v[4][4];
#pragma unroll
    for (int c = 0; c < 4; c++)
#pragma unroll
        for (int h = 0; h < 4; h++)
            v[c][h] = cf{tre[(32 * h + lane) * kTUPad + warp * 4 + c], tim[(32 * h + lane) * kTUPad + warp * 4 + c]};
#pragma unroll
    for (int kb = 0; kb < 4; kb++) {
        // u_kb = inv(L_kb,kb) . a_kb: lane = output row
#pragma unroll
        for (int c = 0; c < 4; c++) xw[c * 32 + lane] = v[c][kb];
        __syncwarp();
        cf acc[4];
#pragma unroll
        for (int c = 0; c < 4; c++) acc[c] = cf{0.f, 0.f};
#pragma unroll 4
        for (int k = 0; k < 32; k++) {
            const cf w = cf{lre[(kb * 32 + lane) * LDS + kb * 32 + k], lim[(kb * 32 + lane) * LDS + kb * 32 + k]};
#pragma unroll
            for (int c = 0; c < 4; c++) {
                const cf ak = xw[c * 32 + k];
                acc[c].re = fmaf(w.re, ak.re, fmaf(-w.im, ak.im, acc[c].re));
                acc[c].im = fmaf(w.re, ak.im, fmaf(w.im, ak.re, acc[c].im));
            }
        }
        __syncwarp();
#pragma unroll
        for (int c = 0; c < 4; c++) {
            v[c][kb] = acc[c];
            xw[c * 32 + lane] = acc[c];
        }
        __syncwarp();
        if (kb < 3) {
#pragma unroll 4
            for (int k = 0; k < 32; k++) {
                cf uk[4];
#pragma unroll
                for (int c = 0; c < 4; c++) uk[c] = xw[c * 32 + k];
#pragma unroll
                for (int h = kb + 1; h < 4; h++) {
                    const cf l = cf{lre[(h * 32 + lane) * LDS + kb * 32 + k], lim[(h * 32 + lane) * LDS + kb * 32 + k]};
#pragma unroll
                    for (int c = 0; c < 4; c++) v[c][h] = zs::cfms(v[c][h], l, uk[c]);
                }
            }
        }
        __syncwarp();
    }
    float *pBr_hi = pack + (int64_t)slot * pack_stride + 2 * zs_pack_plane(n);
    float *pBr_lo = pBr_hi + zs_pack_plane(n);
    float *pBi_hi = pBr_hi + 2 * zs_pack_plane(n);
    float *pBi_lo = pBr_hi + 3 * zs_pack_plane(n);
#pragma unroll
    for (int c = 0; c < 4; c++) {
        const int cc = warp * 4 + c;
        if (cc < ncol) {
            const int64_t j = c0 + cc;
            float *brh = pBr_hi + j * ZS_PACK_K, *brl = pBr_lo + j * ZS_PACK_K;
            float *bih = pBi_hi + j * ZS_PACK_K, *bil = pBi_lo + j * ZS_PACK_K;
#pragma unroll
            for (int h = 0; h < 4; h++) {
                const int i = 32 * h + lane;
                tre[i * kTUPad + cc] = v[c][h].re;
                tim[i * kTUPad + cc] = v[c][h].im;
                pack_put(brh, brl, i, v[c][h].re, mode);
                pack_put(brh, brl, NB + i, -v[c][h].im, mode);
                pack_put(bih, bil, i, v[c][h].im, mode);
                pack_put(bih, bil, NB + i, v[c][h].re, mode);
            }
        }
    }
    __syncthreads();
    for (int idx = tid; idx < NB * kTUCols; idx += kTrsmThreads) {
        const int i = idx >> 6, c = idx & (kTUCols - 1);
        if (c < ncol) {
            const int64_t g = (J + i) * ld + c0 + c;
            re[g] = tre[i * kTUPad + c];
            im[g] = tim[i * kTUPad + c];
        }
    }
}

// ---------------------------------------------------------------- SIMT trailing update

constexpr int kST = 64;        // output tile (complex entries per side)
constexpr int kSK = 32;        // K chunk (real, of the 2*NB packed K)
constexpr int kSPad = kST + 4;

__global__ void __launch_bounds__(256)
k_schur_simt(float *__restrict__ z32, int64_t ld, int64_t plane, int64_t z32_stride, int64_t n, int64_t J,
             const float *__restrict__ pack, int64_t pack_stride, const int *__restrict__ slots) {
    __shared__ __align__(16) float As[kSK][kSPad];
    __shared__ __align__(16) float Brs[kSK][kSPad];
    __shared__ __align__(16) float Bis[kSK][kSPad];
    const int slot = slots[blockIdx.z];
    const int64_t base = J + NB;
    const int64_t i0 = base + (int64_t)blockIdx.y * kST, j0 = base + (int64_t)blockIdx.x * kST;
    const float *pA = pack + (int64_t)slot * pack_stride;
    const float *pBr = pA + 2 * zs_pack_plane(n);
    const float *pBi = pA + 4 * zs_pack_plane(n);
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    float accr[4][4], acci[4][4];
#pragma unroll
    for (int x = 0; x < 4; x++)
#pragma unroll
        for (int y = 0; y < 4; y++) accr[x][y] = acci[x][y] = 0.f;
    const int lr = tid >> 2, lk = (tid & 3) * 8;  // loader: row lr, k lk..lk+7
    const int64_t ar = zs::min64(i0 + lr, n - 1), br = zs::min64(j0 + lr, n - 1);
    for (int kc = 0; kc < ZS_PACK_K; kc += kSK) {
        const float4 *a4 = reinterpret_cast<const float4 *>(pA + ar * ZS_PACK_K + kc + lk);
        const float4 *r4 = reinterpret_cast<const float4 *>(pBr + br * ZS_PACK_K + kc + lk);
        const float4 *m4 = reinterpret_cast<const float4 *>(pBi + br * ZS_PACK_K + kc + lk);
        float4 av[2] = {a4[0], a4[1]}, rv[2] = {r4[0], r4[1]}, mv[2] = {m4[0], m4[1]};
        __syncthreads();
#pragma unroll
        for (int h = 0; h < 2; h++) {
            As[lk + 4 * h + 0][lr] = av[h].x;
            As[lk + 4 * h + 1][lr] = av[h].y;
            As[lk + 4 * h + 2][lr] = av[h].z;
            As[lk + 4 * h + 3][lr] = av[h].w;
            Brs[lk + 4 * h + 0][lr] = rv[h].x;
            Brs[lk + 4 * h + 1][lr] = rv[h].y;
            Brs[lk + 4 * h + 2][lr] = rv[h].z;
            Brs[lk + 4 * h + 3][lr] = rv[h].w;
            Bis[lk + 4 * h + 0][lr] = mv[h].x;
            Bis[lk + 4 * h + 1][lr] = mv[h].y;
            Bis[lk + 4 * h + 2][lr] = mv[h].z;
            Bis[lk + 4 * h + 3][lr] = mv[h].w;
        }
        __syncthreads();
#pragma unroll 8
        for (int k = 0; k < kSK; k++) {
            float4 a = *reinterpret_cast<const float4 *>(&As[k][ty * 4]);
            float4 b = *reinterpret_cast<const float4 *>(&Brs[k][tx * 4]);
            float4 c = *reinterpret_cast<const float4 *>(&Bis[k][tx * 4]);
            float av4[4] = {a.x, a.y, a.z, a.w}, bv4[4] = {b.x, b.y, b.z, b.w}, cv4[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
            for (int x = 0; x < 4; x++)
#pragma unroll
                for (int y = 0; y < 4; y++) {
                    accr[x][y] = fmaf(av4[x], bv4[y], accr[x][y]);
                    acci[x][y] = fmaf(av4[x], cv4[y], acci[x][y]);
                }
        }
    }
    float *re = z32 + (int64_t)slot * z32_stride;
    float *im = re + plane;
#pragma unroll
    for (int x = 0; x < 4; x++) {
        const int64_t i = i0 + ty * 4 + x;
        if (i >= n) continue;
#pragma unroll
        for (int y = 0; y < 4; y++) {
            const int64_t j = j0 + tx * 4 + y;
            if (j < n) {
                re[i * ld + j] -= accr[x][y];
                im[i * ld + j] -= acci[x][y];
            }
        }
    }
}

// ---------------------------------------------------------------- packs for the tensor-core solves

// Operand packs of the block triangular solves (blockIdx.y = 0: rows of A21
// into the A planes; 1: columns of A12, transposed through shared memory,
// into the Br planes), 32 rows or columns per CTA.  sym (a complex-symmetric
// matrix, whose upper part is not kept current): the A planes only, all the
// symmetric block solve reads.
constexpr int kPackThreads = 256;

__global__ void __launch_bounds__(kPackThreads)
k_pack_trsm(const float *__restrict__ z32, int64_t ld, int64_t plane, int64_t z32_stride, int64_t n, int64_t J,
            float *__restrict__ pack, int64_t pack_stride, int mode, int sym, const int *__restrict__ slots) {
    __shared__ float s[ZS_PACK_K][33];
    const int slot = slots[blockIdx.z];
    const float *re = z32 + (int64_t)slot * z32_stride;
    const float *im = re + plane;
    float *pk = pack + (int64_t)slot * pack_stride;
    const int64_t pp = zs_pack_plane(n);
    const int64_t r0 = J + NB + 32 * (int64_t)blockIdx.x;
    const int tid = threadIdx.x;
    if (blockIdx.y == 0) {
        // four consecutive k per thread: 16-byte loads (ld and J are multiples
        // of 32 floats) and stores (pack rows of 256 floats)
        for (int idx = tid; idx < 32 * ZS_PACK_K / 4; idx += kPackThreads) {
            const int r = idx >> 6, k = 4 * (idx & (ZS_PACK_K / 4 - 1));
            const int64_t i = r0 + r;
            if (i >= n) break;  // later idx only move to later rows
            const float4 v = *reinterpret_cast<const float4 *>((k < NB ? re : im) + i * ld + J + (k & (NB - 1)));
            pack_put4(pk, pk + pp, i * ZS_PACK_K + k, v, mode);
        }
    } else {
        for (int idx = tid; idx < 32 * ZS_PACK_K; idx += kPackThreads) {
            const int k = idx >> 5, c = idx & 31;
            const int64_t j = r0 + c;
            s[k][c] = j < n ? (k < NB ? re : im)[(J + (k & (NB - 1))) * ld + j] : 0.f;
        }
        __syncthreads();
        for (int idx = tid; idx < 32 * ZS_PACK_K; idx += kPackThreads) {
            const int c = idx >> 8, k = idx & (ZS_PACK_K - 1);
            const int64_t j = r0 + c;
            if (j >= n) break;
            pack_put(pk + 2 * pp, pk + 3 * pp, j * ZS_PACK_K + k, s[k][c], mode);
        }
    }
}

template <typename K>
cudaError_t set_smem(K kernel, size_t bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

}  // namespace

cudaError_t zs_launch_trsm_l(float *z32, int64_t ld, int64_t plane, int64_t z32_stride, int64_t n,
                             int64_t J, const float *inv32, int64_t inv32_stride, float *pack, int64_t pack_stride,
                             int mode, const int *slots, int nslot, cudaStream_t st) {
    const size_t smem = (2 * NB * NB) * sizeof(float) + 16 * 8 * 32 * sizeof(cf);
    // once per process (thread-safe initialisation of a local static)
    static const cudaError_t attr = set_smem(k_trsm_l, smem);
    if (attr != cudaSuccess) return attr;
    const int64_t m2 = n - J - NB;
    dim3 grid((unsigned)((m2 + kTLRows - 1) / kTLRows), nslot);
    k_trsm_l<<<grid, kTrsmThreads, smem, st>>>(z32, ld, plane, z32_stride, n, J, inv32, inv32_stride, pack,
                                                pack_stride, mode, slots);
    return cudaGetLastError();
}

cudaError_t zs_launch_trsm_u(float *z32, int64_t ld, int64_t plane, int64_t z32_stride, int64_t n,
                             int64_t J, const float *inv32, int64_t inv32_stride, float *pack, int64_t pack_stride,
                             int mode, const int *slots, int nslot, cudaStream_t st) {
    const size_t smem = (2 * NB * LDS + 2 * NB * kTUPad) * sizeof(float) + 16 * 4 * 32 * sizeof(cf);
    // once per process (thread-safe initialisation of a local static)
    static const cudaError_t attr = set_smem(k_trsm_u, smem);
    if (attr != cudaSuccess) return attr;
    const int64_t m2 = n - J - NB;
    dim3 grid((unsigned)((m2 + kTUCols - 1) / kTUCols), nslot);
    k_trsm_u<<<grid, kTrsmThreads, smem, st>>>(z32, ld, plane, z32_stride, n, J, inv32, inv32_stride, pack,
                                                pack_stride, mode, slots);
    return cudaGetLastError();
}

cudaError_t zs_launch_schur_simt(float *z32, int64_t ld, int64_t plane, int64_t z32_stride, int64_t n,
                                 int64_t J, const float *pack, int64_t pack_stride, const int *slots,
                                 int nslot, cudaStream_t st) {
    const int64_t m2 = n - J - NB;
    const unsigned t = (unsigned)((m2 + kST - 1) / kST);
    dim3 grid(t, t, nslot);
    k_schur_simt<<<grid, 256, 0, st>>>(z32, ld, plane, z32_stride, n, J, pack, pack_stride, slots);
    return cudaGetLastError();
}

cudaError_t zs_launch_pack_trsm(const float *z32, int64_t ld, int64_t plane, int64_t z32_stride, int64_t n,
                                int64_t J, float *pack, int64_t pack_stride, int mode, int sym, const int *slots,
                                int nslot, cudaStream_t st) {
    const int64_t m2 = n - J - NB;
    if (m2 <= 0 || nslot <= 0) return cudaSuccess;
    if ((mode != 1 && mode != 2) || sym < 0 || sym > 1) return cudaErrorInvalidValue;
    const dim3 grid((unsigned)((m2 + 31) / 32), sym ? 1 : 2, (unsigned)nslot);
    k_pack_trsm<<<grid, kPackThreads, 0, st>>>(z32, ld, plane, z32_stride, n, J, pack, pack_stride, mode, sym,
                                               slots);
    return cudaGetLastError();
}
