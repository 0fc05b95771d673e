// Diagonal block of the low-precision blocked LU: factorisation of one 128 x
// 128 complex float32 block per frequency and the inverses of its triangular
// factors (malusrfworks.com, "Solving Dense Matrices Fast in the Browser",
// section "Double-precision answers from a GPU without double precision",
// step 1: single-precision LU in blocks of 32, no pivoting).
//
// One CTA (16 warps) per frequency holds the block in shared memory and walks
// it in four 32-column panels p:
//   1. four warps factor the 32 x 32 diagonal sub-block A_pp in registers
//      (lane = column, eight rows per warp, multipliers broadcast by shuffle,
//      pivot rows passed through shared memory between 128-thread barriers);
//   2. all warps invert its triangles, DU_p = U_pp^-1 and DL_p = L_pp^-1
//      (four columns of an inverse per warp, lane = row, substitution with
//      the solved entries broadcast by shuffle);
//   3. all warps form the panel's L and U blocks as products with the
//      inverses, L_ip = A_ip DU_p and U_pj = DL_p A_pj, then the block's own
//      trailing update A_ij -= L_ip U_pj -- register-tiled complex products
//      (8 or 16 rows per warp task, lane = column, rows of the left operand
//      read as broadcast 16-byte loads).
// The factored block goes back to the float32 matrix and the 32 x 32 inverses
// to inv32.  A second kernel (k_block_inv, one CTA per block column of each
// inverse) then builds the 128 x 128 inverses W = U^-1 and V = L^-1 by block
// substitution,
//   U: X_ik = -sum_{m=i+1..k} G_im X_mk,  G_im = DU_i U_im   (i descending)
//   L: X_ik = -sum_{m=k..i-1} G_im X_mk,  G_im = DL_i L_im   (i ascending)
// with X_kk = DU_k resp. DL_k, and writes them out as the dense inverse blocks
// of the triangular solves (dinv) and, when asked, as the tensor-core operand
// packs of the block triangular solves (winv).
//
// Padding: a last block with nb < 128 is completed with the identity, whose
// factors and inverses are the identity again.
#include "common.cuh"

namespace {

using zs::cf;

constexpr int NB = ZS_NB;   // 128
constexpr int P = 32;       // panel / sub-block
constexpr int LDA = NB + 4; // block row stride (floats): 16-byte aligned rows
constexpr int LDD = P + 4;  // inverse sub-block row stride
constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int TMR = 16;     // rows per warp task where results wait for a barrier (one task per warp)
constexpr int TMU = 8;      // rows per warp task of the in-place trailing update

// shared-memory layout (floats)
constexpr int IM_A = NB * LDA;           // re plane -> im plane of the block
constexpr int OFF_D = 2 * NB * LDA;      // inverse sub-blocks [8][P][LDD]: 0-3 DU_p, 4-7 DL_p
constexpr int IM_D = 8 * P * LDD;
constexpr int OFF_R = OFF_D + 2 * IM_D;  // pivot reciprocals [re, im][4][P]
constexpr int OFF_ROW = OFF_R + 8 * P;   // base-LU pivot row, [2 buffers][re, im][P]
constexpr int kSmemFloats = OFF_ROW + 4 * P;
constexpr size_t kSmemBytes = (size_t)kSmemFloats * sizeof(float);

extern __shared__ __align__(16) float smem[];

struct Blk {  // a 32 x 32 complex sub-block: re at smem[off + r ld + c], im at + im
    int off, im, ld;
};
__device__ __forceinline__ Blk blkA(int bi, int bj) { return {bi * P * LDA + bj * P, IM_A, LDA}; }
__device__ __forceinline__ Blk blkDU(int b) { return {OFF_D + b * P * LDD, IM_D, LDD}; }
__device__ __forceinline__ Blk blkDL(int b) { return {OFF_D + (4 + b) * P * LDD, IM_D, LDD}; }
__device__ __forceinline__ cf ld_c(const Blk &B, int r, int c) {
    return {smem[B.off + r * B.ld + c], smem[B.off + B.im + r * B.ld + c]};
}
__device__ __forceinline__ void st_c(const Blk &B, int r, int c, cf v) {
    smem[B.off + r * B.ld + c] = v.re;
    smem[B.off + B.im + r * B.ld + c] = v.im;
}

// Reciprocal of a complex pivot, scaled so the squared modulus stays in
// range, with the hardware's approximate reciprocal (a few ulp: the factor
// is a float32 approximation that the float64 refinement corrects anyway).
// Pivots of modulus near or above 2^126 are flagged by the caller.
__device__ __forceinline__ cf crecip_fast(cf p) {
    const float s = fmaxf(fabsf(p.re), fabsf(p.im));
    const float rs = __fdividef(1.f, s);
    const float a = p.re * rs, b = p.im * rs;
    const float rd = __fdividef(1.f, fmaf(a, a, b * b)) * rs;
    return {a * rd, -b * rd};
}

// acc[t] += sum_k Pm(r0 + t, k) Qm(k, lane), t < TM, k < 32
template <int TM>
__device__ __forceinline__ void mac_rows(const Blk Pm, const Blk Qm, int r0, int lane, cf (&acc)[TM]) {
#pragma unroll 1
    for (int k0 = 0; k0 < P; k0 += 4) {
        float br[4], bi[4];
#pragma unroll
        for (int q = 0; q < 4; q++) {
            br[q] = smem[Qm.off + (k0 + q) * Qm.ld + lane];
            bi[q] = smem[Qm.off + Qm.im + (k0 + q) * Qm.ld + lane];
        }
#pragma unroll
        for (int t = 0; t < TM; t++) {
            const float4 ar = *reinterpret_cast<const float4 *>(&smem[Pm.off + (r0 + t) * Pm.ld + k0]);
            const float4 ai = *reinterpret_cast<const float4 *>(&smem[Pm.off + Pm.im + (r0 + t) * Pm.ld + k0]);
            const float xr[4] = {ar.x, ar.y, ar.z, ar.w}, xi[4] = {ai.x, ai.y, ai.z, ai.w};
#pragma unroll
            for (int q = 0; q < 4; q++) {
                acc[t].re = fmaf(xr[q], br[q], fmaf(-xi[q], bi[q], acc[t].re));
                acc[t].im = fmaf(xr[q], bi[q], fmaf(xi[q], br[q], acc[t].im));
            }
        }
    }
}

template <int TM>
__device__ __forceinline__ void zero(cf (&acc)[TM]) {
#pragma unroll
    for (int t = 0; t < TM; t++) acc[t] = cf{0.f, 0.f};
}

__device__ __forceinline__ void store_rows(const Blk C, int r0, int lane, const cf (&acc)[TMR], float sgn) {
#pragma unroll
    for (int t = 0; t < TMR; t++) st_c(C, r0 + t, lane, cf{sgn * acc[t].re, sgn * acc[t].im});
}

// Step 1: LU of the 32 x 32 diagonal sub-block by warps 0-3: warp w holds
// rows w + 4 t (t < 8) in registers, lane = column; at step k every warp
// reads pivot row k from a double-buffered row in shared memory, updates its
// rows below k (multipliers broadcast from lane k), and the owner of row k+1
// publishes it before a 128-thread barrier.  The step loop stays rolled so
// the code fits the instruction cache.  Returns true if a pivot was tiny or
// not finite.
constexpr int kLuWarps = 4;
constexpr int kLuRows = P / kLuWarps;

__device__ __forceinline__ void lu_barrier() { asm volatile("bar.sync 1, %0;" ::"n"(kLuWarps * 32) : "memory"); }

__device__ bool base_lu(int p, int w, int lane, float tiny) {
    const Blk B = blkA(p, p);
    float *prow = smem + OFF_ROW;
    cf a[kLuRows];
#pragma unroll
    for (int t = 0; t < kLuRows; t++) a[t] = ld_c(B, w + kLuWarps * t, lane);
    if (w == 0) {
        prow[lane] = a[0].re;
        prow[P + lane] = a[0].im;
    }
    lu_barrier();
    bool bad = false;
#pragma unroll 1
    for (int k = 0; k < P; k++) {
        const float *pr = prow + (k & 1) * 2 * P;
        const cf piv = {pr[k], pr[P + k]};
        const cf u = {pr[lane], pr[P + lane]};
        const float pm = fabsf(piv.re) + fabsf(piv.im);
        bad |= !(pm > tiny) || !(pm < 1e37f);
        const cf r = crecip_fast(piv);
        if (w == 0 && lane == k) {
            smem[OFF_R + p * P + k] = r.re;
            smem[OFF_R + 4 * P + p * P + k] = r.im;
        }
        // every row below k: multiplier from lane k; lanes right of k update,
        // lane k keeps the multiplier.  Branch-free so the eight rows' chains overlap.
        const bool right = lane > k, piv_lane = lane == k;
        cf l[kLuRows];
#pragma unroll
        for (int t = 0; t < kLuRows; t++)
            l[t] = cf{__shfl_sync(0xffffffffu, a[t].re, k), __shfl_sync(0xffffffffu, a[t].im, k)};
#pragma unroll
        for (int t = 0; t < kLuRows; t++) {
            const bool below = w + kLuWarps * t > k;
            const cf m = zs::cmul(l[t], r);
            const cf upd = zs::cfms(a[t], m, u);
            const cf nv = right ? upd : (piv_lane ? m : a[t]);
            a[t] = below ? nv : a[t];
        }
        const int kn = k + 1;
        if (kn < P) {
            if (w == (kn & (kLuWarps - 1))) {  // row k+1 is final through step k: publish it
                const int tn = kn / kLuWarps;
                cf v = a[0];
#pragma unroll
                for (int t = 1; t < kLuRows; t++)
                    if (t == tn) v = a[t];
                float *pw = prow + (kn & 1) * 2 * P;
                pw[lane] = v.re;
                pw[P + lane] = v.im;
            }
            lu_barrier();
        }
    }
#pragma unroll
    for (int t = 0; t < kLuRows; t++) st_c(B, w + kLuWarps * t, lane, a[t]);
    return bad;
}

// Step 2: the inverses DU_p = U_pp^-1 and DL_p = L_pp^-1 by all 16 warps:
// warps 0-7 take four columns each of DU_p, warps 8-15 of DL_p; lane = row.
// Column j of the inverse solves U x = e_j (back substitution) resp.
// L x = e_j (forward, unit diagonal); each finished x_k is broadcast from
// lane k and subtracted from the rows still open.
constexpr int kInvCols = 4;

__device__ __forceinline__ void base_inv(int p, int warp, int lane) {
    const Blk B = blkA(p, p);
    const bool upper = warp < 8;
    const int j0 = (warp & 7) * kInvCols;
    cf x[kInvCols];
#pragma unroll
    for (int c = 0; c < kInvCols; c++) x[c] = cf{lane == j0 + c ? 1.f : 0.f, 0.f};
    if (upper) {
#pragma unroll 2
        for (int k = P - 1; k >= 0; k--) {
            const cf r = {smem[OFF_R + p * P + k], smem[OFF_R + 4 * P + p * P + k]};
            const cf u = ld_c(B, lane, k);  // U(lane, k), used by rows lane < k
            const bool open = lane < k, piv_lane = lane == k;
#pragma unroll
            for (int c = 0; c < kInvCols; c++) {
                const cf xf = zs::cmul(x[c], r);  // lane k: x_k is final
                const cf xk = {__shfl_sync(0xffffffffu, xf.re, k), __shfl_sync(0xffffffffu, xf.im, k)};
                const cf upd = zs::cfms(x[c], u, xk);
                x[c].re = open ? upd.re : (piv_lane ? xf.re : x[c].re);
                x[c].im = open ? upd.im : (piv_lane ? xf.im : x[c].im);
            }
        }
    } else {
#pragma unroll 2
        for (int k = 0; k < P; k++) {
            const cf l = ld_c(B, lane, k);  // L(lane, k), used by rows lane > k
            const bool open = lane > k;
#pragma unroll
            for (int c = 0; c < kInvCols; c++) {
                const cf xk = {__shfl_sync(0xffffffffu, x[c].re, k), __shfl_sync(0xffffffffu, x[c].im, k)};
                const cf upd = zs::cfms(x[c], l, xk);
                x[c].re = open ? upd.re : x[c].re;
                x[c].im = open ? upd.im : x[c].im;
            }
        }
    }
    const Blk D = upper ? blkDU(p) : blkDL(p);
#pragma unroll
    for (int c = 0; c < kInvCols; c++) st_c(D, lane, j0 + c, x[c]);
}

__device__ __forceinline__ float tf32_rna(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}

__global__ void __launch_bounds__(kThreads, 1)
k_diag_block(float *__restrict__ z32, int64_t ld, int64_t plane, int64_t z32_stride, int64_t J, int nb,
             const int *__restrict__ slots, int *__restrict__ pivflag, float *__restrict__ inv32,
             int64_t inv32_stride) {
    __shared__ unsigned s_amax;
    __shared__ int s_bad;
    const int slot = slots[blockIdx.x];
    float *gre = z32 + (int64_t)slot * z32_stride;
    float *gim = gre + plane;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        s_amax = 0u;
        s_bad = 0;
    }
    __syncthreads();
    // ---- load (identity padding beyond nb)
    float amax = 0.f;
    for (int idx = tid; idx < NB * NB; idx += kThreads) {
        const int i = idx >> 7, j = idx & (NB - 1);
        float a = (i == j) ? 1.f : 0.f, b = 0.f;
        if (i < nb && j < nb) {
            const int64_t g = (J + i) * ld + J + j;
            a = gre[g];
            b = gim[g];
            amax = fmaxf(amax, fabsf(a) + fabsf(b));
        }
        smem[i * LDA + j] = a;
        smem[IM_A + i * LDA + j] = b;
    }
    if (!(amax <= 3.0e38f)) amax = 3.0e38f;  // non-finite inputs: the pivot test flags them
    atomicMax(&s_amax, __float_as_uint(amax));
    __syncthreads();
    const float tiny = 1e-30f * __uint_as_float(s_amax);

    // ---- LU, one 32-column panel at a time
    for (int p = 0; p < 4; p++) {
        if (warp < kLuWarps && base_lu(p, warp, lane, tiny) && lane == 0) s_bad = 1;
        __syncthreads();
        base_inv(p, warp, lane);
        __syncthreads();
        const int rest = 3 - p;
        if (rest == 0) break;
        // L_ip = A_ip DU_p (tasks 0 .. 2 rest - 1), U_pj = DL_p A_pj (the next 2 rest);
        // tasks read rows of A_pj that other tasks overwrite: write after a barrier
        {
            cf acc[TMR];
            zero(acc);
            const int t = warp, ntask = 4 * rest, b = t >> 1, r0 = (t & 1) * TMR;
            if (t < ntask) {
                const bool lpanel = b < rest;
                mac_rows(lpanel ? blkA(p + 1 + b, p) : blkDL(p), lpanel ? blkDU(p) : blkA(p, p + 1 + b - rest), r0, lane,
                         acc);
            }
            __syncthreads();
            if (t < ntask) store_rows(b < rest ? blkA(p + 1 + b, p) : blkA(p, p + 1 + b - rest), r0, lane, acc, 1.f);
            __syncthreads();
        }
        // A_ij -= L_ip U_pj, i, j > p: each task owns its output rows
        for (int t = warp; t < 4 * rest * rest; t += kWarps) {
            const int b = t >> 2, r0 = (t & 3) * TMU;
            const int bi = p + 1 + b / rest, bj = p + 1 + b % rest;
            cf acc[TMU];
            zero(acc);
            mac_rows(blkA(bi, p), blkA(p, bj), r0, lane, acc);
            const Blk C = blkA(bi, bj);
#pragma unroll
            for (int q = 0; q < TMU; q++) {
                smem[C.off + (r0 + q) * LDA + lane] -= acc[q].re;
                smem[C.off + IM_A + (r0 + q) * LDA + lane] -= acc[q].im;
            }
        }
        __syncthreads();
    }

    // ---- the factor and the 32 x 32 inverses out
    for (int idx = tid; idx < nb * nb; idx += kThreads) {
        const int i = idx / nb, j = idx - i * nb;
        const int64_t g = (J + i) * ld + J + j;
        gre[g] = smem[i * LDA + j];
        gim[g] = smem[IM_A + i * LDA + j];
    }
    {
        float *d32 = inv32 + (int64_t)slot * inv32_stride + (J / NB) * ZS_INV32_STRIDE;
        for (int idx = tid; idx < 8 * P * P; idx += kThreads) {
            const int w = idx >> 10, e = idx & (P * P - 1), i = e >> 5, j = e & 31;
            const int kb = w >> 1, lower = w & 1;  // [kb][U, L]
            const Blk D = lower ? blkDL(kb) : blkDU(kb);
            float *dst = d32 + w * 2 * P * P;
            const cf v = ld_c(D, i, j);
            dst[e] = v.re;
            dst[P * P + e] = v.im;
        }
    }
    if (tid == 0 && s_bad) pivflag[slot] = 1;

}

// ---------------------------------------------------------------- 128 x 128 inverses

// Block column k of W = U^-1 (chain 0-3, k = chain) or of V = L^-1 (chain
// 4-7, k = chain - 4) for one frequency per CTA row.  In local block indices
// l (U: l = i; L: l = 3 - i) both triangles read the same way: nr = number of
// block rows that meet column k, the target row nr - 1 holds X = D_{nr-1},
// and for l = nr-2 down to 0
//   X_l = -sum_{m=l+1..nr-1} G_lm X_m,   G_lm = D_l F_lm,
// with F the factor's off-diagonal sub-blocks (U_im, resp. L_{3-l,3-m}) and D
// the 32 x 32 diagonal inverses the factorisation stored.  Every column block
// is an independent chain; a CTA builds one and writes it to dinv (and winv).
constexpr int SLOT = 2 * P * LDD;  // floats per sub-block slot
constexpr int kInvSlots = 14;      // 6 F (local pairs a < b), 4 D, 4 X
constexpr size_t kInvSmemBytes = (size_t)kInvSlots * SLOT * sizeof(float);

__device__ __forceinline__ Blk slotF(int a, int b) { return {(b * (b - 1) / 2 + a) * SLOT, P * LDD, LDD}; }
__device__ __forceinline__ Blk slotD(int l) { return {(6 + l) * SLOT, P * LDD, LDD}; }
__device__ __forceinline__ Blk slotX(int l) { return {(10 + l) * SLOT, P * LDD, LDD}; }

__global__ void __launch_bounds__(kThreads, 1)
k_block_inv(const float *__restrict__ z32, int64_t ld, int64_t plane, int64_t z32_stride, int64_t J, int nb,
            const float *__restrict__ inv32, int64_t inv32_stride, float *__restrict__ dinv, int64_t dinv_stride,
            float *__restrict__ winv, int mode, const int *__restrict__ slots) {
    const int chain = blockIdx.x, upper = chain < 4, k = chain & 3;
    const int nr = upper ? k + 1 : 4 - k;
    const int slot = slots[blockIdx.y];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float *gre = z32 + (int64_t)slot * z32_stride;
    const float *gim = gre + plane;
    const float *d32 = inv32 + (int64_t)slot * inv32_stride + (J / NB) * ZS_INV32_STRIDE;
    auto gblk = [upper](int l) { return upper ? l : 3 - l; };  // global block index of local l

    // ---- load D_l and the factor sub-blocks F_ab (a < b < nr); padding beyond nb reads as zero
    for (int idx = tid; idx < nr * P * P; idx += kThreads) {
        const int l = idx >> 10, e = idx & (P * P - 1), i = e >> 5, j = e & 31;
        const float *d = d32 + (gblk(l) * 2 + (upper ? 0 : 1)) * 2 * P * P;
        st_c(slotD(l), i, j, cf{d[e], d[P * P + e]});
    }
    const int npair = nr * (nr - 1) / 2;
    for (int idx = tid; idx < npair * P * P; idx += kThreads) {
        const int q = idx >> 10, e = idx & (P * P - 1), i = e >> 5, j = e & 31;
        int b = 1;
        while (b * (b + 1) / 2 <= q) b++;
        const int a = q - b * (b - 1) / 2;
        const int r = gblk(a) * P + i, c = gblk(b) * P + j;  // local (a, b) -> global sub-block
        cf v = {0.f, 0.f};
        if (r < nb && c < nb) v = cf{gre[(J + r) * ld + J + c], gim[(J + r) * ld + J + c]};
        st_c(slotF(a, b), i, j, v);
    }
    __syncthreads();
    // ---- G_ab = D_a F_ab for every pair, in place (each pair: two 16-row tasks)
    {
        const int t = warp, pq = t >> 1, r0 = (t & 1) * TMR;
        int a = 0, b = 1;
        if (t < 2 * npair) {
            while (b * (b + 1) / 2 <= pq) b++;
            a = pq - b * (b - 1) / 2;
        }
        cf acc[TMR];
        zero(acc);
        if (t < 2 * npair) mac_rows(slotD(a), slotF(a, b), r0, lane, acc);
        __syncthreads();
        if (t < 2 * npair) store_rows(slotF(a, b), r0, lane, acc, 1.f);
        __syncthreads();
    }
    // ---- the chain, two rows per warp
    for (int l = nr - 2; l >= 0; l--) {
        cf acc[2];
        zero(acc);
        for (int m = l + 1; m < nr; m++) mac_rows(slotF(l, m), m == nr - 1 ? slotD(nr - 1) : slotX(m), 2 * warp, lane, acc);
#pragma unroll
        for (int q = 0; q < 2; q++) st_c(slotX(l), 2 * warp + q, lane, cf{-acc[q].re, -acc[q].im});
        __syncthreads();
    }
    // ---- dense inverse blocks [L, U][re, im][128][128]: block column k, zeros outside the triangle
    auto value = [&](int row, int col32) -> cf {  // element (row, 32 k + col32) of the inverse
        const int ib = row >> 5, l = upper ? ib : 3 - ib;
        if (l >= nr) return cf{0.f, 0.f};
        return ld_c(l == nr - 1 ? slotD(l) : slotX(l), row & 31, col32);
    };
    float *xr = dinv + (int64_t)slot * dinv_stride + (J / NB) * 4 * NB * NB + (upper ? 2 : 0) * NB * NB;
    for (int idx = tid; idx < NB * P; idx += kThreads) {
        const int row = idx >> 5, c = idx & 31;
        const cf v = value(row, c);
        xr[row * NB + k * P + c] = v.re;
        xr[NB * NB + row * NB + k * P + c] = v.im;
    }
    if (!winv) return;
    // ---- operand packs: pack row r holds column r of W (planes 0-3) resp.
    // row r of V (planes 4-7) as Br = [Re | -Im], Bi = [Im | Re], tf32 hi (+ lo)
    float *pl = winv + (int64_t)slot * ZS_WINV_STRIDE + (upper ? 0 : 4) * ZS_WINV_PLANE;
    for (int idx = tid; idx < NB * P; idx += kThreads) {
        int prow, m;
        cf v;
        if (upper) {  // W(m, 32 k + c) -> pack row 32 k + c, position m
            const int c = idx >> 7;
            m = idx & (NB - 1);
            prow = k * P + c;
            v = value(m, c);
        } else {      // V(r, 32 k + c) -> pack row r, position 32 k + c
            const int c = idx & 31;
            prow = idx >> 5;
            m = k * P + c;
            v = value(prow, c);
        }
        const int64_t o = (int64_t)prow * (2 * NB) + m;
        const float hr = tf32_rna(v.re), hi = tf32_rna(v.im);
        pl[o] = hr;
        pl[o + NB] = -hi;
        pl[2 * ZS_WINV_PLANE + o] = hi;
        pl[2 * ZS_WINV_PLANE + o + NB] = hr;
        if (mode == 2) {
            const float lr = tf32_rna(v.re - hr), li = tf32_rna(v.im - hi);
            pl[ZS_WINV_PLANE + o] = lr;
            pl[ZS_WINV_PLANE + o + NB] = -li;
            pl[3 * ZS_WINV_PLANE + o] = li;
            pl[3 * ZS_WINV_PLANE + o + NB] = lr;
        }
    }
}

}  // namespace

cudaError_t zs_launch_diag_block(float *z32, int64_t ld, int64_t plane, int64_t z32_stride, int64_t J, int nb,
                                 const int *slots, int nslot, int *pivflag, float *inv32, int64_t inv32_stride,
                                 cudaStream_t st) {
    if (nb <= 0 || nb > NB || nslot <= 0) return cudaErrorInvalidValue;
    // once per process (thread-safe initialisation of a local static)
    static const cudaError_t attr = cudaFuncSetAttribute(k_diag_block, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (attr != cudaSuccess) return attr;
    k_diag_block<<<nslot, kThreads, kSmemBytes, st>>>(z32, ld, plane, z32_stride, J, nb, slots, pivflag, inv32,
                                                       inv32_stride);
    return cudaGetLastError();
}

cudaError_t zs_launch_block_inv(const float *z32, int64_t ld, int64_t plane, int64_t z32_stride, int64_t J, int nb,
                                const int *slots, int nslot, const float *inv32, int64_t inv32_stride, float *dinv,
                                int64_t dinv_stride, float *winv, int mode, cudaStream_t st) {
    if (nb <= 0 || nb > NB || nslot <= 0) return cudaErrorInvalidValue;
    if (winv && mode != 1 && mode != 2) return cudaErrorInvalidValue;
    // once per process (thread-safe initialisation of a local static)
    static const cudaError_t attr = cudaFuncSetAttribute(k_block_inv, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kInvSmemBytes);
    if (attr != cudaSuccess) return attr;
    k_block_inv<<<dim3(8, nslot), kThreads, kInvSmemBytes, st>>>(z32, ld, plane, z32_stride, J, nb, inv32,
                                                                  inv32_stride, dinv, dinv_stride, winv, mode, slots);
    return cudaGetLastError();
}
