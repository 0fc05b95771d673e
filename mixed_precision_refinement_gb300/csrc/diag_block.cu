// Diagonal block of the low-precision blocked LU: factorisation of one 128 x
// 128 complex float32 block per frequency and the inverses of its triangular
// factors (malusrfworks.com, "Solving Dense Matrices Fast in the Browser",
// section "Double-precision answers from a GPU without double precision",
// step 1: single-precision LU in blocks of 32, no pivoting).
//
// One CTA (16 warps) per frequency holds the block in shared memory and walks
// it in four 32-column panels p:
//   1. four warps factor the 32 x 32 diagonal sub-block A_pp in registers
//      as a wavefront (lane = column, eight rows per warp, multipliers
//      broadcast by shuffle, rows published through shared memory with a
//      flag each), while the other warps run the inverse window of panel
//      p - 1;
//   2. all warps invert its triangles, DU_p = U_pp^-1 and DL_p = L_pp^-1
//      (four columns of an inverse per warp, lane = row, substitution with
//      the solved entries broadcast by shuffle);
//   3. all warps form the panel's L and U blocks as products with the
//      inverses, L_ip = A_ip DU_p and U_pj = DL_p A_pj, then the block's own
//      trailing update A_ij -= L_ip U_pj -- register-tiled complex products
//      (8 or 16 rows per warp task, lane = column, rows of the left operand
//      read as broadcast 16-byte loads).
// The factored block goes back to the float32 matrix (and, for the FP32
// block solves, the 32 x 32 inverses to inv32).  The same CTA then builds the
// 128 x 128 inverses W = U^-1 and V = L^-1 by block substitution,
//   U: X_ik = -sum_{m=i+1..k} G_im X_mk,  G_im = DU_i U_im   (i descending)
//   L: X_ik = -sum_{m=k..i-1} G_im X_mk,  G_im = DL_i L_im   (i ascending)
// with X_kk = DU_k resp. DL_k: first the twelve G blocks, in place of the
// factor's off-diagonal sub-blocks, then the X blocks by distance from the
// diagonal (6, 4, 2 blocks of all warps' tasks), each round written out as
// the dense inverse blocks of the triangular solves (dinv) and, when asked,
// as the tensor-core operand packs of the block triangular solves (winv).
// The blocks outside the triangles are zero in both; they are set once when
// the buffers are allocated and never written here.
//
// The symmetric mode's instance (SYM = true) takes U = D L^T as the
// definition of the block's U side (D the pivots; an unpivoted LU of a
// complex-symmetric matrix has this form): per panel it forms DL_p alone and
// DU_p = DL_p^T D_p^-1, L_ip = A_ip DU_p and U_pj = D_p L_jp^T, and updates
// only the blocks on and below the diagonal (the next diagonal block first,
// the rest beside the next panel's base LU).  Its windows form V alone and
// emit W = V^T D^-1 from it; no W operand pack is written.
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

// shared-memory layout (floats)
constexpr int IM_A = NB * LDA;           // re plane -> im plane of the block
constexpr int OFF_D = 2 * NB * LDA;      // inverse sub-blocks [8][P][LDD]: 0-3 DU_p, 4-7 DL_p
constexpr int IM_D = 8 * P * LDD;
constexpr int OFF_R = OFF_D + 2 * IM_D;  // pivot reciprocals [re, im][4][P]
constexpr int OFF_ROW = OFF_R + 8 * P;   // base-LU pivot rows of the panel, [P][re, im][P]
constexpr int kSmemFloats = OFF_ROW + 2 * P * P;
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
// The scale is the power of two 2^-e, e the exponent of the larger part,
// made from the bit pattern, so that one reciprocal sits on the wavefront's
// path per pivot.  Zero, subnormal, huge or non-finite pivots are flagged by
// the caller (the result is then not used).
__device__ __forceinline__ cf crecip_fast(cf p) {
    const float s = fmaxf(fabsf(p.re), fabsf(p.im));
    const int e = min(max((__float_as_int(s) >> 23) - 127, -126), 126);
    const float sc = __int_as_float((127 - e) << 23);  // 2^-e
    const float a = p.re * sc, b = p.im * sc;         // the larger in [1, 2)
    const float rd = __fdividef(1.f, fmaf(a, a, b * b)) * sc;
    return {a * rd, -b * rd};
}

// Complex block products on the tensor cores, warp by warp: mma.sync
// m16n8k8 with tf32 operands and float32 accumulation, each real product
// split in three passes (hi*hi + hi*lo + lo*hi, hi = tf32 rounding of x,
// lo = tf32 rounding of x - hi), which is float32-class like the tcgen05
// kernels' 3xTF32.  On this part the legacy mma path retires 0.5 m16n8k8 per
// SM per clock, four times the FP32 FFMA rate, with one instruction per 1024
// products.  A task is 16 rows x 8 NTILE columns of a 32 x 32 block:
//   C(r0 + i, c0 + j) (+)= sum_k Pm(r0 + i, k) Qm(k, c0 + j),  k < 32,
// kept as Re P Re Q, Im P Im Q and the imaginary part (Re C = rr - ii).
// Fragment layout of m16n8k8 (g = lane / 4, t = lane % 4): A a0 (g, t),
// a1 (g+8, t), a2 (g, t+4), a3 (g+8, t+4); B b0 (t, g), b1 (t+4, g);
// C c0 (g, 2t), c1 (g, 2t+1), c2 (g+8, 2t), c3 (g+8, 2t+1).
template <int NTILE>
struct CAcc {
    float rr[NTILE][4], ii[NTILE][4], ri[NTILE][4];
};

template <int NTILE>
__device__ __forceinline__ void cacc_zero(CAcc<NTILE> &c) {
#pragma unroll
    for (int n = 0; n < NTILE; n++)
#pragma unroll
        for (int q = 0; q < 4; q++) c.rr[n][q] = c.ii[n][q] = c.ri[n][q] = 0.f;
}

__device__ __forceinline__ void split_tf32(float x, uint32_t &hi, uint32_t &lo) {
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(hi) : "f"(x));
    const float r = x - __uint_as_float(hi);
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(lo) : "f"(r));
}

__device__ __forceinline__ void mma_tf32(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

template <int NTILE>
__device__ __forceinline__ void cmma(const Blk Pm, const Blk Qm, int r0, int c0, int lane, CAcc<NTILE> &c) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll 1
    for (int k0 = 0; k0 < P; k0 += 8) {
        const int ra = Pm.off + (r0 + g) * Pm.ld + k0 + t;
        uint32_t arh[4], arl[4], aih[4], ail[4];
        const int ao[4] = {0, 8 * Pm.ld, 4, 8 * Pm.ld + 4};
#pragma unroll
        for (int q = 0; q < 4; q++) {
            split_tf32(smem[ra + ao[q]], arh[q], arl[q]);
            split_tf32(smem[Pm.im + ra + ao[q]], aih[q], ail[q]);
        }
#pragma unroll
        for (int n = 0; n < NTILE; n++) {
            const int rb = Qm.off + (k0 + t) * Qm.ld + c0 + 8 * n + g;
            uint32_t brh0, brl0, brh1, brl1, bih0, bil0, bih1, bil1;
            split_tf32(smem[rb], brh0, brl0);
            split_tf32(smem[rb + 4 * Qm.ld], brh1, brl1);
            split_tf32(smem[Qm.im + rb], bih0, bil0);
            split_tf32(smem[Qm.im + rb + 4 * Qm.ld], bih1, bil1);
            mma_tf32(c.rr[n], arh, brh0, brh1);
            mma_tf32(c.rr[n], arh, brl0, brl1);
            mma_tf32(c.rr[n], arl, brh0, brh1);
            mma_tf32(c.ii[n], aih, bih0, bih1);
            mma_tf32(c.ii[n], aih, bil0, bil1);
            mma_tf32(c.ii[n], ail, bih0, bih1);
            mma_tf32(c.ri[n], arh, bih0, bih1);
            mma_tf32(c.ri[n], arh, bil0, bil1);
            mma_tf32(c.ri[n], arl, bih0, bih1);
            mma_tf32(c.ri[n], aih, brh0, brh1);
            mma_tf32(c.ri[n], aih, brl0, brl1);
            mma_tf32(c.ri[n], ail, brh0, brh1);
        }
    }
}

// C(r0 + i, c0 + j) = sgn * product (store) or -= product (sub)
template <int NTILE, bool SUB>
__device__ __forceinline__ void cacc_out(const Blk C, int r0, int c0, int lane, const CAcc<NTILE> &c, float sgn) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int n = 0; n < NTILE; n++)
#pragma unroll
        for (int q = 0; q < 4; q++) {
            const int o = C.off + (r0 + g + (q >> 1) * 8) * C.ld + c0 + 8 * n + 2 * t + (q & 1);
            const float re = c.rr[n][q] - c.ii[n][q], im = c.ri[n][q];
            if (SUB) {
                smem[o] -= re;
                smem[C.im + o] -= im;
            } else {
                smem[o] = sgn * re;
                smem[C.im + o] = sgn * im;
            }
        }
}

// Step 1: LU of the 32 x 32 diagonal sub-block by warps 0-3, as a wavefront:
// warp w holds rows 8w..8w+7 in registers (lane = column).  A row is final
// once the steps of all rows above it are applied; its owner then publishes
// it (and its pivot's reciprocal) to shared memory, raises that row's flag
// to the panel's epoch, and carries on with its own rows below.  A warp
// applies the steps of the rows above its own in order, each after waiting
// for that row's flag only -- no barrier over all four warps per step.
// Multipliers are broadcast from lane k.  Returns true if a pivot was tiny
// or not finite, or a wait gave up (the frequency then takes the float64
// fallback).
constexpr int kLuWarps = 4;
constexpr int kLuRows = P / kLuWarps;

// publication of a row: its stores (by the whole warp, ordered by the warp
// barrier before this) become visible before the flag
__device__ __forceinline__ void row_arrive(uint32_t flag, uint32_t epoch) {
    __threadfence_block();
    asm volatile("st.volatile.shared.u32 [%0], %1;" ::"r"(flag), "r"(epoch) : "memory");
}

// bounded wait for a row's flag.  Every lane polls and the warp leaves
// together: a wait on one lane while the others block at a shuffle made each
// step some microseconds slower on this part.
__device__ __forceinline__ bool row_wait(uint32_t flag, uint32_t epoch) {
    bool ok = false;
    for (unsigned it = 0; it < ZS_SPIN_LIMIT; it++) {
        uint32_t v;
        asm volatile("ld.volatile.shared.u32 %0, [%1];" : "=r"(v) : "r"(flag) : "memory");
        if (__all_sync(0xffffffffu, v == epoch)) {
            ok = true;
            break;
        }
    }
    __threadfence_block();
    return ok;
}

// rows a[t] (t < 8, rows below step k) take step k: multiplier from lane k
// times the pivot reciprocal r; lanes right of k subtract it times u, lane k
// keeps it.  Branch-free so the rows' chains overlap.
__device__ __forceinline__ void lu_step(cf (&a)[kLuRows], int t0, int k, cf r, cf u, int lane) {
    const bool right = lane > k, piv_lane = lane == k;
#pragma unroll
    for (int t = 0; t < kLuRows; t++) {
        if (t < t0) continue;  // t0 is a constant wherever the caller's loop is unrolled
        const cf l = {__shfl_sync(0xffffffffu, a[t].re, k), __shfl_sync(0xffffffffu, a[t].im, k)};
        const cf m = zs::cmul(l, r);
        const cf upd = zs::cfms(a[t], m, u);
        a[t] = right ? upd : (piv_lane ? m : a[t]);
    }
}

__device__ bool base_lu(int p, int w, int lane, float tiny, uint32_t rowflag) {
    const Blk B = blkA(p, p);
    float *rows = smem + OFF_ROW;
    const uint32_t epoch = (uint32_t)(p + 1);  // flags hold the last panel that published the row
    cf a[kLuRows];
#pragma unroll
    for (int t = 0; t < kLuRows; t++) a[t] = ld_c(B, w * kLuRows + t, lane);
    bool bad = false;
    // the rows above this warp's, in order
#pragma unroll 1
    for (int k = 0; k < w * kLuRows; k++) {
        if (!row_wait(rowflag + 4u * k, epoch)) bad = true;
        const cf u = {rows[k * 2 * P + lane], rows[k * 2 * P + P + lane]};
        const cf r = {smem[OFF_R + p * P + k], smem[OFF_R + 4 * P + p * P + k]};
        lu_step(a, 0, k, r, u, lane);
    }
    // this warp's rows: publish row s, then step s on the rows below it
#pragma unroll
    for (int s = 0; s < kLuRows; s++) {
        const int k = w * kLuRows + s;
        const cf piv = {__shfl_sync(0xffffffffu, a[s].re, k), __shfl_sync(0xffffffffu, a[s].im, k)};
        const float pm = fabsf(piv.re) + fabsf(piv.im);
        bad |= !(pm > tiny) || !(pm < 1e37f);
        const cf r = crecip_fast(piv);
        rows[k * 2 * P + lane] = a[s].re;
        rows[k * 2 * P + P + lane] = a[s].im;
        if (lane == 0) {
            smem[OFF_R + p * P + k] = r.re;
            smem[OFF_R + 4 * P + p * P + k] = r.im;
        }
        __syncwarp();
        if (lane == 0) row_arrive(rowflag + 4u * k, epoch);
        lu_step(a, s + 1, k, r, a[s], lane);
    }
#pragma unroll
    for (int t = 0; t < kLuRows; t++) st_c(B, w * kLuRows + t, lane, a[t]);
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
    // steps on rows whose entries of these columns are all zero change
    // nothing: U columns start at their last row, L columns at their first
    if (upper) {
#pragma unroll 2
        for (int k = j0 + kInvCols - 1; k >= 0; k--) {
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
        for (int k = j0; k < P; k++) {
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

// Step 2 of the symmetric mode, where U = D L^T is taken to hold (D the
// pivots; an unpivoted LU of a complex symmetric matrix has this form):
// DL_p = L_pp^-1 only, warp w taking columns w and 31 - w (the forward
// substitution of column j has 32 - j steps, so every warp has 33), and
// DU_p = U_pp^-1 = DL_p^T D_p^-1 from it: DU(i, j) = DL(j, i) / d_j.
__device__ __forceinline__ void base_inv_sym(int p, int warp, int lane) {
    const Blk B = blkA(p, p);
    const int jc[2] = {warp, P - 1 - warp};
    cf x[2];
#pragma unroll
    for (int c = 0; c < 2; c++) x[c] = cf{lane == jc[c] ? 1.f : 0.f, 0.f};
#pragma unroll 2
    for (int k = jc[0]; k < P; k++) {
        const cf l = ld_c(B, lane, k);  // L(lane, k), used by rows lane > k
        const bool open = lane > k;
#pragma unroll
        for (int c = 0; c < 2; c++) {
            const cf xk = {__shfl_sync(0xffffffffu, x[c].re, k), __shfl_sync(0xffffffffu, x[c].im, k)};
            const cf upd = zs::cfms(x[c], l, xk);
            x[c].re = open ? upd.re : x[c].re;
            x[c].im = open ? upd.im : x[c].im;
        }
    }
    const cf rl = {smem[OFF_R + p * P + lane], smem[OFF_R + 4 * P + p * P + lane]};  // 1 / d_lane
#pragma unroll
    for (int c = 0; c < 2; c++) {
        st_c(blkDL(p), lane, jc[c], x[c]);
        st_c(blkDU(p), jc[c], lane, zs::cmul(x[c], rl));
    }
}

__device__ __forceinline__ float tf32_rna(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}

// ---------------------------------------------------------------- inverse windows
//
// The 128 x 128 inverses are built in four windows W(q), q = 0..3.  W(q)
// runs once panel q is final: for q < 3 on warps 4-15 while warps 0-3 factor
// the next panel's diagonal sub-block (and then write DU_q, DL_q out as the
// diagonal blocks of W and V), W(3) on all warps after the last panel.
// (Running the windows on all warps after the wavefront LU instead was
// slower.)  W(q)
//   - writes block row q of the factor (from the diagonal on) and block
//     column q below it back to the float32 matrix (W(3) also DU_3, DL_3);
//   - forms G_U(q, b) = DU_q U_qb (b > q) and G_L(q, m) = DL_q L_qm (m < q)
//     in place of those factor blocks (written back by now);
//   - completes column q of W and row q of V by distance from the diagonal:
//     W_lq = -sum_{m=l+1..q} G_U(l, m) W_mq,  V_qk = -sum_{m=k..q-1} G_L(q, m) V_mk
//     (W_qq = DU_q, V_qq = DL_q), writing each round out.
// Shared-memory slots of the results: a diagonal factor block once written
// back, or an L block whose V row is complete.  V_10, V_21 and V_20 stay for
// W(3); W_23 and W_13 live within W(3).
// Block ids: 4 i + j for A(i, j), 16 + k for DU_k, 20 + k for DL_k.
struct WinOut {
    unsigned char dst, nterm, neg, eu, el, ek;  // eu: 1 = W block (el, ek), 0 = V block, 2 = not written out
    unsigned char tp[3], tq[3];                 // terms Pm(tp) Qm(tq)
};
constexpr int kWinRounds = 10;
__constant__ WinOut kWin[kWinRounds][3] = {
    // W(0): G_U(0,1), G_U(0,2), G_U(0,3)
    {{1, 1, 0, 2, 0, 0, {16}, {1}}, {2, 1, 0, 2, 0, 0, {16}, {2}}, {3, 1, 0, 2, 0, 0, {16}, {3}}},
    // W(1): G_U(1,2), G_U(1,3), G_L(1,0)
    {{6, 1, 0, 2, 0, 0, {17}, {6}}, {7, 1, 0, 2, 0, 0, {17}, {7}}, {4, 1, 0, 2, 0, 0, {21}, {4}}},
    //       W_01 = -G_U(0,1) DU_1 -> A(1,1);  V_10 = -G_L(1,0) DL_0 -> A(0,0)
    {{5, 1, 1, 1, 0, 1, {1}, {17}}, {0, 1, 1, 0, 1, 0, {4}, {20}}},
    // W(2): G_U(2,3), G_L(2,0), G_L(2,1)
    {{11, 1, 0, 2, 0, 0, {18}, {11}}, {8, 1, 0, 2, 0, 0, {22}, {8}}, {9, 1, 0, 2, 0, 0, {22}, {9}}},
    //       W_12 = -G_U(1,2) DU_2 -> A(1,1);  V_21 = -G_L(2,1) DL_1 -> A(2,2)
    {{5, 1, 1, 1, 1, 2, {6}, {18}}, {10, 1, 1, 0, 2, 1, {9}, {21}}},
    //       W_02 = -(G_U(0,1) W_12 + G_U(0,2) DU_2) -> A(1,0)
    //       V_20 = -(G_L(2,1) V_10 + G_L(2,0) DL_0) -> A(2,0)
    {{4, 2, 1, 1, 0, 2, {1, 2}, {5, 18}}, {8, 2, 1, 0, 2, 0, {9, 8}, {0, 20}}},
    // W(3): G_L(3,0), G_L(3,1), G_L(3,2)
    {{12, 1, 0, 2, 0, 0, {23}, {12}}, {13, 1, 0, 2, 0, 0, {23}, {13}}, {14, 1, 0, 2, 0, 0, {23}, {14}}},
    //       W_23 = -G_U(2,3) DU_3 -> A(1,1);  V_32 = -G_L(3,2) DL_2 -> A(1,0)
    {{5, 1, 1, 1, 2, 3, {11}, {19}}, {4, 1, 1, 0, 3, 2, {14}, {22}}},
    //       W_13 = -(G_U(1,2) W_23 + G_U(1,3) DU_3) -> A(2,1)
    //       V_31 = -(G_L(3,2) V_21 + G_L(3,1) DL_1) -> A(3,3)
    {{9, 2, 1, 1, 1, 3, {6, 7}, {5, 19}}, {15, 2, 1, 0, 3, 1, {14, 13}, {10, 21}}},
    //       W_03 = -(G_U(0,1) W_13 + G_U(0,2) W_23 + G_U(0,3) DU_3) -> A(1,0)
    //       V_30 = -(G_L(3,2) V_20 + G_L(3,1) V_10 + G_L(3,0) DL_0) -> A(3,3)
    {{4, 3, 1, 1, 0, 3, {1, 2, 3}, {9, 5, 19}}, {15, 3, 1, 0, 3, 0, {14, 13, 12}, {8, 0, 20}}},
};
__constant__ unsigned char kWinFirst[4] = {0, 1, 3, 6};  // first round of W(q); W(q) has q + 1 rounds
__constant__ unsigned char kWinOuts[kWinRounds] = {3, 3, 2, 3, 2, 2, 3, 2, 2, 2};

// The symmetric mode's windows: the V chain alone (no G_U blocks, no W
// blocks: those are emitted from the V blocks), in the same rounds and
// shared-memory slots as above.  W(0) has nothing to form.
__constant__ WinOut kWinSym[kWinRounds][3] = {
    {},
    // W(1): G_L(1,0);  V_10 = -G_L(1,0) DL_0 -> A(0,0)
    {{4, 1, 0, 2, 0, 0, {21}, {4}}},
    {{0, 1, 1, 0, 1, 0, {4}, {20}}},
    // W(2): G_L(2,0), G_L(2,1);  V_21 = -G_L(2,1) DL_1 -> A(2,2);
    //       V_20 = -(G_L(2,1) V_10 + G_L(2,0) DL_0) -> A(2,0)
    {{8, 1, 0, 2, 0, 0, {22}, {8}}, {9, 1, 0, 2, 0, 0, {22}, {9}}},
    {{10, 1, 1, 0, 2, 1, {9}, {21}}},
    {{8, 2, 1, 0, 2, 0, {9, 8}, {0, 20}}},
    // W(3): G_L(3,0), G_L(3,1), G_L(3,2);  V_32 -> A(1,0);  V_31 -> A(3,3);  V_30 -> A(3,3)
    {{12, 1, 0, 2, 0, 0, {23}, {12}}, {13, 1, 0, 2, 0, 0, {23}, {13}}, {14, 1, 0, 2, 0, 0, {23}, {14}}},
    {{4, 1, 1, 0, 3, 2, {14}, {22}}},
    {{15, 2, 1, 0, 3, 1, {14, 13}, {10, 21}}},
    {{15, 3, 1, 0, 3, 0, {14, 13, 12}, {8, 0, 20}}},
};
__constant__ unsigned char kWinSymOuts[kWinRounds] = {0, 1, 1, 2, 1, 1, 3, 1, 1, 1};

__device__ __forceinline__ Blk blk_id(int id) {
    return id < 16 ? blkA(id >> 2, id & 3) : (id < 20 ? blkDU(id - 16) : blkDL(id - 20));
}

template <int NT, int BAR>
__device__ __forceinline__ void group_sync() {
    asm volatile("bar.sync %0, %1;" ::"n"(BAR), "n"(NT) : "memory");
}

// Block (l, k) of W = U^-1 (upper) or of V = L^-1, held in shared memory at
// S, out to the dense inverse xr ([re, im][128][128] of that triangle) and,
// if pl is set, to the operand packs of the tensor-core block solves: pack
// row r holds column r of W resp. row r of V as Br = [Re | -Im] and
// Bi = [Im | Re], in tf32 hi (planes 0, 2) and, for mode 2, lo (1, 3).
// Blocks outside the triangles are zero in both and are never written.
// Threads t < nt of the calling group take part, four entries each.
__device__ __forceinline__ float4 f4(float a, float b, float c, float d) { return make_float4(a, b, c, d); }
__device__ __forceinline__ float4 tf32_4(const float4 v) {
    return f4(tf32_rna(v.x), tf32_rna(v.y), tf32_rna(v.z), tf32_rna(v.w));
}
__device__ __forceinline__ float4 sub4(const float4 a, const float4 b) { return f4(a.x - b.x, a.y - b.y, a.z - b.z, a.w - b.w); }
__device__ __forceinline__ float4 neg4(const float4 a) { return f4(-a.x, -a.y, -a.z, -a.w); }

__device__ __forceinline__ void emit_one(bool upper, int l, int k, const Blk S, float *xr, float *pl, int mode,
                                         int idx, bool dense) {
    if (dense) {
        const int i = idx >> 3, j = (idx & 7) * 4;
        const float4 re = *reinterpret_cast<const float4 *>(&smem[S.off + i * S.ld + j]);
        const float4 im = *reinterpret_cast<const float4 *>(&smem[S.off + S.im + i * S.ld + j]);
        const int o = (l * P + i) * NB + k * P + j;
        *reinterpret_cast<float4 *>(xr + o) = re;
        *reinterpret_cast<float4 *>(xr + NB * NB + o) = im;
        return;
    }
    // four consecutive pack positions per thread, consecutive threads continue the row
    float4 re, im;
    int o;
    if (upper) {  // W(32 l + i0 + u, 32 k + j) -> pack row 32 k + j, position 32 l + i0 + u
        const int j = idx >> 3, i0 = (idx & 7) * 4;
        const cf v0 = ld_c(S, i0, j), v1 = ld_c(S, i0 + 1, j), v2 = ld_c(S, i0 + 2, j), v3 = ld_c(S, i0 + 3, j);
        re = f4(v0.re, v1.re, v2.re, v3.re);
        im = f4(v0.im, v1.im, v2.im, v3.im);
        o = (k * P + j) * (2 * NB) + l * P + i0;
    } else {      // V(32 l + i, 32 k + j0 + u) -> pack row 32 l + i, position 32 k + j0 + u
        const int i = idx >> 3, j0 = (idx & 7) * 4;
        re = *reinterpret_cast<const float4 *>(&smem[S.off + i * S.ld + j0]);
        im = *reinterpret_cast<const float4 *>(&smem[S.off + S.im + i * S.ld + j0]);
        o = (l * P + i) * (2 * NB) + k * P + j0;
    }
    // the Br planes only (hi, lo): the tensor-core block solve takes Bi from
    // Br's K halves
    const float4 hr = tf32_4(re), hi = tf32_4(im);
    *reinterpret_cast<float4 *>(pl + o) = hr;
    *reinterpret_cast<float4 *>(pl + o + NB) = neg4(hi);
    if (mode == 2) {
        const float4 lr = tf32_4(sub4(re, hr)), li = tf32_4(sub4(im, hi));
        *reinterpret_cast<float4 *>(pl + ZS_WINV_PLANE + o) = lr;
        *reinterpret_cast<float4 *>(pl + ZS_WINV_PLANE + o + NB) = neg4(li);
    }
}

// A W block (lw, kw) at Sw and a V block (lv, kv) at Sv written out together
// (more stores in flight per thread): work items 0..255 the W block, 256..511
// the V block, first the dense inverses, then the packs.
__device__ __noinline__ void emit_pair(int lw, int kw, const Blk Sw, int lv, int kv, const Blk Sv, float *xu,
                                       float *xl, float *pu, float *pv, int mode, int t, int nt) {
    constexpr int NI = P * P / 4;
    for (int idx = t; idx < 2 * NI; idx += nt) {
        if (idx < NI) emit_one(true, lw, kw, Sw, xu, pu, mode, idx, true);
        else emit_one(false, lv, kv, Sv, xl, pv, mode, idx - NI, true);
    }
    if (!pv) return;  // no packs at all (the last diagonal block)
    // the packs; without pu (the symmetric mode, whose block solves read V's alone) V's only
    const int first = pu ? 0 : NI;
    for (int idx = first + t; idx < 2 * NI; idx += nt) {
        if (idx < NI) emit_one(true, lw, kw, Sw, xu, pu, mode, idx, false);
        else emit_one(false, lv, kv, Sv, xl, pv, mode, idx - NI, false);
    }
}

// Symmetric mode: V block (q, k) at Sv (q > k) out as emit_one does, and
// with it W block (k, q) of W = U^-1 = V^T D^-1: W(32k + a, 32q + b) =
// V(32q + b, 32k + a) / d_(32q + b).  Its dense block reads V's columns;
// its pack row 32q + b (column 32q + b of W) is V's pack row 32q + b
// times 1 / d_(32q + b).
__device__ __forceinline__ void emit_w_of_v(int q, int k, const Blk Sv, float *xu, float *pu, int mode, int idx,
                                            bool dense) {
    const float *rre = smem + OFF_R + q * P, *rim = rre + 4 * P;  // 1 / d of V's rows
    if (dense) {
        const int a = idx >> 3, b0 = (idx & 7) * 4;
        cf w[4];
#pragma unroll
        for (int u = 0; u < 4; u++) w[u] = zs::cmul(ld_c(Sv, b0 + u, a), cf{rre[b0 + u], rim[b0 + u]});
        const int o = (k * P + a) * NB + q * P + b0;
        *reinterpret_cast<float4 *>(xu + o) = f4(w[0].re, w[1].re, w[2].re, w[3].re);
        *reinterpret_cast<float4 *>(xu + NB * NB + o) = f4(w[0].im, w[1].im, w[2].im, w[3].im);
        return;
    }
    const int j = idx >> 3, i0 = (idx & 7) * 4;
    const float4 vr = *reinterpret_cast<const float4 *>(&smem[Sv.off + j * Sv.ld + i0]);
    const float4 vi = *reinterpret_cast<const float4 *>(&smem[Sv.off + Sv.im + j * Sv.ld + i0]);
    const float cr = rre[j], ci = rim[j];
    const float4 re = f4(vr.x * cr - vi.x * ci, vr.y * cr - vi.y * ci, vr.z * cr - vi.z * ci, vr.w * cr - vi.w * ci);
    const float4 im = f4(vr.x * ci + vi.x * cr, vr.y * ci + vi.y * cr, vr.z * ci + vi.z * cr, vr.w * ci + vi.w * cr);
    const int o = (q * P + j) * (2 * NB) + k * P + i0;
    const float4 hr = tf32_4(re), hi = tf32_4(im);
    *reinterpret_cast<float4 *>(pu + o) = hr;
    *reinterpret_cast<float4 *>(pu + o + NB) = neg4(hi);
    if (mode == 2) {
        *reinterpret_cast<float4 *>(pu + ZS_WINV_PLANE + o) = tf32_4(sub4(re, hr));
        *reinterpret_cast<float4 *>(pu + ZS_WINV_PLANE + o + NB) = neg4(tf32_4(sub4(im, hi)));
    }
}

__device__ __noinline__ void emit_v_w(int q, int k, const Blk Sv, float *xu, float *xl, float *pu, float *pv, int mode,
                                      int t, int nt) {
    constexpr int NI = P * P / 4;
    for (int idx = t; idx < 2 * NI; idx += nt) {
        if (idx < NI) emit_one(false, q, k, Sv, xl, pv, mode, idx, true);
        else emit_w_of_v(q, k, Sv, xu, pu, mode, idx - NI, true);
    }
    if (!pv) return;
    const int last = pu ? 2 * NI : NI;  // W's pack rows only if someone reads them
    for (int idx = t; idx < last; idx += nt) {
        if (idx < NI) emit_one(false, q, k, Sv, xl, pv, mode, idx, false);
        else emit_w_of_v(q, k, Sv, xu, pu, mode, idx - NI, false);
    }
}

struct WinArgs {
    float *gre, *gim;
    int64_t ld, J;
    int nb, mode;
    float *xu, *xl, *pu, *pv;  // dense inverse of U and L; operand packs of W and V (or null)
};

// One round of W(q): its output blocks, 8 / NTILE tasks of 16 rows x 8 NTILE
// columns each (one task per warp of the group), stored after the group's
// barrier (a result may replace one of its own operands), then written out.
template <int NTILE, int NT, int BAR, bool SYM>
__device__ __forceinline__ void win_round(int r, int t, int lane, const WinArgs &w) {
    constexpr int CPB = 4 / NTILE, TPB = 2 * CPB;  // column groups, tasks per block
    const WinOut(*kWinT)[3] = SYM ? kWinSym : kWin;
    const int nout = SYM ? kWinSymOuts[r] : kWinOuts[r];
    if (nout == 0) return;
    const int wi = t >> 5, b = wi / TPB, rem = wi % TPB, r0 = (rem / CPB) * 16, c0 = (rem % CPB) * 8 * NTILE;
    const bool on = b < nout;
    CAcc<NTILE> acc;
    cacc_zero(acc);
    if (on) {
        const int nterm = kWinT[r][b].nterm;
#pragma unroll 1
        for (int i = 0; i < nterm; i++) cmma(blk_id(kWinT[r][b].tp[i]), blk_id(kWinT[r][b].tq[i]), r0, c0, lane, acc);
    }
    group_sync<NT, BAR>();
    if (on) cacc_out<NTILE, false>(blk_id(kWinT[r][b].dst), r0, c0, lane, acc, kWinT[r][b].neg ? -1.f : 1.f);
    group_sync<NT, BAR>();
    // a chain round's outputs are one W block (0) and one V block (1), or in
    // the symmetric mode one V block, emitted with its W block; G blocks are
    // not written out
    if (SYM) {
        if (kWinT[r][0].eu != 2)
            emit_v_w(kWinT[r][0].el, kWinT[r][0].ek, blk_id(kWinT[r][0].dst), w.xu, w.xl, w.pu, w.pv, w.mode, t, NT);
    } else if (kWinT[r][0].eu != 2) {
        emit_pair(kWinT[r][0].el, kWinT[r][0].ek, blk_id(kWinT[r][0].dst), kWinT[r][1].el, kWinT[r][1].ek,
                  blk_id(kWinT[r][1].dst), w.xu, w.xl, w.pu, w.pv, w.mode, t, NT);
    }
}

// W(q) on a group of NT threads (t = thread index in the group), barrier BAR.
// The G round takes 16 x 16 tasks (12 for its three blocks); the chain
// rounds (two blocks) 16 x 8 TC columns.
template <int NT, int BAR, int TC, bool SYM>
__device__ __noinline__ void inverse_window(int q, int t, int lane, const WinArgs &wa) {
    static_assert(3 * 4 * 32 <= NT && 2 * (8 / TC) * 32 <= NT, "one task per warp");
    const WinArgs w = wa;  // in registers: stores through the pointers cannot alias it
    // write-back: block row q from the diagonal on, then block column q below
    // it, four columns per thread (scalar where the block's last columns stop
    // inside the four); offsets from the block's corner fit in 32 bits
    float *const cre = w.gre + (w.J * w.ld + w.J), *const cim = w.gim + (w.J * w.ld + w.J);
    const int ld = (int)w.ld, nb = w.nb, c0 = q * P;
    auto put = [&](int i, int j) {
        if (i >= nb || j >= nb) return;
        const int g = i * ld + j;
        const float4 re = *reinterpret_cast<const float4 *>(&smem[i * LDA + j]);
        const float4 im = *reinterpret_cast<const float4 *>(&smem[IM_A + i * LDA + j]);
        if (j + 4 <= nb) {
            *reinterpret_cast<float4 *>(cre + g) = re;
            *reinterpret_cast<float4 *>(cim + g) = im;
        } else {
            const float r4[4] = {re.x, re.y, re.z, re.w}, i4[4] = {im.x, im.y, im.z, im.w};
            for (int u = 0; u < nb - j; u++) {
                cre[g + u] = r4[u];
                cim[g + u] = i4[u];
            }
        }
    };
    for (int idx = t; idx < P * (NB / 4); idx += NT) {  // rows c0.., all columns from c0 on
        const int i = c0 + (idx >> 5), j = (idx & 31) * 4;
        if (j >= c0) put(i, j);
    }
    for (int idx = t; idx < (NB - c0 - P) * (P / 4); idx += NT)  // rows below, columns c0..c0+31
        put(c0 + P + (idx >> 3), c0 + (idx & 7) * 4);
    // DU_q and DL_q: by the four LU warps for q < 3 (they finish the next
    // panel's base LU well before the window ends), here for the last panel
    if constexpr (NT == kThreads) emit_pair(q, q, blkDU(q), q, q, blkDL(q), w.xu, w.xl, w.pu, w.pv, w.mode, t, NT);
    const int r0 = kWinFirst[q];
    win_round<2, NT, BAR, SYM>(r0, t, lane, w);
    // the symmetric mode's chain rounds form one block: 16 x 8 tasks
    constexpr int TCR = SYM ? 1 : TC;
#pragma unroll 1
    for (int r = r0 + 1; r <= r0 + q; r++) win_round<TCR, NT, BAR, SYM>(r, t, lane, w);
}

// Symmetric mode: the part of panel q's update that the next panel's base LU
// does not wait for, A_ij -= L_iq U_qj on the blocks q < j <= i except
// (q + 1, q + 1), in 16 x 16 tasks by the threads t < nt of a group.  It
// runs beside the next panel's base LU; that panel's products read it only
// after the barrier that ends the LU.
__device__ __forceinline__ void sym_update_rest(int q, int t, int nt, int lane) {
    const int rest = 3 - q, ntask = 4 * (rest * (rest + 1) / 2 - 1);
    for (int task = t >> 5; task < ntask; task += nt >> 5) {
        const int b = (task >> 2) + 1, r0 = ((task >> 1) & 1) * 16, c0 = (task & 1) * 16;  // b = 0 is the diagonal block
        int i = 0;
        while ((i + 1) * (i + 2) / 2 <= b) i++;
        const int bi = q + 1 + i, bj = q + 1 + b - i * (i + 1) / 2;
        CAcc<2> acc;
        cacc_zero(acc);
        cmma(blkA(bi, q), blkA(q, bj), r0, c0, lane, acc);
        cacc_out<2, true>(blkA(bi, bj), r0, c0, lane, acc, 1.f);
    }
}

template <bool SYM>
__global__ void __launch_bounds__(kThreads, 1)
k_diag_block(float *__restrict__ z32, int64_t ld, int64_t plane, int64_t z32_stride, int64_t J, int nb,
             const int *__restrict__ slots, int *__restrict__ pivflag, float *__restrict__ inv32,
             int64_t inv32_stride, float *__restrict__ dinv, int64_t dinv_stride, float *__restrict__ winv,
             int mode) {
    __shared__ unsigned s_amax;
    __shared__ int s_bad;
    __shared__ unsigned s_rowflag[P];  // publication of the base LU's rows
    const int slot = slots[blockIdx.x];
    float *gre = z32 + (int64_t)slot * z32_stride;
    float *gim = gre + plane;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t rowflag = (uint32_t)__cvta_generic_to_shared(s_rowflag);
    if (tid == 0) {
        s_amax = 0u;
        s_bad = 0;
        for (int k = 0; k < P; k++) s_rowflag[k] = 0u;
    }
    __syncthreads();
    // ---- load (identity padding beyond nb)
    float amax = 0.f;
    if (nb == NB) {
        // a whole block: 16-byte loads (rows of ld floats, ld a multiple of
        // 32, and J a multiple of 128), all of a thread's in flight at once
        const float *bre = gre + J * ld + J, *bim = gim + J * ld + J;
#pragma unroll
        for (int u = 0; u < NB * NB / 4 / kThreads; u++) {
            const int idx = tid + u * kThreads, i = idx >> 5, j = (idx & 31) * 4;
            const float4 a = __ldcg(reinterpret_cast<const float4 *>(bre + i * ld + j));
            const float4 b = __ldcg(reinterpret_cast<const float4 *>(bim + i * ld + j));
            amax = fmaxf(amax, fmaxf(fmaxf(fabsf(a.x) + fabsf(b.x), fabsf(a.y) + fabsf(b.y)),
                                     fmaxf(fabsf(a.z) + fabsf(b.z), fabsf(a.w) + fabsf(b.w))));
            *reinterpret_cast<float4 *>(&smem[i * LDA + j]) = a;
            *reinterpret_cast<float4 *>(&smem[IM_A + i * LDA + j]) = b;
        }
    } else {
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
    }
    if (!(amax <= 3.0e38f)) amax = 3.0e38f;  // non-finite inputs: the pivot test flags them
    atomicMax(&s_amax, __float_as_uint(amax));
    __syncthreads();
    const float tiny = 1e-30f * __uint_as_float(s_amax);

    WinArgs wa;
    wa.gre = gre;
    wa.gim = gim;
    wa.ld = ld;
    wa.J = J;
    wa.nb = nb;
    wa.mode = mode;
    wa.xl = dinv + (int64_t)slot * dinv_stride + (J / NB) * 4 * NB * NB;  // [L, U][re, im][128][128]
    wa.xu = wa.xl + 2 * NB * NB;
    wa.pv = winv ? winv + (int64_t)slot * ZS_WINV_STRIDE + 2 * ZS_WINV_PLANE : nullptr;
    // the symmetric mode's block solves take V's pack alone: no W pack
    wa.pu = winv && !SYM ? winv + (int64_t)slot * ZS_WINV_STRIDE : nullptr;

    // ---- LU, one 32-column panel at a time; W(p - 1) beside the base LU of panel p
    for (int p = 0; p < 4; p++) {
        if (warp < kLuWarps) {
            if (base_lu(p, warp, lane, tiny, rowflag) && lane == 0) s_bad = 1;
            if (p > 0)
                emit_pair(p - 1, p - 1, blkDU(p - 1), p - 1, p - 1, blkDL(p - 1), wa.xu, wa.xl, wa.pu, wa.pv, mode,
                          tid, kLuWarps * 32);
        } else if (p > 0) {
            inverse_window<kThreads - kLuWarps * 32, 2, 2, SYM>(p - 1, tid - kLuWarps * 32, lane, wa);
            if (SYM) sym_update_rest(p - 1, tid - kLuWarps * 32, kThreads - kLuWarps * 32, lane);
        }
        __syncthreads();
        if (SYM) base_inv_sym(p, warp, lane);
        else base_inv(p, warp, lane);
        __syncthreads();
        const int rest = 3 - p;
        if (rest == 0) break;
        if (SYM) {
            // L_ip = A_ip DU_p in 16 x 16 tasks, four per block
            {
                CAcc<2> acc;
                cacc_zero(acc);
                const int t = warp, b = t >> 2, r0 = ((t >> 1) & 1) * 16, c0 = (t & 1) * 16;
                const bool on = t < 4 * rest;
                if (on) cmma(blkA(p + 1 + b, p), blkDU(p), r0, c0, lane, acc);
                __syncthreads();
                if (on) cacc_out<2, false>(blkA(p + 1 + b, p), r0, c0, lane, acc, 1.f);
                __syncthreads();
            }
            // U_pj = D_p L_jp^T, the upper factor's blocks of this panel
            for (int idx = tid; idx < rest * P * P; idx += kThreads) {
                const int jb = idx >> 10, a = (idx >> 5) & 31, c = idx & 31;
                st_c(blkA(p, p + 1 + jb), a, c, zs::cmul(ld_c(blkA(p, p), a, a), ld_c(blkA(p + 1 + jb, p), c, a)));
            }
            __syncthreads();
            // the next diagonal block first, A_(p+1)(p+1) -= L_(p+1)p U_p(p+1), in
            // 16 x 8 tasks; the rest of the update runs beside the next base LU
            if (warp < 8) {
                const int r0 = (warp >> 2) * 16, c0 = (warp & 3) * 8;
                CAcc<1> acc;
                cacc_zero(acc);
                cmma(blkA(p + 1, p), blkA(p, p + 1), r0, c0, lane, acc);
                cacc_out<1, true>(blkA(p + 1, p + 1), r0, c0, lane, acc, 1.f);
            }
            __syncthreads();
            continue;
        }
        // L_ip = A_ip DU_p (tasks 0 .. 2 rest - 1), U_pj = DL_p A_pj (the next 2 rest),
        // 16-row tasks; tasks read rows of A_pj that other tasks overwrite:
        // write after a barrier
        {
            CAcc<4> acc;
            cacc_zero(acc);
            const int t = warp, ntask = 4 * rest, b = t >> 1, r0 = (t & 1) * 16;
            const bool lpanel = b < rest;
            if (t < ntask)
                cmma(lpanel ? blkA(p + 1 + b, p) : blkDL(p), lpanel ? blkDU(p) : blkA(p, p + 1 + b - rest), r0, 0, lane,
                     acc);
            __syncthreads();
            if (t < ntask)
                cacc_out<4, false>(lpanel ? blkA(p + 1 + b, p) : blkA(p, p + 1 + b - rest), r0, 0, lane, acc, 1.f);
            __syncthreads();
        }
        // A_ij -= L_ip U_pj, i, j > p, 16 x 16 tasks: each task owns its output
        for (int t = warp; t < 4 * rest * rest; t += kWarps) {
            const int b = t >> 2, r0 = ((t >> 1) & 1) * 16, c0 = (t & 1) * 16;
            const int bi = p + 1 + b / rest, bj = p + 1 + b % rest;
            CAcc<2> acc;
            cacc_zero(acc);
            cmma(blkA(bi, p), blkA(p, bj), r0, c0, lane, acc);
            cacc_out<2, true>(blkA(bi, bj), r0, c0, lane, acc, 1.f);
        }
        __syncthreads();
    }

    inverse_window<kThreads, 0, 1, SYM>(3, tid, lane, wa);

    // ---- the 32 x 32 inverses, when the FP32 block solves want them
    if (inv32) {
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

}  // namespace

cudaError_t zs_launch_diag_block(float *z32, int64_t ld, int64_t plane, int64_t z32_stride, int64_t J, int nb,
                                 const int *slots, int nslot, int *pivflag, float *inv32, int64_t inv32_stride,
                                 float *dinv, int64_t dinv_stride, float *winv, int mode, int sym, cudaStream_t st) {
    if (nb <= 0 || nb > NB || nslot <= 0 || !dinv) return cudaErrorInvalidValue;
    if (winv && mode != 1 && mode != 2) return cudaErrorInvalidValue;
    // once per process (thread-safe initialisation of a local static)
    static const cudaError_t attr = [] {
        const cudaError_t a = cudaFuncSetAttribute(k_diag_block<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   (int)kSmemBytes);
        return a != cudaSuccess ? a
                                : cudaFuncSetAttribute(k_diag_block<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                       (int)kSmemBytes);
    }();
    if (attr != cudaSuccess) return attr;
    if (sym)
        k_diag_block<true><<<nslot, kThreads, kSmemBytes, st>>>(z32, ld, plane, z32_stride, J, nb, slots, pivflag,
                                                                 inv32, inv32_stride, dinv, dinv_stride, winv, mode);
    else
        k_diag_block<false><<<nslot, kThreads, kSmemBytes, st>>>(z32, ld, plane, z32_stride, J, nb, slots, pivflag,
                                                                  inv32, inv32_stride, dinv, dinv_stride, winv, mode);
    return cudaGetLastError();
}
