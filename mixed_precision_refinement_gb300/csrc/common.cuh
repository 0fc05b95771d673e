// Shared device helpers and launcher declarations for the zsolve kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#define ZS_NB 128           // outer block: columns factored per step of the blocked LU
#define ZS_PANEL 32         // panel width inside the outer block (the page factorises in blocks of 32)
#define ZS_TB 64            // row block of the sequential-diagonal triangular solve
#define ZS_TB2 128          // row block of the inverse-diagonal triangular solve
#define ZS_SPIN_LIMIT (1u << 22)  // bounded waits: polls (>= 64 ns apart) before a wait gives up

// device status bits (one word per context)
#define ZS_DEV_TIMEOUT 1u

namespace zs {

__host__ __device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }

struct cf {  // complex float
    float re, im;
};

__device__ __forceinline__ cf cmul(cf a, cf b) {
    return {a.re * b.re - a.im * b.im, a.re * b.im + a.im * b.re};
}

// a - b*c
__device__ __forceinline__ cf cfms(cf a, cf b, cf c) {
    return {fmaf(-b.re, c.re, fmaf(b.im, c.im, a.re)), fmaf(-b.re, c.im, fmaf(-b.im, c.re, a.im))};
}

// 1/p with a scale to keep the squared modulus in range
__device__ __forceinline__ cf crecip(cf p) {
    float s = fmaxf(fabsf(p.re), fabsf(p.im));
    float a = p.re / s, b = p.im / s;
    float d = s * (a * a + b * b);
    return {a / d, -b / d};
}

__device__ __forceinline__ bool cfinite(cf a) { return isfinite(a.re) && isfinite(a.im); }

// The two 32-bit halves of a double, moved out through PTX so that tests on
// the bit pattern stay integer operations: written on a 64-bit integer, a
// test such as "all bits but the sign are zero" may be turned back into a
// floating-point compare, which on this GPU occupies the slow FP64 pipe.
struct Bits64 {
    unsigned lo, hi;
};
__device__ __forceinline__ Bits64 bits_of(double x) {
    Bits64 b;
    asm("mov.b64 {%0, %1}, %2;" : "=r"(b.lo), "=r"(b.hi) : "d"(x));
    return b;
}
__device__ __forceinline__ double double_of(unsigned lo, unsigned hi) {
    double x;
    asm("mov.b64 %0, {%1, %2};" : "=d"(x) : "r"(lo), "r"(hi));
    return x;
}
__device__ __forceinline__ bool is_zero(Bits64 b) { return ((b.hi << 1) | b.lo) == 0u; }  // +0 or -0
// c ? a : b for doubles as two 32-bit integer selects (no FP64 instruction)
__device__ __forceinline__ double sel_bits(bool c, double a, double b) {
    const Bits64 x = bits_of(a), y = bits_of(b);
    return double_of(c ? x.lo : y.lo, c ? x.hi : y.hi);
}
// -x by flipping the sign bit on the integer side (no FP64 instruction)
__device__ __forceinline__ double neg_bits(double x) {
    const Bits64 b = bits_of(x);
    return double_of(b.lo, b.hi ^ 0x80000000u);
}

// Bounded wait until *flag == want.  Returns false (and raises the timeout bit
// in *status) if it never happens within ZS_SPIN_LIMIT polls.
__device__ __forceinline__ bool wait_flag(const unsigned *flag, unsigned want, unsigned *status) {
    unsigned it = 0;
    while (true) {
        unsigned v;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
        if (v == want) return true;
        if (++it > ZS_SPIN_LIMIT) {
            atomicOr(status, ZS_DEV_TIMEOUT);
            return false;
        }
        // another wait already gave up: stop too, so the launch ends promptly
        if ((it & 1023u) == 0 && (*(volatile const unsigned *)status & ZS_DEV_TIMEOUT)) return false;
        if (it > 64) __nanosleep(256);
    }
}

// In-order progress counters: the 64-bit word holds (epoch << 32) | count,
// where count blocks of this launch's epoch are complete.  Returns the count
// once it exceeds `need` (bounded wait as above), or -1 on give-up.
__device__ __forceinline__ long long progress_read(const unsigned long long *p, unsigned epoch) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return (unsigned)(v >> 32) == epoch ? (long long)(v & 0xffffffffull) : 0;
}

__device__ __forceinline__ long long progress_wait(const unsigned long long *p, unsigned epoch, long long need,
                                                   unsigned *status, unsigned limit = ZS_SPIN_LIMIT) {
    unsigned it = 0;
    while (true) {
        long long c = progress_read(p, epoch);
        if (c > need) return c;
        if (++it > limit) {
            atomicOr(status, ZS_DEV_TIMEOUT | (0x80u << 8));  // site: a triangular-solve progress word
            return -1;
        }
        if ((it & 1023u) == 0 && (*(volatile const unsigned *)status & ZS_DEV_TIMEOUT)) return -1;
        // short sleeps once the block just before the needed one is in work
        if (it > 32) __nanosleep(c == need || it <= 4096 ? 32 : 256);
    }
}

__device__ __forceinline__ void progress_set(unsigned long long *p, unsigned epoch, unsigned count) {
    unsigned long long v = ((unsigned long long)epoch << 32) | count;
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ void set_flag(unsigned *flag, unsigned v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(flag), "r"(v) : "memory");
}

__device__ __forceinline__ bool timed_out(const unsigned *status) {
    return (*(volatile const unsigned *)status & ZS_DEV_TIMEOUT) != 0;
}

}  // namespace zs

// Per-slot parameters of a batch (one slot = one frequency being solved);
// pad carries RN(1/omega), computed on the host.
struct ZsSlotParam {
    double omega, zs_re, zs_im, pad;
};

// Accessors of the solver context for the other translation units (afs.cu).
struct zsolve_ctx;
cudaStream_t zs_ctx_stream(const zsolve_ctx *ctx);
int64_t zs_ctx_n(const zsolve_ctx *ctx);
int zs_ctx_nrhs_max(const zsolve_ctx *ctx);

// ---------------------------------------------------------------- launchers
// All return cudaGetLastError() of the launch.  Matrices of a batch are
// strided by the given slot strides (elements).

// Z64 (c128, ld n) and the complex float32 planes (re at z32, im at z32 + plane;
// z32 = NULL: Z64 alone), rows r0 .. r1-1.  zexp (NULL: not recorded): per slot n ints, the largest
// biased exponent of each row of the slot's Z64.
cudaError_t zs_launch_assemble(const double *L, const double *Psi, const double *G, int64_t n, int64_t r0, int64_t r1,
                               const ZsSlotParam *params, int nslot, double2 *z64, int64_t z64_stride,
                               float *z32, int64_t ld, int64_t plane, int64_t z32_stride,
                               cudaStream_t st, int *zexp = nullptr);
// The float32 planes alone, rows r0 .. r1-1, without float64 arithmetic per
// frequency (double-float evaluation rounded once; assemble.cu)
cudaError_t zs_launch_assemble32(const double *L, const double *Psi, const double *G, int64_t n, int64_t r0,
                                 int64_t r1, const ZsSlotParam *params, int nslot, float *z32, int64_t ld,
                                 int64_t plane, int64_t z32_stride, cudaStream_t st);

// Factorisation steps at outer-block column J for nslot slots listed in slots[].
// inv32: per slot and outer block, ZS_INV32_STRIDE floats:
// [sub-block kb][U, L][re, im][32][32], the inverses of the four 32x32
// diagonal sub-blocks of U and of L (identity padding in a partial block).
#define ZS_INV32_STRIDE (4 * 2 * 2 * 32 * 32)
inline int64_t zs_inv32_slot_stride(int64_t n) { return ((n + 127) / 128) * ZS_INV32_STRIDE; }
// Diagonal block at J (nb <= 128 columns, identity-padded to 128): its LU in
// place in z32; the dense 128x128 inverses of its L and U into dinv (zero
// outside the triangles from the allocation on: only the triangles are
// written) and, if winv != NULL, their operand packs (mode 1: tf32 hi; 2: hi
// + lo); if inv32 != NULL, the 32x32 sub-block inverses.  pivflag[slot] = 1
// on a tiny or non-finite pivot.  sym = 1: the symmetric mode's form, the
// lower blocks alone factored and U = D L^T within the block (its upper
// blocks and U^-1 = L^-T D^-1 formed from L), for a block that is symmetric.
cudaError_t zs_launch_diag_block(float *z32, int64_t ld, int64_t plane, int64_t z32_stride, int64_t J, int nb,
                                 const int *slots, int nslot, int *pivflag, float *inv32, int64_t inv32_stride,
                                 float *dinv, int64_t dinv_stride, float *winv, int mode, int sym,
                                 cudaStream_t st);
// mode: 0 = pack plain fp32 (FFMA), 1 = tf32 rounded (TF32), 2 = tf32 hi + lo (TF32X3)
cudaError_t zs_launch_trsm_l(float *z32, int64_t ld, int64_t plane, int64_t z32_stride, int64_t n,
                             int64_t J, const float *inv32, int64_t inv32_stride, float *pack, int64_t pack_stride,
                             int mode, const int *slots, int nslot, cudaStream_t st);
cudaError_t zs_launch_trsm_u(float *z32, int64_t ld, int64_t plane, int64_t z32_stride, int64_t n,
                             int64_t J, const float *inv32, int64_t inv32_stride, float *pack, int64_t pack_stride,
                             int mode, const int *slots, int nslot, cudaStream_t st);
cudaError_t zs_launch_schur_simt(float *z32, int64_t ld, int64_t plane, int64_t z32_stride, int64_t n,
                                 int64_t J, const float *pack, int64_t pack_stride, const int *slots,
                                 int nslot, cudaStream_t st);

// Operand packs of the block triangular solves on the tensor cores, at outer
// column J: A planes rows i >= J+NB = [Re A21(i,:) | Im A21(i,:)], Br planes
// rows j >= J+NB = [Re A12(:,j) | Im A12(:,j)] (mode 1: tf32 hi; 2: hi + lo).
// sym = 1: Z is complex symmetric and only its lower part is current; the A
// planes only (all the symmetric block solve reads).
cudaError_t zs_launch_pack_trsm(const float *z32, int64_t ld, int64_t plane, int64_t z32_stride, int64_t n,
                                int64_t J, float *pack, int64_t pack_stride, int mode, int sym, const int *slots,
                                int nslot, cudaStream_t st);

// tcgen05 kernels (schur_tc.cu).  Tensor maps are 128-byte CUtensorMap
// objects in host memory, passed by value to the kernels.
cudaError_t zs_tc_pack_map(const float *pack, int64_t n, int nslots, int64_t pack_stride, int box_rows,
                           void *map_out);
cudaError_t zs_tc_winv_map(const float *winv, int nslots, void *map_out);
cudaError_t zs_tc_z32_map(const float *z32, int64_t n, int64_t ld, int64_t plane, int nslots, int64_t z32_stride,
                          void *map_out);
// A22 -= L21 U12 for every listed slot (split: 3xTF32), at most max_grid
// persistent CTAs that take tiles from *ctr (zero before the launch).
// lower: only the tiles on and below the diagonal (complex-symmetric Z).
// part: ZS_PART_ALL, or ZS_PART_COL0 (the first 128-column tile: the next
// step's diagonal block and A21) and ZS_PART_REST (the other tiles).
#define ZS_PART_ALL 0
#define ZS_PART_COL0 1
#define ZS_PART_REST 2
cudaError_t zs_launch_schur_tc(const void *map, const void *cmap, int64_t n, int64_t J, int split, int lower,
                               int part, const int *slots, int nslot, unsigned *ctr, unsigned *status, int max_grid,
                               cudaStream_t st);
// L21 = A21 U11^-1 and U12 = L11^-1 A12 from the packs of zs_launch_pack_trsm
// and zs_launch_diag_block; writes L21, U12 into z32 and their operand packs.
// sym: Z complex symmetric (A12 = A21^T, U11 = D11 L11^T): one product per row
// tile, U12^T = A21 L11^-T, and L21 = U12^T D11^-1 with D11^-1 the diagonal of
// the float32 inverse blocks (dinv, per slot dinv_stride floats); the packs
// then need only A21's rows in the A planes, and the epilogue writes U12 and
// L21 into z32 and the update's one operand pack M = U12^T S, S^2 = D11^-1
// entrywise, into the A planes (the lower update takes both operands from M).
cudaError_t zs_launch_trsm_tc(const void *map, const void *wmap, const void *cmap, const void *pmap, int64_t n,
                              int64_t J, int split, int sym, const float *dinv, int64_t dinv_stride,
                              const int *slots, int nslot, unsigned *ctr, unsigned *status, int num_sms,
                              cudaStream_t st);

// Pack layout (floats), per slot: six planes of n rows x 2*NB:
//   A_hi, A_lo, Br_hi, Br_lo, Bi_hi, Bi_lo
// A row i   = [Re L21(i,:) | Im L21(i,:)]
// Br row j  = [Re U12(:,j) | -Im U12(:,j)]   (Cr = A . Br)
// Bi row j  = [Im U12(:,j) |  Re U12(:,j)]   (Ci = A . Bi; written by the FP32
//                                             path only: the tensor-core update
//                                             takes Bi from Br's K halves)
#define ZS_PACK_K (2 * ZS_NB)
__host__ __device__ inline int64_t zs_pack_plane(int64_t n) { return n * (int64_t)ZS_PACK_K; }

// Triangular solves with the float32 factors: v (c64 interleaved, per active
// slot nrhs rows of n) is overwritten by (LU)^-1 v.
// prog: two in-order progress words (forward, backward) per slot.
// Sequential 64x64 diagonal solves; needs no data beyond the factors.
cudaError_t zs_launch_trsv_seq(const float *z32, int64_t ld, int64_t plane, int64_t z32_stride, int64_t n,
                           float2 *v, int64_t v_stride, int nrhs, const int *slots, int nslot,
                           unsigned long long *prog, unsigned epoch, unsigned *ticket,
                           unsigned *status, int num_sms, cudaStream_t st);

// Inverses of the 128x128 diagonal blocks of L (unit lower) and U (upper):
// per slot [block][L, U][re, im][128][128] floats.  Operand packs of one
// block's inverses for the tensor-core solves, per slot ZS_WINV_STRIDE floats
// = 4 planes of 128 rows x 256:
//   planes 0-1 W = U^-1: Br(j) = [Re W(:,j) | -Im W(:,j)], hi and lo
//   planes 2-3 V = L^-1: Br(k) = [Re V(k,:) | -Im V(k,:)], hi and lo
// No Bi = [Im | Re] plane is kept: the tensor-core block solve takes Bi from
// Br's other K half, with the sign on the MMA's negate-B.
#define ZS_WINV_PLANE (ZS_NB * ZS_PACK_K)
#define ZS_WINV_STRIDE (4 * ZS_WINV_PLANE)
inline int64_t zs_dinv_stride(int64_t n) { return ((n + ZS_TB2 - 1) / ZS_TB2) * 4 * ZS_TB2 * ZS_TB2; }
// Triangular solves with 128-row blocks and the inverse diagonal blocks:
// per slot, ngroup independent groups of nrhs (1, 2 or 4) right-hand sides
// each (group g = rows g*nrhs .. g*nrhs+nrhs-1 of the slot's v), solved as
// separate dependency chains side by side in one launch.
// prog: two progress words per (slot, group), at 2 * (slot * ZS_TRSV_MAX_GROUPS + g).
// wait_limit: polls before a wait for another task's block gives up (raising
// ZS_DEV_TIMEOUT in *status).  first_ticket: the task ticket starts here
// (0 in every solve; a positive value withholds the first tasks, so that the
// bounded waits can be shown to give up -- a testing aid).
#define ZS_TRSV_MAX_GROUPS 8
cudaError_t zs_launch_trsv_inv(const float *z32, int64_t ld, int64_t plane, int64_t z32_stride, int64_t n,
                               const float *dinv, int64_t dinv_stride, float2 *v, int64_t v_stride, int nrhs,
                               int ngroup, const int *slots, int nslot, unsigned long long *prog, unsigned epoch,
                               unsigned *ticket, unsigned *status, int num_sms, cudaStream_t st,
                               unsigned wait_limit = ZS_SPIN_LIMIT, unsigned first_ticket = 0);

// r = b - Z64 x.  out_c64 != NULL: writes float2 (rounded); else writes c128 to out_c128.
// Launches one kernel per chunk of 8/4/2/1 right-hand sides (zs_rhs_chunks).
cudaError_t zs_launch_residual(const double2 *z64, int64_t z64_stride, int64_t n, const double2 *b,
                               const double2 *x, int64_t x_stride, int nrhs, float2 *out_c64,
                               int64_t out64_stride, double2 *out_c128, int64_t out128_stride,
                               const int *slots, int nslot, cudaStream_t st);
inline int zs_rhs_chunks(int nrhs) {
    int c = 0;
    while (nrhs > 0) {
        nrhs -= nrhs >= 8 ? 8 : nrhs >= 4 ? 4 : nrhs >= 2 ? 2 : 1;
        c++;
    }
    return c;
}

// Double-float residual: x split into float4 (Re hi, Re lo, Im hi, Im lo) per element first.
cudaError_t zs_launch_split_x(const double2 *x, int64_t x_stride, int64_t n, int nrhs, float4 *xs, int64_t xs_stride,
                              const int *slots, int nslot, cudaStream_t st);
cudaError_t zs_launch_residual_df(const double2 *z64, int64_t z64_stride, int64_t n, const double2 *b, const float4 *xs,
                                  int64_t xs_stride, int nrhs, float2 *out_c64, int64_t out64_stride,
                                  double2 *out_c128, int64_t out128_stride, const int *slots, int nslot,
                                  cudaStream_t st);
cudaError_t zs_launch_selftest_fill(double2 *z, double2 *x, int64_t n, int zero_re, cudaStream_t st);

// r = b - (j w L x - j Psi x / w + Zs G x) from L, Psi, G (n x n float64) for
// every listed slot (params indexed by slot), groups of frequencies per pass
// over a row (resid_lpg.cu).  Output as zs_launch_residual.
cudaError_t zs_launch_residual_lpg(const double *L, const double *Psi, const double *G, int64_t n,
                                   const ZsSlotParam *params, const double2 *b, const double2 *x, int64_t x_stride,
                                   int nrhs, float2 *out_c64, int64_t out64_stride, double2 *out_c128,
                                   int64_t out128_stride, const int *slots, int nslot, cudaStream_t st);

// Residual from L, Psi, G on the bf16 tensor cores with error-free splitting
// (resid_oz.cu).  The digits of A' = [L; Psi; G] (8 planes, stored tile-major
// in units of 128 rows x 128 K, zs_oz_a_bytes(n) bytes, zero before the first
// use) and their row scales (ea, 3n
// ints) are formed once per set of L, Psi, G, rows r0..r1-1 of each matrix
// per call; amap (a CUtensorMap, 64-byte aligned) describes them.  Per
// evaluation: the digits of x (xdig: 8 planes of ncol_cap rows x n_pad bf16,
// ex: ncol_cap ints, ncol = 2 nslot nrhs <= ncol_cap), the partial products
// (part: part_cap doubles; the product runs on up to num_sms CTAs, fewer if
// a tile's K range would be split into more segments than part holds) and
// then r as zs_launch_residual.
int64_t zs_oz_n_pad(int64_t n);
int64_t zs_oz_a_bytes(int64_t n);  // bytes of A's digits (tile-major, zero padded)
int zs_oz_ncol_alloc(int ncol);
cudaError_t zs_launch_oz_split_a(const double *L, const double *Psi, const double *G, int64_t n, int64_t r0,
                                 int64_t r1, void *dig, int *ea, cudaStream_t st);
cudaError_t zs_oz_a_map(const void *dig, int64_t n, void *map_out);
cudaError_t zs_launch_residual_oz(const void *amap, const int *ea, int64_t n, const ZsSlotParam *params,
                                  const double2 *b, const double2 *x, int64_t x_stride, int nrhs, float2 *out_c64,
                                  int64_t out64_stride, double2 *out_c128, int64_t out128_stride, const int *slots,
                                  int nslot, void *xdig, int *ex, int ncol_cap, double *part, int64_t part_cap,
                                  unsigned *status, int num_sms, cudaStream_t st);

// Fixed-point residual (resid_fx.cu): x split into exact 24-bit limbs per
// right-hand side (xl: per slot xl_stride bytes, zs_fx_x_bytes(n) per right-hand side; xe: per
// (slot, rhs) the scale exponent, index slot * nrhs_max + r), then r = b - Z64 x
// with exact integer products and sums.  zexp: per slot n ints, the largest
// biased exponent of each row of Z64 (written by zs_launch_assemble).
int64_t zs_fx_x_bytes(int64_t n);  // bytes of one right-hand side's limbs
cudaError_t zs_launch_split_fx(const double2 *x, int64_t x_stride, int64_t n, int nrhs, unsigned char *xl,
                               int64_t xl_stride, int *xe, int nrhs_max, const int *slots, int nslot, cudaStream_t st);
// ndf (0..3): of every four 32-column sub-steps, how many take float64 products (DFMA) instead.
cudaError_t zs_launch_residual_fx(const double2 *z64, int64_t z64_stride, const int *zexp, int64_t n, const double2 *b,
                                  const double2 *x, int64_t x_stride, const unsigned char *xl, int64_t xl_stride,
                                  const int *xe, int nrhs_max, int nrhs, float2 *out_c64, int64_t out64_stride,
                                  double2 *out_c128, int64_t out128_stride, const int *slots, int nslot, int ndf,
                                  cudaStream_t st);

// v = (float2) b for every listed slot
cudaError_t zs_launch_cast_rhs(const double2 *b, int64_t n, int nrhs, float2 *v, int64_t v_stride,
                               const int *slots, int nslot, cudaStream_t st);

// x = d (assign) or x += d; partial sums of |d|^2 and |x|^2 per (slot, rhs, chunk)
cudaError_t zs_launch_update(double2 *x, int64_t x_stride, const float2 *d, int64_t d_stride,
                             int64_t n, int nrhs, int assign, double *partials, int nchunks,
                             const int *slots, int nslot, cudaStream_t st);
// relcorr[slot*nrhs + r] = sqrt(sum|d|^2 / sum|x|^2) (inf/nan if non-finite)
cudaError_t zs_launch_relcorr(const double *partials, int nchunks, int nrhs, double *relcorr,
                              const int *slots, int nslot, cudaStream_t st);
int zs_update_chunks(int64_t n);

// d (c128) from v (c64) for the stage-level solve call
cudaError_t zs_launch_widen(const float2 *v, double2 *d, int64_t count, cudaStream_t st);
cudaError_t zs_launch_narrow(const double2 *d, float2 *v, int64_t count, cudaStream_t st);
cudaError_t zs_launch_copy_z32_out(const float *z32, int64_t ld, int64_t plane, int64_t n, float *re,
                                   float *im, cudaStream_t st);

// float64 LU with partial pivoting (the fallback) on a c128 matrix with ld n.
// *launches (if not NULL) is increased by the number of kernels launched.
cudaError_t zs_lu64_factor(double2 *a, int64_t n, int64_t *piv, int *info, cudaStream_t st, int64_t *launches);
cudaError_t zs_lu64_solve(const double2 *lu, int64_t n, const int64_t *piv, double2 *x, int nrhs,
                          cudaStream_t st, int64_t *launches);
