// Trailing (Schur) update of the low-precision LU on the 5th-generation
// tensor cores: A22 -= L21 U12 (malusrfworks.com, "Solving Dense Matrices
// Fast in the Browser", section "Double-precision answers from a GPU without
// double precision", step 1: the factorisation's matrix products, done there
// in 64x64 tiles).
//
// The complex product is two real products over the operand packs written by
// the block triangular solves (K = 2 x 128 real):
//   Re(L21 U12) = A . Br^T,  Im(L21 U12) = A . Bi^T,
//   A = [Re L21 | Im L21],  Br = [Re U12^T | -Im U12^T],  Bi = [Im U12^T | Re U12^T].
// Bi is Br with its K halves swapped and the first half negated, so only Br
// is stored: for a 32-wide K chunk at k, Bi's chunk is -Br's at k + 128 (k <
// 128) or Br's at k - 128.  One CTA owns a 128-row x 128-column complex
// output tile in one fp32 TMEM accumulator of 256 columns: per K step one
// tcgen05.mma of M=128, N=128 for the real part (columns 0-127, B = Br's
// chunk) and one for the imaginary part (columns 128-255, B = Br's other
// chunk, negated by the instruction's negate-B bit where the sign is -).
//   split = 0: kind::tf32, operands rounded to tf32 once;
//   split = 1: 3xTF32 -- x = hi + lo with hi, lo tf32; the product is formed
//              as hi.hi + hi.lo + lo.hi (the lo.lo term is below fp32
//              rounding), which restores float32-class accuracy (Ootomo and
//              Yokota, "Recovering single precision accuracy from Tensor
//              Cores while surpassing the FP32 theoretical peak
//              performance", IJHPCA 2022).
//
// The same kernel runs the two block triangular solves of each step as
// products with the explicit inverses of the diagonal block (kind TRSM):
//   L21   = A21 U11^-1:   A rows i = [Re A21(i,:) | Im A21(i,:)] (A planes),
//                         B = W = U11^-1 as Br(j) = [Re W(:,j) | -Im W(:,j)],
//                         Bi(j) = [Im W(:,j) | Re W(:,j)];
//   U12^T = A12^T L11^-T: A rows j = [Re A12(:,j) | Im A12(:,j)] (Br planes),
//                         B = V = L11^-1 as Br(k) = [Re V(k,:) | -Im V(k,:)],
//                         Bi(k) = [Im V(k,:) | Re V(k,:)].
// Its epilogue stores the result twice with TMA tile stores: into the float32
// factor (U12 transposed on the way through shared memory) and, rounded to
// tf32 hi (+ lo), into the operand packs the trailing update reads next.  A
// tile's epilogue overwrites the very pack rows its own MMAs consumed, which
// is safe: the accumulator is complete only after every load of the tile.
//
// The symmetric mode (kinds SCHUR_LOWER and TRSM_SYM, below) needs one pack
// only: the block solve writes M = U12^T S with S^2 = D11^-1 entrywise into
// the A planes, and since M M^T = L21 U12, the lower update reads both of its
// operands from M's rows: B's real part is [Re M | Im M] with the negate-B
// bit on the second K half, B's imaginary part its K halves swapped, as is.
//
// Warp roles (192 threads, persistent over the tiles of every frequency in
// the batch): warp 0 issues TMA loads (128B-swizzled K-major tiles of 32
// fp32) into a ring of shared-memory stages; warp 1 owns TMEM (512 columns:
// two accumulators, so the epilogue of one tile overlaps the MMAs of the
// next) and issues the MMAs from one thread; warps 2-5 drain the accumulator
// with tcgen05.ld, stage the negated values in shared memory (128B swizzle,
// double-buffered per warp) and subtract them from the float32 trailing
// matrix with TMA reduce-add stores, so the L2 does the read-modify-write and
// the epilogue issues no global loads.  Every
// mbarrier wait is bounded: on give-up the kernel raises a status bit, stops
// all roles, waits (bounded) for its own copies and MMAs and frees TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"

namespace {

constexpr int NB = ZS_NB;
constexpr int KTOT = ZS_PACK_K;   // 256 real K per tile
constexpr int KC = 32;            // fp32 per 128-byte swizzle row
constexpr int NKC = KTOT / KC;    // 8 K chunks
constexpr int TM = 128, TN = 128; // complex output tile
constexpr int kThreads = 192;
constexpr int A_BYTES = TM * KC * 4;       // 16 KB
constexpr int B_BYTES = 2 * TN * KC * 4;   // 32 KB (B rows at chunk k, then the same rows at chunk k +- 128)
constexpr uint32_t TMEM_COLS = 512;
// try_wait polls before a wait gives up: about a second here (a poll that
// finds the phase incomplete suspends for some microseconds)
constexpr uint32_t kWaitLimit = 1u << 19;
constexpr int kTq = 8;  // tile-index queue between the roles (the producer runs at most a few tiles ahead)

enum { PL_A_HI = 0, PL_A_LO = 1, PL_BR_HI = 2, PL_BR_LO = 3, PL_BI_HI = 4, PL_BI_LO = 5 };
// inverse packs: W = U11^-1 in planes 0-1, V = L11^-1 in planes 2-3 (Br hi, Br lo each)
enum { WP_BR_HI = 0, WP_BR_LO = 1, WP_V = 2 };
// KIND_SCHUR_LOWER: the trailing update of a complex-symmetric matrix, whose
// Schur complement stays symmetric: only the tiles on and below the diagonal
// (column tile <= row tile) are formed; the next step reads only those.
// KIND_TRSM_SYM: the block solves of a complex-symmetric matrix in one
// product per row tile: with A12 = A21^T and U11 = D11 L11^T (D11 = diag U11),
// U12^T = A21 L11^-T from the MMAs, and L21 = A21 U11^-1 = U12^T D11^-1 in the
// epilogue, which writes both factors and the update's pack M (half the MMAs
// and operand loads of KIND_TRSM, and a third fewer stores than with
// separate L21 and U12^T packs).
enum { KIND_SCHUR = 0, KIND_TRSM = 1, KIND_SCHUR_LOWER = 2, KIND_TRSM_SYM = 3 };

template <int KIND>
constexpr bool is_trsm() {
    return KIND == KIND_TRSM || KIND == KIND_TRSM_SYM;
}

constexpr int EPI_BOX = 32 * 32 * 4;  // one 32-row x 32-column fp32 box (4 KB)
constexpr int EPI_BYTES = 4 * 2 * EPI_BOX;  // 4 epilogue warps x 2 staging buffers

template <int SPLIT>
struct Cfg {
    static constexpr int STAGE_BYTES = SPLIT ? 2 * (A_BYTES + B_BYTES) : (A_BYTES + B_BYTES);
    static constexpr int STAGES = SPLIT ? 2 : 4;
    static constexpr int SMEM = STAGES * STAGE_BYTES + EPI_BYTES + 1024;  // + alignment slack
};

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

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

// Bounded wait; gives up if another role already did (abort flag) or after
// kWaitLimit polls, raising the device status bit and recording the wait
// site in bits 8-15 of the status word (kernel kind << 4 | role wait 1-5).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                          unsigned *status, unsigned site) {
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

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *map, int c0, int c1, int c2, int c3,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
        "l"((uint64_t)map), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
        : "memory");
}

// Subtract a staged 32x32 box from the trailing matrix: TMA reduce-add (fp32)
__device__ __forceinline__ void tma_reduce_add_4d(const CUtensorMap *map, uint32_t src, int c0, int c1, int c2,
                                                  int c3) {
    asm volatile(
        "cp.reduce.async.bulk.tensor.4d.global.shared::cta.add.tile.bulk_group"
        " [%0, {%1, %2, %3, %4}], [%5];" ::"l"((uint64_t)map),
        "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(src)
        : "memory");
}

// Store a staged 32x32 box (TMA tile store; rows/columns beyond the tensor are dropped)
__device__ __forceinline__ void tma_store_4d(const CUtensorMap *map, uint32_t src, int c0, int c1, int c2, int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.global.shared::cta.tile.bulk_group"
        " [%0, {%1, %2, %3, %4}], [%5];" ::"l"((uint64_t)map),
        "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(src)
        : "memory");
}

__device__ __forceinline__ float tf32_rna(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}

using zs::cf;

// A square root of a complex float (the principal one): with t = sqrt((|a| +
// |z|) / 2), (t, b / 2t) for a >= 0, else (|b| / 2t, +-t) with the sign of b.
// |z| is formed from the larger part so that it does not overflow.  Only
// S^2 = z matters to its one caller, not the branch.
__device__ __forceinline__ cf csqrt_f(cf z) {
    const float a = fabsf(z.re), b = fabsf(z.im), m = fmaxf(a, b);
    if (m == 0.f) return cf{0.f, 0.f};
    const float n = fminf(a, b) / m, mod = m * sqrtf(1.f + n * n);
    const float t = sqrtf(0.5f * (a + mod)), u = 0.5f * b / t;
    return z.re >= 0.f ? cf{t, copysignf(u, z.im)} : cf{u, copysignf(t, z.im)};
}

// Row `lane` of a 32x32 fp32 box in 128B-swizzled shared memory: 16-byte unit
// j of row r sits at unit (j ^ (r & 7)).  sgn = -1 stores the negated values.
__device__ __forceinline__ void stage_row(uint32_t sb, int lane, const float (&v)[32], float sgn) {
#pragma unroll
    for (int j = 0; j < 8; j++) {
        const uint32_t a = sb + (uint32_t)lane * 128u + (uint32_t)((j ^ (lane & 7)) * 16);
        asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(a), "f"(sgn * v[4 * j]),
                     "f"(sgn * v[4 * j + 1]), "f"(sgn * v[4 * j + 2]), "f"(sgn * v[4 * j + 3])
                     : "memory");
    }
}

// Column `lane` of the same box layout (element (t, lane) = v[t]): the transpose.
__device__ __forceinline__ void stage_col(uint32_t sb, int lane, const float (&v)[32]) {
#pragma unroll
    for (int t = 0; t < 32; t++) {
        const uint32_t a = sb + (uint32_t)t * 128u + (uint32_t)((((lane >> 2) ^ (t & 7)) * 16) + (lane & 3) * 4);
        asm volatile("st.shared.f32 [%0], %1;" ::"r"(a), "f"(v[t]) : "memory");
    }
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// wait until at most N committed groups are still reading their shared source
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of
// 128 bytes, 8-row core groups 1024 bytes apart.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr) {
    uint64_t d = 0;
    d |= (uint64_t)((addr >> 4) & 0x3FFF);           // start address
    d |= (uint64_t)1 << 16;                          // leading byte offset (unused for this layout)
    d |= (uint64_t)(1024 >> 4) << 32;                // stride byte offset
    d |= (uint64_t)1 << 46;                          // descriptor version
    d |= (uint64_t)2 << 61;                          // SWIZZLE_128B
    return d;
}

// Instruction descriptor, kind::tf32: D fp32, A/B tf32, both K-major, M=128, N=256.
constexpr uint32_t kIdesc = (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(256 >> 3) << 17) |
                            ((uint32_t)(128 >> 4) << 24);
// the same with N = 128 (one part of a trailing update), and with B negated (bit 14)
constexpr uint32_t kIdesc128 = (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(128 >> 3) << 17) |
                               ((uint32_t)(128 >> 4) << 24);
constexpr uint32_t kIdesc128Neg = kIdesc128 | (1u << 14);

__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t accumulate,
                                         uint32_t idesc = kIdesc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 lanes x 32 consecutive fp32 columns of the accumulator
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),
          "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
          "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; i++) v[i] = __uint_as_float(r[i]);
}

// Tile t of the launch: frequency slot, output row tile, column tile
// (KIND_SCHUR) or solve (KIND_TRSM: 0 = L21, 1 = U12^T, interleaved;
// KIND_TRSM_SYM: both from one product per row tile).
struct Tile {
    int slot, ra, u, rb;
};

// Parts of a trailing update (the Schur kinds): all its tiles, the first
// column tile only (the next outer step's panel: its diagonal block and
// A21), or the others -- so that the next diagonal block can start while the
// rest of the update runs.
enum { PART_ALL = ZS_PART_ALL, PART_COL0 = ZS_PART_COL0, PART_REST = ZS_PART_REST };

template <int KIND>
__host__ __device__ __forceinline__ int tiles_per_slot(int tiles, int part) {
    if (KIND == KIND_SCHUR || KIND == KIND_SCHUR_LOWER) {
        if (part == PART_COL0) return tiles;
        if (part == PART_REST) return KIND == KIND_SCHUR ? tiles * (tiles - 1) : tiles * (tiles - 1) / 2;
    }
    return KIND == KIND_SCHUR         ? tiles * tiles
           : KIND == KIND_SCHUR_LOWER ? tiles * (tiles + 1) / 2
           : KIND == KIND_TRSM_SYM    ? tiles
                                      : 2 * tiles;
}

template <int KIND>
__device__ __forceinline__ Tile tile_of(int t, int tiles, int64_t base, const int *slots, int part) {
    Tile x;
    const int per_slot = tiles_per_slot<KIND>(tiles, part);
    const int si = t / per_slot, rem = t - si * per_slot;
    x.slot = slots[si];
    if ((KIND == KIND_SCHUR || KIND == KIND_SCHUR_LOWER) && part == PART_COL0) {
        x.ra = (int)(base + (int64_t)rem * TM);
        x.rb = (int)base;
        x.u = 0;
    } else if (KIND == KIND_SCHUR_LOWER && part == PART_REST) {
        // row-major over the lower triangle without its first column: row
        // tile tm >= 1 holds tiles tn = 1 .. tm
        int tm = (int)((1.f + sqrtf(8.f * (float)rem + 1.f)) * 0.5f);
        while (tm * (tm - 1) / 2 > rem) tm--;
        while ((tm + 1) * tm / 2 <= rem) tm++;
        const int tn = 1 + rem - tm * (tm - 1) / 2;
        x.ra = (int)(base + (int64_t)tm * TM);
        x.rb = (int)(base + (int64_t)tn * TN);
        x.u = 0;
    } else if (KIND == KIND_SCHUR && part == PART_REST) {
        const int tm = rem / (tiles - 1), tn = 1 + rem - tm * (tiles - 1);
        x.ra = (int)(base + (int64_t)tm * TM);
        x.rb = (int)(base + (int64_t)tn * TN);
        x.u = 0;
    } else if (KIND == KIND_SCHUR_LOWER) {
        // row-major over the lower triangle: row tile tm holds tm + 1 tiles
        int tm = (int)((sqrtf(8.f * (float)rem + 1.f) - 1.f) * 0.5f);
        while ((tm + 1) * (tm + 2) / 2 <= rem) tm++;
        while (tm * (tm + 1) / 2 > rem) tm--;
        const int tn = rem - tm * (tm + 1) / 2;
        x.ra = (int)(base + (int64_t)tm * TM);
        x.rb = (int)(base + (int64_t)tn * TN);
        x.u = 0;
    } else if (KIND == KIND_TRSM_SYM) {
        x.ra = (int)(base + (int64_t)rem * TM);
        x.rb = 0;
        x.u = 0;
    } else if (KIND == KIND_SCHUR) {
        const int tm = rem / tiles, tn = rem - tm * tiles;
        x.ra = (int)(base + (int64_t)tm * TM);
        x.rb = (int)(base + (int64_t)tn * TN);
        x.u = 0;
    } else {
        x.u = rem & 1;
        x.ra = (int)(base + (int64_t)(rem >> 1) * TM);
        x.rb = 0;
    }
    return x;
}

// tmap: operand packs (boxes 32 x 128); wmap: inverse packs (block solves);
// cmap: float32 matrices (boxes 32 x 32); pmap: operand packs (boxes 32 x 32, block-solve stores);
// dinv (KIND_TRSM_SYM): the float32 inverse diagonal blocks, per slot dinv_stride floats.
template <int SPLIT, int KIND>
__global__ void __launch_bounds__(kThreads, 1)
k_cgemm_tc(const __grid_constant__ CUtensorMap tmap, const __grid_constant__ CUtensorMap wmap,
           const __grid_constant__ CUtensorMap cmap, const __grid_constant__ CUtensorMap pmap, int64_t n, int64_t J,
           const int *__restrict__ slots, int nslot, unsigned *__restrict__ ctr, unsigned *__restrict__ status,
           const float *__restrict__ dinv, int64_t dinv_stride, int part) {
    using C = Cfg<SPLIT>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bar_full[C::STAGES], bar_empty[C::STAGES], bar_accf[2], bar_acce[2], bar_drain;
    __shared__ __align__(8) uint64_t bar_tq[kTq];
    __shared__ volatile int s_tq[kTq];  // tile of local tile it at it % kTq; -1 ends the sequence
    __shared__ uint32_t s_tmem;
    __shared__ volatile int s_abort;
    const uint32_t base_addr = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const int64_t base = J + NB;
    const int64_t m2 = n - base;
    const int tiles = (int)((m2 + TM - 1) / TM);
    const int total = tiles_per_slot<KIND>(tiles, part) * nslot;

    if (threadIdx.x == 0) {
        s_abort = 0;
        for (int s = 0; s < C::STAGES; s++) {
            mbar_init(smem_u32(&bar_full[s]), 1);
            mbar_init(smem_u32(&bar_empty[s]), 1);
        }
        for (int b = 0; b < 2; b++) {
            mbar_init(smem_u32(&bar_accf[b]), 1);
            mbar_init(smem_u32(&bar_acce[b]), 4);
        }
        mbar_init(smem_u32(&bar_drain), 1);
        for (int q = 0; q < kTq; q++) mbar_init(smem_u32(&bar_tq[q]), 1);
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

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmap) : "memory");
            if (is_trsm<KIND>()) asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&wmap) : "memory");
            // Tiles are taken dynamically: the first is blockIdx.x, the next
            // ones come from the launch's counter, so CTAs that start late
            // (the SMs busy with another stream's kernel) simply take fewer.
            // Each tile index is published in the queue before its loads; the
            // end of the sequence (-1) occupies one stage with a plain arrive.
            uint32_t g = 0, it = 0;
            int t = (int)blockIdx.x;
            while (true) {
                if (t >= total) t = -1;
                const uint32_t st0 = g % C::STAGES, ph0 = (g / C::STAGES) & 1u;
                if (!mbar_wait(smem_u32(&bar_empty[st0]), ph0 ^ 1u, &s_abort, status, 1u | (KIND << 4))) break;
                s_tq[it % kTq] = t;
                mbar_arrive(smem_u32(&bar_tq[it % kTq]));
                if (t < 0) {
                    mbar_arrive(smem_u32(&bar_full[st0]));
                    g++;
                    break;
                }
                const Tile x = tile_of<KIND>(t, tiles, base, slots, part);
                // A rows: L21 / A21 (A planes) or A12^T (Br planes); B: the pack's
                // own Br rows, or W / V from the inverse packs (their Br planes)
                const int pa = (KIND == KIND_TRSM && x.u) ? PL_BR_HI : PL_A_HI;
                const bool use_v = KIND == KIND_TRSM_SYM || x.u;  // B = L11^-1 (else U11^-1)
                const CUtensorMap *bm = !is_trsm<KIND>() ? &tmap : &wmap;
                // the symmetric update's B is M's own rows (the A planes, see the MMA issue)
                const int pbr = KIND == KIND_SCHUR_LOWER ? PL_A_HI
                                : !is_trsm<KIND>()       ? PL_BR_HI
                                                         : (use_v ? WP_V : 0) + WP_BR_HI;
                bool ok = true;
                for (int kc = 0; kc < NKC; kc++, g++) {
                    const uint32_t st = g % C::STAGES, ph = (g / C::STAGES) & 1u;
                    if (kc > 0 && !mbar_wait(smem_u32(&bar_empty[st]), ph ^ 1u, &s_abort, status, 1u | (KIND << 4))) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = smem_u32(&bar_full[st]);
                    mbar_expect_tx(fb, C::STAGE_BYTES);
                    const uint32_t sa = base_addr + st * C::STAGE_BYTES;
                    const int k0 = kc * KC;
                    // the second B half: Br's other K half (Bi chunk k = -+ Br
                    // chunk k +- 128, the sign applied by the MMA), so that no Bi
                    // plane is written, of the operand packs or the inverse packs
                    const int k2 = (k0 + NB) % KTOT;
                    tma_load_4d(sa, &tmap, k0, x.ra, pa, x.slot, fb);
                    tma_load_4d(sa + A_BYTES, bm, k0, x.rb, pbr, x.slot, fb);
                    tma_load_4d(sa + A_BYTES + B_BYTES / 2, bm, k2, x.rb, pbr, x.slot, fb);
                    if (SPLIT) {  // lo planes follow their hi planes
                        const uint32_t sl = sa + A_BYTES + B_BYTES;
                        tma_load_4d(sl, &tmap, k0, x.ra, pa + 1, x.slot, fb);
                        tma_load_4d(sl + A_BYTES, bm, k0, x.rb, pbr + 1, x.slot, fb);
                        tma_load_4d(sl + A_BYTES + B_BYTES / 2, bm, k2, x.rb, pbr + 1, x.slot, fb);
                    }
                }
                if (!ok) break;
                it++;
                t = (int)gridDim.x + (int)atomicAdd(ctr, 1u);
            }
            // our own copies in flight: wait (bounded) for the last stages to land
            const uint32_t issued = g;
            for (uint32_t q = issued > (uint32_t)C::STAGES ? issued - C::STAGES : 0; q < issued; q++) {
                uint32_t it = 0;
                while (!mbar_try_wait(smem_u32(&bar_full[q % C::STAGES]), (q / C::STAGES) & 1u) &&
                       ++it < kWaitLimit) {
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            uint32_t g = 0, it = 0;
            while (true) {
                // the first stage of the next tile (or the end marker) tells which
                const uint32_t st0 = g % C::STAGES, ph0 = (g / C::STAGES) & 1u;
                if (!mbar_wait(smem_u32(&bar_full[st0]), ph0, &s_abort, status, 2u | (KIND << 4))) break;
                // the accumulator buffer must be free (the epilogue has read the
                // tile two back) also before the end marker completes its next
                // phase: otherwise a slow epilogue could find that barrier two
                // phases on, with the parity it waits for, and wait for ever
                const uint32_t buf = it & 1u, aph = (it >> 1) & 1u;
                if (!mbar_wait(smem_u32(&bar_acce[buf]), aph ^ 1u, &s_abort, status, 3u | (KIND << 4))) break;
                if (s_tq[it % kTq] < 0) {
                    g++;
                    mbar_arrive(smem_u32(&bar_accf[buf]));  // the epilogue's turn to see the end
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + buf * 256u;
                bool ok = true;
                for (int kc = 0; kc < NKC; kc++, g++) {
                    const uint32_t st = g % C::STAGES, ph = (g / C::STAGES) & 1u;
                    if (kc > 0 && !mbar_wait(smem_u32(&bar_full[st]), ph, &s_abort, status, 2u | (KIND << 4))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = base_addr + st * C::STAGE_BYTES;
#pragma unroll
                    for (int ks = 0; ks < KC / 8; ks++) {
                        const uint64_t ah = smem_desc(sa + ks * 32);
                        const uint64_t bh = smem_desc(sa + A_BYTES + ks * 32);
                        const uint32_t acc = (kc | ks) ? 1u : 0u;
                        const uint32_t sl = sa + A_BYTES + B_BYTES;
                        const uint64_t al = smem_desc(sl + ks * 32);
                        const uint64_t bl = smem_desc(sl + A_BYTES + ks * 32);
                        // real part (columns 0-127) from Br, imaginary part
                        // (columns 128-255) from Br's other K half, negated in
                        // the first half of K.  The symmetric update's B rows
                        // are M = [Re M | Im M] (the A planes): Br = [Re M | -Im M]
                        // is them negated in the second half of K, and
                        // Bi = [Im M | Re M] their other K half as it is.
                        const uint64_t bh2 = smem_desc(sa + A_BYTES + B_BYTES / 2 + ks * 32);
                        const uint64_t bl2 = smem_desc(sl + A_BYTES + B_BYTES / 2 + ks * 32);
                        constexpr bool kBfromA = KIND == KIND_SCHUR_LOWER;
                        const uint32_t id1 = kBfromA && kc * KC >= NB ? kIdesc128Neg : kIdesc128;
                        const uint32_t id2 = !kBfromA && kc * KC < NB ? kIdesc128Neg : kIdesc128;
                        if (SPLIT) {
                            mma_tf32(d, al, bh, acc, id1);
                            mma_tf32(d, ah, bl, 1u, id1);
                            mma_tf32(d, ah, bh, 1u, id1);
                            mma_tf32(d + 128u, al, bh2, acc, id2);
                            mma_tf32(d + 128u, ah, bl2, 1u, id2);
                            mma_tf32(d + 128u, ah, bh2, 1u, id2);
                        } else {
                            mma_tf32(d, ah, bh, acc, id1);
                            mma_tf32(d + 128u, ah, bh2, acc, id2);
                        }
                    }
                    mma_commit(smem_u32(&bar_empty[st]));  // stage free once these MMAs finish
                }
                if (!ok) break;
                mma_commit(smem_u32(&bar_accf[buf]));  // accumulator ready
                it++;
            }
            // drain: every MMA issued so far completes before TMEM is freed
            mma_commit(smem_u32(&bar_drain));
            uint32_t w = 0;
            while (!mbar_try_wait(smem_u32(&bar_drain), 0) && ++w < kWaitLimit) {
            }
        }
    } else {
        // ------------------------------------------------ epilogue (warps 2-5)
        const int quad = warp & 3;  // TMEM lanes 32*quad .. 32*quad+31
        const uint32_t stage0 = base_addr + C::STAGES * C::STAGE_BYTES + (uint32_t)(warp - 2) * 2u * EPI_BOX;
        uint32_t it = 0, nbox = 0;
        // next staging buffer of this warp's ring of two: its previous store
        // must have finished reading it
        auto next_box = [&]() -> uint32_t {
            const uint32_t sb = stage0 + (nbox & 1u) * EPI_BOX;
            nbox++;
            if (lane == 0) bulk_wait_read<1>();
            __syncwarp();
            return sb;
        };
        // staged box complete: make it visible to the async proxy, then one lane stores it
        auto publish = [&]() {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
        };
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&cmap) : "memory");
            if (is_trsm<KIND>()) asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&pmap) : "memory");
        }
        for (;; it++) {
            const bool okq = mbar_wait(smem_u32(&bar_tq[it % kTq]), (it / kTq) & 1u, &s_abort, status, 4u | (KIND << 4));
            if (!__all_sync(0xffffffffu, okq)) break;
            const int t = s_tq[it % kTq];
            const uint32_t buf = it & 1u, aph = (it >> 1) & 1u;
            const bool ok = mbar_wait(smem_u32(&bar_accf[buf]), aph, &s_abort, status, 5u | (KIND << 4));
            if (!__all_sync(0xffffffffu, ok) || t < 0) break;
            tc_fence_after();
            const Tile x = tile_of<KIND>(t, tiles, base, slots, part);
            const int row0 = x.ra + quad * 32;  // this warp's 32 output rows
            if (KIND == KIND_TRSM_SYM) {
                // The accumulator holds U12^T for the tile's rows (Re in chunks
                // 0-3, Im in chunks 4-7); per group of 32 columns both parts.
                // D11^-1 is the diagonal of U11^-1 (an upper triangle's inverse
                // has the reciprocal diagonal), taken from the float32 inverses.
                // Out go U12 into the float32 factor, the trailing update's
                // operand rows M = U12^T S, S^2 = D11^-1 (any root of each
                // entry: M M^T = U12^T D11^-1 U12 = L21 U12 whichever), and
                // L21 = M S = U12^T D11^-1 into the factor.
                const float *dre = dinv + (int64_t)x.slot * dinv_stride + (J / NB) * 4 * NB * NB + 2 * NB * NB;
                const float *dim = dre + NB * NB;
#pragma unroll 1
                for (int g = 0; g < 4; g++) {
                    float vr[32], vi[32];
                    const uint32_t tl = tmem + buf * 256u + ((uint32_t)(quad * 32) << 16);
                    tmem_ld32(tl + (uint32_t)(g * 32), vr);
                    tmem_ld32(tl + (uint32_t)((g + 4) * 32), vi);
                    if (g == 3) {  // accumulator fully read: hand it back to the MMA warp
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(smem_u32(&bar_acce[buf]));
                    }
                    const int c32 = g * 32;
                    // S(c32 + lane), one column per lane, shared by shuffles below
                    const cf sg = csqrt_f(cf{__ldg(dre + (c32 + lane) * (NB + 1)), __ldg(dim + (c32 + lane) * (NB + 1))});
#pragma unroll
                    for (int part = 0; part < 2; part++) {
                        // U12(J + c32 + t, i) into the float32 factor (transposed boxes)
                        const uint32_t sb = next_box();
                        stage_col(sb, lane, part ? vi : vr);
                        publish();
                        if (lane == 0) {
                            tma_store_4d(&cmap, sb, row0, (int)J + c32, part, x.slot);
                            bulk_commit();
                        }
                    }
#pragma unroll 2
                    for (int step = 0; step < 2; step++) {
                        // step 0: M = U12^T S (operand rows); step 1: L21 = M S (the factor)
#pragma unroll
                        for (int q = 0; q < 32; q++) {
                            const float sr = __shfl_sync(0xffffffffu, sg.re, q), si = __shfl_sync(0xffffffffu, sg.im, q);
                            const float a = vr[q], b = vi[q];
                            vr[q] = fmaf(a, sr, -b * si);
                            vi[q] = fmaf(a, si, b * sr);
                        }
#pragma unroll
                        for (int part = 0; part < 2; part++) {
                            const float(&v)[32] = part ? vi : vr;
                            if (step == 1) {
                                const uint32_t sb = next_box();
                                stage_row(sb, lane, v, 1.f);
                                publish();
                                if (lane == 0) {
                                    tma_store_4d(&cmap, sb, (int)J + c32, row0, part, x.slot);
                                    bulk_commit();
                                }
                                continue;
                            }
                            // M's rows [Re M | Im M] in the A planes, tf32 hi (and lo)
                            float h[32];
#pragma unroll
                            for (int q = 0; q < 32; q++) h[q] = tf32_rna(v[q]);
#pragma unroll 1
                            for (int lo = 0; lo <= SPLIT; lo++) {
                                if (lo) {
#pragma unroll
                                    for (int q = 0; q < 32; q++) h[q] = tf32_rna(v[q] - h[q]);
                                }
                                const uint32_t sb = next_box();
                                stage_row(sb, lane, h, 1.f);
                                publish();
                                if (lane == 0) {
                                    tma_store_4d(&pmap, sb, part * NB + c32, row0, PL_A_HI + lo, x.slot);
                                    bulk_commit();
                                }
                            }
                        }
                    }
                }
                continue;
            }
#pragma unroll 1
            for (int c = 0; c < 8; c++) {
                float v[32];
                tmem_ld32(tmem + buf * 256u + (uint32_t)(c * 32) + ((uint32_t)(quad * 32) << 16), v);
                if (c == 7) {  // accumulator fully read: hand it back to the MMA warp
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&bar_acce[buf]));
                }
                const int part = c >> 2, c32 = (c & 3) * 32;  // part 0 = real, 1 = imaginary
                if (KIND != KIND_TRSM) {
                    const uint32_t sb = next_box();
                    stage_row(sb, lane, v, -1.f);
                    publish();
                    if (lane == 0) {
                        tma_reduce_add_4d(&cmap, sb, x.rb + c32, row0, part, x.slot);
                        bulk_commit();
                    }
                    continue;
                }
                // ---- KIND_TRSM: the factor itself, then the trailing update's operand packs
                uint32_t sb = next_box();
                if (x.u == 0) stage_row(sb, lane, v, 1.f);  // L21(i, J + c32 + t)
                else stage_col(sb, lane, v);                 // U12(J + c32 + t, j)
                publish();
                if (lane == 0) {
                    if (x.u == 0) tma_store_4d(&cmap, sb, (int)J + c32, row0, part, x.slot);
                    else tma_store_4d(&cmap, sb, row0, (int)J + c32, part, x.slot);
                    bulk_commit();
                }
                float h[32];
#pragma unroll
                for (int q = 0; q < 32; q++) h[q] = tf32_rna(v[q]);
#pragma unroll 1
                for (int lo = 0; lo <= SPLIT; lo++) {
                    if (lo) {
#pragma unroll
                        for (int q = 0; q < 32; q++) h[q] = tf32_rna(v[q] - h[q]);
                    }
                    if (x.u == 0) {  // A row i = [Re L21 | Im L21]: K column = accumulator column
                        sb = next_box();
                        stage_row(sb, lane, h, 1.f);
                        publish();
                        if (lane == 0) {
                            tma_store_4d(&pmap, sb, c * 32, row0, PL_A_HI + lo, x.slot);
                            bulk_commit();
                        }
                    } else {  // Br row j = [Re U12^T | -Im U12^T] (the trailing update derives Bi from it)
                        sb = next_box();
                        stage_row(sb, lane, h, part ? -1.f : 1.f);
                        publish();
                        if (lane == 0) {
                            tma_store_4d(&pmap, sb, part * NB + c32, row0, PL_BR_HI + lo, x.slot);
                            bulk_commit();
                        }
                    }
                }
            }
        }
        if (lane == 0) bulk_wait_all();  // our own stores are complete before exit
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
    }
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

template <int SPLIT, int KIND>
cudaError_t launch_kind(const CUtensorMap &tmap, const CUtensorMap &wmap, const CUtensorMap &cmap,
                        const CUtensorMap &pmap, int64_t n, int64_t J, const int *slots, int nslot, unsigned *ctr,
                        unsigned *status, int max_grid, cudaStream_t st, const float *dinv = nullptr,
                        int64_t dinv_stride = 0, int part = PART_ALL) {
    using C = Cfg<SPLIT>;
    // once per process (thread-safe initialisation of a local static)
    static const cudaError_t attr = cudaFuncSetAttribute(k_cgemm_tc<SPLIT, KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (attr != cudaSuccess) return attr;
    const int64_t m2 = n - J - NB;
    if (m2 <= 0 || nslot <= 0) return cudaSuccess;
    const int tiles = (int)((m2 + TM - 1) / TM);
    const int64_t total = (int64_t)tiles_per_slot<KIND>(tiles, part) * nslot;
    if (total <= 0) return cudaSuccess;
    const int grid = (int)(total < max_grid ? total : max_grid);
    k_cgemm_tc<SPLIT, KIND><<<grid, kThreads, C::SMEM, st>>>(tmap, wmap, cmap, pmap, n, J, slots, nslot, ctr,
                                                             status, dinv, dinv_stride, part);
    return cudaGetLastError();
}

cudaError_t encode_f32_4d(void *map_out, const float *base, const cuuint64_t (&dims)[4], const cuuint64_t (&strides)[3],
                          cuuint32_t box0, cuuint32_t box1) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = get_encode();
    if (!enc) return cudaErrorNotSupported;
    CUtensorMap *map = reinterpret_cast<CUtensorMap *>(map_out);
    cuuint32_t box[4] = {box0, box1, 1, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, (void *)base, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

// Tensor map over the operand packs: dims (K = 256, rows = n, plane = 6,
// slot = S); boxes of 32 K x box_rows rows (128 for operand loads, 32 for
// the triangular solves' stores).
cudaError_t zs_tc_pack_map(const float *pack, int64_t n, int nslots, int64_t pack_stride, int box_rows,
                           void *map_out) {
    const cuuint64_t dims[4] = {(cuuint64_t)KTOT, (cuuint64_t)n, 6, (cuuint64_t)nslots};
    const cuuint64_t strides[3] = {(cuuint64_t)KTOT * 4, (cuuint64_t)zs_pack_plane(n) * 4,
                                   (cuuint64_t)pack_stride * 4};
    return encode_f32_4d(map_out, pack, dims, strides, KC, (cuuint32_t)box_rows);
}

// Tensor map over the inverse packs: dims (K = 256, rows = 128, plane = 4, slot = S), boxes of 32 x 128.
cudaError_t zs_tc_winv_map(const float *winv, int nslots, void *map_out) {
    const cuuint64_t dims[4] = {(cuuint64_t)KTOT, (cuuint64_t)NB, 4, (cuuint64_t)nslots};
    const cuuint64_t strides[3] = {(cuuint64_t)KTOT * 4, (cuuint64_t)ZS_WINV_PLANE * 4,
                                   (cuuint64_t)ZS_WINV_STRIDE * 4};
    return encode_f32_4d(map_out, winv, dims, strides, KC, NB);
}

// Tensor map over the float32 matrices: dims (column = n, row = n,
// plane = 2 (re, im), slot = S), boxes of 32 x 32 for the epilogue stores.
cudaError_t zs_tc_z32_map(const float *z32, int64_t n, int64_t ld, int64_t plane, int nslots, int64_t z32_stride,
                          void *map_out) {
    const cuuint64_t dims[4] = {(cuuint64_t)n, (cuuint64_t)n, 2, (cuuint64_t)nslots};
    const cuuint64_t strides[3] = {(cuuint64_t)ld * 4, (cuuint64_t)plane * 4, (cuuint64_t)z32_stride * 4};
    return encode_f32_4d(map_out, z32, dims, strides, 32, 32);
}

cudaError_t zs_launch_schur_tc(const void *map, const void *cmap, int64_t n, int64_t J, int split, int lower,
                               int part, const int *slots, int nslot, unsigned *ctr, unsigned *status, int max_grid,
                               cudaStream_t st) {
    if (max_grid < 1 || !ctr || part < PART_ALL || part > PART_REST) return cudaErrorInvalidValue;
    const CUtensorMap &m = *reinterpret_cast<const CUtensorMap *>(map);
    const CUtensorMap &c = *reinterpret_cast<const CUtensorMap *>(cmap);
    if (lower) {
        if (split)
            return launch_kind<1, KIND_SCHUR_LOWER>(m, m, c, m, n, J, slots, nslot, ctr, status, max_grid, st, nullptr,
                                                    0, part);
        return launch_kind<0, KIND_SCHUR_LOWER>(m, m, c, m, n, J, slots, nslot, ctr, status, max_grid, st, nullptr, 0,
                                                part);
    }
    if (split)
        return launch_kind<1, KIND_SCHUR>(m, m, c, m, n, J, slots, nslot, ctr, status, max_grid, st, nullptr, 0, part);
    return launch_kind<0, KIND_SCHUR>(m, m, c, m, n, J, slots, nslot, ctr, status, max_grid, st, nullptr, 0, part);
}

cudaError_t zs_launch_trsm_tc(const void *map, const void *wmap, const void *cmap, const void *pmap, int64_t n,
                              int64_t J, int split, int sym, const float *dinv, int64_t dinv_stride,
                              const int *slots, int nslot, unsigned *ctr, unsigned *status, int num_sms,
                              cudaStream_t st) {
    if (!ctr || (sym && !dinv)) return cudaErrorInvalidValue;
    const CUtensorMap &m = *reinterpret_cast<const CUtensorMap *>(map);
    const CUtensorMap &w = *reinterpret_cast<const CUtensorMap *>(wmap);
    const CUtensorMap &c = *reinterpret_cast<const CUtensorMap *>(cmap);
    const CUtensorMap &p = *reinterpret_cast<const CUtensorMap *>(pmap);
    if (sym) {
        if (split)
            return launch_kind<1, KIND_TRSM_SYM>(m, w, c, p, n, J, slots, nslot, ctr, status, num_sms, st, dinv,
                                                 dinv_stride);
        return launch_kind<0, KIND_TRSM_SYM>(m, w, c, p, n, J, slots, nslot, ctr, status, num_sms, st, dinv,
                                             dinv_stride);
    }
    if (split) return launch_kind<1, KIND_TRSM>(m, w, c, p, n, J, slots, nslot, ctr, status, num_sms, st);
    return launch_kind<0, KIND_TRSM>(m, w, c, p, n, J, slots, nslot, ctr, status, num_sms, st);
}
