// C-ABI of the frequency-sweep solver: context, workspaces, the blocked
// factorisation loop, the refinement loop with its convergence and stall
// tests, the fallback trigger and the batched sweep.  See include/zsolve.h
// for the contract of every entry point.
//
// Method (malusrfworks.com, "Solving Dense Matrices Fast in the Browser",
// section "Double-precision answers from a GPU without double precision"):
// factorise in low precision (step 1), solve for x (step 2), form the
// residual in double precision (step 3), solve for a correction with the
// low-precision factors and add it (step 4), repeating steps 3-4 -- the
// page's loop back to step 2 is read as a return to the residual, since the
// first solve happens once -- until the relative correction is below tol.
// A frequency whose refinement does not converge is solved alone by the
// double-precision pivoted LU (same section, paragraph after the steps).
//
// A sweep factors `batch` frequencies together: every launch of the
// factorisation, the solves and the residual covers all of them, so the
// panel and triangular-solve latencies of one frequency overlap with the
// work of the others.  A batch is further split into two lanes -- each with
// its own stream, scratch and host thread -- that run assembly,
// factorisation and refinement side by side: the FP64-pipe-bound kernels of
// one lane (assembly, residual) fill the SMs the other lane leaves idle
// (diagonal blocks on one SM per frequency, tensor-core phases).
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <condition_variable>
#include <mutex>
#include <thread>
#include <vector>

#include "../../include/zsolve.h"
#include "common.cuh"


constexpr int kMaxLanes = 3;

struct zsolve_ctx {
    int64_t n = 0;
    int nrhs_max = 0;
    zsolve_opts opts{};
    int device = 0, num_sms = 0;
    unsigned wait_limit = ZS_SPIN_LIMIT;  // polls before a triangular-solve wait gives up
    // arithmetic of the factorisation in use: 0 FFMA, 1 TF32, 2 TF32X3 (opts.gemm,
    // or for ZSOLVE_GEMM_AUTO the probe's choice, TF32X3 until the probe ran)
    int gemm_eff = 2;
    zsolve_gemm_probe probe{};
    cudaStream_t stream = nullptr;
    int S = 1;  // frequencies held at once
    int64_t ld = 0, plane = 0, z32_stride = 0, z64_stride = 0, pack_stride = 0, v_stride = 0;
    double2 *z64 = nullptr;
    float *z32 = nullptr;
    float *pack = nullptr;
    float *dinv = nullptr;  // inverses of the 128x128 diagonal blocks of L and U
    float *inv32 = nullptr; // inverses of the 32x32 diagonal sub-blocks of the current outer block
    int64_t dinv_stride = 0;
    float *winv = nullptr;  // tensor-core operand packs of the current diagonal block's inverses
    // TMA tensor maps over the two sets of operand packs (32 x 128 boxes for
    // loads; 32 x 32 boxes for stores): outer steps alternate between them when
    // the next step's diagonal block runs ahead of the trailing update
    alignas(64) unsigned char pack_map[2][128] = {};
    alignas(64) unsigned char packst_map[2][128] = {};
    alignas(64) unsigned char winv_map[128] = {};    // TMA tensor map over the inverse packs
    alignas(64) unsigned char z32_map[128] = {};     // TMA tensor map over the float32 matrices
    float2 *v = nullptr;
    float4 *xs = nullptr;  // double-float split of x (residual mode DF)
    // the sweep's L, Psi, G while a sweep runs (residual mode LPG), else null
    const double *cur_L = nullptr, *cur_Psi = nullptr, *cur_G = nullptr;
    ZsSlotParam single{};  // frequency of the last zsolve_assemble
    unsigned char *xl = nullptr;  // fixed-point limbs of x (residual mode FX)
    int *xe = nullptr;     // their scale exponents, per (slot, rhs)
    int *zexp = nullptr;   // residual mode FX: per slot and row of Z64, its largest exponent
    int fx_ndf = 1;        // residual mode FX: sub-steps of four taken in float64 (ZSOLVE_FX_NDF)
    int trsv_r = 0;        // right-hand sides per triangular-solve chain; 0: chosen per solve (ZSOLVE_TRSV_R)
    int lookahead = -1;    // next diagonal block ahead of the trailing update: -1 for few frequencies, 0 never, 1 always (ZSOLVE_LOOKAHEAD)
    int tc_cap = 0;        // testing aid: at most this many CTAs per tcgen05 launch (ZSOLVE_TC_GRID; 0: no cap)
    int trsv_cap = 0;      // tuning aid: CTAs of each lane's triangular solves in a multi-lane batch (ZSOLVE_TRSV_CTAS; 0: SMs / lanes)
    // residual mode OZ: digits of A' = [L; Psi; G] (allocated on first use),
    // their row scales and tensor map; oz_ready while they hold the current
    // sweep's L, Psi, G
    void *oz_a = nullptr;
    int *oz_ea = nullptr;
    alignas(64) unsigned char oz_amap[128] = {};
    bool oz_ready = false;
    // the sweep forms the digits on a stream of their own, beside the first
    // assembly; every residual waits for oz_done
    cudaStream_t oz_stream = nullptr;
    cudaEvent_t oz_start = nullptr, oz_done = nullptr;
    int resid_mode = ZSOLVE_RESID_F64;
    double *partials = nullptr;
    int nchunks = 0;
    double *d_relcorr = nullptr, *h_relcorr = nullptr;
    ZsSlotParam *d_params = nullptr, *h_params = nullptr;
    int *d_all = nullptr;    // 0..S-1
    int *d_pivflag = nullptr, *h_pivflag = nullptr;
    unsigned long long *prog = nullptr;  // triangular-solve progress words, 2 per (slot, right-hand-side group)
    std::atomic<unsigned> epoch{0};      // triangular-solve launches, unique across lanes
    unsigned *d_status = nullptr;
    // fallback workspace (allocated on first use)
    double2 *fb_a = nullptr;
    int64_t *fb_piv = nullptr;
    int *fb_info = nullptr, *h_fb_info = nullptr;
    // device copies for the host-pointer sweep (allocated on first use)
    double *hd_L = nullptr, *hd_Psi = nullptr, *hd_G = nullptr;
    // the host-pointer sweep copies L, Psi, G in row bands on copy_stream;
    // the first assembly waits for each band separately
    static constexpr int kBands = 4;
    cudaStream_t copy_stream = nullptr;
    cudaStream_t copy_aux[2] = {nullptr, nullptr};  // Psi's and G's bands, beside L's
    cudaEvent_t band_ev[kBands] = {}, ev_host = nullptr;
    cudaEvent_t aux_ev[kBands][2] = {};
    int nband = 0;
    double2 *hd_b = nullptr, *hd_x = nullptr;
    size_t hd_x_cap = 0;
    int hd_nrhs_cap = 0;
    // A lane: one group of a batch's frequencies, run on its own stream with
    // its own scratch (lane 0 on the context's stream; the others, for
    // batches of two or more, on streams of their own, each driven by a host
    // thread of its own).
    struct Lane {
        cudaStream_t stream = nullptr;  // lane 0: the context's stream
        cudaStream_t side = nullptr;    // packs the next block solves' operands next to the diagonal block
        bool own_stream = false;
        cudaEvent_t ev[5] = {nullptr, nullptr, nullptr, nullptr, nullptr};
        cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
        cudaEvent_t ev_stag = nullptr;  // this lane's first solve of a two-lane refinement is queued
        int *d_active = nullptr, *h_active = nullptr;  // slots still refining
        unsigned *ticket = nullptr;     // triangular-solve task tickets
        unsigned *tile_ctr = nullptr;   // tile counters of the tcgen05 launches
        unsigned *h_status = nullptr;   // pinned copy of the device status word
        int tc_grid = 0;                // CTAs of this lane's tcgen05 launches
        int trsv_grid = 0;              // CTAs of this lane's triangular solves (0: one per SM)
        bool alone = true;              // no other lane runs beside this one (the next diagonal block may run ahead)
        // residual mode OZ: digits of x, their scales, the partial products
        void *oz_x = nullptr;
        int *oz_ex = nullptr;
        double *oz_part = nullptr;
        int oz_ncol_cap = 0;
        int64_t oz_part_cap = 0;
        // whether this lane's float64 matrices were formed: where the residual
        // works from L, Psi, G alone (OZ, LPG) a sweep assembles the float32
        // planes only, and the fallback then forms a stalled frequency's
        // float64 matrix from the call's inputs
        bool z64_formed = true;
    };
    Lane lane[kMaxLanes];
    int cur_nrhs = 0;  // right-hand sides of the running sweep call
    bool asm32_planes = false;  // testing aid: zsolve_assemble's float32 planes from the float32-only kernel
    int assembled = 0, factored = 0, fb_ready = 0;
    std::mutex err_mu, prof_mu, fb_mu;  // error text; profile records; fallback workspace
    // stage profile: launch counts always, event-timed spans with opts.profile
    int64_t prof_launches[ZSOLVE_NSTAGE] = {};
    double prof_ms[ZSOLVE_NSTAGE] = {};
    struct Span {
        int stage;
        cudaEvent_t a, b;
    };
    std::vector<cudaEvent_t> ev_pool;
    std::vector<Span> pending;
    char err[512] = {0};
};

namespace {

int fail(zsolve_ctx *c, int code, const char *fmt, ...) {
    if (c) {
        std::lock_guard<std::mutex> lock(c->err_mu);
        va_list ap;
        va_start(ap, fmt);
        vsnprintf(c->err, sizeof(c->err), fmt, ap);
        va_end(ap);
    }
    return code;
}

#define ZS_CU(call)                                                                             \
    do {                                                                                        \
        cudaError_t e_ = (call);                                                                \
        if (e_ != cudaSuccess)                                                                  \
            return fail(ctx, ZSOLVE_ECUDA, "%s failed: %s (%s:%d)", #call, cudaGetErrorString(e_), \
                        __FILE__, __LINE__);                                                    \
    } while (0)

#define ZS_TRY(expr)            \
    do {                        \
        int s_ = (expr);        \
        if (s_ != ZSOLVE_OK) return s_; \
    } while (0)

// ------------------------------------------------------------------ stage profile

int prof_resolve_locked(zsolve_ctx *ctx) {
    for (auto &sp : ctx->pending) {
        ZS_CU(cudaEventSynchronize(sp.b));
        float ms = 0.f;
        ZS_CU(cudaEventElapsedTime(&ms, sp.a, sp.b));
        ctx->prof_ms[sp.stage] += ms;
        ctx->ev_pool.push_back(sp.a);
        ctx->ev_pool.push_back(sp.b);
    }
    ctx->pending.clear();
    return ZSOLVE_OK;
}

int prof_resolve(zsolve_ctx *ctx) {
    std::lock_guard<std::mutex> lock(ctx->prof_mu);
    return prof_resolve_locked(ctx);
}

cudaEvent_t prof_take_locked(zsolve_ctx *ctx) {
    if (ctx->ev_pool.empty() && ctx->pending.size() >= 4096) prof_resolve_locked(ctx);
    if (!ctx->ev_pool.empty()) {
        cudaEvent_t e = ctx->ev_pool.back();
        ctx->ev_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

// Brackets the launches of one stage: counts them and, with opts.profile,
// records a pair of events around them on the stream they go to.
struct StageSpan {
    zsolve_ctx *c;
    int stage;
    cudaStream_t s;
    cudaEvent_t a = nullptr;
    StageSpan(zsolve_ctx *ctx, int st, cudaStream_t on) : c(ctx), stage(st), s(on) {
        if (c->opts.profile) {
            std::lock_guard<std::mutex> lock(c->prof_mu);
            a = prof_take_locked(c);
            if (a) cudaEventRecord(a, s);
        }
    }
    void done(int64_t launches) {
        std::lock_guard<std::mutex> lock(c->prof_mu);
        c->prof_launches[stage] += launches;
        if (a) {
            cudaEvent_t b = prof_take_locked(c);
            if (b) {
                cudaEventRecord(b, s);
                c->pending.push_back({stage, a, b});
            } else {
                c->ev_pool.push_back(a);
            }
            a = nullptr;
        }
    }
};

using Lane = zsolve_ctx::Lane;

int gemm_mode(const zsolve_opts &o) {
    switch (o.gemm) {
        case ZSOLVE_GEMM_FFMA: return 0;
        case ZSOLVE_GEMM_TF32: return 1;
        default: return 2;  // TF32X3 and AUTO
    }
}

// ZSOLVE_GEMM_* of an internal mode and back
int gemm_public(int mode) { return mode == 0 ? ZSOLVE_GEMM_FFMA : mode == 1 ? ZSOLVE_GEMM_TF32 : ZSOLVE_GEMM_TF32X3; }
int gemm_internal(int pub) { return pub == ZSOLVE_GEMM_FFMA ? 0 : pub == ZSOLVE_GEMM_TF32 ? 1 : 2; }

size_t slot_bytes(int64_t n, int64_t ld) {
    return (size_t)n * n * sizeof(double2) + (size_t)2 * n * ld * sizeof(float) +
           (size_t)12 * zs_pack_plane(n) * sizeof(float) + (size_t)zs_dinv_stride(n) * sizeof(float) +
           (size_t)zs_inv32_slot_stride(n) * sizeof(float) + (size_t)ZS_WINV_STRIDE * sizeof(float);
}

// ------------------------------------------------------------------ factor

// FP32 (FFMA) path: the steps one after another
int factor_slots_simt(zsolve_ctx *ctx, Lane &ln, const int *slots, int nslot) {
    const int64_t n = ctx->n;
    const int64_t inv32_stride = zs_inv32_slot_stride(n);
    for (int64_t J = 0; J < n; J += ZS_NB) {
        const int nb = (int)std::min<int64_t>(ZS_NB, n - J);
        {
            StageSpan sp(ctx, ZSOLVE_STAGE_DIAG, ln.stream);
            ZS_CU(zs_launch_diag_block(ctx->z32, ctx->ld, ctx->plane, ctx->z32_stride, J, nb, slots, nslot,
                                       ctx->d_pivflag, ctx->inv32, inv32_stride, ctx->dinv, ctx->dinv_stride,
                                       nullptr, 0, 0, ln.stream));
            sp.done(1);
        }
        if (J + nb >= n) break;
        {
            StageSpan sp(ctx, ZSOLVE_STAGE_TRSM, ln.stream);
            ZS_CU(zs_launch_trsm_l(ctx->z32, ctx->ld, ctx->plane, ctx->z32_stride, n, J, ctx->inv32, inv32_stride,
                                   ctx->pack, ctx->pack_stride, 0, slots, nslot, ln.stream));
            ZS_CU(zs_launch_trsm_u(ctx->z32, ctx->ld, ctx->plane, ctx->z32_stride, n, J, ctx->inv32, inv32_stride,
                                   ctx->pack, ctx->pack_stride, 0, slots, nslot, ln.stream));
            sp.done(2);
        }
        StageSpan sp(ctx, ZSOLVE_STAGE_SCHUR, ln.stream);
        ZS_CU(zs_launch_schur_simt(ctx->z32, ctx->ld, ctx->plane, ctx->z32_stride, n, J, ctx->pack, ctx->pack_stride,
                                   slots, nslot, ln.stream));
        sp.done(1);
    }
    return ZSOLVE_OK;
}

// Tensor-core path, one outer block after the other.  The operand packs of
// A21 and A12^T do not depend on the diagonal block, so they are written on
// the side stream while the diagonal block is factored; the tcgen05 block
// solves wait for both.  The tcgen05 kernels take tiles from per-launch
// counters (zeroed once per factorisation).
//
// With few frequencies the chain of diagonal blocks (one CTA per frequency)
// bounds the factorisation.  Then each step's trailing update runs in two
// launches: first its first column tile -- the next step's diagonal block and
// A21 -- after which the side stream factors the next diagonal block and packs
// the next A21 while the main stream finishes the update.  The packs of
// consecutive steps alternate between two buffers, since the next step's are
// written while this step's are still read.
constexpr int kMaxCtr = 512;         // tile counters per factorisation (at most 3 per outer block)
constexpr int kLookaheadSlots = 4;   // frequencies per lane up to which the next diagonal block runs ahead

int tc_grid(const zsolve_ctx *ctx, const Lane &ln) {
    return ctx->tc_cap > 0 ? std::min(ln.tc_grid, ctx->tc_cap) : ln.tc_grid;
}

int factor_slots_tc(zsolve_ctx *ctx, Lane &ln, const int *slots, int nslot) {
    const int64_t n = ctx->n;
    const int mode = ctx->gemm_eff, split = mode == 2 ? 1 : 0, sym = ctx->opts.symmetric;
    const int64_t nblk = (n + ZS_NB - 1) / ZS_NB;
    if (3 * nblk > kMaxCtr) return fail(ctx, ZSOLVE_EINVAL, "n too large for the tile counters");
    ZS_CU(cudaMemsetAsync(ln.tile_ctr, 0, kMaxCtr * sizeof(unsigned), ln.stream));
    unsigned *ctr = ln.tile_ctr;
    // The symmetric mode only: its packs read A21 alone, which the first
    // column tile holds (the full mode's pack of A12 would wait for the rest).
    // By default for a lane that runs alone with few frequencies (beside
    // another lane, that lane's kernels fill the SMs the diagonal chain leaves
    // idle, and running ahead only adds contention), and when the rest of an
    // update is long enough to hide a diagonal block: on average over the
    // steps nslot T^2 / 6 tiles (T = the first step's row tiles), at least two
    // waves of the grid.  (N=8000 with one frequency: 18.4 against 20.0 ms a
    // sweep; N=2157 with one: slower, the rest of each update being short.)
    const int64_t T = (n - 1) / ZS_NB;
    const bool ahead = sym && (ctx->lookahead > 0 ||
                               (ctx->lookahead < 0 && ln.alone && nslot <= kLookaheadSlots &&
                                (int64_t)nslot * T * T >= 12 * (int64_t)tc_grid(ctx, ln)));
    // The symmetric mode's block solve: one product per row tile, its
    // epilogue writing both factors and the update's one operand pack
    // M = U12^T S (S^2 = D11^-1), from which the lower update takes both of
    // its operands.  The full mode's two-product form writes L21 and U12^T
    // packs instead.
    auto pack = [&](int64_t J, int buf, cudaStream_t st) -> int {
        StageSpan sp(ctx, ZSOLVE_STAGE_PACK, st);
        ZS_CU(zs_launch_pack_trsm(ctx->z32, ctx->ld, ctx->plane, ctx->z32_stride, n, J,
                                  ctx->pack + (int64_t)buf * ctx->S * ctx->pack_stride, ctx->pack_stride, mode,
                                  sym, slots, nslot, st));
        sp.done(1);
        return ZSOLVE_OK;
    };
    auto diag = [&](int64_t J, cudaStream_t st) -> int {
        const int nb = (int)std::min<int64_t>(ZS_NB, n - J);
        StageSpan sp(ctx, ZSOLVE_STAGE_DIAG, st);
        ZS_CU(zs_launch_diag_block(ctx->z32, ctx->ld, ctx->plane, ctx->z32_stride, J, nb, slots, nslot,
                                   ctx->d_pivflag, nullptr, 0, ctx->dinv, ctx->dinv_stride,
                                   J + nb >= n ? nullptr : ctx->winv, mode, sym, st));
        sp.done(1);
        return ZSOLVE_OK;
    };
    auto trsm = [&](int64_t J, int buf) -> int {
        StageSpan sp(ctx, ZSOLVE_STAGE_TRSM, ln.stream);
        ZS_CU(zs_launch_trsm_tc(ctx->pack_map[buf], ctx->winv_map, ctx->z32_map, ctx->packst_map[buf], n, J, split,
                                sym, ctx->dinv, ctx->dinv_stride, slots, nslot, ctr++,
                                ctx->d_status, tc_grid(ctx, ln), ln.stream));
        sp.done(1);
        return ZSOLVE_OK;
    };
    auto schur = [&](int64_t J, int buf, int part, int grid) -> int {
        StageSpan sp(ctx, ZSOLVE_STAGE_SCHUR, ln.stream);
        ZS_CU(zs_launch_schur_tc(ctx->pack_map[buf], ctx->z32_map, n, J, split, sym, part, slots, nslot, ctr++,
                                 ctx->d_status, grid, ln.stream));
        sp.done(1);
        return ZSOLVE_OK;
    };
    auto fork = [&]() -> int {  // the side stream follows the main stream from here
        ZS_CU(cudaEventRecord(ln.ev_fork, ln.stream));
        ZS_CU(cudaStreamWaitEvent(ln.side, ln.ev_fork, 0));
        return ZSOLVE_OK;
    };
    if (!ahead) {
        for (int64_t J = 0; J < n; J += ZS_NB) {
            const bool last = J + ZS_NB >= n;
            if (!last) {
                ZS_TRY(fork());
                ZS_TRY(pack(J, 0, ln.side));
                ZS_CU(cudaEventRecord(ln.ev_join, ln.side));
            }
            ZS_TRY(diag(J, ln.stream));
            if (last) break;
            ZS_CU(cudaStreamWaitEvent(ln.stream, ln.ev_join, 0));
            ZS_TRY(trsm(J, 0));
            ZS_TRY(schur(J, 0, ZS_PART_ALL, tc_grid(ctx, ln)));
        }
        return ZSOLVE_OK;
    }
    // step 0's diagonal block and packs; then per step: block solves, the
    // first column tile of the update, the next diagonal block and packs on
    // the side stream beside the rest of the update
    ZS_TRY(fork());
    if (ZS_NB < n) ZS_TRY(pack(0, 0, ln.side));
    ZS_TRY(diag(0, ln.side));
    ZS_CU(cudaEventRecord(ln.ev_join, ln.side));
    for (int64_t J = 0; J + ZS_NB < n; J += ZS_NB) {
        const int buf = (int)((J / ZS_NB) & 1);
        ZS_CU(cudaStreamWaitEvent(ln.stream, ln.ev_join, 0));  // this step's diagonal block and packs
        ZS_TRY(trsm(J, buf));
        ZS_TRY(schur(J, buf, ZS_PART_COL0, tc_grid(ctx, ln)));
        ZS_TRY(fork());
        const int64_t J1 = J + ZS_NB;
        ZS_TRY(diag(J1, ln.side));
        if (J1 + ZS_NB < n) ZS_TRY(pack(J1, buf ^ 1, ln.side));
        ZS_CU(cudaEventRecord(ln.ev_join, ln.side));
        // leave an SM per frequency to the next diagonal block
        ZS_TRY(schur(J, buf, ZS_PART_REST, std::max(1, tc_grid(ctx, ln) - nslot)));
    }
    ZS_CU(cudaStreamWaitEvent(ln.stream, ln.ev_join, 0));  // the last diagonal block
    return ZSOLVE_OK;
}

// slots: device list of nslot slot indices, the first of which is `first`
// with the rest following it (the lane's range)
int factor_slots(zsolve_ctx *ctx, Lane &ln, const int *slots, int nslot, int first) {
    ZS_CU(cudaMemsetAsync(ctx->d_pivflag + first, 0, sizeof(int) * nslot, ln.stream));
    return ctx->gemm_eff == 0 ? factor_slots_simt(ctx, ln, slots, nslot) : factor_slots_tc(ctx, ln, slots, nslot);
}

// ------------------------------------------------------------------ solves

// Right-hand sides per chain of a triangular solve: the largest of 4, 2, 1
// whose chains (slots x groups) hold at least two tasks per CTA of the
// launch (a chain keeps up to n / 128 block tasks in work at once: one per
// block row, each taking the blocks left of it as the wavefront passes), else
// 1.  A chain's critical path is 2 n / 128 dependent block steps, shorter per
// step with fewer right-hand sides; the factors are read once per chain,
// mostly from the L2, since the chains of a slot advance together.
int trsv_rhs_per_chain(const zsolve_ctx *ctx, int left, int nslot, int grid) {
    if (ctx->trsv_r > 0) return std::min(ctx->trsv_r, left >= 4 ? 4 : left >= 2 ? 2 : 1);
    const int64_t nblk = (ctx->n + ZS_TB2 - 1) / ZS_TB2;
    for (int R = 4; R > 1; R >>= 1)
        if (left >= R && (int64_t)nslot * std::min(left / R, ZS_TRSV_MAX_GROUPS) * nblk >= 2 * (int64_t)grid)
            return R;
    return 1;
}

// v <- (LU)^-1 v for the listed slots: the right-hand sides in groups of R
// (4, 2 or 1), up to ZS_TRSV_MAX_GROUPS groups per launch, every (slot,
// group) an independent chain.  first_ticket > 0 withholds the first tasks
// of each launch (testing aid of the bounded waits, zsolve_selftest_wait);
// 0 in every solve.
int lowprec_solve_slots(zsolve_ctx *ctx, Lane &ln, int nrhs, const int *slots, int nslot, unsigned first_ticket = 0) {
    int r0 = 0;
    while (r0 < nrhs) {
        const int left = nrhs - r0;
        const int grid = ln.trsv_grid ? ln.trsv_grid : ctx->num_sms;
        const int R = trsv_rhs_per_chain(ctx, left, nslot, grid);
        const int groups = std::min(left / R, ZS_TRSV_MAX_GROUPS);
        const unsigned epoch = ctx->epoch.fetch_add(1u) + 1u;
        StageSpan sp(ctx, ZSOLVE_STAGE_TRSV, ln.stream);
        ZS_CU(zs_launch_trsv_inv(ctx->z32, ctx->ld, ctx->plane, ctx->z32_stride, ctx->n, ctx->dinv, ctx->dinv_stride,
                                 ctx->v + (int64_t)r0 * ctx->n, ctx->v_stride, R, groups, slots, nslot, ctx->prog,
                                 epoch, ln.ticket, ctx->d_status, grid, ln.stream, ctx->wait_limit, first_ticket));
        sp.done(1);
        r0 += R * groups;
    }
    return ZSOLVE_OK;
}

int check_device_status(zsolve_ctx *ctx, Lane &ln) {
    ZS_CU(cudaMemcpyAsync(ln.h_status, ctx->d_status, sizeof(unsigned), cudaMemcpyDeviceToHost, ln.stream));
    ZS_CU(cudaStreamSynchronize(ln.stream));
    if (*ln.h_status & ZS_DEV_TIMEOUT) {
        const unsigned code = *ln.h_status;
        *ln.h_status = 0;
        ZS_CU(cudaMemsetAsync(ctx->d_status, 0, sizeof(unsigned), ln.stream));
        // bits 8-15: the wait sites that gave up (0x80: a triangular-solve
        // progress word; else tcgen05 kernel kind << 4 | role wait 1-5)
        return fail(ctx, ZSOLVE_ETIMEOUT,
                    "a bounded device-side wait gave up (triangular solve or trailing update; sites 0x%02x)",
                    (code >> 8) & 0xFFu);
    }
    return ZSOLVE_OK;
}

int ensure_fallback(zsolve_ctx *ctx) {
    if (ctx->fb_ready) return ZSOLVE_OK;
    const int64_t n = ctx->n;
    if (cudaMalloc(&ctx->fb_a, (size_t)n * n * sizeof(double2)) != cudaSuccess ||
        cudaMalloc(&ctx->fb_piv, (size_t)n * sizeof(int64_t)) != cudaSuccess ||
        cudaMalloc(&ctx->fb_info, sizeof(int)) != cudaSuccess ||
        cudaMallocHost(&ctx->h_fb_info, sizeof(int)) != cudaSuccess) {
        cudaGetLastError();
        return fail(ctx, ZSOLVE_ENOMEM, "fallback workspace allocation failed (n=%lld)", (long long)n);
    }
    ctx->fb_ready = 1;
    return ZSOLVE_OK;
}

// x (nrhs x n, device) = Z64[slot]^-1 b by the float64 pivoted LU (one
// workspace per context: the lanes take turns)
int fallback_slot(zsolve_ctx *ctx, Lane &ln, int slot, const double2 *b, double2 *x, int nrhs) {
    std::lock_guard<std::mutex> lock(ctx->fb_mu);
    ZS_TRY(ensure_fallback(ctx));
    const int64_t n = ctx->n;
    if (ln.z64_formed) {
        ZS_CU(cudaMemcpyAsync(ctx->fb_a, ctx->z64 + (int64_t)slot * ctx->z64_stride, (size_t)n * n * sizeof(double2),
                              cudaMemcpyDeviceToDevice, ln.stream));
    } else {
        // the sweep assembled the float32 planes alone: this frequency's
        // float64 matrix from the call's inputs, straight into the workspace
        if (!ctx->cur_L || !ctx->cur_Psi || !ctx->cur_G)
            return fail(ctx, ZSOLVE_ESTATE, "fallback without the float64 matrix or the sweep's inputs");
        ZS_CU(zs_launch_assemble(ctx->cur_L, ctx->cur_Psi, ctx->cur_G, n, 0, n, ctx->d_params + slot, 1, ctx->fb_a,
                                 0, nullptr, ctx->ld, ctx->plane, 0, ln.stream));
    }
    int64_t cnt = 0;
    StageSpan sp(ctx, ZSOLVE_STAGE_FALLBACK, ln.stream);
    ZS_CU(zs_lu64_factor(ctx->fb_a, n, ctx->fb_piv, ctx->fb_info, ln.stream, &cnt));
    sp.done(cnt);
    ZS_CU(cudaMemcpyAsync(ctx->h_fb_info, ctx->fb_info, sizeof(int), cudaMemcpyDeviceToHost, ln.stream));
    ZS_CU(cudaStreamSynchronize(ln.stream));
    if (*ctx->h_fb_info != 0)
        return fail(ctx, ZSOLVE_ESINGULAR, "double-precision LU: zero pivot column at %d", *ctx->h_fb_info - 1);
    if (x != b)
        ZS_CU(cudaMemcpyAsync(x, b, (size_t)nrhs * n * sizeof(double2), cudaMemcpyDeviceToDevice, ln.stream));
    cnt = 0;
    StageSpan sp2(ctx, ZSOLVE_STAGE_FALLBACK, ln.stream);
    for (int r0 = 0; r0 < nrhs; r0 += 32)
        ZS_CU(zs_lu64_solve(ctx->fb_a, n, ctx->fb_piv, x + (int64_t)r0 * n, std::min(32, nrhs - r0), ln.stream,
                            &cnt));
    sp2.done(cnt);
    ZS_CU(cudaStreamSynchronize(ln.stream));  // the workspace is free for the other lane only when done
    return ZSOLVE_OK;
}

// Workspaces of the residual mode OZ (on first use): the digits of A' and,
// per lane, those of x for every column a lane can hold (2 S nrhs_max) and
// partial products for up to eight CTAs' segments of a tile's K range.
int ensure_oz(zsolve_ctx *ctx) {
    if (ctx->oz_a) return ZSOLVE_OK;
    const int64_t n = ctx->n, n_pad = zs_oz_n_pad(n);
    const int ncol_cap = zs_oz_ncol_alloc(2 * ctx->S * ctx->nrhs_max);
    // the padding of the tile-major digits (rows past 3n) is never written: zero once
    bool ok = cudaMalloc(&ctx->oz_a, (size_t)zs_oz_a_bytes(n)) == cudaSuccess &&
              cudaMemset(ctx->oz_a, 0, (size_t)zs_oz_a_bytes(n)) == cudaSuccess &&
              cudaMalloc(&ctx->oz_ea, (size_t)3 * n * sizeof(int)) == cudaSuccess &&
              zs_oz_a_map(ctx->oz_a, n, ctx->oz_amap) == cudaSuccess &&
              (ctx->oz_stream || cudaStreamCreateWithFlags(&ctx->oz_stream, cudaStreamNonBlocking) == cudaSuccess) &&
              (ctx->oz_start || cudaEventCreateWithFlags(&ctx->oz_start, cudaEventDisableTiming) == cudaSuccess) &&
              (ctx->oz_done || cudaEventCreateWithFlags(&ctx->oz_done, cudaEventDisableTiming) == cudaSuccess);
    for (auto &ln : ctx->lane) {
        if (!ok) break;
        ln.oz_ncol_cap = ncol_cap;
        ln.oz_part_cap = (int64_t)8 * 3 * n * ncol_cap;  // up to 8 CTAs' segments of a tile
        ok = cudaMalloc(&ln.oz_x, (size_t)8 * ncol_cap * n_pad * 2) == cudaSuccess &&
             cudaMalloc(&ln.oz_ex, (size_t)ncol_cap * sizeof(int)) == cudaSuccess &&
             cudaMalloc(&ln.oz_part, (size_t)ln.oz_part_cap * sizeof(double)) == cudaSuccess;
    }
    if (!ok) {
        cudaGetLastError();
        cudaFree(ctx->oz_a);
        cudaFree(ctx->oz_ea);
        ctx->oz_a = nullptr;
        ctx->oz_ea = nullptr;
        for (auto &ln : ctx->lane) {
            cudaFree(ln.oz_x);
            cudaFree(ln.oz_ex);
            cudaFree(ln.oz_part);
            ln.oz_x = nullptr;
            ln.oz_ex = nullptr;
            ln.oz_part = nullptr;
        }
        return fail(ctx, ZSOLVE_ENOMEM, "residual mode OZ: workspace allocation failed (n=%lld)", (long long)n);
    }
    return ZSOLVE_OK;
}

// The digits of A' = [L; Psi; G], after everything queued so far on `after`,
// on the digits' own stream, so that the first assembly runs beside them;
// oz_done marks their end (every residual waits for it).  While a
// host-pointer sweep's inputs are still being copied, band by band behind the
// copies (as the assembly).
int oz_split_inputs(zsolve_ctx *ctx, const double *L, const double *Psi, const double *G, cudaStream_t after) {
    ZS_TRY(ensure_oz(ctx));
    cudaStream_t st = ctx->oz_stream;
    ZS_CU(cudaEventRecord(ctx->oz_start, after));
    ZS_CU(cudaStreamWaitEvent(st, ctx->oz_start, 0));
    StageSpan sp(ctx, ZSOLVE_STAGE_RESIDUAL, st);
    const int nb = ctx->nband > 0 ? ctx->nband : 1;
    for (int bnd = 0; bnd < nb; bnd++) {
        const int64_t r0 = ctx->n * bnd / nb, r1 = ctx->n * (bnd + 1) / nb;
        if (ctx->nband > 0) ZS_CU(cudaStreamWaitEvent(st, ctx->band_ev[bnd], 0));
        ZS_CU(zs_launch_oz_split_a(L, Psi, G, ctx->n, r0, r1, ctx->oz_a, ctx->oz_ea, st));
    }
    sp.done(nb);
    ZS_CU(cudaEventRecord(ctx->oz_done, st));
    return ZSOLVE_OK;
}

// r = b - Z x for the listed slots in the context's residual arithmetic.
constexpr int kOzMinPairs = 4;  // fewer (frequency, right-hand side) pairs: the OZ mode's GEMV
int residual_slots(zsolve_ctx *ctx, Lane &ln, const double2 *b, const double2 *x, int64_t x_stride, int nrhs,
                   float2 *o64, int64_t o64s, double2 *o128, int64_t o128s, const int *slots, int nslot,
                   StageSpan *sp) {
    const int64_t n = ctx->n;
    // OZ reads its 48 n^2 bytes of digits whatever the number of columns;
    // below four (frequency, right-hand side) pairs the float64 GEMV over Z64
    // (16 n^2 bytes and 2-4 DFMA per entry and pair) is the faster one, where
    // the lane's float64 matrices were formed
    if (ctx->resid_mode == ZSOLVE_RESID_OZ && ctx->oz_ready &&
        ((int64_t)nslot * nrhs >= kOzMinPairs || !ln.z64_formed)) {
        ZS_CU(cudaStreamWaitEvent(ln.stream, ctx->oz_done, 0));
        ZS_CU(zs_launch_residual_oz(ctx->oz_amap, ctx->oz_ea, n, ctx->d_params, b, x, x_stride, nrhs, o64, o64s, o128,
                                    o128s, slots, nslot, ln.oz_x, ln.oz_ex, ln.oz_ncol_cap, ln.oz_part,
                                    ln.oz_part_cap, ctx->d_status, ctx->num_sms, ln.stream));
        sp->done(3);
    } else if (ctx->resid_mode == ZSOLVE_RESID_LPG && ctx->cur_L) {
        ZS_CU(zs_launch_residual_lpg(ctx->cur_L, ctx->cur_Psi, ctx->cur_G, n, ctx->d_params, b, x, x_stride, nrhs, o64,
                                     o64s, o128, o128s, slots, nslot, ln.stream));
        sp->done(nrhs);
    } else if (ctx->resid_mode == ZSOLVE_RESID_FX) {
        const int64_t xl_stride = (int64_t)ctx->nrhs_max * zs_fx_x_bytes(n);
        ZS_CU(zs_launch_split_fx(x, x_stride, n, nrhs, ctx->xl, xl_stride, ctx->xe, ctx->nrhs_max, slots, nslot,
                                 ln.stream));
        ZS_CU(zs_launch_residual_fx(ctx->z64, ctx->z64_stride, ctx->zexp, n, b, x, x_stride, ctx->xl, xl_stride,
                                    ctx->xe, ctx->nrhs_max, nrhs, o64, o64s, o128, o128s, slots, nslot, ctx->fx_ndf,
                                    ln.stream));
        int chunks = 0;
        for (int r = nrhs; r > 0; chunks++) r -= r >= 4 ? 4 : r >= 2 ? 2 : 1;
        sp->done(1 + chunks);
    } else if (ctx->resid_mode == ZSOLVE_RESID_DF) {
        const int64_t xs_stride = (int64_t)ctx->nrhs_max * n;
        ZS_CU(zs_launch_split_x(x, x_stride, n, nrhs, ctx->xs, xs_stride, slots, nslot, ln.stream));
        ZS_CU(zs_launch_residual_df(ctx->z64, ctx->z64_stride, n, b, ctx->xs, xs_stride, nrhs, o64, o64s, o128, o128s,
                                    slots, nslot, ln.stream));
        int chunks = 0;
        for (int r = nrhs; r > 0; chunks++) r -= r >= 4 ? 4 : r >= 2 ? 2 : 1;
        sp->done(1 + chunks);
    } else {
        ZS_CU(zs_launch_residual(ctx->z64, ctx->z64_stride, n, b, x, x_stride, nrhs, o64, o64s, o128, o128s, slots,
                                 nslot, ln.stream));
        sp->done(zs_rhs_chunks(nrhs));
    }
    return ZSOLVE_OK;
}

// Start-up check of the double-float residual against the float64 one on a
// synthetic positive system (two cases: with and without real parts).
int resid_selftest(zsolve_ctx *ctx) {
    const int64_t n = ctx->n;
    double2 *tx = nullptr, *tr = nullptr, *tb = nullptr;
    std::vector<double2> h1(n), h2(n);
    int ok = 1;
    if (cudaMalloc(&tx, n * sizeof(double2)) != cudaSuccess || cudaMalloc(&tr, 2 * n * sizeof(double2)) != cudaSuccess ||
        cudaMalloc(&tb, n * sizeof(double2)) != cudaSuccess) {
        cudaFree(tx);
        cudaFree(tr);
        cudaFree(tb);
        cudaGetLastError();
        return fail(ctx, ZSOLVE_ENOMEM, "residual self-test buffers");
    }
    for (int zero_re = 0; zero_re < 2 && ok; zero_re++) {
        ZS_CU(cudaMemsetAsync(tb, 0, n * sizeof(double2), ctx->lane[0].stream));
        ZS_CU(zs_launch_selftest_fill(ctx->z64, tx, n, zero_re, ctx->lane[0].stream));
        ZS_CU(zs_launch_residual(ctx->z64, ctx->z64_stride, n, tb, tx, 0, 1, nullptr, 0, tr, 0, ctx->d_all, 1,
                                 ctx->lane[0].stream));
        ZS_CU(zs_launch_split_x(tx, 0, n, 1, ctx->xs, 0, ctx->d_all, 1, ctx->lane[0].stream));
        ZS_CU(zs_launch_residual_df(ctx->z64, ctx->z64_stride, n, tb, ctx->xs, 0, 1, nullptr, 0, tr + n, 0, ctx->d_all,
                                    1, ctx->lane[0].stream));
        ZS_CU(cudaMemcpyAsync(h1.data(), tr, n * sizeof(double2), cudaMemcpyDeviceToHost, ctx->lane[0].stream));
        ZS_CU(cudaMemcpyAsync(h2.data(), tr + n, n * sizeof(double2), cudaMemcpyDeviceToHost, ctx->lane[0].stream));
        ZS_CU(cudaStreamSynchronize(ctx->lane[0].stream));
        double err = 0.0, scale = 0.0;
        for (int64_t i = 0; i < n; i++) {
            err = std::max(err, std::max(fabs(h1[i].x - h2[i].x), fabs(h1[i].y - h2[i].y)));
            scale = std::max(scale, std::max(fabs(h1[i].x), fabs(h1[i].y)));
        }
        if (!(err <= 1e-12 * scale)) ok = 0;
    }
    cudaFree(tx);
    cudaFree(tr);
    cudaFree(tb);
    ctx->resid_mode = ok ? ZSOLVE_RESID_DF : ZSOLVE_RESID_F64;
    return ZSOLVE_OK;
}

// Refinement of slots first..first+count-1 on lane ln; x for slot s is at
// x + s*x_stride (x is the batch's base).
// Hand-over between the two lanes of a staggered refinement: the leading
// lane records ev once its first solve is queued and opens the gate; the
// other lane's host thread waits at the gate, then makes its stream wait for
// ev.  The gate is opened on every path, so the waiting thread cannot hang.
struct Stagger {
    std::mutex m;
    std::condition_variable cv;
    bool ready = false;
    cudaEvent_t ev = nullptr;
    void open() {
        {
            std::lock_guard<std::mutex> lock(m);
            ready = true;
        }
        cv.notify_all();
    }
    void wait() {
        std::unique_lock<std::mutex> lock(m);
        cv.wait(lock, [this] { return ready; });
    }
};

int refine_batch(zsolve_ctx *ctx, Lane &ln, const double2 *b, double2 *x, int64_t x_stride, int nrhs, int first,
                 int count, zsolve_info *info, Stagger *lead = nullptr) {
    const int64_t n = ctx->n;
    const zsolve_opts &o = ctx->opts;
    std::vector<int> active, stalled;  // slot indices
    std::vector<double> prev(count, INFINITY), last(count, 1.0);
    std::vector<int> grow(count, 0), iters(count, 0);
    // Slots whose factorisation met a bad pivot go to the fallback.  The flags
    // come back with the first correction norms, so that the first solve is
    // queued behind the factorisation without a wait on the host; a flagged
    // slot's first solve and correction are wasted work, and its x is then
    // the fallback's.  (A forced fallback, or no corrections, reads them here.)
    ZS_CU(cudaMemcpyAsync(ctx->h_pivflag + first, ctx->d_pivflag + first, sizeof(int) * count,
                          cudaMemcpyDeviceToHost, ln.stream));
    bool flags_read = false;
    auto take_flags = [&]() {
        flags_read = true;
        std::vector<int> keep;
        for (int i = 0; i < count; i++) {
            const int s = first + i;
            if (info) info[i].pivot_flag = ctx->h_pivflag[s];
        }
        for (int s : active) {
            if (ctx->h_pivflag[s]) stalled.push_back(s);
            else keep.push_back(s);
        }
        active.swap(keep);
    };
    if (o.force_fallback) {
        ZS_CU(cudaStreamSynchronize(ln.stream));
        for (int i = 0; i < count; i++) stalled.push_back(first + i);
        take_flags();
    } else {
        for (int i = 0; i < count; i++) active.push_back(first + i);
        if (o.max_iter < 1) {
            ZS_CU(cudaStreamSynchronize(ln.stream));
            take_flags();
        }
    }
    auto upload_active = [&]() -> int {
        for (size_t i = 0; i < active.size(); i++) ln.h_active[i] = active[i];
        ZS_CU(cudaMemcpyAsync(ln.d_active, ln.h_active, sizeof(int) * active.size(), cudaMemcpyHostToDevice,
                              ln.stream));
        return ZSOLVE_OK;
    };
    if (!active.empty()) {
        ZS_TRY(upload_active());
        const int na = (int)active.size();
        // step 2: first solve with the low-precision factors
        {
            StageSpan sp(ctx, ZSOLVE_STAGE_UPDATE, ln.stream);
            ZS_CU(zs_launch_cast_rhs(b, n, nrhs, ctx->v, ctx->v_stride, ln.d_active, na, ln.stream));
            sp.done(1);
        }
        ZS_TRY(lowprec_solve_slots(ctx, ln, nrhs, ln.d_active, na));
        if (lead) {
            ZS_CU(cudaEventRecord(lead->ev, ln.stream));
            lead->open();
        }
        StageSpan sp(ctx, ZSOLVE_STAGE_UPDATE, ln.stream);
        ZS_CU(zs_launch_update(x, x_stride, ctx->v, ctx->v_stride, n, nrhs, 1, ctx->partials, ctx->nchunks,
                               ln.d_active, na, ln.stream));
        sp.done(1);
    }
    for (int it = 1; it <= o.max_iter && !active.empty(); it++) {
        const int na = (int)active.size();
        // step 3: residual in double precision, rounded for the low-precision solve
        {
            StageSpan sp(ctx, ZSOLVE_STAGE_RESIDUAL, ln.stream);
            ZS_TRY(residual_slots(ctx, ln, b, x, x_stride, nrhs, ctx->v, ctx->v_stride, nullptr, 0, ln.d_active, na,
                                  &sp));
        }
        // step 4: correction and update
        ZS_TRY(lowprec_solve_slots(ctx, ln, nrhs, ln.d_active, na));
        {
            StageSpan sp(ctx, ZSOLVE_STAGE_UPDATE, ln.stream);
            ZS_CU(zs_launch_update(x, x_stride, ctx->v, ctx->v_stride, n, nrhs, 0, ctx->partials, ctx->nchunks,
                                   ln.d_active, na, ln.stream));
            ZS_CU(zs_launch_relcorr(ctx->partials, ctx->nchunks, nrhs, ctx->d_relcorr, ln.d_active, na, ln.stream));
            sp.done(2);
        }
        ZS_CU(cudaMemcpyAsync(ctx->h_relcorr + (int64_t)first * nrhs, ctx->d_relcorr + (int64_t)first * nrhs,
                              sizeof(double) * (size_t)count * nrhs, cudaMemcpyDeviceToHost, ln.stream));
        ZS_TRY(check_device_status(ctx, ln));  // synchronises
        if (!flags_read) take_flags();  // the flagged slots leave before their norms count
        std::vector<int> next;
        for (int s : active) {
            const int i = s - first;
            double rc = 0.0;
            bool bad = false;
            for (int r = 0; r < nrhs; r++) {
                const double v = ctx->h_relcorr[(int64_t)s * nrhs + r];
                if (!isfinite(v)) bad = true;
                else rc = std::max(rc, v);
            }
            iters[i] = it;
            last[i] = bad ? NAN : rc;
            if (bad) {
                stalled.push_back(s);
                continue;
            }
            if (rc < o.tol) continue;  // converged
            grow[i] = (rc > prev[i]) ? grow[i] + 1 : 0;
            prev[i] = rc;
            if (grow[i] >= 2) stalled.push_back(s);  // diverging
            else next.push_back(s);
        }
        active.swap(next);
        if (!active.empty() && it < o.max_iter) ZS_TRY(upload_active());
    }
    for (int s : active) stalled.push_back(s);  // not converged after max_iter corrections
    std::sort(stalled.begin(), stalled.end());
    for (int i = 0; i < count; i++)
        if (info) {
            info[i].iters = iters[i];
            info[i].relcorr = last[i];
            info[i].fallback = 0;
            info[i].status = ZSOLVE_OK;
            info[i].gemm = gemm_public(ctx->gemm_eff);
        }
    for (int s : stalled) {
        const int i = s - first;
        int st = fallback_slot(ctx, ln, s, b, x + (int64_t)s * x_stride, nrhs);
        if (info) {
            info[i].fallback = 1;
            info[i].status = st;
            info[i].relcorr = 0.0;
        }
        if (st != ZSOLVE_OK && st != ZSOLVE_ESINGULAR) return st;
        if (st == ZSOLVE_ESINGULAR && !info) return st;
    }
    return ZSOLVE_OK;
}

int check_nrhs(zsolve_ctx *ctx, int nrhs) {
    if (nrhs < 1 || nrhs > ctx->nrhs_max)
        return fail(ctx, ZSOLVE_EINVAL, "nrhs=%d outside 1..%d", nrhs, ctx->nrhs_max);
    return ZSOLVE_OK;
}

// A sweep lane of `count` frequencies whose residual reads L, Psi, G rather
// than the float64 matrices: LPG, and OZ where its tensor-core product serves
// (four or more (frequency, right-hand side) pairs; the OZ residual then keeps
// to the product as the lane's frequencies converge).  Its assembly forms the
// float32 planes alone.
bool z32_only(const zsolve_ctx *ctx, int count) {
    if (!ctx->cur_L) return false;
    return ctx->resid_mode == ZSOLVE_RESID_LPG ||
           (ctx->resid_mode == ZSOLVE_RESID_OZ && (int64_t)count * ctx->cur_nrhs >= kOzMinPairs);
}

// Assembly of one lane's share of a batch: slots first..first+count-1.
// While a host-pointer sweep's inputs are still being copied (ctx->nband
// row bands, band b's rows complete at ctx->band_ev[b]), the assembly runs
// band by band behind the copies.
int assemble_lane(zsolve_ctx *ctx, Lane &ln, const double *L, const double *Psi, const double *G, int first,
                  int count) {
    ZS_CU(cudaEventRecord(ln.ev[0], ln.stream));
    StageSpan sp(ctx, ZSOLVE_STAGE_ASSEMBLE, ln.stream);
    const int nb = ctx->nband > 0 ? ctx->nband : 1;
    const bool only32 = z32_only(ctx, count);
    ln.z64_formed = !only32;
    for (int bnd = 0; bnd < nb; bnd++) {
        const int64_t r0 = ctx->n * bnd / nb, r1 = ctx->n * (bnd + 1) / nb;
        if (ctx->nband > 0) ZS_CU(cudaStreamWaitEvent(ln.stream, ctx->band_ev[bnd], 0));
        if (only32)
            ZS_CU(zs_launch_assemble32(L, Psi, G, ctx->n, r0, r1, ctx->d_params + first, count,
                                       ctx->z32 + (int64_t)first * ctx->z32_stride, ctx->ld, ctx->plane,
                                       ctx->z32_stride, ln.stream));
        else
            ZS_CU(zs_launch_assemble(L, Psi, G, ctx->n, r0, r1, ctx->d_params + first, count,
                                     ctx->z64 + (int64_t)first * ctx->z64_stride, ctx->z64_stride,
                                     ctx->z32 + (int64_t)first * ctx->z32_stride, ctx->ld, ctx->plane,
                                     ctx->z32_stride, ln.stream,
                                     ctx->zexp ? ctx->zexp + (int64_t)first * ctx->n : nullptr));
    }
    sp.done(nb);
    ctx->nband = 0;  // the first assembly of a sweep waited for every band
    ZS_CU(cudaEventRecord(ln.ev[1], ln.stream));
    return ZSOLVE_OK;
}

// One lane's share of a batch (slots first..first+count-1): assembled unless
// `assembled`, then factored on ln's stream; ln.ev[0..2] mark the start, the
// end of the assembly and the end of the factorisation.
int factor_lane(zsolve_ctx *ctx, Lane &ln, const double *L, const double *Psi, const double *G, int first,
                int count, bool assembled) {
    if (!assembled) ZS_TRY(assemble_lane(ctx, ln, L, Psi, G, first, count));
    ZS_TRY(factor_slots(ctx, ln, ctx->d_all + first, count, first));
    ZS_CU(cudaEventRecord(ln.ev[2], ln.stream));
    return ZSOLVE_OK;
}

// Refinement of the batch's slots first..first+count-1 on ln's stream, after
// every lane in fl[0..nl) has factored its range [lo[i], lo[i] + cnt[i]) of
// them; then the per-frequency timings.  xb and ib are the batch's base
// (slot 0).  lead: see Stagger.
int refine_lanes(zsolve_ctx *ctx, Lane &ln, const double2 *b, double2 *xb, int nrhs, int first, int count,
                 zsolve_info *ib, Lane *const *fl, const int *lo, const int *cnt, int nl, Stagger *lead = nullptr) {
    ZS_CU(cudaEventRecord(ln.ev[3], ln.stream));  // refinement starts
    const int st = refine_batch(ctx, ln, b, xb, (int64_t)nrhs * ctx->n, nrhs, first, count, ib ? ib + first : nullptr,
                                lead);
    if (st != ZSOLVE_OK && st != ZSOLVE_ESINGULAR) return st;
    ZS_CU(cudaEventRecord(ln.ev[4], ln.stream));
    ZS_CU(cudaEventSynchronize(ln.ev[4]));
    if (ib) {
        float r = 0;
        cudaEventElapsedTime(&r, ln.ev[3], ln.ev[4]);
        for (int k = 0; k < nl; k++) {
            float a = 0, fct = 0;
            cudaEventElapsedTime(&a, fl[k]->ev[0], fl[k]->ev[1]);
            cudaEventElapsedTime(&fct, fl[k]->ev[1], fl[k]->ev[2]);
            for (int i = lo[k]; i < lo[k] + cnt[k]; i++) {
                ib[i].ms_assemble = a / cnt[k];
                ib[i].ms_factor = fct / cnt[k];
                ib[i].ms_refine = r / count;
            }
        }
    }
    return st;
}

// ZSOLVE_GEMM_AUTO: the arithmetic of the factorisation picked by measured
// convergence and speed.  Frequency `f` of the first sweep is solved alone
// (assembly, factorisation, refinement) once in each arithmetic -- TF32,
// TF32X3, FFMA -- on lane 0, with its device time (CUDA events) and its
// correction count recorded; the context then keeps, among the arithmetics
// whose refinement converged without the fallback, the one with the smallest
// time (TF32X3 if none did).  x receives the probe solutions (overwritten by
// the sweep afterwards).
int auto_probe(zsolve_ctx *ctx, const double *L, const double *Psi, const double *G, double omega, double zre,
               double zim, const double2 *b, double2 *x, int nrhs) {
    Lane &ln = ctx->lane[0];
    ctx->h_params[0] = ZsSlotParam{omega, zre, zim, 1.0 / omega};
    ZS_CU(cudaMemcpyAsync(ctx->d_params, ctx->h_params, sizeof(ZsSlotParam), cudaMemcpyHostToDevice, ln.stream));
    zsolve_gemm_probe pr{};
    for (int k = 0; k < 3; k++) {  // index k = ZSOLVE_GEMM_TF32 - 1, TF32X3 - 1, FFMA - 1
        ctx->gemm_eff = gemm_internal(k + 1);
        ln.tc_grid = ctx->num_sms;
        ln.trsv_grid = 0;
        ZS_TRY(factor_lane(ctx, ln, L, Psi, G, 0, 1, false));  // records ln.ev[0] first
        zsolve_info inf{};
        const int st = refine_batch(ctx, ln, b, x, 0, nrhs, 0, 1, &inf);
        if (st != ZSOLVE_OK && st != ZSOLVE_ESINGULAR) return st;
        ZS_CU(cudaEventRecord(ln.ev[4], ln.stream));
        ZS_CU(cudaEventSynchronize(ln.ev[4]));
        float ms = 0.f;
        ZS_CU(cudaEventElapsedTime(&ms, ln.ev[0], ln.ev[4]));
        pr.ms[k] = ms;
        pr.iters[k] = inf.iters;
        pr.fallback[k] = inf.fallback || st != ZSOLVE_OK;
    }
    int best = -1;
    for (int k = 0; k < 3; k++)
        if (!pr.fallback[k] && (best < 0 || pr.ms[k] < pr.ms[best])) best = k;
    pr.done = 1;
    pr.chosen = best < 0 ? ZSOLVE_GEMM_TF32X3 : best + 1;
    ctx->probe = pr;
    ctx->gemm_eff = gemm_internal(pr.chosen);
    return ZSOLVE_OK;
}

int sweep_impl(zsolve_ctx *ctx, const double *L, const double *Psi, const double *G, const double *omega,
               const double *zs, int nf, const double2 *b, double2 *x, int nrhs, zsolve_info *info) {
    const int64_t n = ctx->n;
    for (int f = 0; f < nf; f++)
        if (!(omega[f] > 0.0) || !isfinite(omega[f]) || !isfinite(zs[2 * f]) || !isfinite(zs[2 * f + 1]))
            return fail(ctx, ZSOLVE_EINVAL, "frequency %d: omega must be positive and finite, Zs finite", f);
    ctx->cur_L = L;
    ctx->cur_Psi = Psi;
    ctx->cur_G = G;
    ctx->cur_nrhs = nrhs;
    struct Clear {  // the pointers are borrowed for this call only
        zsolve_ctx *c;
        ~Clear() {
            c->cur_L = c->cur_Psi = c->cur_G = nullptr;
            // on every exit the context's stream follows the digits of L, Psi,
            // G (read from the caller's inputs), so that the caller may reuse them
            if (c->oz_ready) cudaStreamWaitEvent(c->stream, c->oz_done, 0);
            c->oz_ready = false;
        }
    } clear_ptrs{ctx};
    if (ctx->resid_mode == ZSOLVE_RESID_OZ && nf > 0) {
        // before every lane's work: the other lanes start after lane 0's assembly
        ZS_TRY(oz_split_inputs(ctx, L, Psi, G, ctx->lane[0].stream));
        ctx->oz_ready = true;
    }
    if (ctx->opts.gemm == ZSOLVE_GEMM_AUTO && !ctx->probe.done && nf > 0) {
        // the host-pointer sweep's inputs may still be in flight: the probe's
        // assembly waits for every band, the sweep's first one then runs plain
        ZS_TRY(auto_probe(ctx, L, Psi, G, omega[0], zs[0], zs[1], b, x, nrhs));
        ctx->nband = 0;
    }
    Lane &l0 = ctx->lane[0];
    int first_err = ZSOLVE_OK;
    for (int f0 = 0; f0 < nf; f0 += ctx->S) {
        const int count = std::min(ctx->S, nf - f0);
        for (int s = 0; s < count; s++)
            ctx->h_params[s] =
                ZsSlotParam{omega[f0 + s], zs[2 * (f0 + s)], zs[2 * (f0 + s) + 1], 1.0 / omega[f0 + s]};
        ZS_CU(cudaMemcpyAsync(ctx->d_params, ctx->h_params, sizeof(ZsSlotParam) * count, cudaMemcpyHostToDevice,
                              l0.stream));
        double2 *xb = x + (int64_t)f0 * nrhs * n;
        zsolve_info *ib = info ? info + f0 : nullptr;
        int st;
        if (ctx->opts.lanes == 1 || count < 2) {
            l0.tc_grid = ctx->num_sms;
            ZS_TRY(factor_lane(ctx, l0, L, Psi, G, 0, count, false));
            l0.trsv_grid = 0;
            Lane *fl[1] = {&l0};
            const int lo[1] = {0}, cnt[1] = {count};
            st = refine_lanes(ctx, l0, b, xb, nrhs, 0, count, ib, fl, lo, cnt, 1);
        } else {
            // K lanes (2, or 3 with opts.lanes = 3) factor and refine parts of
            // the batch side by side, lane k on its own stream and host thread
            // (lane 0 on the caller's).  Lane k starts after lane k-1's
            // assembly (lane 0 after everything queued before it on the
            // context's stream: inputs, parameters), so that its own FP64-bound
            // assembly runs under the earlier lanes' factorisations and the
            // lanes' outer-block steps stay out of phase.  Its refinement
            // starts when lane k-1's first solve has run, so that the lanes
            // alternate: one lane's triangular solve (latency-bound) beside
            // another's residual (FP64-bound on every SM); the triangular
            // solves take 1/K of the SMs each.
            const int K = (ctx->opts.lanes == 3 && count >= 3) ? 3 : 2;
            int lo[kMaxLanes], cnt[kMaxLanes];
            for (int k = 0, at = 0; k < K; k++) {
                cnt[k] = count / K + (k < count % K ? 1 : 0);
                lo[k] = at;
                at += cnt[k];
            }
            for (int k = 0; k < K; k++) {
                // each lane's persistent tcgen05 grids leave room for the
                // other lanes' diagonal blocks (one CTA per frequency)
                ctx->lane[k].tc_grid = std::max(1, ctx->num_sms - (count - cnt[k]));
                ctx->lane[k].trsv_grid = ctx->trsv_cap > 0 ? ctx->trsv_cap : std::max(1, ctx->num_sms / K);
                ctx->lane[k].alone = false;
            }
            struct Alone {  // lane 0 runs alone again after the batch (the probe, single-system calls)
                zsolve_ctx *c;
                ~Alone() {
                    for (auto &l : c->lane) l.alone = true;
                }
            } alone_again{ctx};
            Stagger asm_gate[kMaxLanes], ref_gate[kMaxLanes];  // lane k's assembly / first solve queued
            int stk[kMaxLanes] = {};
            for (int k = 0; k < K; k++) {
                asm_gate[k].ev = ctx->lane[k].ev[1];  // recorded by assemble_lane at its end
                ref_gate[k].ev = ctx->lane[k].ev_stag;
            }
            // the whole of lane k; opens both of its gates on every path
            auto run_lane = [&](int k) {
                Lane &ln = ctx->lane[k];
                int st_k = ZSOLVE_OK;
                if (k > 0 && cudaSetDevice(ctx->device) != cudaSuccess)
                    st_k = fail(ctx, ZSOLVE_ECUDA, "lane %d: cudaSetDevice failed", k);
                if (k > 0) {
                    asm_gate[k - 1].wait();
                    if (st_k == ZSOLVE_OK && cudaStreamWaitEvent(ln.stream, asm_gate[k - 1].ev, 0) != cudaSuccess)
                        st_k = fail(ctx, ZSOLVE_ECUDA, "lane %d: cudaStreamWaitEvent failed", k);
                }
                if (st_k == ZSOLVE_OK) st_k = assemble_lane(ctx, ln, L, Psi, G, lo[k], cnt[k]);
                asm_gate[k].open();
                if (st_k == ZSOLVE_OK) st_k = factor_lane(ctx, ln, L, Psi, G, lo[k], cnt[k], true);
                if (k > 0) {
                    ref_gate[k - 1].wait();
                    if (st_k == ZSOLVE_OK && cudaStreamWaitEvent(ln.stream, ref_gate[k - 1].ev, 0) != cudaSuccess)
                        st_k = fail(ctx, ZSOLVE_ECUDA, "lane %d: cudaStreamWaitEvent failed", k);
                }
                if (st_k == ZSOLVE_OK) {
                    Lane *fl[1] = {&ln};
                    const int lo1[1] = {lo[k]}, cnt1[1] = {cnt[k]};
                    st_k = refine_lanes(ctx, ln, b, xb, nrhs, lo[k], cnt[k], ib, fl, lo1, cnt1, 1,
                                        k + 1 < K ? &ref_gate[k] : nullptr);
                }
                ref_gate[k].open();
                stk[k] = st_k;
            };
            std::thread workers[kMaxLanes];
            bool threaded[kMaxLanes] = {};
            for (int k = 1; k < K; k++) {
                try {
                    workers[k] = std::thread(run_lane, k);
                    threaded[k] = true;
                } catch (...) {
                    threaded[k] = false;  // no thread: this lane runs after lane 0
                }
            }
            run_lane(0);
            for (int k = 1; k < K; k++) {
                if (threaded[k]) workers[k].join();
                else run_lane(k);
            }
            for (int k = 1; k < K; k++) {
                ZS_CU(cudaEventRecord(ctx->lane[k].ev_join, ctx->lane[k].stream));
                ZS_CU(cudaStreamWaitEvent(l0.stream, ctx->lane[k].ev_join, 0));
            }
            st = ZSOLVE_OK;
            for (int k = 0; k < K; k++)  // the first hard error, else the first singular fallback
                if (stk[k] != ZSOLVE_OK && stk[k] != ZSOLVE_ESINGULAR) {
                    st = stk[k];
                    break;
                }
            if (st == ZSOLVE_OK)
                for (int k = 0; k < K; k++)
                    if (stk[k] != ZSOLVE_OK) {
                        st = stk[k];
                        break;
                    }
        }
        if (st != ZSOLVE_OK && first_err == ZSOLVE_OK) first_err = st;
        if (st != ZSOLVE_OK && st != ZSOLVE_ESINGULAR) return st;
    }
    ctx->assembled = 0;  // slot 0 now holds the last batch's first frequency, not a single system
    ctx->factored = 0;
    return first_err;
}

void free_all(zsolve_ctx *c) {
    cudaFree(c->z64);
    cudaFree(c->z32);
    cudaFree(c->pack);
    cudaFree(c->dinv);
    cudaFree(c->inv32);
    cudaFree(c->winv);
    cudaFree(c->v);
    cudaFree(c->xs);
    cudaFree(c->xl);
    cudaFree(c->xe);
    cudaFree(c->zexp);
    cudaFree(c->oz_a);
    cudaFree(c->oz_ea);
    if (c->oz_stream) cudaStreamDestroy(c->oz_stream);
    if (c->oz_start) cudaEventDestroy(c->oz_start);
    if (c->oz_done) cudaEventDestroy(c->oz_done);
    cudaFree(c->partials);
    cudaFree(c->d_relcorr);
    cudaFreeHost(c->h_relcorr);
    cudaFree(c->d_params);
    cudaFreeHost(c->h_params);
    cudaFree(c->d_all);
    cudaFree(c->d_pivflag);
    cudaFreeHost(c->h_pivflag);
    cudaFree(c->prog);
    cudaFree(c->d_status);
    cudaFree(c->fb_a);
    cudaFree(c->fb_piv);
    cudaFree(c->fb_info);
    cudaFreeHost(c->h_fb_info);
    if (c->copy_stream) cudaStreamDestroy(c->copy_stream);
    for (auto q : c->copy_aux)
        if (q) cudaStreamDestroy(q);
    for (auto &pair : c->aux_ev)
        for (auto e : pair)
            if (e) cudaEventDestroy(e);
    for (auto e : c->band_ev)
        if (e) cudaEventDestroy(e);
    if (c->ev_host) cudaEventDestroy(c->ev_host);
    cudaFree(c->hd_L);
    cudaFree(c->hd_Psi);
    cudaFree(c->hd_G);
    cudaFree(c->hd_b);
    cudaFree(c->hd_x);
    for (auto &ln : c->lane) {
        cudaFree(ln.d_active);
        cudaFreeHost(ln.h_active);
        cudaFree(ln.ticket);
        cudaFree(ln.tile_ctr);
        cudaFreeHost(ln.h_status);
        cudaFree(ln.oz_x);
        cudaFree(ln.oz_ex);
        cudaFree(ln.oz_part);
        for (auto &e : ln.ev)
            if (e) cudaEventDestroy(e);
        if (ln.ev_fork) cudaEventDestroy(ln.ev_fork);
        if (ln.ev_join) cudaEventDestroy(ln.ev_join);
        if (ln.ev_stag) cudaEventDestroy(ln.ev_stag);
        if (ln.side) cudaStreamDestroy(ln.side);
        if (ln.own_stream && ln.stream) cudaStreamDestroy(ln.stream);
    }
    for (auto &sp : c->pending) {
        cudaEventDestroy(sp.a);
        cudaEventDestroy(sp.b);
    }
    for (auto e : c->ev_pool) cudaEventDestroy(e);
    c->pending.clear();
    c->ev_pool.clear();
}

}  // namespace

cudaStream_t zs_ctx_stream(const zsolve_ctx *ctx) { return ctx->stream; }
int64_t zs_ctx_n(const zsolve_ctx *ctx) { return ctx->n; }
int zs_ctx_nrhs_max(const zsolve_ctx *ctx) { return ctx->nrhs_max; }

extern "C" {

int zsolve_default_opts(zsolve_opts *opts) {
    if (!opts) return ZSOLVE_EINVAL;
    opts->tol = 1e-11;
    opts->max_iter = 10;
    opts->gemm = ZSOLVE_GEMM_AUTO;
    opts->outer_block = ZS_NB;
    opts->batch = 0;
    opts->force_fallback = 0;
    opts->profile = 0;
    opts->resid = ZSOLVE_RESID_F64;
    opts->lanes = 0;
    opts->symmetric = 1;
    opts->wait_limit = 0;
    return ZSOLVE_OK;
}

int zsolve_create(zsolve_ctx **out, int64_t n, int nrhs_max, const zsolve_opts *opts) {
    if (!out || n <= 0 || nrhs_max < 1 || nrhs_max > 64) return ZSOLVE_EINVAL;
    *out = nullptr;
    zsolve_ctx *ctx = new (std::nothrow) zsolve_ctx();
    if (!ctx) return ZSOLVE_ENOMEM;
    if (opts) ctx->opts = *opts;
    else zsolve_default_opts(&ctx->opts);
    if (ctx->opts.outer_block == 0) ctx->opts.outer_block = ZS_NB;
    if (ctx->opts.outer_block != ZS_NB || ctx->opts.max_iter < 0 || !(ctx->opts.tol > 0.0) || ctx->opts.gemm < 0 ||
        ctx->opts.gemm > ZSOLVE_GEMM_FFMA || ctx->opts.batch < 0 || ctx->opts.resid < 0 ||
        ctx->opts.resid > ZSOLVE_RESID_OZ || ctx->opts.lanes < 0 || ctx->opts.lanes > 3 || ctx->opts.symmetric < 0 ||
        ctx->opts.symmetric > 1 || ctx->opts.wait_limit < 0) {
        delete ctx;
        return ZSOLVE_EINVAL;
    }
    ctx->n = n;
    ctx->nrhs_max = nrhs_max;
    ctx->gemm_eff = gemm_mode(ctx->opts);
    ctx->probe.chosen = ctx->opts.gemm == ZSOLVE_GEMM_AUTO ? ZSOLVE_GEMM_TF32X3 : ctx->opts.gemm;
    if (ctx->opts.wait_limit > 0) ctx->wait_limit = (unsigned)ctx->opts.wait_limit;
    if (const char *e = getenv("ZSOLVE_FX_NDF")) ctx->fx_ndf = std::min(3, std::max(0, atoi(e)));
    if (const char *e = getenv("ZSOLVE_LOOKAHEAD")) ctx->lookahead = std::min(1, std::max(-1, atoi(e)));
    // testing aid: few CTAs per tcgen05 launch, so that each takes many tiles
    if (const char *e = getenv("ZSOLVE_TC_GRID")) ctx->tc_cap = std::max(0, atoi(e));
    // testing aid: zsolve_assemble rewrites its float32 planes with the kernel
    // that sweeps with the OZ or LPG residual use, so that they can be compared
    if (const char *e = getenv("ZSOLVE_ASM32")) ctx->asm32_planes = atoi(e) != 0;
    if (const char *e = getenv("ZSOLVE_TRSV_CTAS")) ctx->trsv_cap = std::max(0, atoi(e));
    // right-hand sides per triangular-solve chain (1, 2 or 4; unset: chosen per solve)
    if (const char *e = getenv("ZSOLVE_TRSV_R")) {
        const int r = atoi(e);
        ctx->trsv_r = (r == 1 || r == 2 || r == 4) ? r : 0;
    }
    auto bail = [&](int code) {
        free_all(ctx);
        delete ctx;
        return code;
    };
    if (cudaGetDevice(&ctx->device) != cudaSuccess) return bail(ZSOLVE_ECUDA);
    cudaDeviceGetAttribute(&ctx->num_sms, cudaDevAttrMultiProcessorCount, ctx->device);
    ctx->ld = (n + 31) / 32 * 32;
    ctx->plane = n * ctx->ld;
    ctx->z32_stride = 2 * ctx->plane;
    ctx->z64_stride = n * n;
    ctx->pack_stride = 6 * zs_pack_plane(n);
    ctx->v_stride = (int64_t)nrhs_max * n;
    ctx->dinv_stride = zs_dinv_stride(n);
    if (ctx->opts.batch > 0) {
        ctx->S = ctx->opts.batch;
    } else {
        size_t budget = (size_t)8 << 30;
        size_t sb = slot_bytes(n, ctx->ld);
        ctx->S = (int)std::max<size_t>(1, std::min<size_t>(32, budget / sb));
    }
    if (ctx->S > 64) ctx->S = 64;
    const int S = ctx->S;
    ctx->nchunks = zs_update_chunks(n);
#define ALLOC(p, bytes) \
    if (cudaMalloc(&(p), (bytes)) != cudaSuccess) return bail(ZSOLVE_ENOMEM)
#define ALLOCH(p, bytes) \
    if (cudaMallocHost(&(p), (bytes)) != cudaSuccess) return bail(ZSOLVE_ENOMEM)
    ALLOC(ctx->z64, (size_t)S * ctx->z64_stride * sizeof(double2));
    ALLOC(ctx->z32, (size_t)S * ctx->z32_stride * sizeof(float));
    ALLOC(ctx->pack, (size_t)2 * S * ctx->pack_stride * sizeof(float));
    ALLOC(ctx->dinv, (size_t)S * ctx->dinv_stride * sizeof(float));
    // AUTO may pick any arithmetic: it holds the workspaces of both kinds
    const bool is_auto = ctx->opts.gemm == ZSOLVE_GEMM_AUTO;
    if (is_auto || gemm_mode(ctx->opts) == 0) ALLOC(ctx->inv32, (size_t)S * zs_inv32_slot_stride(n) * sizeof(float));
    if (is_auto || gemm_mode(ctx->opts) != 0) ALLOC(ctx->winv, (size_t)S * ZS_WINV_STRIDE * sizeof(float));
    ALLOC(ctx->v, (size_t)S * ctx->v_stride * sizeof(float2));
    ALLOC(ctx->partials, (size_t)S * nrhs_max * ctx->nchunks * 2 * sizeof(double));
    ALLOC(ctx->d_relcorr, (size_t)S * nrhs_max * sizeof(double));
    ALLOCH(ctx->h_relcorr, (size_t)S * nrhs_max * sizeof(double));
    ALLOC(ctx->d_params, S * sizeof(ZsSlotParam));
    ALLOCH(ctx->h_params, S * sizeof(ZsSlotParam));
    ALLOC(ctx->d_all, S * sizeof(int));
    ALLOC(ctx->d_pivflag, S * sizeof(int));
    ALLOCH(ctx->h_pivflag, S * sizeof(int));
    ALLOC(ctx->prog, (size_t)S * 2 * ZS_TRSV_MAX_GROUPS * sizeof(unsigned long long));
    ALLOC(ctx->d_status, sizeof(unsigned));
    for (int l = 0; l < kMaxLanes; l++) {
        Lane &ln = ctx->lane[l];
        ALLOC(ln.d_active, S * sizeof(int));
        ALLOCH(ln.h_active, S * sizeof(int));
        ALLOC(ln.ticket, sizeof(unsigned));
        ALLOC(ln.tile_ctr, kMaxCtr * sizeof(unsigned));
        ALLOCH(ln.h_status, sizeof(unsigned));
        *ln.h_status = 0;
    }
#undef ALLOC
#undef ALLOCH
    for (int l = 0; l < kMaxLanes; l++) {
        Lane &ln = ctx->lane[l];
        for (auto &e : ln.ev)
            if (cudaEventCreate(&e) != cudaSuccess) return bail(ZSOLVE_ECUDA);
        if (cudaStreamCreateWithFlags(&ln.side, cudaStreamNonBlocking) != cudaSuccess ||
            cudaEventCreateWithFlags(&ln.ev_fork, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&ln.ev_join, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&ln.ev_stag, cudaEventDisableTiming) != cudaSuccess)
            return bail(ZSOLVE_ECUDA);
    }
    for (int l = 1; l < kMaxLanes; l++) {
        if (cudaStreamCreateWithFlags(&ctx->lane[l].stream, cudaStreamNonBlocking) != cudaSuccess)
            return bail(ZSOLVE_ECUDA);
        ctx->lane[l].own_stream = true;
    }
    ctx->lane[0].stream = ctx->stream;
    for (auto &ln : ctx->lane) ln.tc_grid = ctx->num_sms;
    if (ctx->winv &&
        (zs_tc_pack_map(ctx->pack, n, S, ctx->pack_stride, 128, ctx->pack_map[0]) != cudaSuccess ||
         zs_tc_pack_map(ctx->pack, n, S, ctx->pack_stride, 32, ctx->packst_map[0]) != cudaSuccess ||
         zs_tc_pack_map(ctx->pack + (int64_t)S * ctx->pack_stride, n, S, ctx->pack_stride, 128, ctx->pack_map[1]) !=
             cudaSuccess ||
         zs_tc_pack_map(ctx->pack + (int64_t)S * ctx->pack_stride, n, S, ctx->pack_stride, 32, ctx->packst_map[1]) !=
             cudaSuccess ||
         zs_tc_winv_map(ctx->winv, S, ctx->winv_map) != cudaSuccess ||
         zs_tc_z32_map(ctx->z32, n, ctx->ld, ctx->plane, S, ctx->z32_stride, ctx->z32_map) != cudaSuccess))
        return bail(ZSOLVE_ECUDA);
    std::vector<int> all(S);
    for (int s = 0; s < S; s++) all[s] = s;
    if (cudaMemcpy(ctx->d_all, all.data(), S * sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemset(ctx->prog, 0, (size_t)S * 2 * ZS_TRSV_MAX_GROUPS * sizeof(unsigned long long)) != cudaSuccess ||
        cudaMemset(ctx->d_status, 0, sizeof(unsigned)) != cudaSuccess ||
        cudaMemset(ctx->d_pivflag, 0, S * sizeof(int)) != cudaSuccess ||
        cudaMemset(ctx->z32, 0, (size_t)S * ctx->z32_stride * sizeof(float)) != cudaSuccess ||
        // the inverse blocks outside the triangles stay zero: the factorisation writes only the triangles
        cudaMemset(ctx->dinv, 0, (size_t)S * ctx->dinv_stride * sizeof(float)) != cudaSuccess ||
        (ctx->winv && cudaMemset(ctx->winv, 0, (size_t)S * ZS_WINV_STRIDE * sizeof(float)) != cudaSuccess))
        return bail(ZSOLVE_ECUDA);
    ctx->resid_mode = (ctx->opts.resid == ZSOLVE_RESID_FX || ctx->opts.resid == ZSOLVE_RESID_LPG ||
                       ctx->opts.resid == ZSOLVE_RESID_OZ)
                          ? ctx->opts.resid
                          : ZSOLVE_RESID_F64;
    if (ctx->opts.resid == ZSOLVE_RESID_OZ && ensure_oz(ctx) != ZSOLVE_OK) return bail(ZSOLVE_ENOMEM);
    if (ctx->opts.resid == ZSOLVE_RESID_FX) {
        if (cudaMalloc(&ctx->xl, (size_t)S * nrhs_max * zs_fx_x_bytes(n)) != cudaSuccess ||
            cudaMalloc(&ctx->xe, (size_t)S * nrhs_max * sizeof(int)) != cudaSuccess ||
            cudaMalloc(&ctx->zexp, (size_t)S * n * sizeof(int)) != cudaSuccess)
            return bail(ZSOLVE_ENOMEM);
    }
    if (ctx->opts.resid == ZSOLVE_RESID_DF) {
        if (cudaMalloc(&ctx->xs, (size_t)S * nrhs_max * n * sizeof(float4)) != cudaSuccess) return bail(ZSOLVE_ENOMEM);
        if (resid_selftest(ctx) != ZSOLVE_OK) return bail(ZSOLVE_ECUDA);
    }
    *out = ctx;
    return ZSOLVE_OK;
}

int zsolve_set_stream(zsolve_ctx *ctx, void *stream) {
    if (!ctx) return ZSOLVE_EINVAL;
    ctx->stream = (cudaStream_t)stream;
    ctx->lane[0].stream = ctx->stream;
    return ZSOLVE_OK;
}

int zsolve_assemble(zsolve_ctx *ctx, const double *L, const double *Psi, const double *G, double omega,
                    double zs_re, double zs_im) {
    if (!ctx || !L || !Psi || !G) return fail(ctx, ZSOLVE_EINVAL, "NULL argument");
    if (!(omega > 0.0) || !isfinite(omega) || !isfinite(zs_re) || !isfinite(zs_im))
        return fail(ctx, ZSOLVE_EINVAL, "omega must be positive and finite, Zs finite");
    ctx->h_params[0] = ZsSlotParam{omega, zs_re, zs_im, 1.0 / omega};
    ctx->single = ctx->h_params[0];
    ZS_CU(cudaMemcpyAsync(ctx->d_params, ctx->h_params, sizeof(ZsSlotParam), cudaMemcpyHostToDevice, ctx->stream));
    StageSpan sp(ctx, ZSOLVE_STAGE_ASSEMBLE, ctx->stream);
    ZS_CU(zs_launch_assemble(L, Psi, G, ctx->n, 0, ctx->n, ctx->d_params, 1, ctx->z64, ctx->z64_stride, ctx->z32,
                             ctx->ld, ctx->plane, ctx->z32_stride, ctx->stream, ctx->zexp));
    if (ctx->asm32_planes)
        ZS_CU(zs_launch_assemble32(L, Psi, G, ctx->n, 0, ctx->n, ctx->d_params, 1, ctx->z32, ctx->ld, ctx->plane,
                                   ctx->z32_stride, ctx->stream));
    sp.done(1);
    ctx->lane[0].z64_formed = true;
    ctx->assembled = 1;
    ctx->factored = 0;
    return ZSOLVE_OK;
}

int zsolve_factor(zsolve_ctx *ctx) {
    if (!ctx) return ZSOLVE_EINVAL;
    if (!ctx->assembled) return fail(ctx, ZSOLVE_ESTATE, "zsolve_factor before zsolve_assemble");
    if (ctx->factored) return ZSOLVE_OK;
    ZS_TRY(factor_slots(ctx, ctx->lane[0], ctx->d_all, 1, 0));
    ctx->factored = 1;
    return ZSOLVE_OK;
}

int zsolve_refine(zsolve_ctx *ctx, const void *b, void *x, int nrhs, zsolve_info *info) {
    if (!ctx || !b || !x) return fail(ctx, ZSOLVE_EINVAL, "NULL argument");
    ZS_TRY(check_nrhs(ctx, nrhs));
    if (!ctx->factored) return fail(ctx, ZSOLVE_ESTATE, "zsolve_refine before zsolve_factor");
    zsolve_info tmp{};
    ZS_CU(cudaEventRecord(ctx->lane[0].ev[2], ctx->stream));
    int st = refine_batch(ctx, ctx->lane[0], (const double2 *)b, (double2 *)x, 0, nrhs, 0, 1, &tmp);
    ZS_CU(cudaEventRecord(ctx->lane[0].ev[3], ctx->stream));
    ZS_CU(cudaEventSynchronize(ctx->lane[0].ev[3]));
    cudaEventElapsedTime(&tmp.ms_refine, ctx->lane[0].ev[2], ctx->lane[0].ev[3]);
    if (info) *info = tmp;
    if (st != ZSOLVE_OK) return st;
    return tmp.status;
}

int zsolve_sweep(zsolve_ctx *ctx, const double *L, const double *Psi, const double *G, const double *omega,
                 const double *zs, int nf, const void *b, void *x, int nrhs, zsolve_info *info) {
    if (!ctx || !L || !Psi || !G || !omega || !zs || !b || !x || nf < 0)
        return fail(ctx, ZSOLVE_EINVAL, "NULL argument or nf < 0");
    ZS_TRY(check_nrhs(ctx, nrhs));
    return sweep_impl(ctx, L, Psi, G, omega, zs, nf, (const double2 *)b, (double2 *)x, nrhs, info);
}

int zsolve_sweep_host(zsolve_ctx *ctx, const double *L, const double *Psi, const double *G, const double *omega,
                      const double *zs, int nf, const void *b, void *x, int nrhs, zsolve_info *info) {
    if (!ctx || !L || !Psi || !G || !omega || !zs || !b || !x || nf < 0)
        return fail(ctx, ZSOLVE_EINVAL, "NULL argument or nf < 0");
    ZS_TRY(check_nrhs(ctx, nrhs));
    const int64_t n = ctx->n;
    const size_t mb = (size_t)n * n * sizeof(double);
    if (!ctx->hd_L) {
        if (cudaMalloc(&ctx->hd_L, mb) != cudaSuccess || cudaMalloc(&ctx->hd_Psi, mb) != cudaSuccess ||
            cudaMalloc(&ctx->hd_G, mb) != cudaSuccess ||
            cudaMalloc(&ctx->hd_b, (size_t)ctx->nrhs_max * n * sizeof(double2)) != cudaSuccess) {
            cudaGetLastError();
            return fail(ctx, ZSOLVE_ENOMEM, "device buffers for host inputs");
        }
    }
    const size_t xb = (size_t)nf * nrhs * n * sizeof(double2);
    if (xb > ctx->hd_x_cap) {
        cudaFree(ctx->hd_x);
        ctx->hd_x = nullptr;
        ctx->hd_x_cap = 0;
        if (xb && cudaMalloc(&ctx->hd_x, xb) != cudaSuccess) {
            cudaGetLastError();
            return fail(ctx, ZSOLVE_ENOMEM, "device buffer for host solutions");
        }
        ctx->hd_x_cap = xb;
    }
    if (!ctx->copy_stream) {
        if (cudaStreamCreateWithFlags(&ctx->copy_stream, cudaStreamNonBlocking) != cudaSuccess ||
            cudaStreamCreateWithFlags(&ctx->copy_aux[0], cudaStreamNonBlocking) != cudaSuccess ||
            cudaStreamCreateWithFlags(&ctx->copy_aux[1], cudaStreamNonBlocking) != cudaSuccess ||
            cudaEventCreateWithFlags(&ctx->ev_host, cudaEventDisableTiming) != cudaSuccess)
            return fail(ctx, ZSOLVE_ECUDA, "copy streams for host inputs");
        for (auto &e : ctx->band_ev)
            if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess)
                return fail(ctx, ZSOLVE_ECUDA, "copy events for host inputs");
        for (auto &pair : ctx->aux_ev)
            for (auto &e : pair)
                if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess)
                    return fail(ctx, ZSOLVE_ECUDA, "copy events for host inputs");
    }
    ZS_CU(cudaMemcpyAsync(ctx->hd_b, b, (size_t)nrhs * n * sizeof(double2), cudaMemcpyHostToDevice, ctx->stream));
    // L, Psi, G in row bands on three copy streams, one per matrix (after
    // everything queued so far on the context's stream); band b is complete
    // at band_ev[b], and the first assembly follows band by band
    ZS_CU(cudaEventRecord(ctx->ev_host, ctx->stream));
    ZS_CU(cudaStreamWaitEvent(ctx->copy_stream, ctx->ev_host, 0));
    for (auto q : ctx->copy_aux) ZS_CU(cudaStreamWaitEvent(q, ctx->ev_host, 0));
    for (int bnd = 0; bnd < zsolve_ctx::kBands; bnd++) {
        const int64_t r0 = n * bnd / zsolve_ctx::kBands, r1 = n * (bnd + 1) / zsolve_ctx::kBands;
        const size_t off = (size_t)r0 * n, len = (size_t)(r1 - r0) * n * sizeof(double);
        ZS_CU(cudaMemcpyAsync(ctx->hd_L + off, L + off, len, cudaMemcpyHostToDevice, ctx->copy_stream));
        ZS_CU(cudaMemcpyAsync(ctx->hd_Psi + off, Psi + off, len, cudaMemcpyHostToDevice, ctx->copy_aux[0]));
        ZS_CU(cudaMemcpyAsync(ctx->hd_G + off, G + off, len, cudaMemcpyHostToDevice, ctx->copy_aux[1]));
        for (int q = 0; q < 2; q++) {
            ZS_CU(cudaEventRecord(ctx->aux_ev[bnd][q], ctx->copy_aux[q]));
            ZS_CU(cudaStreamWaitEvent(ctx->copy_stream, ctx->aux_ev[bnd][q], 0));
        }
        ZS_CU(cudaEventRecord(ctx->band_ev[bnd], ctx->copy_stream));
    }
    ctx->nband = zsolve_ctx::kBands;
    int st = sweep_impl(ctx, ctx->hd_L, ctx->hd_Psi, ctx->hd_G, omega, zs, nf, ctx->hd_b, ctx->hd_x, nrhs, info);
    ctx->nband = 0;
    // the copies are ordered before the context's stream continues, also
    // when the sweep stopped before its first assembly
    ZS_CU(cudaStreamWaitEvent(ctx->stream, ctx->band_ev[zsolve_ctx::kBands - 1], 0));
    if (st != ZSOLVE_OK && st != ZSOLVE_ESINGULAR) return st;
    if (xb) ZS_CU(cudaMemcpyAsync(x, ctx->hd_x, xb, cudaMemcpyDeviceToHost, ctx->stream));
    ZS_CU(cudaStreamSynchronize(ctx->stream));
    return st;
}

int zsolve_residual(zsolve_ctx *ctx, const void *b, const void *x, void *r, int nrhs) {
    if (!ctx || !b || !x || !r) return fail(ctx, ZSOLVE_EINVAL, "NULL argument");
    ZS_TRY(check_nrhs(ctx, nrhs));
    if (!ctx->assembled) return fail(ctx, ZSOLVE_ESTATE, "zsolve_residual before zsolve_assemble");
    StageSpan sp(ctx, ZSOLVE_STAGE_RESIDUAL, ctx->stream);
    ZS_TRY(residual_slots(ctx, ctx->lane[0], (const double2 *)b, (const double2 *)x, 0, nrhs, nullptr, 0, (double2 *)r, 0,
                          ctx->d_all, 1, &sp));
    ZS_CU(cudaStreamSynchronize(ctx->stream));
    return ZSOLVE_OK;
}

int zsolve_residual_lpg(zsolve_ctx *ctx, const double *L, const double *Psi, const double *G, const void *b,
                        const void *x, void *r, int nrhs) {
    if (!ctx || !L || !Psi || !G || !b || !x || !r) return fail(ctx, ZSOLVE_EINVAL, "NULL argument");
    ZS_TRY(check_nrhs(ctx, nrhs));
    if (!ctx->assembled) return fail(ctx, ZSOLVE_ESTATE, "zsolve_residual_lpg before zsolve_assemble");
    ctx->h_params[0] = ctx->single;  // slot 0 holds the single system's frequency again
    ZS_CU(cudaMemcpyAsync(ctx->d_params, ctx->h_params, sizeof(ZsSlotParam), cudaMemcpyHostToDevice, ctx->stream));
    StageSpan sp(ctx, ZSOLVE_STAGE_RESIDUAL, ctx->stream);
    ZS_CU(zs_launch_residual_lpg(L, Psi, G, ctx->n, ctx->d_params, (const double2 *)b, (const double2 *)x, 0, nrhs,
                                 nullptr, 0, (double2 *)r, 0, ctx->d_all, 1, ctx->stream));
    sp.done(nrhs);
    ZS_CU(cudaStreamSynchronize(ctx->stream));
    return ZSOLVE_OK;
}

int zsolve_residual_oz(zsolve_ctx *ctx, const double *L, const double *Psi, const double *G, const void *b,
                       const void *x, void *r, int nrhs) {
    if (!ctx || !L || !Psi || !G || !b || !x || !r) return fail(ctx, ZSOLVE_EINVAL, "NULL argument");
    ZS_TRY(check_nrhs(ctx, nrhs));
    if (!ctx->assembled) return fail(ctx, ZSOLVE_ESTATE, "zsolve_residual_oz before zsolve_assemble");
    ctx->h_params[0] = ctx->single;  // slot 0 holds the single system's frequency again
    ZS_CU(cudaMemcpyAsync(ctx->d_params, ctx->h_params, sizeof(ZsSlotParam), cudaMemcpyHostToDevice, ctx->stream));
    ZS_TRY(oz_split_inputs(ctx, L, Psi, G, ctx->stream));
    ZS_CU(cudaStreamWaitEvent(ctx->stream, ctx->oz_done, 0));
    Lane &ln = ctx->lane[0];
    StageSpan sp(ctx, ZSOLVE_STAGE_RESIDUAL, ctx->stream);
    ZS_CU(zs_launch_residual_oz(ctx->oz_amap, ctx->oz_ea, ctx->n, ctx->d_params, (const double2 *)b,
                                (const double2 *)x, 0, nrhs, nullptr, 0, (double2 *)r, 0, ctx->d_all, 1, ln.oz_x,
                                ln.oz_ex, ln.oz_ncol_cap, ln.oz_part, ln.oz_part_cap, ctx->d_status, ctx->num_sms,
                                ctx->stream));
    sp.done(3);
    return check_device_status(ctx, ln);  // synchronises
}

int zsolve_lowprec_solve(zsolve_ctx *ctx, const void *v, void *d, int nrhs) {
    if (!ctx || !v || !d) return fail(ctx, ZSOLVE_EINVAL, "NULL argument");
    ZS_TRY(check_nrhs(ctx, nrhs));
    if (!ctx->factored) return fail(ctx, ZSOLVE_ESTATE, "zsolve_lowprec_solve before zsolve_factor");
    const int64_t cnt = (int64_t)nrhs * ctx->n;
    {
        StageSpan sp(ctx, ZSOLVE_STAGE_UPDATE, ctx->stream);
        ZS_CU(zs_launch_narrow((const double2 *)v, ctx->v, cnt, ctx->stream));
        sp.done(1);
    }
    ZS_TRY(lowprec_solve_slots(ctx, ctx->lane[0], nrhs, ctx->d_all, 1));
    StageSpan sp(ctx, ZSOLVE_STAGE_UPDATE, ctx->stream);
    ZS_CU(zs_launch_widen(ctx->v, (double2 *)d, cnt, ctx->stream));
    sp.done(1);
    return check_device_status(ctx, ctx->lane[0]);
}

int zsolve_selftest_wait(zsolve_ctx *ctx, int nrhs) {
    if (!ctx) return ZSOLVE_EINVAL;
    ZS_TRY(check_nrhs(ctx, nrhs));
    if (!ctx->factored) return fail(ctx, ZSOLVE_ESTATE, "zsolve_selftest_wait before zsolve_factor");
    // every task of the first chain but its first waits, directly or through
    // the chain, for that chain's first block, which no task computes
    ZS_TRY(lowprec_solve_slots(ctx, ctx->lane[0], nrhs, ctx->d_all, 1, 1u));
    return check_device_status(ctx, ctx->lane[0]);
}

int zsolve_fallback_solve(zsolve_ctx *ctx, const void *b, void *x, int nrhs) {
    if (!ctx || !b || !x) return fail(ctx, ZSOLVE_EINVAL, "NULL argument");
    if (nrhs < 1 || nrhs > ctx->nrhs_max) return fail(ctx, ZSOLVE_EINVAL, "bad nrhs");
    if (!ctx->assembled) return fail(ctx, ZSOLVE_ESTATE, "zsolve_fallback_solve before zsolve_assemble");
    ZS_TRY(fallback_slot(ctx, ctx->lane[0], 0, (const double2 *)b, (double2 *)x, nrhs));
    ZS_CU(cudaStreamSynchronize(ctx->stream));
    return ZSOLVE_OK;
}

int zsolve_get_z64(zsolve_ctx *ctx, void *dst) {
    if (!ctx || !dst) return fail(ctx, ZSOLVE_EINVAL, "NULL argument");
    if (!ctx->assembled) return fail(ctx, ZSOLVE_ESTATE, "nothing assembled");
    ZS_CU(cudaMemcpyAsync(dst, ctx->z64, (size_t)ctx->n * ctx->n * sizeof(double2), cudaMemcpyDeviceToDevice,
                          ctx->stream));
    ZS_CU(cudaStreamSynchronize(ctx->stream));
    return ZSOLVE_OK;
}

int zsolve_get_z32(zsolve_ctx *ctx, float *re, float *im) {
    if (!ctx || !re || !im) return fail(ctx, ZSOLVE_EINVAL, "NULL argument");
    if (!ctx->assembled) return fail(ctx, ZSOLVE_ESTATE, "nothing assembled");
    ZS_CU(zs_launch_copy_z32_out(ctx->z32, ctx->ld, ctx->plane, ctx->n, re, im, ctx->stream));
    ZS_CU(cudaStreamSynchronize(ctx->stream));
    return ZSOLVE_OK;
}

int zsolve_pivot_flag(zsolve_ctx *ctx, int *flag) {
    if (!ctx || !flag) return fail(ctx, ZSOLVE_EINVAL, "NULL argument");
    if (!ctx->factored) return fail(ctx, ZSOLVE_ESTATE, "not factored");
    ZS_CU(cudaMemcpyAsync(ctx->h_pivflag, ctx->d_pivflag, sizeof(int), cudaMemcpyDeviceToHost, ctx->stream));
    ZS_CU(cudaStreamSynchronize(ctx->stream));
    *flag = ctx->h_pivflag[0];
    return ZSOLVE_OK;
}

int zsolve_get_profile(zsolve_ctx *ctx, zsolve_profile *out) {
    if (!ctx || !out) return fail(ctx, ZSOLVE_EINVAL, "NULL argument");
    ZS_TRY(prof_resolve(ctx));
    for (int i = 0; i < ZSOLVE_NSTAGE; i++) {
        out->launches[i] = ctx->prof_launches[i];
        out->ms[i] = ctx->prof_ms[i];
    }
    return ZSOLVE_OK;
}

int zsolve_reset_profile(zsolve_ctx *ctx) {
    if (!ctx) return ZSOLVE_EINVAL;
    ZS_TRY(prof_resolve(ctx));
    for (int i = 0; i < ZSOLVE_NSTAGE; i++) {
        ctx->prof_launches[i] = 0;
        ctx->prof_ms[i] = 0.0;
    }
    return ZSOLVE_OK;
}

int zsolve_get_gemm_choice(zsolve_ctx *ctx, zsolve_gemm_probe *out) {
    if (!ctx || !out) return fail(ctx, ZSOLVE_EINVAL, "NULL argument");
    *out = ctx->probe;
    out->chosen = gemm_public(ctx->gemm_eff);
    return ZSOLVE_OK;
}

int zsolve_get_resid_mode(zsolve_ctx *ctx, int *mode) {
    if (!ctx || !mode) return fail(ctx, ZSOLVE_EINVAL, "NULL argument");
    *mode = ctx->resid_mode;
    return ZSOLVE_OK;
}

const char *zsolve_strerror(int status) {
    switch (status) {
        case ZSOLVE_OK: return "ok";
        case ZSOLVE_EINVAL: return "invalid argument";
        case ZSOLVE_ENOMEM: return "out of memory";
        case ZSOLVE_ECUDA: return "CUDA error";
        case ZSOLVE_ESTATE: return "call out of order (not assembled or not factored)";
        case ZSOLVE_ENONFINITE: return "non-finite input";
        case ZSOLVE_ESINGULAR: return "matrix is singular in double precision";
        case ZSOLVE_ETIMEOUT: return "device-side wait gave up";
        default: return "unknown status";
    }
}

const char *zsolve_last_error(const zsolve_ctx *ctx) { return ctx ? ctx->err : "no context"; }

void zsolve_destroy(zsolve_ctx *ctx) {
    if (!ctx) return;
    free_all(ctx);
    delete ctx;
}

}  // extern "C"
