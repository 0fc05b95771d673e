/*
 * zsolve -- mixed-precision dense complex-symmetric frequency sweeps on GB300.
 *
 * At each frequency the library solves Z(omega) x = b with
 *     Z(omega) = j*omega*L - j*Psi/omega + Zs(omega)*G,
 * L, Psi, G real, symmetric and independent of frequency
 * (malusrfworks.com, "Solving Dense Matrices Fast in the Browser", section
 * "Fewer frequency points: adaptive frequency sampling", the form of Z).
 * The method is mixed-precision iterative refinement (same page, section
 * "Double-precision answers from a GPU without double precision", steps 1-4):
 *   1. factorise Z in low precision without pivoting, LU in blocks of 32;
 *   2. solve with those factors for a first x;
 *   3. form r = b - Z x in double precision;
 *   4. solve for a correction d with the low-precision factors, x += d, and
 *      repeat 3-4 until ||d|| / ||x|| < tol;
 * and a frequency whose refinement does not converge is solved alone by a
 * double-precision LU with partial pivoting (same section, the paragraph
 * after the steps; section "Measure first" for partial pivoting as the
 * fallback).  All of it runs on one GPU.
 *
 * Conventions for every entry point:
 *  - Matrices are n x n, row-major, dense.  L, Psi, G are real float64.
 *    Complex vectors are interleaved (re, im) float64 ("c128"); a block of
 *    nrhs right-hand sides is nrhs rows of n c128 values.
 *  - Pointers to matrices and vectors are DEVICE pointers unless the name of
 *    the entry point ends in _host.  They are borrowed for the duration of
 *    the call; the library keeps no reference to them.
 *  - Work is enqueued on the context's stream (zsolve_set_stream; default
 *    the legacy default stream).  zsolve_assemble and zsolve_factor return
 *    without synchronising.  zsolve_refine, zsolve_sweep and the other
 *    solve calls synchronise the stream once per refinement step (to read
 *    the convergence test) and return with their outputs complete.
 *  - The context owns every workspace (about 24 n^2 bytes per concurrently
 *    factored frequency plus O(n * nrhs)); nothing is allocated after
 *    zsolve_create except the fallback workspace on its first use.
 *  - A context is not thread-safe; use one per host thread.
 *  - Every call returns ZSOLVE_OK (0) or a negative status; the message of
 *    the last failure is kept in the context (zsolve_last_error).  After
 *    ZSOLVE_ECUDA the CUDA context may be unusable.
 */
#ifndef ZSOLVE_H
#define ZSOLVE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* status codes */
#define ZSOLVE_OK 0
#define ZSOLVE_EINVAL (-1)     /* invalid argument (n <= 0, nrhs > nrhs_max, NULL, omega <= 0) */
#define ZSOLVE_ENOMEM (-2)     /* device or host allocation failed */
#define ZSOLVE_ECUDA (-3)      /* CUDA runtime error */
#define ZSOLVE_ESTATE (-4)     /* call out of order: not assembled / not factored */
#define ZSOLVE_ENONFINITE (-5) /* non-finite value in an input */
#define ZSOLVE_ESINGULAR (-6)  /* the double-precision fallback met an exactly zero pivot column */
#define ZSOLVE_ETIMEOUT (-7)   /* a bounded device-side wait gave up (dependency never satisfied) */

/* arithmetic of the trailing (Schur) update of the low-precision factorisation */
#define ZSOLVE_GEMM_AUTO 0   /* picked per context by measured convergence and speed (zsolve_get_gemm_choice) */
#define ZSOLVE_GEMM_TF32 1   /* one tf32 tensor-core product per term (tcgen05) */
#define ZSOLVE_GEMM_TF32X3 2 /* split hi/lo tf32, three products per term (tcgen05) */
#define ZSOLVE_GEMM_FFMA 3   /* FP32 fused multiply-add on the CUDA cores */

/* arithmetic of the residual r = b - Z x (step 3) */
#define ZSOLVE_RESID_F64 0 /* float64 multiply-adds (DFMA); default */
#define ZSOLVE_RESID_DF 1  /* double-float on the FP32 pipes, about 46 bits (the page's GPU residual);
                              checked against the float64 kernel when the context is created */
#define ZSOLVE_RESID_FX 2  /* float64-accurate on the integer pipes: Z and x turned exactly into
                              72-bit fixed point (three 24-bit limbs), products and sums exact in
                              64-bit integers, each lane's sum rounded once to float64 */
#define ZSOLVE_RESID_LPG 3 /* zsolve_sweep: r = b - (j w L x - j Psi x / w + Zs G x) in float64 from
                              the sweep's L, Psi, G, several frequencies per pass over them, without
                              the assembled float64 Z (zsolve_residual_lpg); calls on the single
                              system of zsolve_assemble keep the float64 GEMV (F64) */
#define ZSOLVE_RESID_OZ 4  /* zsolve_sweep: the same form, L x, Psi x, G x of all of a batch's
                              frequencies as one product on the bf16 tensor cores with error-free
                              splitting (8 digits of 7 bits per value, exact digit products and
                              sums, one rounding to float64 per output; zsolve_residual_oz);
                              evaluations of fewer than 4 (frequency, right-hand side) pairs, and
                              calls on the single system, take the float64 GEMV (F64) */

typedef struct zsolve_ctx zsolve_ctx; /* opaque */

typedef struct {
    double tol;         /* stop when every RHS has ||d||_2/||x||_2 < tol (default 1e-11) */
    int max_iter;       /* corrections after the first solve before declaring a stall (10) */
    int gemm;           /* ZSOLVE_GEMM_* (default AUTO) */
    int outer_block;    /* columns per outer block of the factorisation; 128 (only value) */
    int batch;          /* frequencies factored together by zsolve_sweep; 0 = automatic */
    int force_fallback; /* testing aid: treat every frequency as stalled (default 0) */
    int profile;        /* 1: time every stage with CUDA events (zsolve_get_profile); default 0 */
    int resid;          /* ZSOLVE_RESID_* (default F64) */
    int lanes;          /* 0 (default) or 2: a sweep batch of 2 or more frequencies runs as two
                           concurrent lanes (streams and host threads); 3: three lanes for a
                           batch of 3 or more; 1: one lane */
    int symmetric;      /* 1 (default): use that Z is complex symmetric (same page, section "Measure
                           first": exploiting the symmetry halves the factorisation's work
                           against LU).  The trailing update forms only the tiles on and below the
                           diagonal, and each step's U12 solve takes A12^T from A21, so the
                           factors are those of the unpivoted LU of the matrix the lower
                           triangle defines (U = D L^T in exact arithmetic).  The double-
                           precision residual still uses all of Z, so a Z that is not
                           symmetric is still solved (refinement or the fallback).  Tensor-
                           core modes only (ignored with ZSOLVE_GEMM_FFMA); 0: the full update */
    int wait_limit;     /* polls before a wait of the triangular solve for another task's block gives
                           up with ZSOLVE_ETIMEOUT (0, the default: 2^22, about a second); a small
                           value lets a test see a wait give up quickly (zsolve_selftest_wait) */
} zsolve_opts;

/* stages of the path, for zsolve_get_profile */
#define ZSOLVE_STAGE_ASSEMBLE 0 /* fused float64 assembly + float32 cast */
#define ZSOLVE_STAGE_DIAG 1     /* diagonal-block LU, 32-column panels */
#define ZSOLVE_STAGE_TRSM 2     /* L21 = A21 U11^-1 and U12 = L11^-1 A12 */
#define ZSOLVE_STAGE_SCHUR 3    /* trailing update A22 -= L21 U12 */
#define ZSOLVE_STAGE_TRSV 4     /* forward/back substitution with the float32 factors */
#define ZSOLVE_STAGE_RESIDUAL 5 /* r = b - Z x in float64 */
#define ZSOLVE_STAGE_UPDATE 6   /* rounding of b, x += d, correction norms */
#define ZSOLVE_STAGE_FALLBACK 7 /* float64 pivoted LU and its substitution */
#define ZSOLVE_STAGE_PACK 8     /* tensor-core operand packs of A21 and A12^T */
#define ZSOLVE_NSTAGE 9

typedef struct {
    int64_t launches[ZSOLVE_NSTAGE]; /* kernels launched per stage (always counted) */
    double ms[ZSOLVE_NSTAGE];        /* device time per stage (only with opts.profile = 1) */
} zsolve_profile;

typedef struct {
    int iters;         /* corrections applied after the first solve */
    int fallback;      /* 1 if x came from the double-precision pivoted LU */
    int status;        /* ZSOLVE_OK, or the error that ended this frequency */
    int pivot_flag;    /* 1 if the low-precision factorisation met a tiny or non-finite pivot */
    double relcorr;    /* final max over RHS of ||d||_2/||x||_2 (0 after a fallback) */
    float ms_assemble; /* device time of the stages (batched: the batch's time / batch size) */
    float ms_factor;
    float ms_refine;
    int gemm;          /* arithmetic of this frequency's factors: ZSOLVE_GEMM_TF32, _TF32X3 or _FFMA */
} zsolve_info;

/* The choice of ZSOLVE_GEMM_AUTO.  The first zsolve_sweep of a context
 * created with gemm = AUTO solves its first frequency alone once in each
 * arithmetic (assembly, factorisation and refinement, timed with CUDA events
 * on the context's stream) and keeps, among the arithmetics whose refinement
 * converged without the fallback, the fastest (TF32X3 if none converged).
 * Until then, and for contexts with a fixed arithmetic, `chosen` is the
 * arithmetic in use and the rest is zero.  Arrays are indexed by
 * ZSOLVE_GEMM_TF32 - 1, ZSOLVE_GEMM_TF32X3 - 1, ZSOLVE_GEMM_FFMA - 1.
 * Passage: section "Double-precision answers from a GPU without double
 * precision" -- how low the factorisation's precision may go is set by
 * whether the refinement still converges; the page factorises in float32. */
typedef struct {
    int done;        /* 1 once the probe has run */
    int chosen;      /* ZSOLVE_GEMM_TF32, _TF32X3 or _FFMA: the arithmetic in use */
    float ms[3];     /* probe: device time of assembly + factorisation + refinement */
    int iters[3];    /* probe: corrections made */
    int fallback[3]; /* probe: 1 if the refinement stalled (the float64 fallback solved it) */
} zsolve_gemm_probe;

/* Fill *opts with the defaults listed above. */
int zsolve_default_opts(zsolve_opts *opts);

/* Create a context for n x n systems with up to nrhs_max right-hand sides.
 * opts may be NULL (defaults).  Allocates the device workspaces.
 * Passage: section "Double-precision answers from a GPU without double
 * precision" (the factors, residual and correction the steps keep) and
 * section "Measure first" (the memory a dense complex system of size n takes). */
int zsolve_create(zsolve_ctx **ctx, int64_t n, int nrhs_max, const zsolve_opts *opts);

/* Enqueue subsequent work on `stream` (a cudaStream_t; NULL = default stream).
 * No passage: the page runs one queue of GPU work; this names it. */
int zsolve_set_stream(zsolve_ctx *ctx, void *stream);

/* Z(omega) = j*omega*L - j*Psi/omega + Zs*G, written in float64 (kept for the
 * residual) and rounded to complex float32 (to be factorised), in one pass
 * over L, Psi, G (device, n x n float64).  omega > 0; zs_re + j*zs_im is
 * Zs(omega), computed by the caller.
 * Passage: section "Fewer frequency points: adaptive frequency sampling", the
 * form of Z with L, Psi, G independent of frequency. */
int zsolve_assemble(zsolve_ctx *ctx, const double *L, const double *Psi, const double *G,
                    double omega, double zs_re, double zs_im);

/* Unpivoted LU of the complex float32 copy of the assembled Z, in place:
 * 32-column panels inside 128-column outer blocks, trailing update by the
 * opts.gemm arithmetic.  Records whether a pivot was tiny or non-finite.
 * Passage: section "Double-precision answers from a GPU without double
 * precision", step 1 (single-precision LU in blocks of 32, no pivoting). */
int zsolve_factor(zsolve_ctx *ctx);

/* Refine x for nrhs right-hand sides b (device c128, nrhs x n) against the
 * assembled and factored Z; x (device c128, nrhs x n) is output only.  A
 * stalled refinement or a flagged pivot switches this call to the float64
 * pivoted LU (info->fallback = 1).  info (host) may be NULL.
 * Passage: section "Double-precision answers from a GPU without double
 * precision", steps 2-4 and the paragraph after them (the stopping test and
 * the switch to a direct solve when the refinement does not converge). */
int zsolve_refine(zsolve_ctx *ctx, const void *b, void *x, int nrhs, zsolve_info *info);

/* The whole sweep: for each of nf frequencies omega[f] (host array) with
 * surface impedance zs[2f] + j*zs[2f+1] (host array), assemble, factor and
 * refine.  b (device c128, nrhs x n) is shared by all frequencies; x (device
 * c128, nf x nrhs x n) receives the solutions; info (host, nf entries) may be
 * NULL.  Frequencies are processed opts.batch at a time.  Unless opts.lanes
 * is 1, a batch of two or more frequencies is split into two lanes that run
 * concurrently on the context's stream and on a second stream of the
 * context, each driven by its own host thread (the second one created and
 * joined inside the call).  Each lane assembles, factors and refines its
 * half; the second lane's refinement starts once the first lane's first
 * solve has run, so that one lane's triangular solves run beside the other's
 * residuals.  The call returns when all of it is done and the context's
 * stream is ordered after it.  Returns the first error; a frequency that
 * needed the fallback is not an error. */
/* Passage: the page's introduction and section "Fewer frequency points" (a
 * sweep is the same solve at every frequency of a list), with the steps of
 * zsolve_assemble, zsolve_factor and zsolve_refine at each frequency. */
int zsolve_sweep(zsolve_ctx *ctx, const double *L, const double *Psi, const double *G,
                 const double *omega, const double *zs, int nf, const void *b, void *x,
                 int nrhs, zsolve_info *info);

/* zsolve_sweep with HOST pointers for L, Psi, G, b and x: copies the inputs
 * to context-owned device buffers, sweeps, and copies the solutions back.
 * L, Psi and G are copied in row bands on a copy stream of the context, and
 * the first assembly follows them band by band, so the copy overlaps it.
 * Pinned host memory gives asynchronous, full-speed copies. */
int zsolve_sweep_host(zsolve_ctx *ctx, const double *L, const double *Psi, const double *G,
                      const double *omega, const double *zs, int nf, const void *b, void *x,
                      int nrhs, zsolve_info *info);

/* ---- stage-level calls on the single system of zsolve_assemble/factor ---- */

/* r = b - Z x with the float64 Z (step 3).  b, x, r: device c128, nrhs x n. */
int zsolve_residual(zsolve_ctx *ctx, const void *b, const void *x, void *r, int nrhs);

/* r = b - Z x for the single system of zsolve_assemble (its omega and Zs),
 * computed from L, Psi, G (device, n x n float64, as passed to
 * zsolve_assemble) without the assembled Z: r = b - (j w L x - j Psi x / w +
 * Zs G x), three float64 products per entry (the residual mode
 * ZSOLVE_RESID_LPG of the sweeps).  b, x, r: device c128, nrhs x n.
 * Passage: step 3 (the residual in double precision) with the form of Z of
 * section "Fewer frequency points: adaptive frequency sampling". */
int zsolve_residual_lpg(zsolve_ctx *ctx, const double *L, const double *Psi, const double *G, const void *b,
                        const void *x, void *r, int nrhs);

/* r = b - Z x for the single system of zsolve_assemble (its omega and Zs),
 * from L, Psi, G (device, n x n float64, as passed to zsolve_assemble) by
 * the residual mode ZSOLVE_RESID_OZ: the products L x, Psi x, G x on the
 * bf16 tensor cores with error-free splitting (Ozaki et al., "Error-free
 * transformations of matrix multiplication by using fast routines of matrix
 * multiplication and its applications", 2012), then r = b - (j w L x -
 * j Psi x / w + Zs G x) in float64.  Error: that of the float64 combination,
 * plus at most 2^-54 of each row's largest |entry| times sum |x| (and of
 * x's largest |entry| times the row's sum |entry|).  A non-finite value in a
 * row of L, Psi, G or in x gives NaN residuals for it.  The first call
 * allocates about 48 n^2 bytes of digits; each call forms them from L, Psi,
 * G again.  b, x, r: device c128, nrhs x n.  Returns ZSOLVE_ETIMEOUT if a
 * bounded device-side wait gave up.  Passage: step 3 (the residual in double
 * precision) with the form of Z of section "Fewer frequency points: adaptive
 * frequency sampling". */
int zsolve_residual_oz(zsolve_ctx *ctx, const double *L, const double *Psi, const double *G, const void *b,
                       const void *x, void *r, int nrhs);

/* d = (L U)^-1 v with the low-precision factors (steps 2 and 4): v is
 * rounded to complex float32, solved in float32, and d returned as c128.
 * v, d: device c128, nrhs x n. */
int zsolve_lowprec_solve(zsolve_ctx *ctx, const void *v, void *d, int nrhs);

/* Check of the bounded device-side waits (failure detection without a GPU
 * fault): runs the low-precision solve of the factored single system with
 * its first task withheld, so that every other task waits for a block that no
 * task computes.  Each wait gives up after opts.wait_limit polls and raises
 * the device status bit; the call returns ZSOLVE_ETIMEOUT, the expected
 * result (ZSOLVE_OK would mean that a wait did not give up).  The status bit
 * is cleared on return, so the context stays usable.  The contents of the
 * context's solve buffer are left undefined. */
int zsolve_selftest_wait(zsolve_ctx *ctx, int nrhs);

/* x = Z^-1 b by the float64 LU with partial pivoting of the assembled Z (the
 * fallback on its own).  b, x: device c128, nrhs x n. */
int zsolve_fallback_solve(zsolve_ctx *ctx, const void *b, void *x, int nrhs);

/* The arithmetic of the factorisation in use and, for ZSOLVE_GEMM_AUTO, the
 * measurements it was picked on (zsolve_gemm_probe). */
int zsolve_get_gemm_choice(zsolve_ctx *ctx, zsolve_gemm_probe *out);

/* Residual arithmetic in use (ZSOLVE_RESID_*) in *mode.  A context created
 * with ZSOLVE_RESID_DF first compares the double-float residual with the
 * float64 one on a synthetic system (the page's start-up self-test, section
 * "The shader compiler was erasing the error"); if they disagree by more than
 * 1e-12 relative, the context uses ZSOLVE_RESID_F64. */
int zsolve_get_resid_mode(zsolve_ctx *ctx, int *mode);

/* Copy the float64 Z (device c128, n x n) of the single system to dst. */
int zsolve_get_z64(zsolve_ctx *ctx, void *dst);

/* Copy the complex float32 matrix of the single system -- Z after
 * zsolve_assemble, the packed L\U factors after zsolve_factor -- into the
 * device float planes re and im (n x n each, row-major). */
int zsolve_get_z32(zsolve_ctx *ctx, float *re, float *im);

/* Tiny or non-finite pivot seen by the last zsolve_factor (0 or 1) in *flag. */
int zsolve_pivot_flag(zsolve_ctx *ctx, int *flag);

/* Launch counts and (with opts.profile) per-stage device times accumulated
 * since zsolve_create or the last zsolve_reset_profile.  Synchronises the
 * context's stream to resolve pending timings. */
int zsolve_get_profile(zsolve_ctx *ctx, zsolve_profile *out);

/* Zero the counters of zsolve_get_profile. */
int zsolve_reset_profile(zsolve_ctx *ctx);

/* Allocation-free low-precision solve.  The page has no counterpart: this
 * entry point exists for callers that cannot allocate device memory where
 * they need a solve -- a memory-pool-managed application that forbids stray
 * cudaMalloc calls, a real-time loop that may not allocate (or trigger the
 * implicit synchronisation an allocation can cause), a plug-in whose host
 * framework owns all device memory.  It applies float32 factors the caller
 * already holds (for instance copied out with zsolve_get_z32) and allocates
 * nothing: no cudaMalloc, no cudaFree, no allocating library call.
 *
 *   z32        device: system s has its real plane at z32 + s*sys_stride and
 *              its imaginary plane at z32 + s*sys_stride + plane, each n rows
 *              of stride ld floats, holding the packed unit-lower L and upper
 *              U of the unpivoted LU (the layout zsolve_get_z32 writes with
 *              ld = n, plane = n*n)
 *   v          device, complex float32 interleaved (re, im): system s holds
 *              nrhs rows of n values at v + s*v_stride (complex elements);
 *              overwritten by (L U)^-1 v
 *   nsys       1 .. 64 systems solved together (more: ZSOLVE_EINVAL)
 *   stream     cudaStream_t, NULL = default stream
 *
 * Its scratch (progress words, work ticket, status word, system list) is a
 * statically sized __device__ array of about 1.3 KB inside the library,
 * held by every GPU that loads the library until the process exits.  The
 * first call on a device sets the array up (looks up its device address and
 * writes the system list) with that device current; make that first call
 * before any stream capture.  Every call shares the array and each call
 * clears what must start at zero, so calls that overlap on the GPU (two
 * streams, two host threads) race: serialise them.  Returns after the solve
 * has finished (it synchronises `stream`); ZSOLVE_ETIMEOUT if a bounded
 * device-side wait gave up. */
int zsolve_lowprec_solve_noalloc(const float *z32, int64_t ld, int64_t plane, int64_t sys_stride, int64_t n,
                                 int nsys, void *v, int64_t v_stride, int nrhs, void *stream);

/* ---------------------------------------------------------------------------
 * Adaptive frequency sampling (AFS): a reduced-order model of the sweep
 * (malusrfworks.com, "Solving Dense Matrices Fast in the Browser", section
 * "Fewer frequency points: adaptive frequency sampling", steps 1-4):
 *   1. full solves (zsolve_sweep on the context) at a few candidates; the
 *      real and imaginary parts of their solutions, made orthonormal, are
 *      the columns of a real basis V (n x q);
 *   2. the q x q system Z_r(omega) = j*omega*V^T L V - j*V^T Psi V/omega
 *      + Zs*V^T G V;
 *   3. at every candidate, y from Z_r y = V^T b and an estimate of the
 *      relative residual ||Z(omega) V y - b|| / ||b|| built from q-sized
 *      quantities only; the candidate (not yet fully solved) with the worst
 *      estimate gets the next full solve;
 *   4. the loop ends once every estimate is below opts.tol.
 * Readings of what the page leaves open: the first exact solves are at the
 * two ends of the candidate list; the residual is relative and a candidate's
 * estimate is the largest over its right-hand sides; the basis is built by
 * two passes of classical Gram-Schmidt, dropping a vector whose norm after
 * them is at most opts.drop times its norm before; the loop also ends when
 * opts.max_solves exact solves have been made or the basis is full
 * (info.converged = 0).  The output at every candidate, the exactly solved
 * ones included, is V y.
 * ------------------------------------------------------------------------- */
#define ZSOLVE_AFS_MAX_BASIS 96

typedef struct zsolve_afs zsolve_afs;

typedef struct {
    double tol;     /* stop when every estimated relative residual is below tol (default 1e-4) */
    int max_solves; /* exact solves at most, >= 1 (default 32) */
    int max_basis;  /* basis vectors at most, 1 .. ZSOLVE_AFS_MAX_BASIS (default 96) */
    double drop;    /* orthogonalisation drop threshold, 0 <= drop < 1 (default 1e-8) */
} zsolve_afs_opts;

typedef struct {
    int n_exact;      /* exact solves made */
    int q;            /* basis vectors */
    int converged;    /* 1 if every final estimate is below tol */
    int basis_full;   /* 1 if a solution vector was left out because the basis was full */
    int evals;        /* evaluations of the whole candidate list */
    int fallbacks;    /* exact solves that needed the double-precision fallback */
    double max_resid; /* largest final estimate */
    double eval_gflop; /* algorithmic work of the evaluations: per candidate and pass,
                          8/3 q^3 (complex LU, real flops) + 44 q^2 per right-hand side
                          (8 q^2 elimination and substitution, 36 q^2 the quadratic form) */
    float ms_exact, ms_basis, ms_eval, ms_expand; /* device time of each phase, summed */
} zsolve_afs_info;

/* Defaults listed in zsolve_afs_opts. */
int zsolve_afs_default_opts(zsolve_afs_opts *opts);

/* A handle for AFS sweeps of the system size of ctx (whose solver makes the
 * exact solves and whose stream carries all of the work).  It owns the basis
 * and its products (about 4 n max_basis float64 values), the reduced terms,
 * and per-candidate buffers grown on demand.  ctx must outlive it.  The exact
 * solves take at most two frequencies at a time, so a context created with
 * opts.batch = 2 holds all the factorisation memory AFS uses.  Like a
 * context, a handle is not thread-safe; its sweeps use the context's solver,
 * so two handles on one context must not run at the same time.
 * ZSOLVE_EINVAL for bad options, or if the reduced system of max_basis
 * unknowns and the context's nrhs_max right-hand sides does not fit in
 * 227 KB of shared memory ((q (q + nrhs) + 4 q) x 16 bytes). */
int zsolve_afs_create(zsolve_afs **afs, zsolve_ctx *ctx, const zsolve_afs_opts *opts);

/* AFS over the m candidates omega[m] (host, rad/s, > 0) with surface
 * impedances zs[2m] (host, interleaved re, im), for the right-hand sides b
 * (device c128, nrhs x n, the same at every candidate).
 *   x        device c128, m x nrhs x n: the reduced-order solution V y at
 *            every candidate (NULL: not formed)
 *   sampled  host, room for min(m, max_solves) ints: candidate indices solved
 *            exactly, in order (NULL allowed)
 *   resid    host, m doubles: the final residual estimates (NULL allowed)
 *   info     host (NULL allowed)
 * L, Psi, G are device pointers as for zsolve_sweep.  Returns after all
 * work is done.  ZSOLVE_EINVAL for bad arguments; an exact solve's failure
 * status (ZSOLVE_ESINGULAR, ...) is returned as is. */
int zsolve_afs_sweep(zsolve_afs *afs, const double *L, const double *Psi, const double *G, const double *omega,
                     const double *zs, int m, const void *b, void *x, int nrhs, int *sampled, double *resid,
                     zsolve_afs_info *info);

/* Kernel launches the handle has made (exact solves not included). */
int64_t zsolve_afs_launches(const zsolve_afs *afs);

/* Message of the handle's last failure ("" if none). */
const char *zsolve_afs_last_error(const zsolve_afs *afs);

/* Release the handle's buffers.  NULL is allowed. */
void zsolve_afs_destroy(zsolve_afs *afs);

/* Static string for a status code.  No passage: error reporting of the library. */
const char *zsolve_strerror(int status);

/* Message of the last failure in this context ("" if none). */
const char *zsolve_last_error(const zsolve_ctx *ctx);

/* Release every workspace.  NULL is allowed.  No passage: resource release. */
void zsolve_destroy(zsolve_ctx *ctx);

#ifdef __cplusplus
}
#endif

#endif /* ZSOLVE_H */
