// Forward and back substitution with the complex float32 factors, using
// explicit inverses of the 128 x 128 diagonal blocks (malusrfworks.com,
// "Solving Dense Matrices Fast in the Browser", section "Double-precision
// answers from a GPU without double precision", steps 2 and 4: solve with the
// single-precision factorisation).
//
// The inverses of the 128 x 128 diagonal blocks (X = L_bb^-1, unit lower, and
// X = U_bb^-1, upper) come from the factorisation (diag_block.cu).
//
// k_trsv_inv (per solve): the same ticketed, in-order task scheme as the
// sequential kernel, with 128-row blocks (half the dependency chain) and the
// block's own triangle applied as a dense 128 x 128 product with the inverse
// (all warps, no sequential steps) instead of a one-warp substitution.  Every
// task waits only on tasks with smaller tickets, claimed by running CTAs; each
// wait is bounded and raises the status bit instead of hanging.
//
// The chains of one launch are (slot, right-hand-side group) pairs: with few
// frequencies and several right-hand sides, groups of fewer right-hand sides
// give more chains side by side (each a short latency-bound critical path),
// at the price of reading the slot's factors once per group; the groups of a
// slot advance together, so most of those repeated reads hit the L2.
//
// Bound: HBM for the off-diagonal blocks (8 n^2 bytes per frequency per
// solve) plus the dependency chain's latency (n / 128 steps per direction).
#include "common.cuh"

namespace {

using zs::cf;

constexpr int TB = ZS_TB2;  // 128
// lane 0 waits until more than `need` blocks are complete; the warp barrier
// orders the other lanes' loads after its acquire
__device__ __forceinline__ long long warp_progress(const unsigned long long *p, unsigned epoch, long long need,
                                                   unsigned *status, int lane, unsigned limit) {
    long long c = 0;
    if (lane == 0) c = zs::progress_wait(p, epoch, need, status, limit);
    c = __shfl_sync(0xffffffffu, c, 0);
    __syncwarp();
    return c;
}

// Sum of each of NV values over the warp's 32 lanes, as a reduce-scatter:
// at every level a lane keeps half of its values and adds the partner's
// copy of that half (16 + 8 + ... shuffles instead of 5 NV).  Afterwards
// lane l holds the sums with indices ((l >> s) & (NV / K - 1)) * K + u,
// u < K, in v[0..K), K = max(NV / 32, 1), s = log2(32 K / NV) (lanes that
// differ in their low s bits hold the same sums).
template <int NV, int M = 16>
__device__ __forceinline__ void reduce_scatter(float (&v)[NV], int lane) {
    if constexpr (M >= 1) {
        if constexpr (NV >= 2) {
            constexpr int H = NV / 2;
            const bool hi = (lane & M) != 0;
            float w[H];
#pragma unroll
            for (int k = 0; k < H; k++) {
                const float send = hi ? v[k] : v[k + H];
                const float keep = hi ? v[k + H] : v[k];
                w[k] = keep + __shfl_xor_sync(0xffffffffu, send, M);
            }
            if constexpr (M > 1) {
                reduce_scatter<H, M / 2>(w, lane);
            }
#pragma unroll
            for (int k = 0; k < H; k++) v[k] = w[k];
        } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], M);
            if constexpr (M > 1) reduce_scatter<NV, M / 2>(v, lane);
        }
    }
}

// After reduce_scatter<16 R>: the number of sums a lane holds, and the index
// of its first one (values are laid out [row 0..7][rhs][re, im]).
template <int R>
struct Scatter {
    static constexpr int NV = 16 * R;
    static constexpr int K = NV >= 32 ? NV / 32 : 1;
    static constexpr int SHIFT = NV >= 32 ? 0 : (NV == 16 ? 1 : (NV == 8 ? 2 : 3));
    __device__ static int first(int lane) { return ((lane >> SHIFT) & (NV / K - 1)) * K; }
    // one lane of each group of equal holders writes
    __device__ static bool writer(int lane) { return (lane & ((1 << SHIFT) - 1)) == 0; }
};

constexpr int kThreads = 512;  // 16 warps, 8 rows each
constexpr size_t kSmemBytes = (size_t)2 * TB * TB * sizeof(float);  // the task's inverse block, re and im

// The critical step of a task is its last chunk (the block just before it in
// the chain) and then the product with its inverse block.  Everything that
// does not depend on that block's solution is started first: the inverse
// block is copied into shared memory at the start of the task (cp.async),
// the task's right-hand side is loaded as soon as it is final, and each
// chunk's factor rows are loaded into registers before the wait for the
// chunk's solution (with one right-hand side; more keep the loads after the
// wait to stay in registers).
template <int R>
__global__ void __launch_bounds__(kThreads, 1)
k_trsv_inv(const float *__restrict__ z32, int64_t ld, int64_t plane, int64_t z32_stride, int64_t n,
           const float *__restrict__ dinv, int64_t dinv_stride, float2 *__restrict__ v, int64_t v_stride,
           int ngroup, const int *__restrict__ slots, int nslot, unsigned long long *__restrict__ prog,
           unsigned epoch, unsigned *ticket, unsigned *status, unsigned wait_limit) {
    constexpr bool kPreload = R == 1;
    extern __shared__ __align__(16) float sinv[];  // [re, im][TB][TB]
    __shared__ cf part[TB][R];
    __shared__ cf rv[TB][R];
    __shared__ unsigned s_task, s_stop;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nblk = (int)((n + TB - 1) / TB);
    const unsigned nchain = (unsigned)nslot * (unsigned)ngroup;
    const unsigned total = 2u * (unsigned)nblk * nchain;
    const uint32_t sinv_addr = (uint32_t)__cvta_generic_to_shared(sinv);
    while (true) {
        __syncthreads();
        if (tid == 0) {
            s_task = atomicAdd(ticket, 1u);
            s_stop = zs::timed_out(status) ? 1u : 0u;
        }
        __syncthreads();
        const unsigned t = s_task;
        if (t >= total || s_stop) break;
        const int phase = (int)(t / ((unsigned)nblk * nchain));
        const unsigned rem = t - (unsigned)phase * nblk * nchain;
        const int ci = (int)(rem % nchain);  // chain: slot si, group g
        const int bq = (int)(rem / nchain);
        const int b = phase == 0 ? bq : nblk - 1 - bq;
        const int si = ci / ngroup, g = ci - si * ngroup;
        const int slot = slots[si];
        const float *re = z32 + (int64_t)slot * z32_stride;
        const float *im = re + plane;
        const float *ir = dinv + (int64_t)slot * dinv_stride + (int64_t)b * 4 * TB * TB + (int64_t)phase * 2 * TB * TB;
        float2 *vs = v + (int64_t)slot * v_stride + (int64_t)g * R * n;
        unsigned long long *pf = prog + 2 * ((int64_t)slot * ZS_TRSV_MAX_GROUPS + g), *pb = pf + 1;
        const int64_t r0 = (int64_t)b * TB;
        const int rows = (int)zs::min64(TB, n - r0);
        const int64_t wrow = (r0 + warp * 8) * ld;  // offset of the warp's first row
        // the inverse block (re and im planes are contiguous) into shared memory
        for (int q = tid; q < 2 * TB * TB / 4; q += kThreads)
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sinv_addr + 16u * q), "l"(ir + 4 * q)
                         : "memory");
        asm volatile("cp.async.commit_group;" ::: "memory");
        cf acc[8][R];
#pragma unroll
        for (int i = 0; i < 8; i++)
#pragma unroll
            for (int r = 0; r < R; r++) acc[i][r] = cf{0.f, 0.f};
        bool ok = true;
        if (phase == 1) ok = warp_progress(pf, epoch, b, status, lane, wait_limit) >= 0;  // own forward result
        // the block's right-hand side (final now: the input, resp. the forward result)
        cf vb = cf{0.f, 0.f};
        const int ei = tid / R, er = tid - ei * R;
        if (tid < TB * R && ei < rows && ok) {
            const float2 t2 = __ldcg(&vs[er * n + r0 + ei]);
            vb = cf{t2.x, t2.y};
        }
        const int nchunk = phase == 0 ? b : nblk - 1 - b;
        long long ready = 0;
        for (int q = 0; q < nchunk && ok; q++) {
            const int c = phase == 0 ? q : nblk - 1 - q;
            // lane owns 4 consecutive columns: one 16-byte load per row and plane
            const int64_t col = (int64_t)c * TB + 4 * lane;
            const bool full = col + 3 < n;
            float4 ar4[8], ai4[8];
            // the warp's 8 rows of the chunk, by pointer steps (rows past the
            // block's end read its first row; their sums are not stored)
            const float *pc = re + wrow + col;
            if (kPreload && full) {
                const float *pr = pc;
#pragma unroll
                for (int i = 0; i < 8; i++) {
                    const float *ps = warp * 8 + i < rows ? pr : re + r0 * ld + col;
                    ar4[i] = __ldg(reinterpret_cast<const float4 *>(ps));
                    ai4[i] = __ldg(reinterpret_cast<const float4 *>(ps + plane));
                    pr += ld;
                }
            }
            if (q >= ready) {
                ready = warp_progress(phase == 0 ? pf : pb, epoch, q, status, lane, wait_limit);
                if (ready < 0) {
                    ok = false;
                    break;
                }
            }
            if (full) {
                cf y[4][R];
#pragma unroll
                for (int e = 0; e < 4; e++)
#pragma unroll
                    for (int r = 0; r < R; r++) {
                        const float2 t2 = __ldcg(&vs[r * n + col + e]);
                        y[e][r] = cf{t2.x, t2.y};
                    }
                const float *pr = pc;
#pragma unroll
                for (int i = 0; i < 8; i++) {
                    if (!kPreload) {
                        const float *ps = warp * 8 + i < rows ? pr : re + r0 * ld + col;
                        ar4[i] = __ldg(reinterpret_cast<const float4 *>(ps));
                        ai4[i] = __ldg(reinterpret_cast<const float4 *>(ps + plane));
                        pr += ld;
                    }
                    const cf a[4] = {cf{ar4[i].x, ai4[i].x}, cf{ar4[i].y, ai4[i].y}, cf{ar4[i].z, ai4[i].z},
                                     cf{ar4[i].w, ai4[i].w}};
#pragma unroll
                    for (int e = 0; e < 4; e++)
#pragma unroll
                        for (int r = 0; r < R; r++) {
                            acc[i][r].re = fmaf(a[e].re, y[e][r].re, fmaf(-a[e].im, y[e][r].im, acc[i][r].re));
                            acc[i][r].im = fmaf(a[e].re, y[e][r].im, fmaf(a[e].im, y[e][r].re, acc[i][r].im));
                        }
                }
            } else {
                for (int e = 0; e < 4; e++) {
                    if (col + e >= n) break;
                    cf y[R];
#pragma unroll
                    for (int r = 0; r < R; r++) {
                        const float2 t2 = __ldcg(&vs[r * n + col + e]);
                        y[r] = cf{t2.x, t2.y};
                    }
#pragma unroll
                    for (int i = 0; i < 8; i++) {
                        const int li = warp * 8 + i;
                        const int64_t g = (r0 + (li < rows ? li : 0)) * ld + col + e;
                        const cf a = cf{__ldg(re + g), __ldg(im + g)};
#pragma unroll
                        for (int r = 0; r < R; r++) {
                            acc[i][r].re = fmaf(a.re, y[r].re, fmaf(-a.im, y[r].im, acc[i][r].re));
                            acc[i][r].im = fmaf(a.re, y[r].im, fmaf(a.im, y[r].re, acc[i][r].im));
                        }
                    }
                }
            }
        }
        {
            float s[16 * R];
#pragma unroll
            for (int i = 0; i < 8; i++)
#pragma unroll
                for (int r = 0; r < R; r++) {
                    s[(i * R + r) * 2] = acc[i][r].re;
                    s[(i * R + r) * 2 + 1] = acc[i][r].im;
                }
            reduce_scatter(s, lane);
            float *pw = reinterpret_cast<float *>(&part[warp * 8][0]);
            if (Scatter<R>::writer(lane)) {
                const int f = Scatter<R>::first(lane);
#pragma unroll
                for (int u = 0; u < Scatter<R>::K; u++) pw[f + u] = s[u];
            }
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
        if (!__syncthreads_and(ok ? 1 : 0)) continue;  // a wait gave up: uniform skip
        // right-hand side of the block's own triangle
        if (tid < TB * R) rv[ei][er] = ei < rows ? cf{vb.re - part[ei][er].re, vb.im - part[ei][er].im} : cf{0.f, 0.f};
        __syncthreads();
        // y = inverse block . rv: warp w rows 8w..8w+7, lanes over columns
        cf acc2[8][R];
#pragma unroll
        for (int i = 0; i < 8; i++)
#pragma unroll
            for (int r = 0; r < R; r++) acc2[i][r] = cf{0.f, 0.f};
        {
            const int j0 = 4 * lane;  // 4 consecutive columns of the inverse block
            cf y[4][R];
#pragma unroll
            for (int e = 0; e < 4; e++)
#pragma unroll
                for (int r = 0; r < R; r++) y[e][r] = rv[j0 + e][r];
#pragma unroll
            for (int i = 0; i < 8; i++) {
                const int li = warp * 8 + i;
                const float4 ar4 = *reinterpret_cast<const float4 *>(&sinv[li * TB + j0]);
                const float4 ai4 = *reinterpret_cast<const float4 *>(&sinv[TB * TB + li * TB + j0]);
                const cf a[4] = {cf{ar4.x, ai4.x}, cf{ar4.y, ai4.y}, cf{ar4.z, ai4.z}, cf{ar4.w, ai4.w}};
#pragma unroll
                for (int e = 0; e < 4; e++)
#pragma unroll
                    for (int r = 0; r < R; r++) {
                        acc2[i][r].re = fmaf(a[e].re, y[e][r].re, fmaf(-a[e].im, y[e][r].im, acc2[i][r].re));
                        acc2[i][r].im = fmaf(a[e].re, y[e][r].im, fmaf(a[e].im, y[e][r].re, acc2[i][r].im));
                    }
            }
        }
        {
            float s[16 * R];
#pragma unroll
            for (int i = 0; i < 8; i++)
#pragma unroll
                for (int r = 0; r < R; r++) {
                    s[(i * R + r) * 2] = acc2[i][r].re;
                    s[(i * R + r) * 2 + 1] = acc2[i][r].im;
                }
            reduce_scatter(s, lane);
            if (Scatter<R>::writer(lane)) {
                const int f = Scatter<R>::first(lane);
#pragma unroll
                for (int u = 0; u < Scatter<R>::K; u++) {
                    const int idx = f + u, c = idx & 1, r = (idx >> 1) % R, li = warp * 8 + (idx >> 1) / R;
                    if (li < rows) __stcg(reinterpret_cast<float *>(&vs[r * n + r0 + li]) + c, s[u]);
                }
            }
        }
        // the barrier orders every warp's stores before thread 0's release,
        // which (being cumulative) publishes them with the progress word
        __syncthreads();
        if (tid == 0) zs::progress_set(phase == 0 ? pf : pb, epoch, (unsigned)(phase == 0 ? b + 1 : bq + 1));
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
}

template <int R>
cudaError_t launch_inv(const float *z32, int64_t ld, int64_t plane, int64_t z32_stride, int64_t n, const float *dinv,
                       int64_t dinv_stride, float2 *v, int64_t v_stride, int ngroup, const int *slots, int nslot,
                       unsigned long long *prog, unsigned epoch, unsigned *ticket, unsigned *status, int num_sms,
                       cudaStream_t st, unsigned wait_limit, unsigned first_ticket) {
    // once per process and instance (thread-safe initialisation of a local static)
    static const cudaError_t attr =
        cudaFuncSetAttribute(k_trsv_inv<R>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (attr != cudaSuccess) return attr;
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_trsv_inv<R>, kThreads, kSmemBytes);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    const int64_t nblk = (n + TB - 1) / TB;
    int64_t grid = (int64_t)per_sm * num_sms;
    const int64_t tasks = 2 * nblk * nslot * ngroup;
    if (grid > tasks) grid = tasks;
    if (first_ticket == 0) {
        e = cudaMemsetAsync(ticket, 0, sizeof(unsigned), st);
    } else {
        // withheld tasks (testing aid): the value is staged by the copy
        // before the call returns, so a local is a valid source
        const unsigned t0 = first_ticket;
        e = cudaMemcpyAsync(ticket, &t0, sizeof(unsigned), cudaMemcpyHostToDevice, st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    }
    if (e != cudaSuccess) return e;
    // A plain launch: a task waits only on tasks with smaller tickets, which
    // CTAs that are already running have claimed, so the solve progresses
    // with any number of resident CTAs -- also while another stream's kernels
    // hold part of the GPU.
    k_trsv_inv<R><<<(unsigned)grid, kThreads, kSmemBytes, st>>>(z32, ld, plane, z32_stride, n, dinv, dinv_stride, v,
                                                                v_stride, ngroup, slots, nslot, prog, epoch, ticket,
                                                                status, wait_limit);
    return cudaGetLastError();
}

}  // namespace

cudaError_t zs_launch_trsv_inv(const float *z32, int64_t ld, int64_t plane, int64_t z32_stride, int64_t n,
                               const float *dinv, int64_t dinv_stride, float2 *v, int64_t v_stride, int nrhs,
                               int ngroup, const int *slots, int nslot, unsigned long long *prog, unsigned epoch,
                               unsigned *ticket, unsigned *status, int num_sms, cudaStream_t st, unsigned wait_limit,
                               unsigned first_ticket) {
    if (ngroup < 1 || ngroup > ZS_TRSV_MAX_GROUPS || nslot < 1) return cudaErrorInvalidValue;
    switch (nrhs) {
        case 1:
            return launch_inv<1>(z32, ld, plane, z32_stride, n, dinv, dinv_stride, v, v_stride, ngroup, slots, nslot,
                                 prog, epoch, ticket, status, num_sms, st, wait_limit, first_ticket);
        case 2:
            return launch_inv<2>(z32, ld, plane, z32_stride, n, dinv, dinv_stride, v, v_stride, ngroup, slots, nslot,
                                 prog, epoch, ticket, status, num_sms, st, wait_limit, first_ticket);
        case 4:
            return launch_inv<4>(z32, ld, plane, z32_stride, n, dinv, dinv_stride, v, v_stride, ngroup, slots, nslot,
                                 prog, epoch, ticket, status, num_sms, st, wait_limit, first_ticket);
        default:
            return cudaErrorInvalidValue;
    }
}
