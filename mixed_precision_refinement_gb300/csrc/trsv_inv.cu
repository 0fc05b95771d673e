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
// Bound: HBM for the off-diagonal blocks (8 n^2 bytes per frequency per
// solve) plus the dependency chain's latency (n / 128 steps per direction).
#include "common.cuh"

namespace {

using zs::cf;

constexpr int TB = ZS_TB2;  // 128
// lane 0 waits until more than `need` blocks are complete; the warp barrier
// orders the other lanes' loads after its acquire
__device__ __forceinline__ long long warp_progress(const unsigned long long *p, unsigned epoch, long long need,
                                                   unsigned *status, int lane) {
    long long c = 0;
    if (lane == 0) c = zs::progress_wait(p, epoch, need, status);
    c = __shfl_sync(0xffffffffu, c, 0);
    __syncwarp();
    return c;
}

constexpr int kThreads = 512;  // 16 warps, 8 rows each

template <int R>
__global__ void __launch_bounds__(kThreads, 1)
k_trsv_inv(const float *__restrict__ z32, int64_t ld, int64_t plane, int64_t z32_stride, int64_t n,
           const float *__restrict__ dinv, int64_t dinv_stride, float2 *__restrict__ v, int64_t v_stride,
           const int *__restrict__ slots, int nslot, unsigned long long *__restrict__ prog, unsigned epoch,
           unsigned *ticket, unsigned *status) {
    __shared__ cf part[TB][R];
    __shared__ cf rv[TB][R];
    __shared__ unsigned s_task, s_stop;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nblk = (int)((n + TB - 1) / TB);
    const unsigned total = 2u * (unsigned)nblk * (unsigned)nslot;
    while (true) {
        __syncthreads();
        if (tid == 0) {
            s_task = atomicAdd(ticket, 1u);
            s_stop = zs::timed_out(status) ? 1u : 0u;
        }
        __syncthreads();
        const unsigned t = s_task;
        if (t >= total || s_stop) break;
        const int phase = (int)(t / ((unsigned)nblk * nslot));
        const unsigned rem = t - (unsigned)phase * nblk * nslot;
        const int si = (int)(rem % (unsigned)nslot);
        const int bq = (int)(rem / (unsigned)nslot);
        const int b = phase == 0 ? bq : nblk - 1 - bq;
        const int slot = slots[si];
        const float *re = z32 + (int64_t)slot * z32_stride;
        const float *im = re + plane;
        const float *ir = dinv + (int64_t)slot * dinv_stride + (int64_t)b * 4 * TB * TB + (int64_t)phase * 2 * TB * TB;
        const float *ii = ir + TB * TB;
        float2 *vs = v + (int64_t)slot * v_stride;
        unsigned long long *pf = prog + 2 * (int64_t)slot, *pb = pf + 1;
        const int64_t r0 = (int64_t)b * TB;
        const int rows = (int)zs::min64(TB, n - r0);
        // the inverse block is needed last: start pulling it into L2 now
        {
            const char *p0 = reinterpret_cast<const char *>(ir);
            for (int q = tid; q < 2 * TB * TB * 4 / 128; q += kThreads)
                asm volatile("prefetch.global.L2 [%0];" ::"l"(p0 + (int64_t)q * 128));
        }
        cf acc[8][R];
#pragma unroll
        for (int i = 0; i < 8; i++)
#pragma unroll
            for (int r = 0; r < R; r++) acc[i][r] = cf{0.f, 0.f};
        bool ok = true;
        if (phase == 1) ok = warp_progress(pf, epoch, b, status, lane) >= 0;  // own forward result
        const int nchunk = phase == 0 ? b : nblk - 1 - b;
        long long ready = 0;
        for (int q = 0; q < nchunk && ok;) {
            if (q >= ready) {
                ready = warp_progress(phase == 0 ? pf : pb, epoch, q, status, lane);
                if (ready < 0) {
                    ok = false;
                    break;
                }
            }
            const int qend = (int)(ready < nchunk ? ready : nchunk);
            for (; q < qend; q++) {
                const int c = phase == 0 ? q : nblk - 1 - q;
                // lane owns 4 consecutive columns: one 16-byte load per row and plane
                const int64_t col = (int64_t)c * TB + 4 * lane;
                if (col + 3 < n) {
                    cf y[4][R];
#pragma unroll
                    for (int e = 0; e < 4; e++)
#pragma unroll
                        for (int r = 0; r < R; r++) {
                            const float2 t2 = __ldcg(&vs[r * n + col + e]);
                            y[e][r] = cf{t2.x, t2.y};
                        }
#pragma unroll
                    for (int i = 0; i < 8; i++) {
                        const int li = warp * 8 + i;
                        const int64_t g = (r0 + (li < rows ? li : 0)) * ld + col;
                        const float4 ar4 = __ldg(reinterpret_cast<const float4 *>(re + g));
                        const float4 ai4 = __ldg(reinterpret_cast<const float4 *>(im + g));
                        const cf a[4] = {cf{ar4.x, ai4.x}, cf{ar4.y, ai4.y}, cf{ar4.z, ai4.z}, cf{ar4.w, ai4.w}};
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
        }
#pragma unroll
        for (int i = 0; i < 8; i++)
#pragma unroll
            for (int r = 0; r < R; r++) {
                float x = acc[i][r].re, y = acc[i][r].im;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    x += __shfl_xor_sync(0xffffffffu, x, o);
                    y += __shfl_xor_sync(0xffffffffu, y, o);
                }
                if (lane == 0) part[warp * 8 + i][r] = cf{x, y};
            }
        if (!__syncthreads_and(ok ? 1 : 0)) continue;  // a wait gave up: uniform skip
        // right-hand side of the block's own triangle
        for (int e = tid; e < TB * R; e += kThreads) {
            const int i = e / R, r = e - i * R;
            cf val = cf{0.f, 0.f};
            if (i < rows) {
                const float2 t2 = __ldcg(&vs[r * n + r0 + i]);
                val = cf{t2.x - part[i][r].re, t2.y - part[i][r].im};
            }
            rv[i][r] = val;
        }
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
                const float4 ar4 = __ldg(reinterpret_cast<const float4 *>(ir + li * TB + j0));
                const float4 ai4 = __ldg(reinterpret_cast<const float4 *>(ii + li * TB + j0));
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
#pragma unroll
        for (int i = 0; i < 8; i++)
#pragma unroll
            for (int r = 0; r < R; r++) {
                float x = acc2[i][r].re, y = acc2[i][r].im;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    x += __shfl_xor_sync(0xffffffffu, x, o);
                    y += __shfl_xor_sync(0xffffffffu, y, o);
                }
                const int li = warp * 8 + i;
                if (lane == 0 && li < rows) __stcg(&vs[r * n + r0 + li], make_float2(x, y));
            }
        __threadfence();
        __syncthreads();
        if (tid == 0) zs::progress_set(phase == 0 ? pf : pb, epoch, (unsigned)(phase == 0 ? b + 1 : bq + 1));
    }
}

template <int R>
cudaError_t launch_inv(const float *z32, int64_t ld, int64_t plane, int64_t z32_stride, int64_t n, const float *dinv,
                       int64_t dinv_stride, float2 *v, int64_t v_stride, const int *slots, int nslot,
                       unsigned long long *prog, unsigned epoch, unsigned *ticket, unsigned *status, int num_sms,
                       cudaStream_t st) {
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_trsv_inv<R>, kThreads, 0);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    const int64_t nblk = (n + TB - 1) / TB;
    int64_t grid = (int64_t)per_sm * num_sms;
    const int64_t tasks = 2 * nblk * nslot;
    if (grid > tasks) grid = tasks;
    e = cudaMemsetAsync(ticket, 0, sizeof(unsigned), st);
    if (e != cudaSuccess) return e;
    // A plain launch: a task waits only on tasks with smaller tickets, which
    // CTAs that are already running have claimed, so the solve progresses
    // with any number of resident CTAs -- also while another stream's kernels
    // hold part of the GPU.
    k_trsv_inv<R><<<(unsigned)grid, kThreads, 0, st>>>(z32, ld, plane, z32_stride, n, dinv, dinv_stride, v, v_stride,
                                                       slots, nslot, prog, epoch, ticket, status);
    return cudaGetLastError();
}

}  // namespace

cudaError_t zs_launch_trsv_inv(const float *z32, int64_t ld, int64_t plane, int64_t z32_stride, int64_t n,
                               const float *dinv, int64_t dinv_stride, float2 *v, int64_t v_stride, int nrhs,
                               const int *slots, int nslot, unsigned long long *prog, unsigned epoch, unsigned *ticket,
                               unsigned *status, int num_sms, cudaStream_t st) {
    switch (nrhs) {
        case 1:
            return launch_inv<1>(z32, ld, plane, z32_stride, n, dinv, dinv_stride, v, v_stride, slots, nslot, prog,
                                 epoch, ticket, status, num_sms, st);
        case 2:
            return launch_inv<2>(z32, ld, plane, z32_stride, n, dinv, dinv_stride, v, v_stride, slots, nslot, prog,
                                 epoch, ticket, status, num_sms, st);
        case 4:
            return launch_inv<4>(z32, ld, plane, z32_stride, n, dinv, dinv_stride, v, v_stride, slots, nslot, prog,
                                 epoch, ticket, status, num_sms, st);
        default:
            return cudaErrorInvalidValue;
    }
}
