// Forward and back substitution with the complex float32 factors
// (malusrfworks.com, "Solving Dense Matrices Fast in the Browser", section
// "Double-precision answers from a GPU without double precision", steps 2
// and 4: solve with the single-precision factorisation).
//
// v <- U^-1 L^-1 v for every (frequency, right-hand side) of a batch, in ONE
// cooperative launch.  The rows are cut into blocks of ZS_TB = 64.  Work
// items ("tasks") are the forward blocks 0..nb-1 followed by the backward
// blocks nb-1..0, interleaved over the frequencies of the batch; a CTA takes
// the next task from a ticket counter.  Task (b) accumulates the products of
// its 64 rows of L (or U) with the already-solved blocks, oldest first,
// then solves its own 64 x 64 triangle in shared memory.  Blocks of one
// (frequency, direction) complete in order, so each publishes a single
// progress word (epoch, blocks done): one acquire load tells a task how many
// solved blocks it may read.  Every task waits only on tasks with smaller
// tickets, which were claimed by CTAs already running, so the wait chain
// always ends; each wait is also bounded (ZS_SPIN_LIMIT) and raises a status
// bit instead of hanging.  The words carry the launch's epoch, so they are
// never cleared.
//
// Bound: HBM (each launch reads both triangles once: 8 n^2 bytes per
// frequency) plus the latency of the dependency chain.
#include <cooperative_groups.h>

#include "common.cuh"

namespace {

using zs::cf;

constexpr int TB = ZS_TB;
constexpr int kThreads = 256;  // 8 warps, 8 rows each
constexpr int kLdd = TB + 1;

// lane 0 of the warp waits until more than `need` blocks are complete; the
// warp barrier orders the other lanes' loads after its acquire
__device__ __forceinline__ long long warp_progress(const unsigned long long *p, unsigned epoch, long long need,
                                                   unsigned *status, int lane) {
    long long c = 0;
    if (lane == 0) c = zs::progress_wait(p, epoch, need, status);
    c = __shfl_sync(0xffffffffu, c, 0);
    __syncwarp();
    return c;
}

template <int R>
__global__ void __launch_bounds__(kThreads)
k_trsv_seq(const float *__restrict__ z32, int64_t ld, int64_t plane, int64_t z32_stride, int64_t n,
       float2 *__restrict__ v, int64_t v_stride, const int *__restrict__ slots, int nslot,
       unsigned long long *__restrict__ prog, unsigned epoch, unsigned *ticket, unsigned *status) {
    __shared__ float dre[TB * kLdd], dim_[TB * kLdd];  // diagonal block
    __shared__ cf part[TB][R];                         // accumulated off-diagonal products
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
        if (t >= total || s_stop) break;  // uniform across the CTA
        const int phase = (int)(t / ((unsigned)nblk * nslot));  // 0 forward, 1 backward
        const unsigned rem = t - (unsigned)phase * nblk * nslot;
        const int si = (int)(rem % (unsigned)nslot);
        const int bq = (int)(rem / (unsigned)nslot);
        const int b = phase == 0 ? bq : nblk - 1 - bq;
        const int slot = slots[si];
        const float *re = z32 + (int64_t)slot * z32_stride;
        const float *im = re + plane;
        float2 *vs = v + (int64_t)slot * v_stride;
        unsigned long long *pf = prog + 2 * (int64_t)slot, *pb = pf + 1;
        const int64_t r0 = (int64_t)b * TB;
        const int rows = (int)zs::min64(TB, n - r0);
        // diagonal block into shared memory (independent of other tasks)
        for (int idx = tid; idx < TB * TB; idx += kThreads) {
            int i = idx / TB, j = idx - i * TB;
            float a = 0.f, c = 0.f;
            if (i < rows && j < rows) {
                a = re[(r0 + i) * ld + r0 + j];
                c = im[(r0 + i) * ld + r0 + j];
            }
            dre[i * kLdd + j] = a;
            dim_[i * kLdd + j] = c;
        }
        // off-diagonal products: lanes stride columns, warp w owns rows 8w..8w+7
        cf acc[8][R];
#pragma unroll
        for (int i = 0; i < 8; i++)
#pragma unroll
            for (int r = 0; r < R; r++) acc[i][r] = cf{0.f, 0.f};
        // solved blocks, oldest first: forward c = 0..b-1, backward c = nblk-1..b+1
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
#pragma unroll 2
            for (; q < qend; q++) {
                const int c = phase == 0 ? q : nblk - 1 - q;
#pragma unroll
                for (int h = 0; h < 2; h++) {
                    const int64_t col = (int64_t)c * TB + lane + 32 * h;
                    if (col < n) {
                        cf y[R];
#pragma unroll
                        for (int r = 0; r < R; r++) {
                            float2 t2 = __ldcg(&vs[r * n + col]);
                            y[r] = cf{t2.x, t2.y};
                        }
#pragma unroll
                        for (int i = 0; i < 8; i++) {
                            const int li = warp * 8 + i;
                            if (li < rows) {
                                const int64_t g = (r0 + li) * ld + col;
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
        }
        // reduce across lanes
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
        // solve the diagonal triangle: warp 0, lane l owns rows l and l + 32
        if (warp == 0) {
            cf x[2][R];
#pragma unroll
            for (int q = 0; q < 2; q++) {
                const int li = lane + 32 * q;
#pragma unroll
                for (int r = 0; r < R; r++) {
                    if (li < rows) {
                        float2 t2 = __ldcg(&vs[r * n + r0 + li]);
                        x[q][r] = cf{t2.x - part[li][r].re, t2.y - part[li][r].im};
                    } else {
                        x[q][r] = cf{0.f, 0.f};
                    }
                }
            }
            if (phase == 0) {  // unit lower: columns in increasing order
#pragma unroll
                for (int q = 0; q < 2; q++) {
                    for (int kl = 0; kl < 32; kl++) {
                        const int k = 32 * q + kl;
                        if (k >= rows) break;
#pragma unroll
                        for (int r = 0; r < R; r++) {
                            cf yk;
                            yk.re = __shfl_sync(0xffffffffu, x[q][r].re, kl);
                            yk.im = __shfl_sync(0xffffffffu, x[q][r].im, kl);
#pragma unroll
                            for (int q2 = q; q2 < 2; q2++) {
                                const int li = lane + 32 * q2;
                                if (li > k && li < rows)
                                    x[q2][r] = zs::cfms(x[q2][r], cf{dre[li * kLdd + k], dim_[li * kLdd + k]}, yk);
                            }
                        }
                    }
                }
            } else {  // upper with diagonal: columns in decreasing order
#pragma unroll
                for (int q = 1; q >= 0; q--) {
                    for (int kl = 31; kl >= 0; kl--) {
                        const int k = 32 * q + kl;
                        if (k >= rows) continue;
                        const cf dinv = zs::crecip(cf{dre[k * kLdd + k], dim_[k * kLdd + k]});
#pragma unroll
                        for (int r = 0; r < R; r++) {
                            if (lane == kl) x[q][r] = zs::cmul(x[q][r], dinv);
                            cf zk;
                            zk.re = __shfl_sync(0xffffffffu, x[q][r].re, kl);
                            zk.im = __shfl_sync(0xffffffffu, x[q][r].im, kl);
#pragma unroll
                            for (int q2 = 0; q2 <= q; q2++) {
                                const int li = lane + 32 * q2;
                                if (li < k) x[q2][r] = zs::cfms(x[q2][r], cf{dre[li * kLdd + k], dim_[li * kLdd + k]}, zk);
                            }
                        }
                    }
                }
            }
#pragma unroll
            for (int q = 0; q < 2; q++) {
                const int li = lane + 32 * q;
                if (li < rows)
#pragma unroll
                    for (int r = 0; r < R; r++) __stcg(&vs[r * n + r0 + li], make_float2(x[q][r].re, x[q][r].im));
            }
            __threadfence();
            __syncwarp();
            if (lane == 0) zs::progress_set(phase == 0 ? pf : pb, epoch, (unsigned)(phase == 0 ? b + 1 : bq + 1));
        }
    }
}

template <int R>
cudaError_t launch_seq(const float *z32, int64_t ld, int64_t plane, int64_t z32_stride, int64_t n, float2 *v,
                     int64_t v_stride, const int *slots, int nslot, unsigned long long *prog,
                     unsigned epoch, unsigned *ticket, unsigned *status, int num_sms, cudaStream_t st) {
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_trsv_seq<R>, kThreads, 0);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    const int64_t nblk = (n + TB - 1) / TB;
    int64_t grid = (int64_t)per_sm * num_sms;
    const int64_t tasks = 2 * nblk * nslot;
    if (grid > tasks) grid = tasks;
    e = cudaMemsetAsync(ticket, 0, sizeof(unsigned), st);
    if (e != cudaSuccess) return e;
    void *args[] = {(void *)&z32, (void *)&ld, (void *)&plane, (void *)&z32_stride, (void *)&n,
                    (void *)&v, (void *)&v_stride, (void *)&slots, (void *)&nslot, (void *)&prog,
                    (void *)&epoch, (void *)&ticket, (void *)&status};
    e = cudaLaunchCooperativeKernel((const void *)k_trsv_seq<R>, dim3((unsigned)grid), dim3(kThreads), args, 0, st);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

cudaError_t zs_launch_trsv_seq(const float *z32, int64_t ld, int64_t plane, int64_t z32_stride, int64_t n,
                           float2 *v, int64_t v_stride, int nrhs, const int *slots, int nslot,
                           unsigned long long *prog, unsigned epoch, unsigned *ticket,
                           unsigned *status, int num_sms, cudaStream_t st) {
    switch (nrhs) {
        case 1:
            return launch_seq<1>(z32, ld, plane, z32_stride, n, v, v_stride, slots, nslot, prog,
                               epoch, ticket, status, num_sms, st);
        case 2:
            return launch_seq<2>(z32, ld, plane, z32_stride, n, v, v_stride, slots, nslot, prog,
                               epoch, ticket, status, num_sms, st);
        case 4:
            return launch_seq<4>(z32, ld, plane, z32_stride, n, v, v_stride, slots, nslot, prog,
                               epoch, ticket, status, num_sms, st);
        case 8:
            return launch_seq<8>(z32, ld, plane, z32_stride, n, v, v_stride, slots, nslot, prog,
                               epoch, ticket, status, num_sms, st);
        default:
            return cudaErrorInvalidValue;
    }
}
