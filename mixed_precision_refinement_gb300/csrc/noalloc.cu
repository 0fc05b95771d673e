// Allocation-free variant of the low-precision triangular solve.
//
// Some callers cannot allocate device memory at the point where they need a
// solve: code inside a memory-pool-managed application that forbids stray
// cudaMalloc calls, real-time loops where an allocation (and the implicit
// device synchronisation it can cause) is not allowed, or a plug-in running
// under a host framework that owns all device memory.  For them this entry
// point applies already-computed float32 factors using only the buffers the
// caller passes (factors and right-hand sides) plus a small scratch area that
// lives in this file as a statically sized __device__ array.
//
// The scratch holds what the batched solve needs besides its inputs and
// outputs: the in-order progress words (two per system), the work ticket,
// the timeout status word and the list of system indices.  Every GPU that
// loads the library holds this array (about 1.3 KB) until the process exits.
// All calls share it, so calls that overlap on the GPU (e.g. on two streams)
// race; serialise them.  The array keeps the last call's contents, so each
// call clears the parts that must start at zero.
#include <stdio.h>

#include <mutex>

#include "../../include/zsolve.h"
#include "common.cuh"

#define ZS_NOALLOC_MAX_SYS 64

namespace {

struct NoallocScratch {
    unsigned long long prog[2 * ZS_NOALLOC_MAX_SYS];  // progress words, 2 per system
    unsigned ticket;
    unsigned status;
    int slots[ZS_NOALLOC_MAX_SYS];
};

// The scratch itself.  In host code this name is only a stand-in for the
// device array: its address must be obtained with cudaGetSymbolAddress.
static __device__ __align__(256) NoallocScratch zs_noalloc_scratch;

constexpr int kMaxDevices = 64;
NoallocScratch *g_scratch[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};
std::mutex g_mu;

// Once per device, with that device current: the device address of the
// scratch array and the constant system-index list.
int setup(int dev, NoallocScratch **out, int *sms) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, zs_noalloc_scratch) != cudaSuccess) return ZSOLVE_ECUDA;
        int idx[ZS_NOALLOC_MAX_SYS];
        for (int i = 0; i < ZS_NOALLOC_MAX_SYS; i++) idx[i] = i;
        NoallocScratch *sp = static_cast<NoallocScratch *>(p);
        if (cudaMemcpy(sp->slots, idx, sizeof(idx), cudaMemcpyHostToDevice) != cudaSuccess) return ZSOLVE_ECUDA;
        int n_sms = 0;
        if (cudaDeviceGetAttribute(&n_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return ZSOLVE_ECUDA;
        g_sms[dev] = n_sms;
        g_scratch[dev] = sp;
    }
    *out = g_scratch[dev];
    *sms = g_sms[dev];
    return ZSOLVE_OK;
}

}  // namespace

extern "C" int zsolve_lowprec_solve_noalloc(const float *z32, int64_t ld, int64_t plane, int64_t sys_stride,
                                            int64_t n, int nsys, void *v, int64_t v_stride, int nrhs, void *stream) {
    if (!z32 || !v || n <= 0 || ld < n || plane < n * ld || nsys < 1 || nrhs < 1) return ZSOLVE_EINVAL;
    if (nsys > ZS_NOALLOC_MAX_SYS) return ZSOLVE_EINVAL;  // more systems than the static scratch holds
    if (nsys > 1 && sys_stride < 2 * plane) return ZSOLVE_EINVAL;
    if (v_stride < (int64_t)nrhs * n && nsys > 1) return ZSOLVE_EINVAL;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ZSOLVE_ECUDA;
    NoallocScratch *sp = nullptr;
    int sms = 0;
    int st = setup(dev, &sp, &sms);
    if (st != ZSOLVE_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    // progress words and status must start at zero (the ticket is cleared per launch)
    if (cudaMemsetAsync(sp, 0, offsetof(NoallocScratch, slots), s) != cudaSuccess) return ZSOLVE_ECUDA;
    float2 *vv = static_cast<float2 *>(v);
    unsigned epoch = 0;
    for (int r0 = 0; r0 < nrhs;) {
        const int left = nrhs - r0;
        const int R = left >= 8 ? 8 : left >= 4 ? 4 : left >= 2 ? 2 : 1;
        epoch++;
        if (zs_launch_trsv_seq(z32, ld, plane, sys_stride, n, vv + (int64_t)r0 * n, v_stride, R, sp->slots, nsys,
                           sp->prog, epoch, &sp->ticket, &sp->status, sms, s) != cudaSuccess)
            return ZSOLVE_ECUDA;
        r0 += R;
    }
    unsigned h_status = 0;
    if (cudaMemcpyAsync(&h_status, &sp->status, sizeof(unsigned), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return ZSOLVE_ECUDA;
    return (h_status & ZS_DEV_TIMEOUT) ? ZSOLVE_ETIMEOUT : ZSOLVE_OK;
}
