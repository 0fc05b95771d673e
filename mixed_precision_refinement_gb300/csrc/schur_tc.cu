// tcgen05 trailing update: placeholder until the tensor-core kernel lands.
#include "common.cuh"

cudaError_t zs_launch_schur_tc(float *, int64_t, int64_t, int64_t, int64_t, int64_t, const float *, int64_t, int,
                               const int *, int, cudaStream_t) {
    return cudaErrorNotSupported;
}
