// k_selftest.cu -- the failure path of the bounded waits, exercised for real.
//
// Every wait of the tensor-core kernels is an mbarrier try_wait loop bounded
// by a cycle limit; when it runs out the kernel records kDevErrTimeout in the
// caller's workspace and returns instead of hanging.  This kernel waits, with
// that same primitive, on an mbarrier nothing ever arrives on: no copy, MMA or
// TMEM is involved, so running out is harmless, and the host can check that
// the error word is set and the context stays usable.
#include "rkv_common.cuh"
#include "rkv_internal.h"
#include "tcgen05.cuh"

namespace rkv {
namespace {

__global__ void wait_timeout_kernel(DeviceStatus* st) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        tc::mbar_init(&bar, 1);
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x == 0 && !tc::mbar_wait(&bar, 0, &abort_flag))
        set_error(st, kDevErrTimeout, 0xfffu);
}

}  // namespace

cudaError_t launch_wait_timeout(DeviceStatus* st, cudaStream_t s) {
    wait_timeout_kernel<<<1, 32, 0, s>>>(st);
    return cudaGetLastError();
}

}  // namespace rkv
