// rkv_noalloc.cu -- rkv_compress_noalloc: the compression step with its
// scratch memory inside the library instead of a caller workspace.
//
// Some callers cannot hand the library a workspace: code that runs inside an
// inference engine's plugin or custom-op hook, where the engine owns every
// byte of device memory and its contract forbids allocating (or growing a
// memory pool) while requests execute, or a process whose memory is fully
// reserved up front for the KV cache so that an extra allocation would fail or
// fragment the pool.  For them this entry point keeps its scratch in a
// file-scope __device__ array of fixed size, RKV_NOALLOC_SCRATCH_BYTES, which
// every GPU that loads the library holds until the process exits.
//
// The array's name is only a host-side stand-in in host code, so every call
// looks up the device address with cudaGetSymbolAddress on the current device
// (a host-side lookup once the module is loaded; not caching it means a
// context that was torn down and created again, which may place the module
// elsewhere, is never written through a stale pointer).  The call never
// allocates or frees device memory.  Every call shares the one array: its
// device error word is cleared by each call once the arguments have passed
// their checks (the other scratch regions are fully written before they are
// read), and two calls that may run at the same time on the GPU (different
// streams, or different host threads) race on it.  The error word is read
// back, and cleared, by rkv_noalloc_device_status.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/rkv.h"
#include "rkv_common.cuh"
#include "rkv_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[RKV_NOALLOC_SCRATCH_BYTES];

// Device address of the scratch array on the current device.
cudaError_t scratch_for_current_device(void** out) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    *out = p;
    return cudaSuccess;
}

}  // namespace

extern "C" int rkv_compress_noalloc(const rkv_desc* desc, const void* K, const void* V,
                                    const void* Q_obs, int n_cached, int budget, int n_obs,
                                    float lambda, int beta, float tau, void* out_K, void* out_V,
                                    int32_t* out_idx, void* stream) {
    if (!desc) return RKV_ERR_INVALID_ARG;
    const size_t need = rkv_workspace_size(desc, n_cached > 0 ? n_cached : 1, n_obs);
    if (need == 0) return RKV_ERR_INVALID_ARG;
    if (need > (size_t)RKV_NOALLOC_SCRATCH_BYTES) return RKV_ERR_TOO_LARGE;
    void* scratch = nullptr;
    if (scratch_for_current_device(&scratch) != cudaSuccess) return RKV_ERR_CUDA;
    return rkv::compress_call(desc, K, V, Q_obs, n_cached, budget, n_obs, lambda, beta, tau,
                              nullptr, out_K, out_V, out_idx, scratch,
                              (size_t)RKV_NOALLOC_SCRATCH_BYTES, stream, true,
                              false);  // creating partitions may allocate
}

extern "C" int rkv_noalloc_device_status(void* stream) {
    void* scratch = nullptr;
    if (scratch_for_current_device(&scratch) != cudaSuccess) return RKV_ERR_CUDA;
    return rkv_get_device_status(scratch, stream);
}

extern "C" int rkv_noalloc_selftest_wait_timeout(void* stream) {
    void* scratch = nullptr;
    if (scratch_for_current_device(&scratch) != cudaSuccess) return RKV_ERR_CUDA;
    return rkv_selftest_wait_timeout(scratch, stream);
}
