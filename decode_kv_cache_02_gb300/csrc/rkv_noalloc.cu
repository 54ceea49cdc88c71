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
// The array's name is only a host-side stand-in in host code, so the device
// address is looked up with cudaGetSymbolAddress, once per device, on the
// first call made while that device is current, and cached.  The call never
// allocates or frees device memory.  Every call shares the one array: its
// device error word is cleared at the start of each call (the other scratch
// regions are fully written before they are read), and two calls that may run
// at the same time on the GPU (different streams, or different host threads)
// race on it.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/rkv.h"
#include "rkv_common.cuh"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[RKV_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {nullptr};
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device (looked up once).
cudaError_t scratch_for_current_device(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
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
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(scratch, 0, sizeof(rkv::DeviceStatus), s) != cudaSuccess)
        return RKV_ERR_CUDA;
    return rkv_compress(desc, K, V, Q_obs, n_cached, budget, n_obs, lambda, beta, tau, out_K,
                        out_V, out_idx, scratch, (size_t)RKV_NOALLOC_SCRATCH_BYTES, stream);
}
