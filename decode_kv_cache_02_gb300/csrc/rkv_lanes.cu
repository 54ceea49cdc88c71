// rkv_lanes.cu -- two disjoint SM partitions of one GPU, each with a stream
// of its own (driver green contexts): the tensor-bound Gram of one group of
// problems runs on one partition while the HBM-bound importance and
// compaction of other groups run on the other, so the step's two bottlenecks
// (tensor pipe, HBM) are busy at the same time instead of one after the other.
//
// Events are created in the context of the stream they are recorded on (a
// green context's stream takes only that context's events); waits may cross
// contexts.  Everything is created once per (device, split) and kept for the
// life of the process.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <map>
#include <mutex>
#include <utility>

#include "rkv_internal.h"

namespace rkv {
namespace {

struct Driver {
    PFN_cuDeviceGet_v2000 device_get = nullptr;
    PFN_cuDeviceGetDevResource_v12040 get_resource = nullptr;
    PFN_cuDevSmResourceSplitByCount_v12040 split = nullptr;
    PFN_cuDevResourceGenerateDesc_v12040 gen_desc = nullptr;
    PFN_cuGreenCtxCreate_v12040 create = nullptr;
    PFN_cuCtxFromGreenCtx_v12040 to_ctx = nullptr;
    PFN_cuGreenCtxStreamCreate_v12050 stream_create = nullptr;
    PFN_cuCtxPushCurrent_v4000 push = nullptr;
    PFN_cuCtxPopCurrent_v4000 pop = nullptr;
    bool ok = false;
};

template <typename T>
bool entry(const char* name, int version, T* out) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &p, version, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !p)
        return false;
    *out = reinterpret_cast<T>(p);
    return true;
}

const Driver& driver() {
    static Driver d;
    static std::once_flag once;
    std::call_once(once, [] {
        d.ok = entry("cuDeviceGet", 2000, &d.device_get) &&
               entry("cuDeviceGetDevResource", 12040, &d.get_resource) &&
               entry("cuDevSmResourceSplitByCount", 12040, &d.split) &&
               entry("cuDevResourceGenerateDesc", 12040, &d.gen_desc) &&
               entry("cuGreenCtxCreate", 12040, &d.create) &&
               entry("cuCtxFromGreenCtx", 12040, &d.to_ctx) &&
               entry("cuGreenCtxStreamCreate", 12050, &d.stream_create) &&
               entry("cuCtxPushCurrent", 4000, &d.push) &&
               entry("cuCtxPopCurrent", 4000, &d.pop);
    });
    return d;
}

// SMs per group of the split (the partitions' granularity)
constexpr unsigned kGroupSms = 4;
constexpr int kMaxGroups = 64;

bool make_lane(const Driver& d, CUdevice dev, CUdevResource* res, unsigned n, Lane* lane) {
    CUdevResourceDesc desc = nullptr;
    CUgreenCtx g = nullptr;
    CUcontext ctx = nullptr;
    CUstream st = nullptr;
    if (d.gen_desc(&desc, res, n) != CUDA_SUCCESS) return false;
    if (d.create(&g, desc, dev, CU_GREEN_CTX_DEFAULT_STREAM) != CUDA_SUCCESS) return false;
    if (d.to_ctx(&ctx, g) != CUDA_SUCCESS) return false;
    if (d.stream_create(&st, g, CU_STREAM_NON_BLOCKING, 0) != CUDA_SUCCESS) return false;
    lane->ctx = ctx;
    lane->stream = reinterpret_cast<cudaStream_t>(st);
    lane->sms = 0;
    for (unsigned i = 0; i < n; ++i) lane->sms += (int)res[i].sm.smCount;
    return lane->sms > 0;
}

// Splits the current device: `tensor_sms` (rounded down to whole groups) for
// the tensor lane, the rest (with any SMs the split leaves over) for the
// other.  Returns false when the driver or the device offers no split.
bool make_lanes(int tensor_sms, Lanes* out) {
    const Driver& d = driver();
    if (!d.ok) return false;
    int ord = 0;
    if (cudaGetDevice(&ord) != cudaSuccess) return false;
    cudaFree(nullptr);  // the primary context exists before green contexts refer to it
    CUdevice dev;
    if (d.device_get(&dev, ord) != CUDA_SUCCESS) return false;
    CUdevResource all{};
    if (d.get_resource(dev, &all, CU_DEV_RESOURCE_TYPE_SM) != CUDA_SUCCESS) return false;
    CUdevResource groups[kMaxGroups];
    CUdevResource rest{};
    unsigned n = all.sm.smCount / kGroupSms;
    if (n > (unsigned)kMaxGroups) n = kMaxGroups;
    if (d.split(groups, &n, &all, &rest, CU_DEV_SM_RESOURCE_SPLIT_IGNORE_SM_COSCHEDULING,
                kGroupSms) != CUDA_SUCCESS)
        return false;
    if (n < 2 || groups[0].sm.smCount == 0) return false;
    // the split may round the group size up
    const unsigned want = (unsigned)tensor_sms / groups[0].sm.smCount;
    if (want < 1 || want >= n) return false;
    // the tensor lane: the first `want` groups; the other: the remaining
    // groups and the split's remainder
    out->tensor.id = 1;
    out->hbm.id = 2;
    if (!make_lane(d, dev, groups, want, &out->tensor)) return false;
    CUdevResource other[kMaxGroups + 1];
    unsigned m = 0;
    for (unsigned i = want; i < n; ++i) other[m++] = groups[i];
    if (rest.sm.smCount > 0) other[m++] = rest;
    return make_lane(d, dev, other, m, &out->hbm);
}

}  // namespace

const Lanes* lanes_for_current_device(int tensor_sms) {
    static std::mutex mu;
    static std::map<std::pair<int, int>, Lanes*> cache;
    int ord = 0;
    if (cudaGetDevice(&ord) != cudaSuccess) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    const auto key = std::make_pair(ord, tensor_sms);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    Lanes* l = new Lanes();
    if (!make_lanes(tensor_sms, l)) {
        delete l;
        l = nullptr;
    }
    cache[key] = l;  // a failed split is not retried
    return l;
}

LaneScope::LaneScope(const Lane* lane) : pushed_(false) {
    if (!lane) return;
    const Driver& d = driver();
    pushed_ = d.push(static_cast<CUcontext>(lane->ctx)) == CUDA_SUCCESS;
}

LaneScope::~LaneScope() {
    if (!pushed_) return;
    CUcontext c;
    driver().pop(&c);
}

}  // namespace rkv
