// rkv_common.cuh -- device helpers shared by the librkv kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define RKV_DEV __device__ __forceinline__

namespace rkv {

// Device error word, stored at the start of the caller's workspace.
struct DeviceStatus {
    unsigned int code;  // 0 = ok, else one of the kDevErr* codes
    unsigned int info;  // kernel-specific detail (which wait / which index)
};

enum : unsigned int {
    kDevErrNone = 0,
    kDevErrTimeout = 1,  // a bounded mbarrier wait gave up
    kDevErrIndex = 2,    // an index was found outside its buffer
};

// Record an error; the first one wins.
RKV_DEV void set_error(DeviceStatus* st, unsigned int code, unsigned int info) {
    if (st == nullptr) return;
    if (atomicCAS(&st->code, 0u, code) == 0u) atomicExch(&st->info, info);
}

// Element loads as fp32 (bf16 -> fp32 is exact).
template <typename T> struct Elem;
template <> struct Elem<float> {
    static RKV_DEV float to_f(float x) { return x; }
};
template <> struct Elem<__nv_bfloat16> {
    static RKV_DEV float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
};

// 8 consecutive elements as fp32 from a 16-byte (bf16) or two 16-byte (fp32)
// aligned loads.
RKV_DEV void load8(const __nv_bfloat16* p, float* o) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        o[2 * t] = __uint_as_float(w[t] << 16);
        o[2 * t + 1] = __uint_as_float(w[t] & 0xffff0000u);
    }
}
RKV_DEV void load8(const float* p, float* o) {
    const float4 a = *reinterpret_cast<const float4*>(p);
    const float4 b = *reinterpret_cast<const float4*>(p + 4);
    o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
    o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
}

// Monotone map float -> uint32: a < b  <=>  key(a) < key(b).  -0 is mapped
// to the key of +0 so that the two compare equal, as they do as floats.
RKV_DEV uint32_t orderable(float z) {
    uint32_t b = __float_as_uint(z + 0.0f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

RKV_DEV float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
RKV_DEV float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

}  // namespace rkv
