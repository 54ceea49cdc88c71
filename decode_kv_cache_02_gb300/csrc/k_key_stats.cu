// k_key_stats.cu -- per-key norms and the plain similarity sums.
//
// R-KV review (yoonschallenge.tistory.com/1236), question 2, cause 3: "key
// vector normalisation" precedes the all-pairs cosine similarity.  Redundancy
// (summary-table row "redundancy") needs, for every key i,
//     sum_i = sum_{j != i} S_ij,   S_ij = khat_i . khat_j,  khat = k / max(|k|, eps).
// The unthresholded part of that sum is linear in the keys:
//     sum_i = khat_i . s - khat_i . khat_i,   s = sum_j khat_j,
// so it costs O(N d) per problem, not O(N^2 d).  The Gram kernels then only
// handle the thresholded part (pairs with S_ij > tau).
//
// One CTA per problem, 8 warps; each warp owns whole rows (d/32 values per
// lane, coalesced 128/256-byte row reads).  Pass 1 writes inv_norm and builds
// s in fp32 (per-warp partials, then a fixed-order sum over warps); pass 2
// re-reads the rows (from L2) and writes sum_i.
#include "rkv_common.cuh"
#include "rkv_internal.h"
#include "../../include/rkv.h"

namespace rkv {
namespace {

constexpr int kWarps = 8;

template <typename T, int D>
__global__ void __launch_bounds__(kWarps * 32)
key_stats_kernel(const T* __restrict__ K, int n_cap, int N, float* __restrict__ inv_norm,
                 float* __restrict__ sum_s, int64_t ld) {
    constexpr int VPL = D / 32;  // values per lane
    __shared__ float s_part[kWarps][D];
    __shared__ float s_vec[D];
    const int64_t p = blockIdx.x;
    const T* Kp = K + (size_t)p * n_cap * D;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    float acc[VPL];
#pragma unroll
    for (int t = 0; t < VPL; ++t) acc[t] = 0.f;
    for (int i = warp; i < N; i += kWarps) {
        float v[VPL];
#pragma unroll
        for (int t = 0; t < VPL; ++t) v[t] = Elem<T>::to_f(Kp[(size_t)i * D + lane * VPL + t]);
        float n2 = 0.f;
#pragma unroll
        for (int t = 0; t < VPL; ++t) n2 = fmaf(v[t], v[t], n2);
        n2 = warp_sum(n2);
        const float inv = 1.0f / fmaxf(sqrtf(n2), 1e-12f);
        if (lane == 0) inv_norm[p * ld + i] = inv;
#pragma unroll
        for (int t = 0; t < VPL; ++t) acc[t] = fmaf(v[t], inv, acc[t]);
    }
#pragma unroll
    for (int t = 0; t < VPL; ++t) s_part[warp][lane * VPL + t] = acc[t];
    __syncthreads();
    for (int c = threadIdx.x; c < D; c += blockDim.x) {
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) s += s_part[w][c];
        s_vec[c] = s;
    }
    __syncthreads();
    float sv[VPL];
#pragma unroll
    for (int t = 0; t < VPL; ++t) sv[t] = s_vec[lane * VPL + t];
    for (int i = warp; i < N; i += kWarps) {
        float v[VPL];
#pragma unroll
        for (int t = 0; t < VPL; ++t) v[t] = Elem<T>::to_f(Kp[(size_t)i * D + lane * VPL + t]);
        float n2 = 0.f, ds = 0.f;
#pragma unroll
        for (int t = 0; t < VPL; ++t) {
            n2 = fmaf(v[t], v[t], n2);
            ds = fmaf(v[t], sv[t], ds);
        }
        n2 = warp_sum(n2);
        ds = warp_sum(ds);
        const float inv = 1.0f / fmaxf(sqrtf(n2), 1e-12f);
        if (lane == 0) sum_s[p * ld + i] = ds * inv - (n2 * inv) * inv;
    }
}

template <typename T, int D>
cudaError_t launch_t(const ScoreArgs& a, cudaStream_t s) {
    key_stats_kernel<T, D><<<(unsigned)a.P, kWarps * 32, 0, s>>>(
        static_cast<const T*>(a.K), a.n_cap, a.N, a.inv_norm, a.sum_s, a.ld_ws);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_key_stats(const ScoreArgs& a, cudaStream_t s) {
    if (a.P == 0) return cudaSuccess;
    if (a.dtype == RKV_DTYPE_BF16)
        return a.d == 128 ? launch_t<__nv_bfloat16, 128>(a, s) : launch_t<__nv_bfloat16, 64>(a, s);
    return a.d == 128 ? launch_t<float, 128>(a, s) : launch_t<float, 64>(a, s);
}

}  // namespace rkv
