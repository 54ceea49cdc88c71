// k_select.cu -- per-problem top-k of the combined score, ascending indices.
//
// R-KV review (yoonschallenge.tistory.com/1236), opening notes ("keep the
// newest 8, score the rest, select only the top tokens that fit the
// budget") and question 2, cause 3 ("top-k token selection").  Ties in Z go to
// the larger (more recent) index; the output is the kept candidates in
// ascending order followed by the n_obs observation tokens.
//
// One CTA per problem.  Candidate scores are mapped to order-preserving
// 32-bit keys and kept in shared memory.  An MSB-first radix select (four
// 8-bit digits, shared-memory histograms, a warp-parallel bin search) finds the
// k-th largest key u_k exactly; every key above u_k is kept, and of the keys
// equal to u_k the ones with the largest indices fill the rest.  Two block
// scans in index order then place each kept index at its output position, so
// the result is deterministic and needs no sort.
#include "rkv_common.cuh"
#include "rkv_internal.h"
#include "../../include/rkv.h"

namespace rkv {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;

// Exclusive scan of one int per thread over the block; returns the thread's
// prefix and writes the block total to *total.
__device__ int block_exclusive_scan(int v, int* s_warp, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = lane < kWarps ? s_warp[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < kWarps) s_warp[lane] = w;  // inclusive warp prefix
    }
    __syncthreads();
    const int base = warp > 0 ? s_warp[warp - 1] : 0;
    *total = s_warp[kWarps - 1];
    __syncthreads();
    return base + x - v;
}

__global__ void __launch_bounds__(kThreads)
select_kernel(const float* __restrict__ Z, int64_t ldz, int N, int n_obs, int budget,
              int32_t* __restrict__ idx) {
    extern __shared__ uint32_t s_key[];  // [C]
    __shared__ uint32_t s_hist[256];
    __shared__ int s_warp[kWarps];
    __shared__ uint32_t s_prefix;
    __shared__ int s_krem;
    const int64_t p = blockIdx.x;
    const int C = N - n_obs, k = budget - n_obs;
    const float* zp = Z + p * ldz;
    int32_t* out = idx + p * (int64_t)budget;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

    for (int r = threadIdx.x; r < n_obs; r += kThreads) out[k + r] = C + r;
    if (k <= 0) return;

    for (int i = threadIdx.x; i < C; i += kThreads) s_key[i] = orderable(zp[i]);
    if (threadIdx.x == 0) {
        s_prefix = 0;
        s_krem = k;
    }
    // radix select of the k-th largest key
    uint32_t mask = 0;
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int b = threadIdx.x; b < 256; b += kThreads) s_hist[b] = 0;
        __syncthreads();
        const uint32_t prefix = s_prefix;
        for (int i = threadIdx.x; i < C; i += kThreads) {
            const uint32_t u = s_key[i];
            if ((u & mask) == prefix) atomicAdd(&s_hist[(u >> shift) & 255u], 1u);
        }
        __syncthreads();
        if (warp == 0) {
            // lane L owns bins 8L .. 8L+7; count of all bins above lane L's
            uint32_t h[8], tot = 0;
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                h[t] = s_hist[lane * 8 + t];
                tot += h[t];
            }
            uint32_t incl = tot;  // inclusive suffix sum over lanes >= lane
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_down_sync(0xffffffffu, incl, o);
                if (lane + o < 32) incl += y;
            }
            uint32_t above = incl - tot;  // keys in bins of higher lanes
            const uint32_t krem = (uint32_t)s_krem;
            if (above < krem && krem <= incl) {
#pragma unroll
                for (int t = 7; t >= 0; --t) {
                    if (above + h[t] >= krem) {
                        s_prefix = prefix | ((uint32_t)(lane * 8 + t) << shift);
                        s_krem = (int)(krem - above);
                        break;
                    }
                    above += h[t];
                }
            }
        }
        mask |= 255u << shift;
        __syncthreads();
    }
    const uint32_t uk = s_prefix;
    const int need_eq = s_krem;  // keys equal to uk that are kept (>= 1)

    // contiguous items per thread, in index order
    const int ipt = (C + kThreads - 1) / kThreads;
    const int lo = min(C, (int)threadIdx.x * ipt), hi = min(C, lo + ipt);
    int n_eq = 0;
    for (int i = lo; i < hi; ++i) n_eq += (s_key[i] == uk);
    int eq_total;
    int eq_before = block_exclusive_scan(n_eq, s_warp, &eq_total);
    const int eq_cut = eq_total - need_eq;  // ties with rank >= eq_cut are kept
    int n_keep = 0;
    {
        int e = eq_before;
        for (int i = lo; i < hi; ++i) {
            const uint32_t u = s_key[i];
            if (u > uk) ++n_keep;
            else if (u == uk) { n_keep += (e >= eq_cut); ++e; }
        }
    }
    int keep_total;
    int pos = block_exclusive_scan(n_keep, s_warp, &keep_total);
    {
        int e = eq_before;
        for (int i = lo; i < hi; ++i) {
            const uint32_t u = s_key[i];
            bool keep = false;
            if (u > uk) keep = true;
            else if (u == uk) { keep = (e >= eq_cut); ++e; }
            if (keep && pos < k) out[pos++] = i;
        }
    }
    (void)lane;
}

}  // namespace

cudaError_t launch_select(int64_t P, int N, const float* Z, int64_t ldz, int n_obs, int budget,
                          int32_t* idx, DeviceStatus* st, cudaStream_t s) {
    (void)st;
    if (P == 0) return cudaSuccess;
    const size_t smem = sizeof(uint32_t) * (size_t)(N - n_obs > 0 ? N - n_obs : 1);
    cudaError_t e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    select_kernel<<<(unsigned)P, kThreads, smem, s>>>(Z, ldz, N, n_obs, budget, idx);
    return cudaGetLastError();
}

namespace {
__global__ void identity_idx_kernel(int64_t total, int n, int budget, int32_t* idx) {
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int r = (int)(e % budget);
        idx[e] = r < n ? r : -1;
    }
}
}  // namespace

cudaError_t launch_identity_idx(int64_t P, int n, int budget, int32_t* idx, cudaStream_t s) {
    const int64_t total = P * (int64_t)budget;
    if (total == 0) return cudaSuccess;
    const int64_t blocks = (total + 255) / 256;
    identity_idx_kernel<<<(unsigned)(blocks < 152 * 32 ? blocks : 152 * 32), 256, 0, s>>>(total, n,
                                                                                       budget, idx);
    return cudaGetLastError();
}

}  // namespace rkv
