// k_select.cu -- per-problem top-k of the combined score, ascending indices.
//
// R-KV review (yoonschallenge.tistory.com/1236), opening notes (the newest 8
// tokens always stay; the other tokens are scored and the best ones that fit
// the budget are kept) and question 2, cause 3 (top-k over the scores).  Ties in Z go to
// the larger (more recent) index; the output is the kept candidates in
// ascending order followed by the n_obs observation tokens.
//
// Up to 2048 candidates: one warp per problem (below).  Larger problems: one
// CTA per problem.  Candidate scores are mapped to order-preserving
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

// ------------------------------------------------------------------------
// One warp per problem, for C <= 32 * MAXI candidates: the scores stay in
// registers (element t of lane l is candidate 32 t + l, so the loads are
// coalesced and all in flight together) and the warp needs no block barrier.
// A first pass counts the scores in 256 buckets linear in the score between
// the problem's smallest and largest (a warp-private histogram in shared
// memory); bucket(z) never decreases with z, so the bucket that holds the k-th
// largest score is the only one that needs an exact look.  Its scores, as
// order-preserving integers, are compacted into a warp-private list and
// ranked directly (up to 32 of them) or by radix passes.  Keys above the
// k-th largest u_k are kept, and of the keys equal to u_k those with the
// largest indices; output positions come from a ballot per row of 32
// candidates, which keeps them in index order.
constexpr int kWarpSelWarps = 4;
constexpr int kWarpSelMaxC = 2048;

// The bin of the krem-th largest key in hist[0..255]: the digit, the rank left
// inside the bin and the bin's count, in every lane.
RKV_DEV void find_bin(const uint32_t* hist, uint32_t& krem, uint32_t& digit, uint32_t& bin_count) {
    const int lane = threadIdx.x & 31;
    uint32_t h[8], tot = 0;
#pragma unroll
    for (int b = 0; b < 8; ++b) {
        h[b] = hist[lane * 8 + b];
        tot += h[b];
    }
    uint32_t incl = tot;  // keys in the bins of lanes >= lane
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_down_sync(0xffffffffu, incl, o);
        if (lane + o < 32) incl += y;
    }
    uint32_t above = incl - tot;
    uint32_t d = 0, kn = 0, c = 0;
    const bool mine = above < krem && krem <= incl;
    if (mine) {
#pragma unroll
        for (int b = 7; b >= 0; --b) {
            if (above + h[b] >= krem) {
                d = (uint32_t)(lane * 8 + b);
                kn = krem - above;
                c = h[b];
                break;
            }
            above += h[b];
        }
    }
    const int src = __ffs(__ballot_sync(0xffffffffu, mine)) - 1;
    digit = __shfl_sync(0xffffffffu, d, src);
    krem = __shfl_sync(0xffffffffu, kn, src);
    bin_count = __shfl_sync(0xffffffffu, c, src);
}

template <int MAXI>
__global__ void __launch_bounds__(32 * kWarpSelWarps)
select_warp_kernel(const float* __restrict__ Z, int64_t ldz, int64_t P, int N, int n_obs,
                   int budget, int32_t* __restrict__ idx) {
    __shared__ uint32_t s_hist[kWarpSelWarps][256];
    extern __shared__ uint32_t s_list_all[];  // [kWarpSelWarps][C]
    const int lane = threadIdx.x & 31, wl = threadIdx.x >> 5;
    const int64_t p = (int64_t)blockIdx.x * kWarpSelWarps + wl;
    if (p >= P) return;
    uint32_t* hist = s_hist[wl];
    const int C = N - n_obs, k = budget - n_obs;
    uint32_t* list = s_list_all + (size_t)wl * C;
    const float* zp = Z + p * ldz;
    int32_t* out = idx + p * (int64_t)budget;
    for (int r = lane; r < n_obs; r += 32) out[k + r] = C + r;
    if (k <= 0) return;
    const int rows = (C + 31) / 32;
    const uint32_t lt = (1u << lane) - 1u;

    // all loads first (clamped, unpredicated) so that they are in flight together
    float z[MAXI];
#pragma unroll
    for (int t = 0; t < MAXI; ++t) z[t] = __ldg(zp + min(t * 32 + lane, C - 1));
    float zmin = INFINITY, zmax = -INFINITY;
#pragma unroll
    for (int t = 0; t < MAXI; ++t) {
        if (t < rows && t * 32 + lane < C) {
            zmin = fminf(zmin, z[t]);
            zmax = fmaxf(zmax, z[t]);
        }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        zmin = fminf(zmin, __shfl_xor_sync(0xffffffffu, zmin, o));
        zmax = fmaxf(zmax, __shfl_xor_sync(0xffffffffu, zmax, o));
    }
    // 256 buckets linear in the score: bucket(z) = floor((z - zmin) * scale)
    // never decreases with z, so every score in a higher bucket is larger and
    // only the bucket of the k-th largest needs an exact look
    const float range = zmax - zmin;
    const float scale = range > 0.f ? 255.5f / range : 0.f;
#pragma unroll
    for (int b = 0; b < 8; ++b) hist[lane * 8 + b] = 0u;
    __syncwarp();
#pragma unroll
    for (int t = 0; t < MAXI; ++t) {
        if (t < rows && t * 32 + lane < C) {
            const int bk = min(255, max(0, (int)((z[t] - zmin) * scale)));
            atomicAdd(&hist[bk], 1u);
        }
    }
    __syncwarp();
    uint32_t krem = (uint32_t)k, bucket, m;
    find_bin(hist, krem, bucket, m);
    // the bucket's keys (order-preserving integers) into the list
    {
        uint32_t w = 0;
#pragma unroll
        for (int t = 0; t < MAXI; ++t) {
            const bool in = t < rows && t * 32 + lane < C &&
                            (uint32_t)min(255, max(0, (int)((z[t] - zmin) * scale))) == bucket;
            const uint32_t bm = __ballot_sync(0xffffffffu, in);
            if (in) list[w + __popc(bm & lt)] = orderable(z[t]);
            w += __popc(bm);
        }
    }
    __syncwarp();
    // the krem-th largest of the m keys in the list: uk, how many keys equal
    // it (eq_count) and how many of those are kept (need_eq)
    uint32_t uk, eq_count, need_eq;
    if (m <= 32) {
        const uint32_t mine = lane < (int)m ? list[lane] : 0u;
        uint32_t gt = 0, eq = 0;
        for (uint32_t x = 0; x < m; ++x) {
            const uint32_t o = __shfl_sync(0xffffffffu, mine, x);
            gt += o > mine;
            eq += o == mine;
        }
        const bool it = lane < (int)m && gt < krem && krem <= gt + eq;
        const int src = __ffs(__ballot_sync(0xffffffffu, it)) - 1;
        uk = __shfl_sync(0xffffffffu, mine, src);
        eq_count = __shfl_sync(0xffffffffu, eq, src);
        need_eq = krem - __shfl_sync(0xffffffffu, gt, src);
    } else {
        // radix passes over the list, from the highest bit where its keys differ
        uint32_t lmin = 0xffffffffu, lmax = 0u;
        for (uint32_t x = lane; x < m; x += 32) {
            lmin = min(lmin, list[x]);
            lmax = max(lmax, list[x]);
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            lmin = min(lmin, __shfl_xor_sync(0xffffffffu, lmin, o));
            lmax = max(lmax, __shfl_xor_sync(0xffffffffu, lmax, o));
        }
        int top = lmin == lmax ? 0 : 32 - __clz(lmin ^ lmax);
        uint32_t prefix = top == 32 ? 0u : lmax & ~((1u << top) - 1u);
        eq_count = m;
        __syncwarp();  // the histogram is read before it is cleared again
        while (top > 0) {
            const int sh = top >= 8 ? top - 8 : 0;
            const uint32_t dm = top >= 8 ? 255u : ((1u << top) - 1u);
            const uint32_t pm = top == 32 ? 0u : ~((1u << top) - 1u);
#pragma unroll
            for (int b = 0; b < 8; ++b) hist[lane * 8 + b] = 0u;
            __syncwarp();
            for (uint32_t x = lane; x < m; x += 32) {
                const uint32_t u = list[x];
                if ((u & pm) == prefix) atomicAdd(&hist[(u >> sh) & dm], 1u);
            }
            __syncwarp();
            uint32_t dg;
            find_bin(hist, krem, dg, eq_count);
            prefix |= dg << sh;
            top = sh;
            __syncwarp();
        }
        uk = prefix;
        need_eq = krem;
    }
    // keys above uk are kept; of the eq_count keys equal to uk, the need_eq
    // with the largest indices
    const uint32_t eq_cut = eq_count - need_eq;
    uint32_t eq_before = 0, pos = 0;
#pragma unroll
    for (int t = 0; t < MAXI; ++t) {
        const int i = t * 32 + lane;
        const bool valid = t < rows && i < C;
        const uint32_t key = valid ? orderable(z[t]) : 0u;
        bool keep;
        if (eq_cut == 0) {
            keep = valid && key >= uk;
        } else {
            const bool eq = valid && key == uk;
            const uint32_t eqm = __ballot_sync(0xffffffffu, eq);
            keep = valid && (key > uk || (eq && eq_before + __popc(eqm & lt) >= eq_cut));
            eq_before += __popc(eqm);
        }
        const uint32_t km = __ballot_sync(0xffffffffu, keep);
        const uint32_t at = pos + __popc(km & lt);
        if (keep && at < (uint32_t)k) out[at] = i;
        pos += __popc(km);
    }
}

}  // namespace

cudaError_t launch_select(int64_t P, int N, const float* Z, int64_t ldz, int n_obs, int budget,
                          int32_t* idx, DeviceStatus* st, cudaStream_t s) {
    (void)st;
    if (P == 0) return cudaSuccess;
    const int C = N - n_obs;
    if (C >= 1 && C <= kWarpSelMaxC) {
        const int64_t blocks = (P + kWarpSelWarps - 1) / kWarpSelWarps;
        const size_t list_bytes = sizeof(uint32_t) * (size_t)kWarpSelWarps * C;
        auto kern = C <= 32 * 40 ? select_warp_kernel<40> : select_warp_kernel<64>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)list_bytes);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
        if (e != cudaSuccess) return e;
        kern<<<(unsigned)blocks, 32 * kWarpSelWarps, list_bytes, s>>>(Z, ldz, P, N, n_obs, budget, idx);
        return cudaGetLastError();
    }
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
