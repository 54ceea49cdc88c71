// k_importance.cu -- attention importance of every cached key.
//
// R-KV review (yoonschallenge.tistory.com/1236), summary-table row
// "importance": the weight the recent observation tokens give each past key
// in attention; under GQA the query heads that share one KV head are
// max-pooled so a strong signal is not averaged away.  Computed here as
//     l_{g,q,j} = (q_{g,q} . k_j) / sqrt(d)      for j <= N - n_obs + q
//     p_{g,q,j} = softmax_j(l_{g,q,.})
//     I_j       = max_g (1/n_obs) sum_q p_{g,q,j}
// (mean over the observation queries; the observation tokens are causal
// among themselves).
//
// SIMT version: one CTA per problem, 128 threads, fp32 FMAs from shared
// memory.  Pass 1 streams the keys in tiles of 128 and keeps a running
// (max, sum) per query row; pass 2 recomputes the logits and forms I.
#include "rkv_common.cuh"
#include "rkv_internal.h"
#include "../../include/rkv.h"

namespace rkv {
namespace {

constexpr int kThreads = 128;  // keys per tile, one per thread
constexpr int kMaxRows = 128;  // G * n_obs

template <int D>
struct ImpSmem {
    static constexpr int kPad = D + 4;  // row pitch of the key tile (floats)
    static size_t bytes(int rows) {
        return sizeof(float) * ((size_t)rows * D + (size_t)kThreads * kPad +
                                (size_t)rows * kThreads + 2 * (size_t)rows);
    }
};

// logits of key (tile base j0 + thread) against every query row -> sL[r][t]
template <int D>
__device__ void tile_logits(const float* sQ, const float* sKt, float* sL, int rows, int n_obs,
                            int N, int j, float scale) {
    const float4* kr = reinterpret_cast<const float4*>(sKt + threadIdx.x * ImpSmem<D>::kPad);
    for (int r = 0; r < rows; ++r) {
        const float4* qr = reinterpret_cast<const float4*>(sQ + r * D);
        float acc = 0.f;
#pragma unroll 8
        for (int c = 0; c < D / 4; ++c) {
            const float4 a = qr[c], b = kr[c];
            acc = fmaf(a.x, b.x, acc);
            acc = fmaf(a.y, b.y, acc);
            acc = fmaf(a.z, b.z, acc);
            acc = fmaf(a.w, b.w, acc);
        }
        const int q = r % n_obs;
        const bool valid = (j < N) && (j <= N - n_obs + q);
        sL[r * kThreads + threadIdx.x] = valid ? acc * scale : -INFINITY;
    }
}

template <typename T, int D>
__device__ void load_tile(const T* Kp, int j0, int N, float* sKt) {
    // rows j0 .. j0+127 of the problem, zero past N
    for (int e = threadIdx.x * 8; e < kThreads * D; e += kThreads * 8) {
        const int row = e / D, col = e % D;
        float v[8];
        if (j0 + row < N) {
            load8(Kp + (size_t)(j0 + row) * D + col, v);
        } else {
#pragma unroll
            for (int t = 0; t < 8; ++t) v[t] = 0.f;
        }
        float* dst = sKt + row * ImpSmem<D>::kPad + col;
#pragma unroll
        for (int t = 0; t < 8; ++t) dst[t] = v[t];
    }
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads)
importance_simt_kernel(const T* __restrict__ K, const T* __restrict__ Q, int G, int n_cap,
                       int N, int n_obs, float* __restrict__ I, int64_t ld) {
    extern __shared__ float4 smem4[];
    float* smem = reinterpret_cast<float*>(smem4);
    const int rows = G * n_obs;
    float* sQ = smem;                                  // [rows][D]
    float* sKt = sQ + rows * D;                        // [128][D+4]
    float* sL = sKt + kThreads * ImpSmem<D>::kPad;     // [rows][128]
    float* sM = sL + rows * kThreads;                  // [rows] running max
    float* sS = sM + rows;                             // [rows] running sum
    const int64_t p = blockIdx.x;
    const T* Kp = K + (size_t)p * n_cap * D;
    const T* Qp = Q + (size_t)p * rows * D;
    const float scale = 1.0f / sqrtf((float)D);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    for (int e = threadIdx.x * 8; e < rows * D; e += kThreads * 8) load8(Qp + e, sQ + e);
    for (int r = threadIdx.x; r < rows; r += kThreads) {
        sM[r] = -INFINITY;
        sS[r] = 0.f;
    }
    __syncthreads();

    // pass 1: running max and sum per query row
    for (int j0 = 0; j0 < N; j0 += kThreads) {
        load_tile<T, D>(Kp, j0, N, sKt);
        __syncthreads();
        tile_logits<D>(sQ, sKt, sL, rows, n_obs, N, j0 + threadIdx.x, scale);
        __syncthreads();
        for (int r = warp; r < rows; r += kThreads / 32) {
            float v[kThreads / 32];
            float mt = -INFINITY;
#pragma unroll
            for (int c = 0; c < kThreads / 32; ++c) {
                v[c] = sL[r * kThreads + lane + 32 * c];
                mt = fmaxf(mt, v[c]);
            }
            mt = warp_max(mt);
            const float m_old = sM[r];
            const float m_new = fmaxf(m_old, mt);
            float e = 0.f;
#pragma unroll
            for (int c = 0; c < kThreads / 32; ++c) e += (v[c] == -INFINITY) ? 0.f : expf(v[c] - m_new);
            e = warp_sum(e);
            if (lane == 0) {
                const float keep = (m_old == -INFINITY) ? 0.f : sS[r] * expf(m_old - m_new);
                sS[r] = keep + e;
                sM[r] = m_new;
            }
        }
        __syncthreads();
    }

    // pass 2: probabilities, mean over queries, max over heads
    for (int j0 = 0; j0 < N; j0 += kThreads) {
        load_tile<T, D>(Kp, j0, N, sKt);
        __syncthreads();
        const int j = j0 + threadIdx.x;
        tile_logits<D>(sQ, sKt, sL, rows, n_obs, N, j, scale);
        __syncthreads();
        if (j < N) {
            float best = -INFINITY;
            for (int g = 0; g < G; ++g) {
                float acc = 0.f;
                for (int q = 0; q < n_obs; ++q) {
                    const int r = g * n_obs + q;
                    const float l = sL[r * kThreads + threadIdx.x];
                    acc += (l == -INFINITY) ? 0.f : expf(l - sM[r]) / sS[r];
                }
                best = fmaxf(best, acc / (float)n_obs);
            }
            I[p * ld + j] = best;
        }
        __syncthreads();
    }
}

template <typename T, int D>
cudaError_t launch_t(const ScoreArgs& a, cudaStream_t s) {
    const int rows = a.G * a.n_obs;
    const size_t smem = ImpSmem<D>::bytes(rows);
    auto kern = importance_simt_kernel<T, D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)a.P, kThreads, smem, s>>>(static_cast<const T*>(a.K), static_cast<const T*>(a.Q),
                                               a.G, a.n_cap, a.N, a.n_obs, a.I, a.ld_out);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_importance(const ScoreArgs& a, cudaStream_t s) {
    if (a.P == 0) return cudaSuccess;
    if (a.G * a.n_obs > kMaxRows) return cudaErrorInvalidValue;
    if (a.dtype == RKV_DTYPE_BF16)
        return a.d == 128 ? launch_t<__nv_bfloat16, 128>(a, s) : launch_t<__nv_bfloat16, 64>(a, s);
    return a.d == 128 ? launch_t<float, 128>(a, s) : launch_t<float, 64>(a, s);
}

}  // namespace rkv
