// k_gram_simt.cu -- thresholded key Gram, recency protection, R and Z
// (CUDA-core version; fp32 inputs and any supported shape).
//
// R-KV review (yoonschallenge.tistory.com/1236), summary-table rows
// "redundancy" and "final selection criterion"; question 2, cause 3.  With
// S_ij = (k_i . k_j) * inv_i * inv_j (inv = 1/max(|k|, eps)), for every
// candidate i:
//     sim_i   = sum_{j != i, S_ij > tau} S_ij
//     newer_i = #{ j > i : S_ij > tau }
//     protected_i = newer_i < beta          (the beta most recent of a
//                                            similar group keep their score)
//     R_i = (sum_i - [protected_i] * sim_i) / (N - 1)
//     Z_i = lambda * I_i - (1 - lambda) * R_i
// sum_i comes from the key-stats kernel; the observation tokens get R = 0 and
// Z = +inf (always kept).
//
// Layout: grid (row tiles of 64, P); 256 threads as 16 x 16, each owning a
// 4 x 4 block of the 64 x 64 output tile; both operand tiles are staged in
// shared memory transposed ([c][row]) so that a thread reads its 4 rows /
// 4 columns as one float4.
#include "rkv_common.cuh"
#include "rkv_internal.h"
#include "../../include/rkv.h"

namespace rkv {
namespace {

constexpr int kTile = 64;
constexpr int kThreads = 256;

template <typename T, int D>
__device__ void stage_transposed(const T* Kp, int r0, int N, float* sT) {
    // sT[c * kTile + row] = K[r0 + row][c], zero past N
    for (int e = threadIdx.x; e < kTile * (D / 8); e += kThreads) {
        const int row = e % kTile, c8 = (e / kTile) * 8;
        float v[8];
        if (r0 + row < N) {
            load8(Kp + (size_t)(r0 + row) * D + c8, v);
        } else {
#pragma unroll
            for (int t = 0; t < 8; ++t) v[t] = 0.f;
        }
#pragma unroll
        for (int t = 0; t < 8; ++t) sT[(c8 + t) * kTile + row] = v[t];
    }
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads)
gram_simt_kernel(const T* __restrict__ K, int n_cap, int N, int n_obs, float lambda, int beta,
                 float tau, const float* __restrict__ inv_norm, const float* __restrict__ sum_s,
                 int64_t ld_ws, const float* __restrict__ I, float* __restrict__ R,
                 float* __restrict__ Z, int64_t ld_out) {
    extern __shared__ float4 smem4[];
    float* sA = reinterpret_cast<float*>(smem4);  // [D][64] rows i
    float* sB = sA + D * kTile;                    // [D][64] rows j
    const int64_t p = blockIdx.y;
    const int i0 = blockIdx.x * kTile;
    const T* Kp = K + (size_t)p * n_cap * D;
    const float* invp = inv_norm + p * ld_ws;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;

    stage_transposed<T, D>(Kp, i0, N, sA);
    float inv_i[4];
    int gi[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        gi[u] = i0 + ty * 4 + u;
        inv_i[u] = gi[u] < N ? invp[gi[u]] : 0.f;
    }
    float sim[4] = {0.f, 0.f, 0.f, 0.f};
    int newer[4] = {0, 0, 0, 0};

    for (int j0 = 0; j0 < N; j0 += kTile) {
        __syncthreads();  // previous sB fully consumed
        stage_transposed<T, D>(Kp, j0, N, sB);
        __syncthreads();
        float acc[4][4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int v = 0; v < 4; ++v) acc[u][v] = 0.f;
#pragma unroll 4
        for (int c = 0; c < D; ++c) {
            const float4 a = *reinterpret_cast<const float4*>(sA + c * kTile + ty * 4);
            const float4 b = *reinterpret_cast<const float4*>(sB + c * kTile + tx * 4);
            const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int v = 0; v < 4; ++v) acc[u][v] = fmaf(av[u], bv[v], acc[u][v]);
        }
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const int j = j0 + tx * 4 + v;
            if (j >= N) continue;
            const float inv_j = invp[j];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                if (gi[u] >= N || j == gi[u]) continue;
                const float s = acc[u][v] * inv_i[u] * inv_j;
                if (s > tau) {
                    sim[u] += s;
                    if (j > gi[u]) newer[u] += 1;
                }
            }
        }
    }
    // reduce over the 16 threads (tx) that share rows ty*4 .. ty*4+3
#pragma unroll
    for (int u = 0; u < 4; ++u) {
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) {
            sim[u] += __shfl_xor_sync(0xffffffffu, sim[u], o);
            newer[u] += __shfl_xor_sync(0xffffffffu, newer[u], o);
        }
    }
    if (tx == 0) {
        const int C = N - n_obs;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int i = gi[u];
            if (i >= N) continue;
            float r = 0.f, z = INFINITY;
            if (i < C) {
                const float tot = sum_s[p * ld_ws + i];
                r = (tot - (newer[u] < beta ? sim[u] : 0.f)) / (float)(N - 1);
                z = lambda * I[p * ld_out + i] - (1.0f - lambda) * r;
            }
            if (R) R[p * ld_out + i] = r;
            Z[p * ld_out + i] = z;
        }
    }
}

template <typename T, int D>
cudaError_t launch_t(const ScoreArgs& a, cudaStream_t s) {
    const size_t smem = sizeof(float) * 2 * D * kTile;
    auto kern = gram_simt_kernel<T, D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((a.N + kTile - 1) / kTile, (unsigned)a.P);
    kern<<<grid, kThreads, smem, s>>>(static_cast<const T*>(a.K), a.n_cap, a.N, a.n_obs, a.lambda,
                                      a.beta, a.tau, a.inv_norm, a.sum_s, a.ld_ws, a.I, a.R, a.Z,
                                      a.ld_out);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gram_simt(const ScoreArgs& a, cudaStream_t s) {
    if (a.P == 0) return cudaSuccess;
    if (a.P > 65535) {
        // grid.y limit: split the problems
        ScoreArgs b = a;
        for (int64_t p0 = 0; p0 < a.P; p0 += 65535) {
            b.P = a.P - p0 < 65535 ? a.P - p0 : 65535;
            const size_t es = a.dtype == RKV_DTYPE_BF16 ? 2 : 4;
            b.K = static_cast<const char*>(a.K) + (size_t)p0 * a.n_cap * a.d * es;
            b.inv_norm = a.inv_norm + p0 * a.ld_ws;
            b.sum_s = a.sum_s + p0 * a.ld_ws;
            b.I = a.I + p0 * a.ld_out;
            b.R = a.R ? a.R + p0 * a.ld_out : nullptr;
            b.Z = a.Z + p0 * a.ld_out;
            cudaError_t e = launch_gram_simt(b, s);
            if (e != cudaSuccess) return e;
        }
        return cudaSuccess;
    }
    if (a.dtype == RKV_DTYPE_BF16)
        return a.d == 128 ? launch_t<__nv_bfloat16, 128>(a, s) : launch_t<__nv_bfloat16, 64>(a, s);
    return a.d == 128 ? launch_t<float, 128>(a, s) : launch_t<float, 64>(a, s);
}

}  // namespace rkv
