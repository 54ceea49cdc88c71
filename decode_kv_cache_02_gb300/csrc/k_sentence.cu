// k_sentence.cu -- sentence representations and sentence-level penalties.
//
// SkipKV review (yoonschallenge.tistory.com/1230), summary-table row "Method 1:
// Sentence-level KV Storage Skipping": a sentence is represented by the mean
// of its tokens' last-layer hidden states (no separate sentence encoder), and
// when two sentences' cosine similarity exceeds tau the earlier one is treated
// as redundant and evicted first; row "Final eviction score": the tokens of a
// redundant sentence get the sentence similarity as an extra penalty.
//
//   reps[s, a]  = mean of hidden[s, t] over the tokens t of sentence a
//   pen[s, a]   = max { cos(a, b) : a < b < count[s], cos(a, b) > tau }, 0 if none
//   cos(a, b)   = (r_a . r_b) / (max(|r_a|, eps) * max(|r_b|, eps)),  eps = 1e-12
//
// Both are small next to the step (a few dozen sentences of a few thousand
// hidden units per sequence); they run on the CUDA cores in fp32.
#include "rkv_common.cuh"
#include "rkv_internal.h"
#include "../../include/rkv.h"

namespace rkv {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

// One CTA per (sequence, sentence a): rep a in shared memory, each warp takes
// later sentences b in turn and reduces r_a . r_b and |r_b|^2 over the hidden
// units (float4 loads, coalesced along the row).
__global__ void __launch_bounds__(kThreads)
sentence_penalty_kernel(const float* __restrict__ reps, const int32_t* __restrict__ count,
                        int max_sent, int hidden, float tau, float* __restrict__ pen) {
    extern __shared__ float4 s_a[];  // hidden / 4
    __shared__ float s_red[kWarps];
    const int64_t s = blockIdx.x / max_sent;
    const int a = (int)(blockIdx.x - s * max_sent);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n = min(max(count[s], 0), max_sent);
    float* out = pen + s * max_sent + a;
    if (a >= n) {
        if (tid == 0) *out = 0.f;
        return;
    }
    const int h4 = hidden / 4;
    const float4* ra = reinterpret_cast<const float4*>(reps + (s * max_sent + a) * (int64_t)hidden);
    float nn = 0.f;
    for (int c = tid; c < h4; c += kThreads) {
        const float4 x = ra[c];
        s_a[c] = x;
        nn = fmaf(x.x, x.x, fmaf(x.y, x.y, fmaf(x.z, x.z, fmaf(x.w, x.w, nn))));
    }
    nn = warp_sum(nn);
    if (lane == 0) s_red[warp] = nn;
    __syncthreads();
    float na = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) na += s_red[w];
    const float inv_a = 1.0f / fmaxf(sqrtf(na), 1e-12f);
    __syncthreads();  // s_red is reused below
    float best = -INFINITY;
    for (int b = a + 1 + warp; b < n; b += kWarps) {
        const float4* rb =
            reinterpret_cast<const float4*>(reps + (s * max_sent + b) * (int64_t)hidden);
        float dot = 0.f, nb = 0.f;
        for (int c = lane; c < h4; c += 32) {
            const float4 y = rb[c], x = s_a[c];
            dot = fmaf(x.x, y.x, fmaf(x.y, y.y, fmaf(x.z, y.z, fmaf(x.w, y.w, dot))));
            nb = fmaf(y.x, y.x, fmaf(y.y, y.y, fmaf(y.z, y.z, fmaf(y.w, y.w, nb))));
        }
        dot = warp_sum(dot);
        nb = warp_sum(nb);
        const float cs = dot * inv_a * (1.0f / fmaxf(sqrtf(nb), 1e-12f));
        if (cs > tau) best = fmaxf(best, cs);
    }
    if (lane == 0) s_red[warp] = best;
    __syncthreads();
    if (tid == 0) {
        float m = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) m = fmaxf(m, s_red[w]);
        *out = m > -INFINITY ? m : 0.f;
    }
}

template <typename T> RKV_DEV float4 load4(const T* p);
template <> RKV_DEV float4 load4<float>(const float* p) {
    return *reinterpret_cast<const float4*>(p);
}
template <> RKV_DEV float4 load4<__nv_bfloat16>(const __nv_bfloat16* p) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                       __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
}

// One CTA per (sequence, column chunk); each thread sums 4 hidden units over the
// tokens in order, writing a sentence's mean when its run of tokens ends (a
// sentence's tokens are consecutive).
template <typename T>
__global__ void __launch_bounds__(kThreads)
sentence_reps_kernel(const T* __restrict__ hidden, const int32_t* __restrict__ token_seg, int T_len,
                     int hdim, int max_sent, int chunks, float* __restrict__ reps) {
    const int64_t s = blockIdx.x / chunks;
    const int chunk = (int)(blockIdx.x - s * chunks);
    const int c = (chunk * kThreads + threadIdx.x) * 4;
    if (c >= hdim) return;
    const int32_t* seg = token_seg + s * T_len;
    const T* hs = hidden + s * (int64_t)T_len * hdim + c;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    int cur = -1, cnt = 0;
    auto flush = [&]() {
        if (cur >= 0 && cur < max_sent && cnt > 0) {
            const float inv = 1.0f / (float)cnt;
            *reinterpret_cast<float4*>(reps + (s * max_sent + cur) * (int64_t)hdim + c) =
                make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
        }
    };
    for (int t = 0; t < T_len; ++t) {
        const int a = seg[t];
        if (a != cur) {
            flush();
            cur = a;
            cnt = 0;
            acc = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        if (a < 0 || a >= max_sent) continue;
        const float4 x = load4<T>(hs + (int64_t)t * hdim);
        acc.x += x.x;
        acc.y += x.y;
        acc.z += x.z;
        acc.w += x.w;
        ++cnt;
    }
    flush();
}

}  // namespace

cudaError_t launch_sentence_penalty(int64_t S, int max_sent, int hidden, const float* reps,
                                    const int32_t* count, float tau, float* pen, cudaStream_t s) {
    if (S == 0) return cudaSuccess;
    const size_t smem = sizeof(float) * (size_t)hidden;
    cudaError_t e = cudaFuncSetAttribute(sentence_penalty_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    sentence_penalty_kernel<<<(unsigned)(S * max_sent), kThreads, smem, s>>>(
        reps, count, max_sent, hidden, tau, pen);
    return cudaGetLastError();
}

cudaError_t launch_sentence_reps(const void* hidden, int dtype, const int32_t* token_seg,
                                 int64_t S, int T, int hidden_dim, int max_sent, float* reps,
                                 cudaStream_t s) {
    if (S == 0) return cudaSuccess;
    cudaError_t e = cudaMemsetAsync(reps, 0, sizeof(float) * (size_t)S * max_sent * hidden_dim, s);
    if (e != cudaSuccess || T == 0) return e;
    const int chunks = (hidden_dim / 4 + kThreads - 1) / kThreads;
    const unsigned grid = (unsigned)(S * chunks);
    if (dtype == RKV_DTYPE_BF16)
        sentence_reps_kernel<__nv_bfloat16><<<grid, kThreads, 0, s>>>(
            static_cast<const __nv_bfloat16*>(hidden), token_seg, T, hidden_dim, max_sent, chunks,
            reps);
    else
        sentence_reps_kernel<float><<<grid, kThreads, 0, s>>>(
            static_cast<const float*>(hidden), token_seg, T, hidden_dim, max_sent, chunks, reps);
    return cudaGetLastError();
}

}  // namespace rkv
