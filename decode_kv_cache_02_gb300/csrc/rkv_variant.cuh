// rkv_variant.cuh -- per-problem arithmetic of the scoring variants, shared
// by the stand-alone variant kernel and the fused select + gather, so that
// both give the same Z bit for bit.
//
// R-KV review (yoonschallenge.tistory.com/1236): question 2, cause 3 lists a
// softmax of the redundancy; the summary table's comparison method SnapKV
// pools its importance over neighbouring positions.
//   R'_i = exp(R_i - m) * (1 / sum_{j<C} exp(R_j - m)),  m = max_{j<C} R_j
//   I'_i = max { I_j : j < C, |j - i| <= half }
//   Z_i  = lambda * I'_i - (1 - lambda) * R'_i
// The reductions stride the candidates by the block size and fold lanes by
// xor shuffles, then warps in order: the same order in every kernel that
// includes this header with the same block size.
#pragma once

#include "rkv_common.cuh"
#include "rkv_internal.h"

namespace rkv {

// Block-wide max (kMax) or sum of v; every thread gets the result.  s_red
// holds kThreads / 32 floats.
template <int kThreads, bool kMax>
__device__ float variant_block_reduce(float v, float* s_red) {
    constexpr int kWarps = kThreads / 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        const float y = __shfl_xor_sync(0xffffffffu, v, o);
        v = kMax ? fmaxf(v, y) : v + y;
    }
    if (lane == 0) s_red[warp] = v;
    __syncthreads();
    float t = s_red[0];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) t = kMax ? fmaxf(t, s_red[w]) : t + s_red[w];
    __syncthreads();  // s_red may be reused right after
    return t;
}

struct SoftmaxStats {
    float m;        // max of R over the candidates
    float inv_sum;  // 1 / sum of exp(R - m)
};

// Softmax statistics of R[0..C) (global or shared memory).  Contains block
// barriers: every thread of the block must call it.
template <int kThreads>
__device__ SoftmaxStats softmax_stats(const float* R, int C, float* s_red) {
    float mx = -INFINITY;
    for (int i = threadIdx.x; i < C; i += kThreads) mx = fmaxf(mx, R[i]);
    SoftmaxStats st;
    st.m = variant_block_reduce<kThreads, true>(mx, s_red);
    float sum = 0.f;
    for (int i = threadIdx.x; i < C; i += kThreads) sum += expf(R[i] - st.m);
    // the largest candidate contributes exp(0) = 1, so the sum is >= 1
    st.inv_sum = 1.0f / variant_block_reduce<kThreads, false>(sum, s_red);
    return st;
}

// I'_i: the maximum of I over the candidates within `half` positions of i.
RKV_DEV float pooled_importance(const float* I, int i, int C, int half) {
    float v = I[i];
    const int lo = max(0, i - half), hi = min(C - 1, i + half);
    for (int j = lo; j <= hi; ++j) v = fmaxf(v, I[j]);
    return v;
}

RKV_DEV float softmax_term(float r, const SoftmaxStats& st) {
    return __fmul_rn(expf(__fsub_rn(r, st.m)), st.inv_sum);
}

// Z from the variant's terms, rounded the same way wherever it is computed
// (no contraction into a fused multiply-add).
RKV_DEV float variant_z(float lambda, float ip, float rs) {
    return __fsub_rn(__fmul_rn(lambda, ip), __fmul_rn(__fsub_rn(1.0f, lambda), rs));
}

// The sentence penalty of row i of problem p (SkipKV review, row "Final
// eviction score"): pen[s, a] for the row's sentence a, 0 for rows outside a
// sentence or without sentence information.
RKV_DEV float row_penalty(const VariantIn& v, int64_t p, int i) {
    if (v.pen == nullptr) return 0.f;
    const int64_t s = (p / v.heads) % v.num_seqs;
    const int a = v.seg[p * v.ld_seg + i];
    const int n = min(v.count[s], v.max_sent);
    return (a >= 0 && a < n) ? v.pen[s * v.max_sent + a] : 0.f;
}

// Z of candidate i with every variant term.
RKV_DEV float variant_score(const VariantIn& v, int64_t p, int i, float ip, float rs) {
    return __fsub_rn(variant_z(v.lambda, ip, rs), row_penalty(v, p, i));
}

}  // namespace rkv
