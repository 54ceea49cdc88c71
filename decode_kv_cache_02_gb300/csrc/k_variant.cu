// k_variant.cu -- variants of the combined score: a softmax of the
// redundancy over the candidates and a pooling window on the importance.
//
// R-KV review (yoonschallenge.tistory.com/1236): question 2, cause 3 lists a
// softmax of the redundancy among the operations of each compression round;
// the summary table compares R-KV with SnapKV, the attention-only method whose
// importance is pooled over neighbouring positions.  Row "final selection
// criterion" combines the two as Z = lambda*I - (1-lambda)*R.
//
// Per problem (C = N - n_obs candidates, h = (w-1)/2):
//   R'_i = exp(R_i - m) / sum_{j<C} exp(R_j - m),  m = max_{j<C} R_j
//          (the softmax; subtracting m changes nothing but the range)
//   I'_i = max { I_j : j < C, |j - i| <= h }
//   Z_i  = lambda*I'_i - (1-lambda)*R'_i - pen_i   for i < C
//          (pen_i: the sentence penalty of row i's sentence, see k_sentence.cu)
// Observation tokens (i >= C) keep their I, get R = 0 and Z = +inf.
//
// One CTA per problem: a block maximum and a block sum over the candidates'
// R (both reads of the row after the first hit L1/L2), then one pass that
// writes Z (and I', R' when asked).  Bound by HBM: read I and R, write Z.
// rkv_compress folds the same arithmetic into its select + gather kernel; this
// one serves rkv_score_ex and problems too large for that kernel.
#include "rkv_common.cuh"
#include "rkv_internal.h"
#include "rkv_variant.cuh"

namespace rkv {
namespace {

constexpr int kThreads = 256;

// I_out and R_out may be null.  R_out may equal R (each thread rewrites only
// the rows it read after both reductions); I_out must not overlap I.
__global__ void __launch_bounds__(kThreads)
variant_kernel(VariantIn v, float* __restrict__ Z, float* __restrict__ I_out, float* R_out,
               int64_t ld_out, int N, int n_obs) {
    __shared__ float s_red[kThreads / 32];
    const int64_t p = blockIdx.x;
    const int C = N - n_obs;
    const float* Ip = v.I + p * v.ld;
    const float* Rp = v.R + p * v.ld;
    SoftmaxStats st{0.f, 1.f};
    if (v.softmax) st = softmax_stats<kThreads>(Rp, C, s_red);
    for (int i = threadIdx.x; i < N; i += kThreads) {
        const int64_t o = p * ld_out + i;
        if (i < C) {
            const float ip = pooled_importance(Ip, i, C, v.half);
            const float r = Rp[i];
            const float rs = v.softmax ? softmax_term(r, st) : r;
            Z[o] = variant_score(v, p, i, ip, rs);
            if (I_out) I_out[o] = ip;
            if (R_out) R_out[o] = rs;
        } else {
            Z[o] = INFINITY;
            if (I_out) I_out[o] = Ip[i];
            if (R_out) R_out[o] = 0.f;
        }
    }
}

}  // namespace

cudaError_t launch_variant(int64_t P, int N, int n_obs, const VariantIn& v, float* Z,
                           float* I_out, float* R_out, int64_t ld_out, cudaStream_t s) {
    if (P == 0) return cudaSuccess;
    variant_kernel<<<(unsigned)P, kThreads, 0, s>>>(v, Z, I_out, R_out, ld_out, N, n_obs);
    return cudaGetLastError();
}

}  // namespace rkv
