// k_gram_tc.cu -- thresholded key Gram on the sm_103a tensor cores (tcgen05,
// TMEM accumulators, TMA-fed shared memory), with recency protection, R and
// Z computed in the epilogue.  The Gram itself never leaves the SM.
//
// R-KV review (yoonschallenge.tistory.com/1236): summary-table row
// "redundancy" (cosine similarity of key vectors in one head; the beta most
// recent similar tokens are protected), row "final selection criterion"
// (Z = lambda*I - (1-lambda)*R), question 2, cause 3 (all-pairs cosine
// similarity, O(B^2) in the budget -- the one dense contraction of the step).
//
// What is computed per problem (one KV head of one sequence and layer), with
// S_ij = (k_i . k_j) * inv_i * inv_j and inv = 1/max(|k|, eps) from the
// key-stats kernel:
//   sim_i   = sum_{j != i, S_ij > tau} S_ij
//   newer_i = #{ j > i : S_ij > tau }
//   R_i = (sum_i - [newer_i < beta] * sim_i) / (N - 1),  Z_i = lambda*I_i - (1-lambda)*R_i
// where sum_i = sum_{j != i} S_ij also comes from the key-stats kernel (it is
// linear in the keys), so the Gram epilogue only has to find the pairs above
// tau.
//
// Design (one persistent CTA per SM, problems strided over CTAs):
//   * The problem's keys are cut into T = ceil(N/128) row blocks of 128.  Only
//     the upper-triangular block pairs (I, J >= I) are multiplied: S is
//     symmetric, so a pair found in block (I, J), J > I, counts for row i
//     directly and for row j through a shared-memory atomic (rare: only
//     similar pairs).  newer_j never changes there because i < j.
//   * warp 0, one lane: TMA producer.  Block I (the A operand, 2 slots) and
//     blocks J > I (the B operand, a ring of stages) are fetched with
//     cp.async.bulk.tensor (3-D map [P][N][d], 128B swizzle, rows past N
//     zero-filled).  No multicast.
//   * warp 1: owns 256 TMEM columns (two 128x128 fp32 accumulators); one lane
//     issues tcgen05.mma.cta_group::1.kind::f16 (bf16 x bf16 -> fp32, M = N =
//     128, K = 16 per instruction, exact products) and tcgen05.commit.
//   * warps 2..5 (128 threads, one per accumulator row / TMEM lane): the
//     epilogue.  tcgen05.ld brings 32 columns at a time into registers;
//     t = acc * inv_j, and a warp-wide max test skips the 32x32 sub-tile unless
//     some t exceeds tau / inv_i.  Diagonal blocks take the exact path for
//     every element (self-pair excluded).
//   * Every mbarrier wait is bounded; on timeout the kernel records
//     kDevErrTimeout in the device status, stops issuing work, waits (bounded)
//     for its own copies and MMAs in flight, frees its TMEM and returns.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/rkv.h"
#include "rkv_common.cuh"
#include "rkv_internal.h"
#include "tcgen05.cuh"

namespace rkv {
namespace {

using namespace tc;

constexpr int kRows = 128;           // rows (and columns) of one Gram tile
constexpr int kChunkElems = 64;      // bf16 elements per 128-byte swizzle row
constexpr int kChunkBytes = kRows * 128;  // one [128 x 64] bf16 TMA box
constexpr int kMaxBlocks = 34;       // N <= 4352
constexpr int kThreads = 192;        // producer warp, MMA warp, 4 epilogue warps
constexpr int kEpiThreads = 128;
constexpr uint32_t kTmemCols = 256;  // two 128-column fp32 accumulators

template <int D>
struct Cfg {
    static constexpr int KC = D / kChunkElems;  // swizzle chunks per row block
    static constexpr int kBlockBytes = KC * kChunkBytes;
    static constexpr int kAStages = 2;
    static constexpr int kBStages = D == 128 ? 3 : 6;
    static constexpr size_t kBarOff = (size_t)(kAStages + kBStages) * kBlockBytes +
                                      2 * (size_t)kMaxBlocks * kRows * sizeof(float);
    static constexpr int kNumBars = 2 * kAStages + 2 * kBStages + 4 + 2;
    static constexpr size_t kSmemBytes = 1024 + kBarOff + 8 * kNumBars + 16;
};

struct Params {
    int64_t P;
    int N, n_obs, beta;
    float lambda, tau;
    const float* inv_norm;
    const float* sum_s;
    int64_t ld_ws;
    const float* I;
    float* R;
    float* Z;
    int64_t ld_out;
    DeviceStatus* status;
};

// Instruction descriptor: D fp32, A and B bf16, both K-major, M = N = 128.
constexpr uint32_t kIdesc = tc::idesc_bf16(kRows, kRows);

// ---------------------------------------------------------------- kernel --
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
gram_tc_kernel(const __grid_constant__ CUtensorMap tmap, const Params prm) {
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sA = smem;
    uint8_t* sB = sA + C::kAStages * C::kBlockBytes;
    float* s_inv = reinterpret_cast<float*>(sB + C::kBStages * C::kBlockBytes);
    float* s_sim = s_inv + kMaxBlocks * kRows;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
    uint64_t* a_full = bars;
    uint64_t* a_empty = a_full + C::kAStages;
    uint64_t* b_full = a_empty + C::kAStages;
    uint64_t* b_empty = b_full + C::kBStages;
    uint64_t* acc_full = b_empty + C::kBStages;
    uint64_t* acc_empty = acc_full + 2;
    uint64_t* epi_bar = acc_empty + 2;   // 128 epilogue threads meet here
    uint64_t* drain_bar = epi_bar + 1;   // MMA completion at exit
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(drain_bar + 1);
    volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int N = prm.N;
    const int T = (N + kRows - 1) / kRows;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kAStages; ++s) {
            mbar_init(&a_full[s], 1);
            mbar_init(&a_empty[s], 1);
        }
        for (int s = 0; s < C::kBStages; ++s) {
            mbar_init(&b_full[s], 1);
            mbar_init(&b_empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&acc_full[s], 1);
            mbar_init(&acc_empty[s], kEpiThreads);
        }
        mbar_init(epi_bar, kEpiThreads);
        mbar_init(drain_bar, 1);
        *s_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap))
                     : "memory");
    }
    if (warp == 1) {
        tmem_alloc(s_tmem, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;

    if (warp == 0) {
        // ------------------------------------------------------ producer --
        if (lane == 0) {
            uint32_t ka = 0, kb = 0;
            bool ok = true;
            for (int64_t p = blockIdx.x; ok && p < prm.P; p += gridDim.x) {
                for (int I = 0; ok && I < T; ++I) {
                    const int sa = ka % C::kAStages;
                    if (!(ok = mbar_wait(&a_empty[sa], ((ka / C::kAStages) & 1) ^ 1, s_abort)))
                        break;
                    mbar_arrive_expect_tx(&a_full[sa], C::kBlockBytes);
                    for (int c = 0; c < C::KC; ++c)
                        tma_load_3d(sA + sa * C::kBlockBytes + c * kChunkBytes, &tmap, &a_full[sa],
                                    c * kChunkElems, I * kRows, (int)p);
                    ++ka;
                    for (int J = I + 1; ok && J < T; ++J) {
                        const int sb = kb % C::kBStages;
                        if (!(ok = mbar_wait(&b_empty[sb], ((kb / C::kBStages) & 1) ^ 1, s_abort)))
                            break;
                        mbar_arrive_expect_tx(&b_full[sb], C::kBlockBytes);
                        for (int c = 0; c < C::KC; ++c)
                            tma_load_3d(sB + sb * C::kBlockBytes + c * kChunkBytes, &tmap,
                                        &b_full[sb], c * kChunkElems, J * kRows, (int)p);
                        ++kb;
                    }
                }
            }
            if (!ok) {
                *s_abort = 1;
                set_error(prm.status, kDevErrTimeout, 1u);
                // let the copies already issued land before the CTA exits
                volatile int never = 0;
                for (uint32_t u = ka > (uint32_t)C::kAStages ? ka - C::kAStages : 0; u < ka; ++u)
                    mbar_wait(&a_full[u % C::kAStages], (u / C::kAStages) & 1, &never);
                for (uint32_t u = kb > (uint32_t)C::kBStages ? kb - C::kBStages : 0; u < kb; ++u)
                    mbar_wait(&b_full[u % C::kBStages], (u / C::kBStages) & 1, &never);
            }
        }
    } else if (warp == 1) {
        // ----------------------------------------------------- MMA issuer --
        if (lane == 0) {
            uint32_t ka = 0, kb = 0, kacc = 0;
            bool ok = true;
            for (int64_t p = blockIdx.x; ok && p < prm.P; p += gridDim.x) {
                for (int I = 0; ok && I < T; ++I) {
                    const int sa = ka % C::kAStages;
                    if (!(ok = mbar_wait(&a_full[sa], (ka / C::kAStages) & 1, s_abort))) break;
                    const uint8_t* a_base = sA + sa * C::kBlockBytes;
                    for (int J = I; ok && J < T; ++J) {
                        const uint8_t* b_base = a_base;
                        int sb = -1;
                        if (J > I) {
                            sb = kb % C::kBStages;
                            if (!(ok = mbar_wait(&b_full[sb], (kb / C::kBStages) & 1, s_abort)))
                                break;
                            b_base = sB + sb * C::kBlockBytes;
                        }
                        const int acc = kacc & 1;
                        if (!(ok = mbar_wait(&acc_empty[acc], ((kacc >> 1) & 1) ^ 1, s_abort)))
                            break;
                        tc_fence_after();
                        const uint32_t d_tmem = tmem + (uint32_t)(acc * kRows);
#pragma unroll
                        for (int c = 0; c < C::KC; ++c) {
                            const uint64_t ad = sdesc_sw128(a_base + c * kChunkBytes);
                            const uint64_t bd = sdesc_sw128(b_base + c * kChunkBytes);
#pragma unroll
                            for (int k = 0; k < kChunkElems / 16; ++k)
                                mma_bf16(d_tmem, ad + 2 * k, bd + 2 * k, kIdesc, (c | k) != 0);
                        }
                        mma_commit(&acc_full[acc]);
                        if (sb >= 0) {
                            mma_commit(&b_empty[sb]);
                            ++kb;
                        }
                        ++kacc;
                    }
                    if (!ok) break;
                    mma_commit(&a_empty[sa]);
                    ++ka;
                }
            }
            if (!ok) {
                *s_abort = 1;
                set_error(prm.status, kDevErrTimeout, 2u);
            }
            // every MMA issued so far has completed before TMEM is released
            mma_commit(drain_bar);
            volatile int never = 0;
            mbar_wait(drain_bar, 0, &never);
        }
    } else {
        // ------------------------------------------------------- epilogue --
        const int et = threadIdx.x - 64;      // 0..127
        const int q = warp & 3;               // TMEM lane quarter of this warp
        const int row = q * 32 + lane;        // accumulator row of this thread
        const uint32_t t_row = tmem + ((uint32_t)(q * 32) << 16);
        const int Cn = N - prm.n_obs;
        const float inv_nm1 = 1.0f / (float)(N - 1);
        uint32_t kacc = 0, kepi = 0;
        bool ok = true;
        for (int64_t p = blockIdx.x; ok && p < prm.P; p += gridDim.x) {
            const float* invp = prm.inv_norm + p * prm.ld_ws;
            for (int x = et; x < T * kRows; x += kEpiThreads) {
                s_inv[x] = x < N ? invp[x] : 0.f;
                s_sim[x] = 0.f;
            }
            mbar_arrive(epi_bar);
            ok = __all_sync(0xffffffffu, mbar_wait(epi_bar, kepi & 1, s_abort));
            ++kepi;
            for (int I = 0; ok && I < T; ++I) {
                const int i = I * kRows + row;
                const bool valid_i = i < N;
                const float inv_i = valid_i ? s_inv[i] : 0.f;
                const float thr = valid_i ? prm.tau / inv_i : INFINITY;
                float sim_row = 0.f;
                int newer = 0;
                for (int J = I; J < T; ++J) {
                    const int acc = kacc & 1;
                    ok = __all_sync(0xffffffffu, mbar_wait(&acc_full[acc], (kacc >> 1) & 1, s_abort));
                    if (!ok) break;
                    tc_fence_after();
                    const bool diag = (J == I);
#pragma unroll 1
                    for (int c = 0; c < kRows / 32; ++c) {
                        uint32_t r[32];
                        tmem_ld_32cols(t_row + (uint32_t)(acc * kRows + c * 32), r);
                        tmem_ld_wait();
                        const float* ij = s_inv + J * kRows + c * 32;
                        float t[32];
                        float m = -INFINITY;
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            t[e] = __uint_as_float(r[e]) * ij[e];
                            m = fmaxf(m, t[e]);
                        }
                        if (__any_sync(0xffffffffu, diag || m > thr)) {
                            const int jb = J * kRows + c * 32;
#pragma unroll
                            for (int e = 0; e < 32; ++e) {
                                const int j = jb + e;
                                if (t[e] > thr && j < N && j != i) {
                                    const float s = t[e] * inv_i;
                                    sim_row += s;
                                    newer += (j > i);
                                    if (!diag) atomicAdd(&s_sim[j], s);
                                }
                            }
                        }
                    }
                    tc_fence_before();
                    mbar_arrive(&acc_empty[acc]);
                    ++kacc;
                }
                if (!ok) break;
                // all column contributions to block I are in s_sim now
                mbar_arrive(epi_bar);
                ok = __all_sync(0xffffffffu, mbar_wait(epi_bar, kepi & 1, s_abort));
                ++kepi;
                if (!ok) break;
                if (valid_i) {
                    const float sim_i = s_sim[i] + sim_row;
                    float rr = 0.f, z = INFINITY;
                    if (i < Cn) {
                        const float tot = prm.sum_s[p * prm.ld_ws + i];
                        rr = (tot - (newer < prm.beta ? sim_i : 0.f)) * inv_nm1;
                        z = prm.lambda * prm.I[p * prm.ld_out + i] - (1.0f - prm.lambda) * rr;
                    }
                    if (prm.R) prm.R[p * prm.ld_out + i] = rr;
                    prm.Z[p * prm.ld_out + i] = z;
                }
            }
            if (!ok) break;
            // s_inv / s_sim are reset for the next problem only after every
            // thread has read them
            mbar_arrive(epi_bar);
            ok = __all_sync(0xffffffffu, mbar_wait(epi_bar, kepi & 1, s_abort));
            ++kepi;
        }
        if (!ok) {
            *s_abort = 1;
            set_error(prm.status, kDevErrTimeout, 3u);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------ host --
template <int D>
cudaError_t launch_t(const ScoreArgs& a, cudaStream_t s) {
    using C = Cfg<D>;
    CUtensorMap map;
    if (!make_map_3d_bf16(&map, a.K, D, a.N, a.P, D, (int64_t)a.n_cap * D, kRows))
        return cudaErrorInvalidValue;
    Params prm{a.P,      a.N,     a.n_obs,   a.beta, a.lambda, a.tau,    a.inv_norm,
               a.sum_s,  a.ld_ws, a.I,       a.R,    a.Z,      a.ld_out, a.status};
    auto kern = gram_tc_kernel<D>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmemBytes);
    if (e != cudaSuccess) return e;
    const int64_t sms = sm_count();
    const int64_t grid = a.P < sms ? a.P : sms;
    kern<<<(unsigned)grid, kThreads, C::kSmemBytes, s>>>(map, prm);
    return cudaGetLastError();
}

}  // namespace

bool gram_tc_supported(const ScoreArgs& a) {
    return a.dtype == RKV_DTYPE_BF16 && (a.d == 64 || a.d == 128) && a.N >= 2 &&
           a.N <= kMaxBlocks * kRows && a.P <= 0x7fffffff && encode_fn() != nullptr;
}

cudaError_t launch_gram_tc(const ScoreArgs& a, cudaStream_t s) {
    if (a.P == 0) return cudaSuccess;
    return a.d == 128 ? launch_t<128>(a, s) : launch_t<64>(a, s);
}

}  // namespace rkv
