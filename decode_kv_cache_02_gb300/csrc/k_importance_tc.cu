// k_importance_tc.cu -- attention importance on the sm_103a tensor cores.
//
// R-KV review (yoonschallenge.tistory.com/1236), summary-table row
// "importance": the attention the recent observation queries give each past
// key, max-pooled over the query heads of a GQA group.  With R = G * n_obs
// query rows (g, q) per problem:
//     l_{c,j} = (q_c . k_j) / sqrt(d)          c = g*n_obs + q, j <= N - n_obs + q
//     I_j     = max_g (1/n_obs) sum_q softmax_j(l_{c,.})
//
// The logits of a block of 128 keys are one tcgen05.mma chain: A = the key
// block (M = 128, K-major bf16 from TMA), B = the problem's R query rows
// followed by s = sum_j khat_j as two bf16 rows (hi, lo) and zero rows, N =
// RP = 48, fp32 accumulators in TMEM.  The s columns give k_i . s, which
// completes the redundancy row sum sum_i = inv_i (k_i . s) - |khat_i|^2 (the
// key-stats kernel leaves |khat_i|^2 in sum_i) without another pass over K.
// One epilogue thread owns one key row of a block; two groups of four warps
// take alternate blocks (the MMA order's even and odd accumulators), so two
// warps per scheduler hide the latency of the exponentials.  Two passes over
// the problem's keys; the second reads the blocks in reverse order, so the
// ones the first read last (the most likely to be in L2) come first, and the
// first pass's copies ask L2 to keep their lines (evict_last), the second's to
// drop them first:
//   pass 1  per-thread online (max, sum of exp) per query row, then a block
//           reduction (warp shuffles + shared memory) to the row's max M_c and
//           1 / sum_j exp(l - M_c);
//   pass 2  p = exp(l - M_c) / S_c, mean over q, max over g -> I_j.
// Warp 0 (one lane) issues the TMA loads, warp 1 owns TMEM and one lane issues
// the MMAs, the other warps are the epilogue; one persistent CTA per SM, with
// a five-stage ring of key blocks so the next problem's keys stream in while
// the epilogue reduces.  All waits are bounded.  When all of a problem's
// logits fit in TMEM the resident variant below reads the keys only once.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/rkv.h"
#include "rkv_common.cuh"
#include "rkv_internal.h"
#include "tcgen05.cuh"

namespace rkv {
namespace {

using namespace tc;

constexpr int kRows = 128;
constexpr int kChunkElems = 64;
constexpr int kChunkBytes = kRows * 128;
constexpr int kThreads = 320;
constexpr int kEpi = 256;  // two groups of four warps taking alternate key blocks
constexpr int kAcc = 4;            // accumulators in flight
constexpr int kAccCols = 64;       // TMEM columns per accumulator
constexpr uint32_t kTmemCols = 256;
constexpr int kMaxQueryRows = 46;  // G * n_obs handled here (plus the two s rows)

template <int D, int RP>
struct ICfg {
    static constexpr int KC = D / kChunkElems;
    static constexpr int kBlockBytes = KC * kChunkBytes;
    static constexpr int kQChunkBytes = RP * 128;
    static constexpr int kStages = D == 128 ? 5 : 10;
    static constexpr size_t kQOff = (size_t)kStages * kBlockBytes;
    static constexpr size_t kRedOff = kQOff + (size_t)KC * kQChunkBytes;
    static constexpr size_t kBarOff = kRedOff + sizeof(float) * 16 * RP;
    static constexpr int kNumBars = 2 * kStages + 2 + 2 * kAcc + 2;
    static constexpr size_t kSmemBytes = 1024 + kBarOff + 8 * kNumBars + 16;
};

constexpr int kMaxObs = kMaxQueryRows;

struct IParams {
    int64_t P;
    int N, n_obs, G;
    int R;         // query rows G * n_obs; B rows R, R+1 hold s (hi, lo)
    float scale;
    float scale2;  // log2(e) / sqrt(d)
    float* I;
    int64_t ld;
    // sum_i = inv_i (k_i . s) - |khat_i|^2: the key-stats kernel leaves
    // |khat_i|^2 in sum_s, this kernel completes it
    float* inv_norm;  // written by the resident variant with the statistics folded in
    float* sum_s;
    int64_t ld_ws;
    DeviceStatus* status;
    KeySource ks;  // contiguous keys, or the paged pool read through the table
    // resident variant with the key statistics folded in: s = sum_j khat_j
    // (fp32) per problem, stride ld_s floats
    float* s32;
    int64_t ld_s;
    // bit c of colmask[k]: query row c exists and its query index c % n_obs
    // is >= k (so it sees a key k positions past N - n_obs); bit c of
    // lastmask: c is the last query row of its head.
    unsigned long long colmask[kMaxObs + 1];
    unsigned long long lastmask;
    int ns;  // resident variant: logit slots in TMEM
};

RKV_DEV void tmem_ld_16cols(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

// one TMEM column (no wait)
RKV_DEV uint32_t tmem_ld_1col(uint32_t taddr) {
    uint32_t r;
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(r) : "r"(taddr));
    return r;
}

// 2^x and log2(x) by the approximate PTX instructions (flush-to-zero)
RKV_DEV float ex2_fast(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
RKV_DEV float lg2_fast(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <int D, int RP>
__global__ void __launch_bounds__(kThreads, 1)
importance_tc_kernel(const __grid_constant__ KeyMaps kmap,
                     const __grid_constant__ CUtensorMap qmap,
                     const __grid_constant__ CUtensorMap smap, const IParams prm) {
    using C = ICfg<D, RP>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sK = smem;
    uint8_t* sQ = smem + C::kQOff;
    float* redM = reinterpret_cast<float*>(smem + C::kRedOff);  // [8][RP]
    float* redS = redM + 8 * RP;                                 // [8][RP]
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
    uint64_t* k_full = bars;
    uint64_t* k_empty = k_full + C::kStages;
    uint64_t* q_full = k_empty + C::kStages;
    uint64_t* q_empty = q_full + 1;
    uint64_t* acc_full = q_empty + 1;
    uint64_t* acc_empty = acc_full + kAcc;
    uint64_t* epi_bar = acc_empty + kAcc;
    uint64_t* drain_bar = epi_bar + 1;
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(drain_bar + 1);
    volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
    __shared__ unsigned long long s_colmask[kMaxObs + 1];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int N = prm.N, n_obs = prm.n_obs;
    for (int k = threadIdx.x; k <= n_obs && k <= kMaxObs; k += blockDim.x) s_colmask[k] = prm.colmask[k];
    const int T = (N + kRows - 1) / kRows;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&k_full[s], 1);
            mbar_init(&k_empty[s], 1);
        }
        mbar_init(q_full, 1);
        mbar_init(q_empty, 1);
        for (int a = 0; a < kAcc; ++a) {
            mbar_init(&acc_full[a], 1);
            mbar_init(&acc_empty[a], kEpi / 64);  // the four warps of one group
        }
        mbar_init(epi_bar, kEpi / 32);
        mbar_init(drain_bar, 1);
        *s_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
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
        if (lane == 0) {
            uint32_t kk = 0, kq = 0;
            bool ok = true;
            for (int64_t p = blockIdx.x; ok && p < prm.P; p += gridDim.x) {
                if (!(ok = mbar_wait(q_empty, (kq & 1) ^ 1, s_abort))) break;
                mbar_arrive_expect_tx(q_full, C::KC * C::kQChunkBytes);
                for (int c = 0; c < C::KC; ++c) {
                    tma_load_3d(sQ + c * C::kQChunkBytes, &qmap, q_full, c * kChunkElems, 0, (int)p);
                    tma_load_3d(sQ + c * C::kQChunkBytes + prm.R * 128, &smap, q_full,
                                c * kChunkElems, 0, (int)p);
                }
                ++kq;
                for (int pass = 0; ok && pass < 2; ++pass) {
                    const uint64_t policy = pass == 0 ? l2_policy_evict_last() : l2_policy_evict_first();
                    for (int i = 0; i < T; ++i) {
                        const int b = pass == 0 ? i : T - 1 - i;
                        const int s = kk % C::kStages;
                        if (!(ok = mbar_wait(&k_empty[s], ((kk / C::kStages) & 1) ^ 1, s_abort)))
                            break;
                        mbar_arrive_expect_tx(&k_full[s], C::kBlockBytes);
                        load_key_rows(sK + s * C::kBlockBytes, kChunkBytes, C::KC, &kmap, &k_full[s],
                                      p, b * kRows, kRows, prm.ks, policy);
                        ++kk;
                    }
                }
            }
            if (!ok) {
                *s_abort = 1;
                set_error(prm.status, kDevErrTimeout, 11u);
                volatile int never = 0;
                for (uint32_t u = kk > (uint32_t)C::kStages ? kk - C::kStages : 0; u < kk; ++u)
                    mbar_wait(&k_full[u % C::kStages], (u / C::kStages) & 1, &never);
                if (kq > 0) mbar_wait(q_full, (kq - 1) & 1, &never);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16(kRows, RP);
            uint32_t kk = 0, kq = 0, ka = 0;
            bool ok = true;
            for (int64_t p = blockIdx.x; ok && p < prm.P; p += gridDim.x) {
                if (!(ok = mbar_wait(q_full, kq & 1, s_abort))) break;
                for (int pass = 0; ok && pass < 2; ++pass) {
                    for (int b = 0; b < T; ++b) {
                        const int s = kk % C::kStages;
                        if (!(ok = mbar_wait(&k_full[s], (kk / C::kStages) & 1, s_abort))) break;
                        const int a = ka % kAcc;
                        if (!(ok = mbar_wait(&acc_empty[a], ((ka / kAcc) & 1) ^ 1, s_abort))) break;
                        tc_fence_after();
                        const uint32_t d_tmem = tmem + (uint32_t)(a * kAccCols);
#pragma unroll
                        for (int c = 0; c < C::KC; ++c) {
                            const uint64_t ad = sdesc_sw128(sK + s * C::kBlockBytes + c * kChunkBytes);
                            const uint64_t bd = sdesc_sw128(sQ + c * C::kQChunkBytes);
#pragma unroll
                            for (int k = 0; k < kChunkElems / 16; ++k)
                                mma_bf16(d_tmem, ad + 2 * k, bd + 2 * k, idesc, (c | k) != 0);
                        }
                        mma_commit(&acc_full[a]);
                        mma_commit(&k_empty[s]);
                        ++kk;
                        ++ka;
                    }
                }
                if (!ok) break;
                mma_commit(q_empty);
                ++kq;
            }
            if (!ok) {
                *s_abort = 1;
                set_error(prm.status, kDevErrTimeout, 12u);
            }
            mma_commit(drain_bar);
            volatile int never = 0;
            mbar_wait(drain_bar, 0, &never);
        }
    } else {
        const int qd = warp & 3;            // TMEM lane quarter
        const int ew = warp - 2;            // 0..7
        const int grp = ew >> 2;            // takes the blocks of accumulator counter parity grp
        const int row = qd * 32 + lane;
        const uint32_t t_row = tmem + ((uint32_t)(qd * 32) << 16);
        const int lim = N - n_obs;  // key j is seen by query q iff j <= lim + q
        // blocks whose rows all lie at or before N - n_obs: every query row
        // sees every key there, no mask
        const int full_blocks = (lim + 1) / kRows;
        const float scale2 = prm.scale2;  // log2(e) / sqrt(d): logits in log2 units
        const float log2_nobs = lg2_fast((float)n_obs);
        const unsigned long long lastmask = prm.lastmask;
        uint32_t ka = 0, ke = 0;
        bool ok = true;
        for (int64_t p = blockIdx.x; ok && p < prm.P; p += gridDim.x) {
            float m[RP], s[RP];
#pragma unroll
            for (int c = 0; c < RP; ++c) {
                m[c] = -INFINITY;
                s[c] = 0.f;
            }
            // ---- pass 1: online max / sum of exp per query row (log2 units)
            const uint32_t ka1 = ka;  // accumulator counter of the pass's block 0
            for (int b = (grp + (int)(ka1 & 1)) & 1; b < T; b += 2) {
                const uint32_t kb = ka1 + (uint32_t)b;
                const int a = kb % kAcc;
                ok = __all_sync(0xffffffffu, mbar_wait(&acc_full[a], (kb / kAcc) & 1, s_abort));
                if (!ok) break;
                tc_fence_after();
                const int j = b * kRows + row;
                const unsigned long long vm =
                    b < full_blocks ? ~0ull
                                    : (j <= lim ? s_colmask[0] : (j < N ? s_colmask[j - lim] : 0ull));
#pragma unroll
                for (int cc = 0; cc < RP / 16; ++cc) {
                    uint32_t r[16];
                    tmem_ld_16cols(t_row + (uint32_t)(a * kAccCols + cc * 16), r);
                    tmem_ld_wait();
                    if (b < full_blocks) {
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const int c = cc * 16 + e;
                            const float l = __uint_as_float(r[e]) * scale2;
                            const float mn = fmaxf(m[c], l);
                            s[c] = fmaf(s[c], ex2_fast(m[c] - mn), ex2_fast(l - mn));
                            m[c] = mn;
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const int c = cc * 16 + e;
                            if ((vm >> c) & 1ull) {
                                const float l = __uint_as_float(r[e]) * scale2;
                                const float mn = fmaxf(m[c], l);
                                s[c] = fmaf(s[c], ex2_fast(m[c] - mn), ex2_fast(l - mn));
                                m[c] = mn;
                            }
                        }
                    }
                }
                tc_fence_before();
                mbar_arrive_warp(&acc_empty[a]);
            }
            if (!ok) break;
            ka = ka1 + (uint32_t)T;
            // ---- block reduction: row max, then the rescaled sums
#pragma unroll
            for (int c = 0; c < RP; ++c) {
                const float mx = warp_max(m[c]);
                if (lane == 0) redM[ew * RP + c] = mx;
            }
            mbar_arrive_warp(epi_bar);
            ok = __all_sync(0xffffffffu, mbar_wait(epi_bar, ke & 1, s_abort));
            ++ke;
            if (!ok) break;
#pragma unroll
            for (int c = 0; c < RP; ++c) {
                float M = redM[c];
#pragma unroll
                for (int w = 1; w < kEpi / 32; ++w) M = fmaxf(M, redM[w * RP + c]);
                const float part = (m[c] == -INFINITY) ? 0.f : s[c] * ex2_fast(m[c] - M);
                const float ws = warp_sum(part);
                if (lane == 0) redS[ew * RP + c] = ws;
                m[c] = M;
            }
            mbar_arrive_warp(epi_bar);
            ok = __all_sync(0xffffffffu, mbar_wait(epi_bar, ke & 1, s_abort));
            ++ke;
            if (!ok) break;
            // fold 1 / (sum * n_obs) into the exponent: p / n_obs = exp2(l - m')
#pragma unroll
            for (int c = 0; c < RP; ++c) {
                float S = 0.f;
#pragma unroll
                for (int w = 0; w < kEpi / 32; ++w) S += redS[w * RP + c];
                m[c] += lg2_fast(S) + log2_nobs;
            }
            // ---- pass 2: probabilities -> importance (blocks in reverse order)
            const uint32_t ka2 = ka;
            for (int i = (grp + (int)(ka2 & 1)) & 1; i < T; i += 2) {
                const uint32_t kb = ka2 + (uint32_t)i;
                const int b = T - 1 - i;
                const int a = kb % kAcc;
                ok = __all_sync(0xffffffffu, mbar_wait(&acc_full[a], (kb / kAcc) & 1, s_abort));
                if (!ok) break;
                tc_fence_after();
                const int j = b * kRows + row;
                const unsigned long long vm =
                    b < full_blocks ? ~0ull
                                    : (j <= lim ? s_colmask[0] : (j < N ? s_colmask[j - lim] : 0ull));
                float iv = 0.f, self = 0.f;
                if (j < N) {
                    iv = prm.inv_norm[p * prm.ld_ws + j];
                    self = prm.sum_s[p * prm.ld_ws + j];
                }
                // k_j . s: the two s columns (R, R + 1) of the accumulator
                const uint32_t s_hi = tmem_ld_1col(t_row + (uint32_t)(a * kAccCols + prm.R));
                const uint32_t s_lo = tmem_ld_1col(t_row + (uint32_t)(a * kAccCols + prm.R + 1));
                float best = -INFINITY, acc = 0.f;
#pragma unroll
                for (int cc = 0; cc < RP / 16; ++cc) {
                    uint32_t r[16];
                    tmem_ld_16cols(t_row + (uint32_t)(a * kAccCols + cc * 16), r);
                    tmem_ld_wait();
                    if (b < full_blocks) {
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const int c = cc * 16 + e;
                            acc += ex2_fast(fmaf(__uint_as_float(r[e]), scale2, -m[c]));
                            if ((lastmask >> c) & 1ull) {  // last query row of a head
                                best = fmaxf(best, acc);
                                acc = 0.f;
                            }
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const int c = cc * 16 + e;
                            if ((vm >> c) & 1ull)
                                acc += ex2_fast(fmaf(__uint_as_float(r[e]), scale2, -m[c]));
                            if ((lastmask >> c) & 1ull) {
                                best = fmaxf(best, acc);
                                acc = 0.f;
                            }
                        }
                    }
                }
                const float dot = __uint_as_float(s_hi) + __uint_as_float(s_lo);
                tc_fence_before();
                mbar_arrive_warp(&acc_empty[a]);
                if (j < N) {
                    prm.I[p * prm.ld + j] = best;
                    prm.sum_s[p * prm.ld_ws + j] = iv * dot - self;
                }
            }
            ka = ka2 + (uint32_t)T;
        }
        if (!ok) {
            *s_abort = 1;
            set_error(prm.status, kDevErrTimeout, 13u);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------------
// Resident variant: when a problem's logits fit in TMEM, each key block is
// multiplied once and its logits stay in TMEM while the epilogue sweeps them
// three times (row max, sum of exponentials, probabilities); the keys are
// read from memory once.  TMEM is a ring of NS slots of SC columns (the query
// rows, padded); sweep 2 writes each exponential back over its logit
// (tcgen05.st), so sweep 3 only scales them, and sweep 3 releases a block's
// slot, so the MMAs of the next problem run while this one is swept and the
// key stream keeps going.
// NS >= T keeps the ring free of deadlock (a problem never waits for one of
// its own slots).  The query rows are double-buffered.
//
// The tensor pipe takes about as long for one M = 128 MMA of N = 16 as of
// N = 128, so k_i . s (which completes sum_i) is not a second MMA per K step:
// two dot warps read each key block from shared memory, take the dot product
// with s in fp32, and release the stage together with the MMA.
//
// Warps: 0 TMA producer, 1 MMA issuer (and TMEM owner), 2..9 the epilogue in
// two groups taking alternate key blocks, 10..11 the dot warps.
constexpr int kREpi = 256;
constexpr int kRDotWarps = 4;
constexpr int kRThreads = 64 + kREpi + 32 * kRDotWarps;
constexpr uint32_t kRTmemCols = 512;
constexpr int kRMaxSlots = 16;
constexpr int kSRows = 2;  // s_hi, s_lo: the rows of s the dot warps read
constexpr uint32_t kSAccCols = 32;  // two s accumulators of 16 columns (statistics mode, d = 128)

// Shared-memory descriptor of a key block read as an MN-major operand (its
// rows are keys, the contraction runs over them): 128-byte swizzle atoms of
// 64 consecutive dimensions x 8 keys (1024 bytes), the next 8 keys 1024 bytes
// on (stride), the next 64 dimensions one chunk (16 KB) on (leading).
RKV_DEV uint64_t sdesc_sw128_mn(const void* p) {
    const uint64_t a = smem_u32(p);
    uint64_t d = (a >> 4) & 0x3FFFull;
    d |= (uint64_t)(kChunkBytes >> 4) << 16;  // leading byte offset: the next 64 dimensions
    d |= (uint64_t)(1024 >> 4) << 32;         // stride byte offset: the next 8 keys
    d |= 1ull << 46;
    d |= 2ull << 61;
    return d;
}
constexpr size_t kSmemLimit = 232448;  // 227 KB of opt-in shared memory per CTA

template <int D, int SC>
struct RCfg {
    static constexpr int KC = D / kChunkElems;
    static constexpr int kBlockBytes = KC * kChunkBytes;
    static constexpr int kQChunkBytes = SC * 128;
    static constexpr int kSChunkBytes = 1024;  // kSRows rows used; 1024-byte aligned
    static constexpr int kBBytes = KC * (kQChunkBytes + kSChunkBytes);  // one problem's B operands
    // two tiles of the s MMA's B operand (inv_hi, inv_lo of a block's keys,
    // 14 zero rows): 16 rows x 128 keys bf16, 128-byte swizzle
    static constexpr int kInvTileBytes = 2 * 16 * 128;
    static constexpr int kFixedBars = 4 + 2 * kRMaxSlots + 2 + 8;
    static constexpr size_t kRedBytes = sizeof(float) * (16 * SC + kRDotWarps * D);
    static constexpr size_t kFixed =
        1024 + 2 * (size_t)kInvTileBytes + 2 * (size_t)kBBytes + kRedBytes + 8 * kFixedBars + 16;
    static constexpr int kFit = (int)((kSmemLimit - kFixed) / (kBlockBytes + 16));
    static constexpr int kStages = kFit < 12 ? kFit : 12;
    static constexpr size_t kInvOff = (size_t)kStages * kBlockBytes;
    static constexpr size_t kBOff = kInvOff + 2 * (size_t)kInvTileBytes;
    static constexpr size_t kRedOff = kBOff + 2 * (size_t)kBBytes;
    static constexpr size_t kBarOff = kRedOff + kRedBytes;
    static constexpr int kNumBars = 2 * kStages + kFixedBars;
    static constexpr size_t kSmemBytes = 1024 + kBarOff + 8 * kNumBars + 16;
    static_assert(kStages >= 4 && kSmemBytes <= kSmemLimit, "shared memory plan");
};

// 16 TMEM columns into r[OFF .. OFF+15] (constant indices keep r in registers)
template <int OFF, int RP>
RKV_DEV void tmem_ld16_at(uint32_t taddr, uint32_t (&r)[RP]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[OFF + 0]), "=r"(r[OFF + 1]), "=r"(r[OFF + 2]), "=r"(r[OFF + 3]),
          "=r"(r[OFF + 4]), "=r"(r[OFF + 5]), "=r"(r[OFF + 6]), "=r"(r[OFF + 7]),
          "=r"(r[OFF + 8]), "=r"(r[OFF + 9]), "=r"(r[OFF + 10]), "=r"(r[OFF + 11]),
          "=r"(r[OFF + 12]), "=r"(r[OFF + 13]), "=r"(r[OFF + 14]), "=r"(r[OFF + 15])
        : "r"(taddr + (uint32_t)OFF));
}

// the SC query columns of one key row (no wait)
template <int SC>
RKV_DEV void tmem_ld_row_nowait(uint32_t taddr, uint32_t (&r)[SC]) {
    tmem_ld16_at<0, SC>(taddr, r);
    tmem_ld16_at<16, SC>(taddr, r);
    if constexpr (SC > 32) tmem_ld16_at<32, SC>(taddr, r);
}

// r[OFF .. OFF+15] into 16 TMEM columns
template <int OFF, int RP>
RKV_DEV void tmem_st16_at(uint32_t taddr, const uint32_t (&r)[RP]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(
            taddr + (uint32_t)OFF),
        "r"(r[OFF + 0]), "r"(r[OFF + 1]), "r"(r[OFF + 2]), "r"(r[OFF + 3]), "r"(r[OFF + 4]),
        "r"(r[OFF + 5]), "r"(r[OFF + 6]), "r"(r[OFF + 7]), "r"(r[OFF + 8]), "r"(r[OFF + 9]),
        "r"(r[OFF + 10]), "r"(r[OFF + 11]), "r"(r[OFF + 12]), "r"(r[OFF + 13]), "r"(r[OFF + 14]),
        "r"(r[OFF + 15])
        : "memory");
}

// the SC columns of one row back into TMEM
template <int SC>
RKV_DEV void tmem_st_row(uint32_t taddr, const uint32_t (&r)[SC]) {
    tmem_st16_at<0, SC>(taddr, r);
    tmem_st16_at<16, SC>(taddr, r);
    if constexpr (SC > 32) tmem_st16_at<32, SC>(taddr, r);
}

RKV_DEV void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

struct OpMax {
    RKV_DEV float operator()(float a, float b) const { return fmaxf(a, b); }
};
struct OpAdd {
    RKV_DEV float operator()(float a, float b) const { return a + b; }
};

// Warp reduce-scatter of v[OFF .. OFF+NV) (NV = 16 or 32): rounds of halving
// width, each lane keeping the half its lane bit selects and folding in the
// partner's other half.  On return lane l holds the reduction over the warp of
// column OFF + (l mod NV); v is clobbered.
template <int OFF, int NV, int SC, class Op>
RKV_DEV float warp_reduce_scatter(float (&v)[SC], Op op) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int h = NV / 2; h >= 1; h >>= 1) {
        const bool up = (lane & h) != 0;
#pragma unroll
        for (int i = 0; i < h; ++i) {
            const float send = up ? v[OFF + i] : v[OFF + i + h];
            const float keep = up ? v[OFF + i + h] : v[OFF + i];
            v[OFF + i] = op(keep, __shfl_xor_sync(0xffffffffu, send, h));
        }
    }
    float r = v[OFF];
#pragma unroll
    for (int h = NV; h < 32; h <<= 1) r = op(r, __shfl_xor_sync(0xffffffffu, r, h));
    return r;
}

// Row statistics over the eight epilogue warps: each warp reduce-scatters its
// per-thread partials, lane l posts column l (and 32 + l mod 16 when SC = 48),
// and after the barrier every lane folds its column over the warps.
template <int SC, class Op>
RKV_DEV void post_partials(float (&v)[SC], float* red, int ew, Op op) {
    const int lane = threadIdx.x & 31;
    const float lo = warp_reduce_scatter<0, 32, SC>(v, op);
    red[ew * SC + lane] = lo;
    if constexpr (SC > 32) {
        const float hi = warp_reduce_scatter<32, SC - 32, SC>(v, op);
        if (lane < SC - 32) red[ew * SC + 32 + lane] = hi;
    }
}

template <int SC, class Op>
RKV_DEV void fold_partials(const float* red, float& lo, float& hi, Op op) {
    const int lane = threadIdx.x & 31;
    lo = red[lane];
#pragma unroll
    for (int w = 1; w < 8; ++w) lo = op(lo, red[w * SC + lane]);
    hi = 0.f;
    if constexpr (SC > 32) {
        const int c = 32 + (lane & (SC - 33));
        hi = red[c];
#pragma unroll
        for (int w = 1; w < 8; ++w) hi = op(hi, red[w * SC + c]);
    }
}

// every lane gets all SC column values back from the lanes that own them
template <int SC>
RKV_DEV void broadcast_columns(float (&v)[SC], float lo, float hi) {
#pragma unroll
    for (int c = 0; c < 32; ++c) v[c] = __shfl_sync(0xffffffffu, lo, c);
#pragma unroll
    for (int c = 32; c < SC; ++c) v[c] = __shfl_sync(0xffffffffu, hi, c - 32);
}

// |k|^2 over the D elements of row r of a key block (fp32, packed FMAs)
template <int KC>
RKV_DEV float row_norm2(const uint8_t* blk, int r) {
    unsigned long long acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
    for (int c = 0; c < KC; ++c) {
        const uint8_t* tile = blk + c * kChunkBytes;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const uint4 k = swizzled_unit(tile, r, u);
            const unsigned long long k0 = bf16x2_to_f32x2(k.x), k1 = bf16x2_to_f32x2(k.y);
            const unsigned long long k2 = bf16x2_to_f32x2(k.z), k3 = bf16x2_to_f32x2(k.w);
            fma_f32x2(acc[0], k0, k0);
            fma_f32x2(acc[1], k1, k1);
            fma_f32x2(acc[2], k2, k2);
            fma_f32x2(acc[3], k3, k3);
        }
    }
    return (f32x2_sum(acc[0]) + f32x2_sum(acc[1])) + (f32x2_sum(acc[2]) + f32x2_sum(acc[3]));
}

RKV_DEV void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// HEAD > 0: the query rows form SC / HEAD heads of HEAD rows (R == SC), so a
// head's last row is known at compile time; HEAD == 0 reads it from lastmask.
// kStats: the key statistics are taken here too (no separate pass over K):
// the dot warps write inv_i and |khat_i|^2 for every key and s = sum_j khat_j
// per problem, and leave k_i . s to the Gram kernel.
template <int D, int SC, int HEAD, bool kStats>
__global__ void __launch_bounds__(kRThreads, 1)
importance_tcr_kernel(const __grid_constant__ KeyMaps kmap,
                      const __grid_constant__ CUtensorMap qmap,
                      const __grid_constant__ CUtensorMap smap, const IParams prm) {
    using C = RCfg<D, SC>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sK = smem;
    uint8_t* sB = smem + C::kBOff;  // [2][ KC query chunks | KC s chunks ]
    float* redM = reinterpret_cast<float*>(smem + C::kRedOff);  // [8][SC]
    float* redS = redM + 8 * SC;                                 // [8][SC]
    float* sDot = redS + 8 * SC;                                 // [kRDotWarps][D]: s in fp32
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
    uint64_t* k_full = bars;
    uint64_t* k_empty = k_full + C::kStages;
    uint64_t* q_full = k_empty + C::kStages;    // [2]
    uint64_t* q_empty = q_full + 2;             // [2]
    uint64_t* blk_full = q_empty + 2;           // [kRMaxSlots]
    uint64_t* tmem_free = blk_full + kRMaxSlots;  // [kRMaxSlots]
    uint64_t* epi_bar = tmem_free + kRMaxSlots;
    uint64_t* drain_bar = epi_bar + 1;
    // statistics mode at d = 128: s = sum_j khat_j on the tensor core
    uint64_t* inv_full = drain_bar + 1;    // [2] a block's inv rows written
    uint64_t* inv_empty = inv_full + 2;    // [2] their s MMAs done
    uint64_t* sacc_full = inv_empty + 2;   // [2] a problem's s accumulated
    uint64_t* sacc_empty = sacc_full + 2;  // [2] read by the dot warps
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(sacc_empty + 2);
    volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
    __shared__ unsigned long long s_colmask[kMaxObs + 1];
    // kSMma: s = K_blk^T (inv_hi + inv_lo) per block, accumulated in TMEM
    // (lanes = dimensions, two 16-column accumulators after the logit ring):
    // A = the key block read MN-major, B = the block's inverse norms as two
    // bf16 rows (hi, lo) and 14 zero rows
    constexpr bool kSMma = kStats && D == 128;
    uint8_t* sInv = smem + C::kInvOff;  // [2][C::kInvTileBytes]
    const uint32_t sacc_col = kRTmemCols - kSAccCols;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int N = prm.N, n_obs = prm.n_obs;
    const uint32_t NS = (uint32_t)prm.ns;
    for (int k = threadIdx.x; k <= n_obs && k <= kMaxObs; k += blockDim.x) s_colmask[k] = prm.colmask[k];
    const int T = (N + kRows - 1) / kRows;

    if (kSMma) {
        // the s MMA's B tiles: rows 2..15 stay zero, rows 0 and 1 are rewritten
        // for every block
        for (int i = threadIdx.x; i < 2 * C::kInvTileBytes / 16; i += blockDim.x)
            reinterpret_cast<uint4*>(sInv)[i] = make_uint4(0u, 0u, 0u, 0u);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    // query rows R .. SC-1 of both B buffers are never loaded: zero them once
    // (their logit columns are never used, zeros keep them finite)
    if (prm.R < SC) {
        const int pad = (SC - prm.R) * 128;
        for (int i = threadIdx.x; i < 2 * C::KC * pad / 16; i += blockDim.x) {
            const int chunk = i / (pad / 16), off = i % (pad / 16);
            const int buf = chunk / C::KC, c = chunk % C::KC;
            *reinterpret_cast<uint4*>(sB + buf * C::kBBytes + c * C::kQChunkBytes + prm.R * 128 +
                                      off * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&k_full[s], 1);
            mbar_init(&k_empty[s], 1 + kRDotWarps);  // the MMAs' commit and each dot warp
        }
        for (int q = 0; q < 2; ++q) {
            mbar_init(&q_full[q], 1);
            mbar_init(&q_empty[q], kStats ? 1 : 1 + kRDotWarps);  // the dot warps read s
        }
        for (int b = 0; b < kRMaxSlots; ++b) {
            mbar_init(&blk_full[b], 1);
            mbar_init(&tmem_free[b], kREpi / 64);  // the group (its warps) that reads the block
        }
        mbar_init(epi_bar, kREpi / 32);
        mbar_init(drain_bar, 1);
        for (int t = 0; t < 2; ++t) {
            mbar_init(&inv_full[t], kRDotWarps);
            mbar_init(&inv_empty[t], 1);
            mbar_init(&sacc_full[t], 1);
            mbar_init(&sacc_empty[t], kRDotWarps);
        }
        *s_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        tmem_alloc(s_tmem, kRTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;

    if (warp == 0) {
        if (lane == 0) {
            uint32_t kk = 0, kq = 0;
            bool ok = true;
            const uint32_t q_tx = (uint32_t)(C::KC * (prm.R + (kStats ? 0 : kSRows)) * 128);
            for (int64_t p = blockIdx.x; ok && p < prm.P; p += gridDim.x) {
                const int qb = kq & 1;
                if (!(ok = mbar_wait(&q_empty[qb], ((kq >> 1) & 1) ^ 1, s_abort))) break;
                mbar_arrive_expect_tx(&q_full[qb], q_tx);
                uint8_t* b_buf = sB + qb * C::kBBytes;
                for (int c = 0; c < C::KC; ++c) {
                    tma_load_3d(b_buf + c * C::kQChunkBytes, &qmap, &q_full[qb], c * kChunkElems, 0,
                                (int)p);
                    if (!kStats)
                        tma_load_3d(b_buf + C::KC * C::kQChunkBytes + c * C::kSChunkBytes, &smap,
                                    &q_full[qb], c * kChunkElems, 0, (int)p);
                }
                ++kq;
                for (int b = 0; b < T; ++b) {
                    const int s = kk % C::kStages;
                    if (!(ok = mbar_wait(&k_empty[s], ((kk / C::kStages) & 1) ^ 1, s_abort))) break;
                    mbar_arrive_expect_tx(&k_full[s], C::kBlockBytes);
                    // with the statistics folded in nothing else reads the
                    // table before the compaction: check its ids here
                    load_key_rows(sK + s * C::kBlockBytes, kChunkBytes, C::KC, &kmap, &k_full[s], p,
                                  b * kRows, kRows, prm.ks, 0, kStats ? prm.status : nullptr);
                    ++kk;
                }
            }
            if (!ok) {
                *s_abort = 1;
                set_error(prm.status, kDevErrTimeout, 21u);
            }
            // let every copy this warp started land before the CTA exits
            volatile int never = 0;
            for (uint32_t u = kk > (uint32_t)C::kStages ? kk - C::kStages : 0; u < kk; ++u)
                mbar_wait(&k_full[u % C::kStages], (u / C::kStages) & 1, &never);
            for (uint32_t u = kq > 2u ? kq - 2u : 0u; u < kq; ++u)
                mbar_wait(&q_full[u & 1], (u >> 1) & 1, &never);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc_q = idesc_bf16(kRows, SC);
            // the s MMA: M = 128 dimensions (A transposed: MN-major), N = 16
            constexpr uint32_t idesc_s = idesc_bf16(128, 16) | (1u << 15);
            uint32_t u = 0, kp = 0;
            bool ok = true;
            for (int64_t p = blockIdx.x; ok && p < prm.P; p += gridDim.x, ++kp) {
                const int qb = kp & 1;
                if (!(ok = mbar_wait(&q_full[qb], (kp >> 1) & 1, s_abort))) break;
                const uint8_t* b_buf = sB + qb * C::kBBytes;
                const int sbuf = kp & 1;
                // the dot warps have read this accumulator's previous problem
                if (kSMma && !(ok = mbar_wait(&sacc_empty[sbuf], ((kp >> 1) & 1) ^ 1, s_abort))) break;
                for (int b = 0; b < T; ++b, ++u) {
                    const int s = u % C::kStages;
                    if (!(ok = mbar_wait(&k_full[s], (u / C::kStages) & 1, s_abort))) break;
                    const uint32_t slot = u % NS;
                    // the slot's previous block has been swept
                    if (!(ok = mbar_wait(&tmem_free[slot], ((u / NS) & 1) ^ 1, s_abort))) break;
                    tc_fence_after();
                    const uint32_t d_q = tmem + slot * (uint32_t)SC;
#pragma unroll
                    for (int c = 0; c < C::KC; ++c) {
                        const uint64_t ad = sdesc_sw128(sK + s * C::kBlockBytes + c * kChunkBytes);
                        const uint64_t bq = sdesc_sw128(b_buf + c * C::kQChunkBytes);
#pragma unroll
                        for (int k = 0; k < kChunkElems / 16; ++k)
                            mma_bf16(d_q, ad + 2 * k, bq + 2 * k, idesc_q, (c | k) != 0);
                    }
                    mma_commit(&blk_full[slot]);
                    if (kSMma) {
                        // s += K_blk^T (inv_hi, inv_lo): 16 keys per instruction
                        const int t = u & 1;
                        if (!(ok = mbar_wait(&inv_full[t], (u >> 1) & 1, s_abort))) break;
                        tc_fence_after();
                        const uint8_t* inv_tile = sInv + t * C::kInvTileBytes;
#pragma unroll
                        for (int ks = 0; ks < kRows / 16; ++ks) {
                            const uint64_t ad = sdesc_sw128_mn(sK + s * C::kBlockBytes + ks * 2048);
                            const uint64_t bd =
                                sdesc_sw128(inv_tile + (ks >> 2) * (16 * 128)) + 2 * (ks & 3);
                            mma_bf16(tmem + sacc_col + (uint32_t)(sbuf * 16), ad, bd, idesc_s,
                                     (b | ks) != 0);
                        }
                        mma_commit(&inv_empty[t]);
                        if (b == T - 1) mma_commit(&sacc_full[sbuf]);
                    }
                    mma_commit(&k_empty[s]);
                }
                if (!ok) break;
                mma_commit(&q_empty[qb]);
            }
            if (!ok) {
                *s_abort = 1;
                set_error(prm.status, kDevErrTimeout, 22u);
            }
            mma_commit(drain_bar);
            volatile int never = 0;
            mbar_wait(drain_bar, 0, &never);
        }
    } else if (kStats && warp >= 2 + kREpi / 32) {
        // ---- statistics warps: inv_i = 1 / max(|k_i|, eps) and |khat_i|^2 of
        // row dw * 32 + lane of every key block, and s = sum_j khat_j: lane l
        // adds columns l * CPL .. l * CPL + CPL - 1 of the warp's 32 rows (each
        // row's inv_i handed over by shuffle); the four warps' partial s meet
        // in shared memory at the problem's end, in a fixed order
        constexpr int CPL = D / 32;
        const int dw = warp - (2 + kREpi / 32);
        const int r0 = dw * 32 + lane;
        const int c0 = lane * CPL;  // this lane's first column of s
        const int cchunk = c0 / kChunkElems, cunit = (c0 % kChunkElems) >> 3, celem = c0 & 7;
        uint32_t kk = 0, kp = 0;
        bool ok = true;
        // kSMma: this lane's key in the inverse-norm tiles (row 0 hi, row 1 lo;
        // 16-byte unit u of row r at unit u ^ r)
        const int ichunk = r0 >> 6, iel = r0 & 63;
        const int ioff0 = ichunk * 16 * 128 + (((iel >> 3) ^ 0) << 4) + (iel & 7) * 2;
        const int ioff1 = ichunk * 16 * 128 + 128 + (((iel >> 3) ^ 1) << 4) + (iel & 7) * 2;
        for (int64_t p = blockIdx.x; ok && p < prm.P; p += gridDim.x, ++kp) {
            float sacc[CPL];
#pragma unroll
            for (int t = 0; t < CPL; ++t) sacc[t] = 0.f;
            for (int b = 0; b < T; ++b, ++kk) {
                const int st = kk % C::kStages;
                ok = __all_sync(0xffffffffu, mbar_wait(&k_full[st], (kk / C::kStages) & 1, s_abort));
                if (!ok) break;
                const uint8_t* blk = sK + st * C::kBlockBytes;
                const int j0 = b * kRows + r0;
                const float n2 = row_norm2<C::KC>(blk, r0);
                // rows past N are TMA zero fill; they add nothing to s
                const float inv = j0 < N ? 1.0f / fmaxf(sqrtf(n2), 1e-12f) : 0.f;
                if constexpr (kSMma) {
                    // inv as bf16 hi + lo into the block's B tile for the s MMA
                    const int t = kk & 1;
                    ok = __all_sync(0xffffffffu,
                                    mbar_wait(&inv_empty[t], ((kk >> 1) & 1) ^ 1, s_abort));
                    if (!ok) break;
                    const __nv_bfloat16 hi = __float2bfloat16_rn(inv);
                    const __nv_bfloat16 lo = __float2bfloat16_rn(inv - __bfloat162float(hi));
                    uint8_t* tile_t = sInv + t * C::kInvTileBytes;
                    *reinterpret_cast<__nv_bfloat16*>(tile_t + ioff0) = hi;
                    *reinterpret_cast<__nv_bfloat16*>(tile_t + ioff1) = lo;
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(&inv_full[t]);
                        mbar_arrive(&k_empty[st]);
                    }
                } else {
                    const uint8_t* tile = blk + cchunk * kChunkBytes;
#pragma unroll 8
                    for (int rr = 0; rr < 32; ++rr) {
                        const float iv = __shfl_sync(0xffffffffu, inv, rr);
                        const int r = dw * 32 + rr;
                        const uint8_t* src = tile + r * 128 + ((cunit ^ (r & 7)) << 4) + celem * 2;
                        if constexpr (CPL == 4) {
                            const uint2 v = *reinterpret_cast<const uint2*>(src);
                            sacc[0] = fmaf(__uint_as_float(v.x << 16), iv, sacc[0]);
                            sacc[1] = fmaf(__uint_as_float(v.x & 0xffff0000u), iv, sacc[1]);
                            sacc[2] = fmaf(__uint_as_float(v.y << 16), iv, sacc[2]);
                            sacc[3] = fmaf(__uint_as_float(v.y & 0xffff0000u), iv, sacc[3]);
                        } else {
                            const uint32_t v = *reinterpret_cast<const uint32_t*>(src);
                            sacc[0] = fmaf(__uint_as_float(v << 16), iv, sacc[0]);
                            sacc[1] = fmaf(__uint_as_float(v & 0xffff0000u), iv, sacc[1]);
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&k_empty[st]);
                }
                if (j0 < N) {
                    prm.inv_norm[p * prm.ld_ws + j0] = inv;
                    // |khat_i|^2; the Gram kernel completes sum_i from it
                    prm.sum_s[p * prm.ld_ws + j0] = (n2 * inv) * inv;
                }
            }
            if (!ok) break;
            if constexpr (kSMma) {
                // s of this warp's 32 dimensions (its TMEM lane quarter), once
                // the problem's s MMAs are done
                const int sbuf = kp & 1;
                ok = __all_sync(0xffffffffu, mbar_wait(&sacc_full[sbuf], (kp >> 1) & 1, s_abort));
                if (!ok) break;
                tc_fence_after();
                const uint32_t taddr = tmem + ((uint32_t)((warp & 3) * 32) << 16) + sacc_col +
                                       (uint32_t)(sbuf * 16);
                const uint32_t shi = tmem_ld_1col(taddr), slo = tmem_ld_1col(taddr + 1);
                tmem_ld_wait();
                tc_fence_before();
                mbar_arrive_warp(&sacc_empty[sbuf]);
                prm.s32[p * prm.ld_s + (warp & 3) * 32 + lane] =
                    __uint_as_float(shi) + __uint_as_float(slo);
            } else {
#pragma unroll
                for (int t = 0; t < CPL; ++t) sDot[dw * D + c0 + t] = sacc[t];
                named_bar_sync(1, 32 * kRDotWarps);
                if (dw == 0) {
                    for (int c = lane; c < D; c += 32) {
                        float v = 0.f;
#pragma unroll
                        for (int w = 0; w < kRDotWarps; ++w) v += sDot[w * D + c];
                        prm.s32[p * prm.ld_s + c] = v;
                    }
                }
                named_bar_sync(1, 32 * kRDotWarps);
            }
        }
        if (!ok) {
            *s_abort = 1;
            set_error(prm.status, kDevErrTimeout, 25u);
        }
    } else if (warp >= 2 + kREpi / 32) {
        // ---- dot warps: sum_i = inv_i (k_i . s) - |khat_i|^2 (the key-stats
        // kernel leaves |khat_i|^2 in sum_s), rows dw * 64 + lane and + 32 of
        // every key block.  inv_i and |khat_i|^2 are loaded two blocks ahead
        // (a cursor over (problem, block) pairs) so that no store waits on them.
        const int dw = warp - (2 + kREpi / 32);
        const int r0 = dw * 32 + lane;
        float* s32 = sDot + dw * D;
        auto fetch = [&](int64_t q, int c, float (&v)[2]) {
            const int j0 = c * kRows + r0;
            v[0] = v[1] = 0.f;
            if (q < prm.P && j0 < N) {
                v[0] = prm.inv_norm[q * prm.ld_ws + j0];
                v[1] = prm.sum_s[q * prm.ld_ws + j0];
            }
        };
        auto advance = [&](int64_t& q, int& c) {
            if (++c == T) {
                c = 0;
                q += gridDim.x;
            }
        };
        int64_t p = blockIdx.x, fq = blockIdx.x;
        int b = 0, fc = 0;
        uint32_t kk = 0, kp = 0;
        bool ok = true;
        float va[2], vb[2];
        fetch(fq, fc, va);
        advance(fq, fc);
        fetch(fq, fc, vb);
        advance(fq, fc);
        // one key block of problem p with its prefetched inv / |khat|^2
        auto dot_block = [&](float (&v)[2]) {
            if (b == 0) {
                // s = s_hi + s_lo in fp32: rows 0 and 1 of each s chunk (row
                // r's 16-byte unit u at unit u ^ r)
                const int qb = kp & 1;
                ok = __all_sync(0xffffffffu, mbar_wait(&q_full[qb], (kp >> 1) & 1, s_abort));
                if (!ok) return;
                const uint8_t* s_buf = sB + qb * C::kBBytes + C::KC * C::kQChunkBytes;
                __syncwarp();  // the previous problem's reads of s32 are done
                for (int e = lane; e < D; e += 32) {
                    const int c = e / kChunkElems, x = e % kChunkElems, u = x >> 3, w = x & 7;
                    const uint8_t* ch = s_buf + c * C::kSChunkBytes;
                    const __nv_bfloat16 hi =
                        reinterpret_cast<const __nv_bfloat16*>(ch + ((u ^ 0) << 4))[w];
                    const __nv_bfloat16 lo =
                        reinterpret_cast<const __nv_bfloat16*>(ch + 128 + ((u ^ 1) << 4))[w];
                    s32[e] = __bfloat162float(hi) + __bfloat162float(lo);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&q_empty[qb]);
            }
            const int st = kk % C::kStages;
            ok = __all_sync(0xffffffffu, mbar_wait(&k_full[st], (kk / C::kStages) & 1, s_abort));
            if (!ok) return;
            const uint8_t* blk = sK + st * C::kBlockBytes;
            const float d0 = row_dot<C::KC>(blk, r0, s32);
            __syncwarp();
            if (lane == 0) mbar_arrive(&k_empty[st]);
            const int j0 = b * kRows + r0;
            if (j0 < N) prm.sum_s[p * prm.ld_ws + j0] = v[0] * d0 - v[1];
            ++kk;
            if (b + 1 == T) ++kp;
            advance(p, b);
        };
        while (ok && p < prm.P) {
            dot_block(va);
            fetch(fq, fc, va);
            advance(fq, fc);
            if (!ok || p >= prm.P) break;
            dot_block(vb);
            fetch(fq, fc, vb);
            advance(fq, fc);
        }
        if (!ok) {
            *s_abort = 1;
            set_error(prm.status, kDevErrTimeout, 24u);
        }
    } else {
        const int ew = warp - 2;           // 0..7
        const int grp = ew >> 2;           // blocks b with b % 2 == grp
        const int qd = warp & 3;           // TMEM lane quarter
        const int row = qd * 32 + lane;
        const uint32_t lane_off = (uint32_t)(qd * 32) << 16;
        const int lim = N - n_obs;
        // blocks whose rows all lie at or before N - n_obs: every query row
        // sees every key there, no mask.  Columns R .. SC-1 (zero query rows)
        // need none either: they never reach a head's mean.
        const int full_blocks = (lim + 1) / kRows;
        const unsigned long long lastmask = prm.lastmask;
        const float scale2 = prm.scale2;   // log2(e) / sqrt(d)
        uint32_t ub = 0, ke = 0;           // ub: ring index of the problem's block 0
        bool ok = true;
        for (int64_t p = blockIdx.x; ok && p < prm.P; p += gridDim.x, ub += (uint32_t)T) {
            float m[SC];
#pragma unroll
            for (int c = 0; c < SC; ++c) m[c] = -INFINITY;
            // ---- sweep 1: largest raw logit per query row
            for (int b = grp; b < T; b += 2) {
                const uint32_t u = ub + (uint32_t)b;
                const uint32_t slot = u % NS;
                const int j = b * kRows + row;
                ok = __all_sync(0xffffffffu, mbar_wait(&blk_full[slot], (u / NS) & 1, s_abort));
                if (!ok) break;
                tc_fence_after();
                uint32_t r[SC];
                tmem_ld_row_nowait<SC>(tmem + lane_off + slot * (uint32_t)SC, r);
                tmem_ld_wait();
                if (b < full_blocks) {
#pragma unroll
                    for (int c = 0; c < SC; ++c) m[c] = fmaxf(m[c], __uint_as_float(r[c]));
                } else {
                    const unsigned long long vm =
                        j <= lim ? s_colmask[0] : (j < N ? s_colmask[j - lim] : 0ull);
#pragma unroll
                    for (int c = 0; c < SC; ++c)
                        if ((vm >> c) & 1ull) m[c] = fmaxf(m[c], __uint_as_float(r[c]));
                }
            }
            if (!ok) break;
            post_partials<SC>(m, redM, ew, OpMax{});
            mbar_arrive_warp(epi_bar);
            ok = __all_sync(0xffffffffu, mbar_wait(epi_bar, ke & 1, s_abort));
            ++ke;
            if (!ok) break;
            float mlo, mhi;  // this lane's columns: row max in log2 units
            fold_partials<SC>(redM, mlo, mhi, OpMax{});
            mlo *= scale2;
            mhi *= scale2;
            broadcast_columns<SC>(m, mlo, mhi);
            // ---- sweep 2: sum of exponentials; each exponential (0 where the
            // query does not see the key) replaces its logit in TMEM, so that
            // sweep 3 only scales them
            float sm[SC];
#pragma unroll
            for (int c = 0; c < SC; ++c) sm[c] = 0.f;
            for (int b = grp; b < T; b += 2) {
                const uint32_t slot = (ub + (uint32_t)b) % NS;
                const uint32_t taddr = tmem + lane_off + slot * (uint32_t)SC;
                tc_fence_after();
                uint32_t r[SC];
                tmem_ld_row_nowait<SC>(taddr, r);
                tmem_ld_wait();
                if (b < full_blocks) {
#pragma unroll
                    for (int c = 0; c < SC; ++c) {
                        const float e = ex2_fast(fmaf(__uint_as_float(r[c]), scale2, -m[c]));
                        sm[c] += e;
                        r[c] = __float_as_uint(e);
                    }
                } else {
                    const int j = b * kRows + row;
                    const unsigned long long vm =
                        j <= lim ? s_colmask[0] : (j < N ? s_colmask[j - lim] : 0ull);
#pragma unroll
                    for (int c = 0; c < SC; ++c) {
                        const float e =
                            ((vm >> c) & 1ull)
                                ? ex2_fast(fmaf(__uint_as_float(r[c]), scale2, -m[c]))
                                : 0.f;
                        sm[c] += e;
                        r[c] = __float_as_uint(e);
                    }
                }
                tmem_st_row<SC>(taddr, r);
            }
            tmem_st_wait();
            post_partials<SC>(sm, redS, ew, OpAdd{});
            mbar_arrive_warp(epi_bar);
            ok = __all_sync(0xffffffffu, mbar_wait(epi_bar, ke & 1, s_abort));
            ++ke;
            if (!ok) break;
            // p / n_obs = e * (1 / (sum * n_obs)): m now holds the column scales
            {
                float slo, shi;
                fold_partials<SC>(redS, slo, shi, OpAdd{});
                const float ilo = 1.0f / (slo * (float)n_obs);
                const float ihi = SC > 32 ? 1.0f / (shi * (float)n_obs) : 0.f;
                broadcast_columns<SC>(m, ilo, ihi);
            }
            // ---- sweep 3: probabilities -> importance; frees the slot
            for (int b = grp; b < T; b += 2) {
                const uint32_t slot = (ub + (uint32_t)b) % NS;
                tc_fence_after();
                const int j = b * kRows + row;
                uint32_t r[SC];
                tmem_ld_row_nowait<SC>(tmem + lane_off + slot * (uint32_t)SC, r);
                tmem_ld_wait();
                tc_fence_before();
                mbar_arrive_warp(&tmem_free[slot]);
                float best = -INFINITY, acc = 0.f;
#pragma unroll
                for (int c = 0; c < SC; ++c) {
                    acc = fmaf(__uint_as_float(r[c]), m[c], acc);
                    if (HEAD > 0 ? (c % (HEAD > 0 ? HEAD : 1) == HEAD - 1) : ((lastmask >> c) & 1ull)) {
                        best = fmaxf(best, acc);  // last query row of a head
                        acc = 0.f;
                    }
                }
                if (j < N) prm.I[p * prm.ld + j] = best;
            }
        }
        if (!ok) {
            *s_abort = 1;
            set_error(prm.status, kDevErrTimeout, 23u);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kRTmemCols);
}

// Ring size of the resident variant for T key blocks of SC logit columns:
// as many slots as TMEM holds; false when a problem does not fit.
bool resident_ring(int T, int SC, int* ns, bool s_mma) {
    // with the s MMA, its two 16-column accumulators take the last 32 columns
    int n = (int)(kRTmemCols - (s_mma ? kSAccCols : 0)) / SC;
    if (n > kRMaxSlots) n = kRMaxSlots;
    if (T > n) return false;
    *ns = n;
    return true;
}

template <int D, int RP>
cudaError_t launch_t(const ScoreArgs& a, cudaStream_t s) {
    using C = ICfg<D, RP>;
    const int R = a.G * a.n_obs;
    IParams prm{};
    prm.P = a.P;
    prm.N = a.N;
    prm.n_obs = a.n_obs;
    prm.G = a.G;
    prm.R = R;
    prm.scale = 1.0f / sqrtf((float)D);
    prm.scale2 = (float)(1.4426950408889634 / sqrt((double)D));
    prm.I = a.I;
    prm.ld = a.ld_out;
    prm.inv_norm = a.inv_norm;
    prm.sum_s = a.sum_s;
    prm.ld_ws = a.ld_ws;
    prm.status = a.status;
    for (int k = 0; k <= a.n_obs && k <= kMaxObs; ++k) {
        unsigned long long m = 0;
        for (int c = 0; c < R; ++c)
            if (c % a.n_obs >= k) m |= 1ull << c;
        prm.colmask[k] = m;
    }
    for (int c = 0; c < R; ++c)
        if (c % a.n_obs == a.n_obs - 1) prm.lastmask |= 1ull << c;
    const int64_t cap = a.sms > 0 ? a.sms : (int64_t)sm_count();
    const int64_t grid = a.P < cap ? a.P : cap;
    const int T = (a.N + kRows - 1) / kRows;
    KeyMaps kmap;
    CUtensorMap qmap, smap;
    if (!make_key_map(&kmap, a, D, kRows, &prm.ks)) return cudaErrorInvalidValue;
    if (!make_map_3d_bf16(&qmap, a.Q, D, R, a.P, D, (int64_t)R * D, R))
        return cudaErrorInvalidValue;
    const int SC = R <= 32 ? 32 : 48;
    if (resident_ring(T, SC, &prm.ns, a.fused_stats && D == 128)) {
        // s rows hi, lo for the dot warps
        if (!make_map_3d_bf16(&smap, a.s_rows, D, 16, a.P, D, (int64_t)16 * D, kSRows))
            return cudaErrorInvalidValue;
        // with the statistics folded in, s (fp32) goes where the s rows were
        prm.s32 = static_cast<float*>(a.s_rows);
        prm.ld_s = (int64_t)16 * D / 2;
        const bool st = a.fused_stats;
        if (SC == 32) {
            using RC = RCfg<D, 32>;
            auto kern = (R == 32 && a.n_obs == 8)
                            ? (st ? importance_tcr_kernel<D, 32, 8, true> : importance_tcr_kernel<D, 32, 8, false>)
                            : (st ? importance_tcr_kernel<D, 32, 0, true> : importance_tcr_kernel<D, 32, 0, false>);
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)RC::kSmemBytes);
            if (e != cudaSuccess) return e;
            kern<<<(unsigned)grid, kRThreads, RC::kSmemBytes, s>>>(kmap, qmap, smap, prm);
        } else {
            using RC = RCfg<D, 48>;
            auto kern = st ? importance_tcr_kernel<D, 48, 0, true> : importance_tcr_kernel<D, 48, 0, false>;
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)RC::kSmemBytes);
            if (e != cudaSuccess) return e;
            kern<<<(unsigned)grid, kRThreads, RC::kSmemBytes, s>>>(kmap, qmap, smap, prm);
        }
        return cudaGetLastError();
    }
    // two-pass variant: the query rows, then s (hi, lo) and zeros up to RP rows
    if (!make_map_3d_bf16(&smap, a.s_rows, D, 16, a.P, D, (int64_t)16 * D, RP - R))
        return cudaErrorInvalidValue;
    auto kern = importance_tc_kernel<D, RP>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmemBytes);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)grid, kThreads, C::kSmemBytes, s>>>(kmap, qmap, smap, prm);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const ScoreArgs& a, cudaStream_t s) {
    // the query rows plus the two rows of s, padded to the MMA's N step of 16
    return launch_t<D, 48>(a, s);
}

}  // namespace

bool importance_tc_shape_ok(const ScoreArgs& a) {
    return a.dtype == RKV_DTYPE_BF16 && (a.d == 64 || a.d == 128) &&
           a.G * a.n_obs <= kMaxQueryRows && (a.G * a.n_obs) % 8 == 0 &&
           a.N >= 2 && a.P <= 0x7fffffff;
}

bool importance_tc_supported(const ScoreArgs& a) {
    return importance_tc_shape_ok(a) && encode_fn() != nullptr;
}

bool importance_tc_resident(const ScoreArgs& a) {
    int ns = 0;
    return importance_tc_shape_ok(a) &&
           resident_ring((a.N + kRows - 1) / kRows, a.G * a.n_obs <= 32 ? 32 : 48, &ns, a.d == 128);
}

cudaError_t launch_importance_tc(const ScoreArgs& a, cudaStream_t s) {
    if (a.P == 0) return cudaSuccess;
    return a.d == 128 ? launch_d<128>(a, s) : launch_d<64>(a, s);
}

}  // namespace rkv
