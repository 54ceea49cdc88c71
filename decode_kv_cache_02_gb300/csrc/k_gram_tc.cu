// k_gram_tc.cu -- thresholded key Gram on the sm_103a tensor cores (tcgen05,
// TMEM accumulators, TMA-fed shared memory), with recency protection, R and
// Z computed in the epilogue, for N <= 2048 (longer rows: k_gram_tc_pairs.cu).
// The Gram itself never leaves the SM.
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
//     directly and for row j through a warp reduce-scatter of the sub-tile's
//     columns and one shared-memory atomic per column (only in sub-tiles that
//     hold a similar pair).  newer_j never changes there because i < j.
//   * warp 0, one lane: TMA producer.  Block I (the A operand, 2 slots) and
//     blocks J > I (the B operand, a ring of stages) are fetched with
//     cp.async.bulk.tensor (3-D map [P][N][d], 128B swizzle, rows past N
//     zero-filled); the problem's inverse norms arrive by cp.async.bulk into a
//     double buffer one problem ahead.  No multicast.
//   * warp 1: owns all 512 TMEM columns (two 128x256 fp32 accumulators); one
//     lane issues tcgen05.mma.cta_group::1.kind::f16 (bf16 x bf16 -> fp32,
//     M = 128, N = 256 -- two column blocks per instruction -- K = 16 per
//     instruction, exact products) and tcgen05.commit.
//   * warps 2..17 (512 threads, four per scheduler for latency hiding): the
//     epilogue.  Warp w reads TMEM lanes 32*(w%4).. (one accumulator row per
//     thread) and one 32-column quarter of the tile, then filters the 32x32
//     sub-tile -- the largest accumulator of the row's 32 columns (returned by
//     the TMEM load itself, tcgen05.ld.red .max) times the largest inverse
//     norm of the 32 columns -- and skips the sub-tile unless some S could
//     exceed tau (the sub-tile holding the row's own column always runs).  The
//     exact path is branch-free: a per-lane hit mask, row sums in registers,
//     popc for the newer count.
//   * Row-side partials (sum of above-tau S, count of newer similar tokens)
//     of the two column halves meet in shared memory through atomics; the
//     count is kept as one saturating byte per row (exact for beta <= 63), so
//     R and Z are written once per problem, with no barrier per row block.
//   * Every mbarrier wait is bounded; on timeout the kernel records
//     kDevErrTimeout in the device status, stops issuing work, waits (bounded)
//     for its own copies and MMAs in flight, frees its TMEM and returns.
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

constexpr int kRows = 128;                // rows (and columns) of one Gram tile
constexpr int kChunkElems = 64;           // bf16 elements per 128-byte swizzle row
constexpr int kChunkBytes = kRows * 128;  // one [128 x 64] bf16 TMA box
constexpr int kMaxBlocksLarge = 34;       // N <= 4352
constexpr int kMaxBlocksSmall = 16;       // N <= 2048: room for one more B stage
constexpr int kEpiWarps = 16;
constexpr int kEpiThreads = 32 * kEpiWarps;
constexpr int kColGroups = kEpiWarps / 4;        // warps sharing one TMEM lane quarter
constexpr int kChunksPerWarp = 4 / kColGroups;   // 32-column chunks per warp per tile
constexpr int kNewerCap = 255 / kColGroups;      // per-group cap of the newer count
constexpr int kThreads = 64 + kEpiThreads;  // producer warp, MMA warp, epilogue
constexpr int kDotWarps = 2;  // with the statistics folded into importance: k_i . s
constexpr uint32_t kTmemCols = 512;  // all of TMEM: 4 accumulators of 128 columns or 2 of 256
constexpr int kPrefetch = 5;  // finalize rows per thread loaded at problem start (N <= 1280)

// W: column blocks per tile.  A tile multiplies row block I with W column
// blocks J0 .. J0+W-1 at once (one MMA of N = 128 W), so the MMA issuer's
// fixed cost per tile -- barrier waits and commits between tiles, during which
// the tensor pipe idles because issuing an MMA blocks until the pipe takes it
// -- is spread over W blocks.
template <int D, int MB, int W>
struct Cfg {
    static constexpr int kMaxBlocks = MB;
    static constexpr int kInvFloats = MB * kRows;
    static constexpr int KC = D / kChunkElems;  // swizzle chunks per row block
    static constexpr int kBlockBytes = KC * kChunkBytes;
    static constexpr int kAccBufs = 4 / W;      // accumulators of 128 W columns
    static constexpr int kAStages = 2;
    // B stages of W blocks each (the same shared memory as 3 or 4 single blocks)
    static constexpr int kBStages =
        ((D == 128 ? 3 : 6) + (MB <= kMaxBlocksSmall ? (D == 128 ? 1 : 2) : 0)) / W;
    static constexpr int kBStageBytes = W * kBlockBytes;
    static constexpr int kBChunkBytes = W * kChunkBytes;  // one chunk of W blocks
    static constexpr size_t kInvOff = (size_t)kAStages * kBlockBytes + (size_t)kBStages * kBStageBytes;
    static constexpr size_t kSimOff = kInvOff + 2 * sizeof(float) * kInvFloats;
    static constexpr size_t kNewerOff = kSimOff + sizeof(float) * kInvFloats;
    static constexpr size_t kInvMaxOff = kNewerOff + kInvFloats;  // one byte per row
    static constexpr size_t kBarOff = kInvMaxOff + 2 * sizeof(float) * kMaxBlocks * 4;
    static constexpr int kNumBars = 2 * kAStages + 2 * kBStages + 2 * 4 + 4 + 2 + 4;
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
    KeySource ks;  // contiguous keys, or the paged pool read through the table
};

constexpr uint32_t kIdesc = idesc_bf16(kRows, kRows);
constexpr uint32_t kIdesc2 = idesc_bf16(kRows, 2 * kRows);

// Fixed-point scale of the shared-memory similarity sums (integer atomics are
// native in shared memory): a similarity is stored in units of 2^-18, so a row
// sum of up to 4352 similarities fits in 31 bits and each addition rounds by
// at most 2^-19.
constexpr float kSimScale = 262144.0f;

// Reduce-scatter over the warp of fp32 values kept as bits in v (the raw
// accumulator registers, reused): on return, lane L holds in v[0] the sum over
// all lanes of their v[L].
RKV_DEV float warp_column_sums_bits(uint32_t (&v)[32], int lane) {
#pragma unroll
    for (int w = 16; w >= 1; w >>= 1) {
        const bool upper = (lane & w) != 0;
#pragma unroll
        for (int k = 0; k < w; ++k) {
            const float send = __uint_as_float(upper ? v[k] : v[k + w]);
            const float keep = __uint_as_float(upper ? v[k + w] : v[k]);
            v[k] = __float_as_uint(keep + __shfl_xor_sync(0xffffffffu, send, w));
        }
    }
    return __uint_as_float(v[0]);
}

RKV_DEV void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// ---------------------------------------------------------------- kernel --
// kDot: two more warps complete sum_i = inv_i (k_i . s) - |khat_i|^2 from each
// row block while it sits in shared memory as the A operand (the importance
// kernel then takes the key statistics and no pass over K is spent on them).
template <int D, int MB, int W, bool kDot>
__global__ void __launch_bounds__(kThreads + (kDot ? 32 * kDotWarps : 0), 1)
gram_tc_kernel(const __grid_constant__ KeyMaps tmap, const __grid_constant__ KeyMaps bmap,
               const Params prm, const float* __restrict__ s32) {
    using C = Cfg<D, MB, W>;
    constexpr int kAccBufs = C::kAccBufs;
    constexpr int kMaxBlocks = C::kMaxBlocks;
    constexpr int kInvFloats = C::kInvFloats;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sA = smem;
    uint8_t* sB = sA + C::kAStages * C::kBlockBytes;
    float* s_inv = reinterpret_cast<float*>(smem + C::kInvOff);        // [2][kInvFloats]
    // above-tau similarity sums per row, fixed point (kSimScale units)
    int* s_sim = reinterpret_cast<int*>(smem + C::kSimOff);            // [kInvFloats]
    // newer-similar counts, one saturating byte per row, four rows per word
    unsigned int* s_newer = reinterpret_cast<unsigned int*>(smem + C::kNewerOff);
    float* s_invmax = reinterpret_cast<float*>(smem + C::kInvMaxOff);  // [2][kMaxBlocks*4]
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
    uint64_t* a_full = bars;
    uint64_t* a_empty = a_full + C::kAStages;
    uint64_t* b_full = a_empty + C::kAStages;
    uint64_t* b_empty = b_full + C::kBStages;
    uint64_t* acc_full = b_empty + C::kBStages;
    uint64_t* acc_empty = acc_full + kAccBufs;
    uint64_t* inv_full = acc_empty + kAccBufs;  // [2]
    uint64_t* inv_empty = inv_full + 2;         // [2]
    uint64_t* epi_bar = inv_empty + 2;
    uint64_t* drain_bar = epi_bar + 1;
    // kDot: a problem's sum_i are written (sum_ready) / the epilogue has read
    // them (sum_free), one pair per problem parity
    uint64_t* sum_ready = drain_bar + 1;  // [2]
    uint64_t* sum_free = sum_ready + 2;   // [2]
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(sum_free + 2);
    volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int N = prm.N;
    const int T = (N + kRows - 1) / kRows;
    const uint32_t inv_bytes = (uint32_t)((N + 3) / 4) * 16;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kAStages; ++s) {
            mbar_init(&a_full[s], 1);
            mbar_init(&a_empty[s], kDot ? 1 + kDotWarps : 1);  // the MMAs, and the dot warps
        }
        for (int s = 0; s < C::kBStages; ++s) {
            mbar_init(&b_full[s], 1);
            mbar_init(&b_empty[s], 1);
        }
        for (int s = 0; s < kAccBufs; ++s) {
            mbar_init(&acc_full[s], 1);
            mbar_init(&acc_empty[s], kEpiWarps);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&inv_full[s], 1);
            mbar_init(&inv_empty[s], kEpiWarps);
        }
        mbar_init(epi_bar, kEpiWarps);
        mbar_init(drain_bar, 1);
        for (int t = 0; t < 2; ++t) {
            mbar_init(&sum_ready[t], kDotWarps);
            mbar_init(&sum_free[t], kEpiWarps);
        }
        *s_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        prefetch_key_maps(&tmap);
        prefetch_key_maps(&bmap);
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
            uint32_t ka = 0, kb = 0, kinv = 0;
            bool ok = true;
            // inverse norms of the first problem
            if (blockIdx.x < prm.P) {
                mbar_arrive_expect_tx(&inv_full[0], inv_bytes);
                bulk_copy_g2s(s_inv, prm.inv_norm + (int64_t)blockIdx.x * prm.ld_ws, inv_bytes,
                              &inv_full[0]);
                kinv = 1;
            }
            for (int64_t p = blockIdx.x; ok && p < prm.P; p += gridDim.x) {
                for (int I = 0; ok && I < T; ++I) {
                    const int sa = ka % C::kAStages;
                    if (!(ok = mbar_wait(&a_empty[sa], ((ka / C::kAStages) & 1) ^ 1, s_abort)))
                        break;
                    mbar_arrive_expect_tx(&a_full[sa], C::kBlockBytes);
                    load_key_rows(sA + sa * C::kBlockBytes, kChunkBytes, C::KC, &tmap, &a_full[sa], p,
                                  I * kRows, kRows, prm.ks);
                    ++ka;
                    // the column blocks of the row's tiles: J > I one at a time (the
                    // diagonal tile reuses block I), or W at a time from J = I
                    for (int J = W == 1 ? I + 1 : I; ok && J < T; J += W) {
                        const int sb = kb % C::kBStages;
                        if (!(ok = mbar_wait(&b_empty[sb], ((kb / C::kBStages) & 1) ^ 1, s_abort)))
                            break;
                        mbar_arrive_expect_tx(&b_full[sb], C::kBStageBytes);
                        load_key_rows(sB + sb * C::kBStageBytes, C::kBChunkBytes, C::KC, &bmap,
                                      &b_full[sb], p, J * kRows, W * kRows, prm.ks);
                        ++kb;
                    }
                    if (ok && I == 0 && p + gridDim.x < prm.P) {
                        // inverse norms of the next problem into the other buffer
                        const int ib = kinv & 1;
                        if (!(ok = mbar_wait(&inv_empty[ib], ((kinv >> 1) & 1) ^ 1, s_abort))) break;
                        mbar_arrive_expect_tx(&inv_full[ib], inv_bytes);
                        bulk_copy_g2s(s_inv + ib * kInvFloats,
                                      prm.inv_norm + (p + gridDim.x) * prm.ld_ws, inv_bytes,
                                      &inv_full[ib]);
                        ++kinv;
                    }
                }
            }
            if (!ok) {
                *s_abort = 1;
                set_error(prm.status, kDevErrTimeout, 1u);
            }
            // every copy issued has landed before the CTA may exit
            volatile int never = 0;
            for (uint32_t u = ka > (uint32_t)C::kAStages ? ka - C::kAStages : 0; u < ka; ++u)
                mbar_wait(&a_full[u % C::kAStages], (u / C::kAStages) & 1, &never);
            for (uint32_t u = kb > (uint32_t)C::kBStages ? kb - C::kBStages : 0; u < kb; ++u)
                mbar_wait(&b_full[u % C::kBStages], (u / C::kBStages) & 1, &never);
            for (uint32_t u = kinv > 2u ? kinv - 2 : 0; u < kinv; ++u)
                mbar_wait(&inv_full[u & 1], (u >> 1) & 1, &never);
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
                    for (int J = I; ok && J < T; J += W) {
                        const uint8_t* b_base = a_base;
                        int sb = -1;
                        if (W > 1 || J > I) {
                            sb = kb % C::kBStages;
                            if (!(ok = mbar_wait(&b_full[sb], (kb / C::kBStages) & 1, s_abort)))
                                break;
                            b_base = sB + sb * C::kBStageBytes;
                        }
                        const int acc = kacc % kAccBufs;
                        if (!(ok = mbar_wait(&acc_empty[acc], ((kacc / kAccBufs) & 1) ^ 1, s_abort)))
                            break;
                        tc_fence_after();
                        const uint32_t d_tmem = tmem + (uint32_t)(acc * W * kRows);
#pragma unroll
                        for (int c = 0; c < C::KC; ++c) {
                            const uint64_t ad = sdesc_sw128(a_base + c * kChunkBytes);
                            const uint64_t bd = sdesc_sw128(b_base + c * (W > 1 ? C::kBChunkBytes : kChunkBytes));
#pragma unroll
                            for (int k = 0; k < kChunkElems / 16; ++k)
                                mma_bf16(d_tmem, ad + 2 * k, bd + 2 * k, W > 1 ? kIdesc2 : kIdesc,
                                         (c | k) != 0);
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
    } else if (kDot && warp >= 2 + kEpiWarps) {
        // -------------------------------------------------------- dot warps --
        // rows dw * 64 + lane and + 32 of each row block, read from the A slot
        // in the MMA's order; the slot is released by the MMAs' commit and one
        // arrival per dot warp
        // kDot: s = sum_j khat_j in fp32 per problem (16 D / 2 floats apart)
        // from the importance kernel; sum_s holds |khat_i|^2, turned into
        // sum_i in place
        __shared__ float s_vec[kDotWarps][D];
        float* sum_w = const_cast<float*>(prm.sum_s);
        const int dw = warp - (2 + kEpiWarps);
        uint32_t ka = 0, kprob = 0;
        bool ok = true;
        for (int64_t p = blockIdx.x; ok && p < prm.P; p += gridDim.x, ++kprob) {
            __syncwarp();  // the previous problem's reads of s_vec are done
            for (int c = lane; c < D; c += 32) s_vec[dw][c] = s32[p * (16 * D / 2) + c];
            __syncwarp();
            for (int I = 0; ok && I < T; ++I, ++ka) {
                // inverse norms and |khat_i|^2 of the two rows, on their way
                const int i0 = I * kRows + dw * 64 + lane, i1 = i0 + 32;
                float iv[2] = {0.f, 0.f}, kh[2] = {0.f, 0.f};
                if (i0 < N) {
                    iv[0] = prm.inv_norm[p * prm.ld_ws + i0];
                    kh[0] = sum_w[p * prm.ld_ws + i0];
                }
                if (i1 < N) {
                    iv[1] = prm.inv_norm[p * prm.ld_ws + i1];
                    kh[1] = sum_w[p * prm.ld_ws + i1];
                }
                const int sa = ka % C::kAStages;
                ok = __all_sync(0xffffffffu, mbar_wait(&a_full[sa], (ka / C::kAStages) & 1, s_abort));
                if (!ok) break;
                const uint8_t* blk = sA + sa * C::kBlockBytes;
                const float d0 = row_dot_lean<C::KC>(blk, dw * 64 + lane, s_vec[dw]);
                const float d1 = row_dot_lean<C::KC>(blk, dw * 64 + 32 + lane, s_vec[dw]);
                __syncwarp();
                if (lane == 0) mbar_arrive(&a_empty[sa]);
                if (i0 < N) sum_w[p * prm.ld_ws + i0] = iv[0] * d0 - kh[0];
                if (i1 < N) sum_w[p * prm.ld_ws + i1] = iv[1] * d1 - kh[1];
            }
            if (!ok) break;
            // this problem's sum_i are in memory (release at CTA scope), once
            // the epilogue has read the ones of two problems back
            const int sb = kprob & 1;
            ok = __all_sync(0xffffffffu, mbar_wait(&sum_free[sb], ((kprob >> 1) & 1) ^ 1, s_abort));
            if (!ok) break;
            __syncwarp();
            if (lane == 0) mbar_arrive(&sum_ready[sb]);
        }
        if (!ok) {
            *s_abort = 1;
            set_error(prm.status, kDevErrTimeout, 4u);
        }
    } else {
        // ------------------------------------------------------- epilogue --
        const int et = threadIdx.x - 64;      // 0..255
        const int q = warp & 3;               // TMEM lane quarter of this warp
        const int cg = (warp - 2) >> 2;       // which column group of the 128 columns
        const int row = q * 32 + lane;        // accumulator row of this thread
        const uint32_t t_lane = tmem + ((uint32_t)(q * 32) << 16);
        const int Cn = N - prm.n_obs;
        const bool tau_pos = prm.tau > 0.f;
        const float inv_nm1 = 1.0f / (float)(N - 1);
        uint32_t kacc = 0, kepi = 0, kinv = 0, kprob = 0;
        bool ok = true;
        for (int x = et; x < kInvFloats; x += kEpiThreads) s_sim[x] = 0;
        for (int x = et; x < kInvFloats / 4; x += kEpiThreads) s_newer[x] = 0u;
        for (int64_t p = blockIdx.x; ok && p < prm.P; p += gridDim.x) {
            const int ib = kinv & 1;
            ok = __all_sync(0xffffffffu, mbar_wait(&inv_full[ib], (kinv >> 1) & 1, s_abort));
            if (!ok) break;
            const float* inv = s_inv + ib * kInvFloats;
            float* invmax = s_invmax + ib * kMaxBlocks * 4;
            // finalize inputs of this thread's first rows, loaded now, used
            // after the problem's last tile
            float pre_tot[kPrefetch], pre_imp[kPrefetch];
#pragma unroll
            for (int u = 0; u < kPrefetch; ++u) {
                const int i = et + u * kEpiThreads;
                pre_tot[u] = i < Cn ? prm.sum_s[p * prm.ld_ws + i] : 0.f;
                pre_imp[u] = i < Cn ? prm.I[p * prm.ld_out + i] : 0.f;
            }
            // largest inverse norm of each 32-column chunk: one warp per chunk
            // (a lane per column), chunks spread over the epilogue warps
            for (int x = (warp - 2); x < T * 4; x += kEpiWarps) {
                const int j = x * 32 + lane;
                float m = j < N ? inv[j] : -INFINITY;
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
                if (lane == 0) invmax[x] = m;
            }
            // the previous problem's s_sim / s_newer entries are zero again
            mbar_arrive_warp(epi_bar);
            ok = __all_sync(0xffffffffu, mbar_wait(epi_bar, kepi & 1, s_abort));
            ++kepi;
            for (int I = 0; ok && I < T; ++I) {
                const int i = I * kRows + row;
                const bool valid_i = i < N;
                const float inv_i = valid_i ? inv[i] : 0.f;
                const float thr = valid_i ? prm.tau / inv_i : INFINITY;
                float sim_row = 0.f;
                int newer = 0;
                for (int J0 = I; J0 < T; J0 += W) {
                  const int acc = kacc % kAccBufs;
                  ok = __all_sync(0xffffffffu,
                                  mbar_wait(&acc_full[acc], (kacc / kAccBufs) & 1, s_abort));
                  if (!ok) break;
                  tc_fence_after();
                  ++kacc;
                  // the tile's column blocks one after another, with one
                  // register buffer; the accumulator is released after the last
                  for (int w = 0; w < W; ++w) {
                    const int J = J0 + w;
                    // the warp's column group rotates with J so that the hot
                    // sub-tiles next to the diagonal do not always land on the
                    // same warps
                    const int cgr = (cg + J) % kColGroups;
                    uint32_t r[kChunksPerWarp][32];
                    float rmax[kChunksPerWarp];  // the row's largest accumulator per chunk
#pragma unroll
                    for (int h = 0; h < kChunksPerWarp; ++h)
                        tmem_ld_32cols_max(t_lane + (uint32_t)(acc * W * kRows + w * kRows +
                                                               (cgr * kChunksPerWarp + h) * 32),
                                           r[h], rmax[h]);
                    tmem_ld_wait();
                    if (w == W - 1) {
                        tc_fence_before();
                        mbar_arrive_warp(&acc_empty[acc]);  // the accumulator is in registers now
                    }
                    if (J >= T) continue;  // past the problem's last block (zero keys)
                    const bool diag = (J == I);
#pragma unroll
                    for (int h = 0; h < kChunksPerWarp; ++h) {
                        const int cq = cgr * kChunksPerWarp + h;  // 32-column chunk within the tile
                        const int chunk = J * 4 + cq;             // chunk of the problem
                        const int jb = chunk * 32;
                        if (tau_pos) {
                            // tau > 0: key rows past N are zero (TMA fill), so
                            // their S is 0 and never passes; only the row's own
                            // column needs excluding, and it lies in the chunk of
                            // a diagonal tile that matches the warp's lane
                            // quarter, at column e = lane
                            const bool self_chunk = diag && cq == q;
                            bool hot = self_chunk;  // S_ii > tau there anyway
                            // (rmax <= 0 never passes: thr > 0)
                            if (!hot) hot = rmax[h] * invmax[chunk] > thr;
                            if (__any_sync(0xffffffffu, hot)) {
                                const float4* iv4 = reinterpret_cast<const float4*>(inv + jb);
                                uint32_t hits = 0;
                                float rs = 0.f;  // the row's hits before inv_i
                                if (!diag) {
                                    // the hits first: the filter's bound is loose, and
                                    // most chunks it passes hold no pair above tau
#pragma unroll
                                    for (int e4 = 0; e4 < 8; ++e4) {
                                        const float4 w4 = iv4[e4];
                                        const float iv[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                                        for (int u = 0; u < 4; ++u) {
                                            const int e = e4 * 4 + u;
                                            const float t = __uint_as_float(r[h][e]) * iv[u];
                                            hits |= (t > thr) ? (1u << e) : 0u;
                                        }
                                    }
                                    if (__any_sync(0xffffffffu, hits != 0u)) {
#pragma unroll
                                        for (int e4 = 0; e4 < 8; ++e4) {
                                            const float4 w4 = iv4[e4];
                                            const float iv[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                                            for (int u = 0; u < 4; ++u) {
                                                const int e = e4 * 4 + u;
                                                const float t = __uint_as_float(r[h][e]) * iv[u];
                                                const bool hit = (hits >> e) & 1u;
                                                rs += hit ? t : 0.f;
                                                // S_ij of the hits, in the registers of the raw values
                                                r[h][e] = __float_as_uint(hit ? t * inv_i : 0.f);
                                            }
                                        }
                                        // column side: lane L adds column jb+L over the warp's rows
                                        const float cs = warp_column_sums_bits(r[h], lane);
                                        if (cs != 0.f)
                                            atomicAdd(&s_sim[jb + lane], __float2int_rn(cs * kSimScale));
                                        newer += __popc(hits);  // every column is newer
                                    }
                                } else if (self_chunk) {
#pragma unroll
                                    for (int e4 = 0; e4 < 8; ++e4) {
                                        const float4 w4 = iv4[e4];
                                        const float iv[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                                        for (int u = 0; u < 4; ++u) {
                                            const int e = e4 * 4 + u;
                                            const float t = __uint_as_float(r[h][e]) * iv[u];
                                            const bool hit = t > thr && e != lane;
                                            rs += hit ? t : 0.f;
                                            hits |= hit ? (1u << e) : 0u;
                                        }
                                    }
                                    newer += __popc(hits & (lane == 31 ? 0u : (0xffffffffu << (lane + 1))));
                                } else {
#pragma unroll
                                    for (int e4 = 0; e4 < 8; ++e4) {
                                        const float4 w4 = iv4[e4];
                                        const float iv[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                                        for (int u = 0; u < 4; ++u) {
                                            const int e = e4 * 4 + u;
                                            const float t = __uint_as_float(r[h][e]) * iv[u];
                                            const bool hit = t > thr;
                                            rs += hit ? t : 0.f;
                                            hits |= hit ? (1u << e) : 0u;
                                        }
                                    }
                                    // chunks right of the row's own chunk hold newer tokens
                                    if (cq > q) newer += __popc(hits);
                                }
                                sim_row += rs * inv_i;
                            }
                        } else {
                            // tau <= 0: every existing pair counts; columns past N
                            // and the row's own column are excluded one by one
                            const int e_self = diag ? i - jb : -1;
                            const int e_end = min(32, N - jb);
                            const float4* iv4 = reinterpret_cast<const float4*>(inv + jb);
                            uint32_t hits = 0;
                            float row_sum = 0.f;
#pragma unroll
                            for (int e4 = 0; e4 < 8; ++e4) {
                                const float4 w4 = iv4[e4];
                                const float iv[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                                for (int u = 0; u < 4; ++u) {
                                    const int e = e4 * 4 + u;
                                    const float t = __uint_as_float(r[h][e]) * iv[u];
                                    const bool hit = (t > thr) && (e < e_end) && (e != e_self);
                                    const float v = hit ? t * inv_i : 0.f;
                                    row_sum += v;
                                    hits |= (hit ? 1u : 0u) << e;
                                    r[h][e] = __float_as_uint(v);
                                }
                            }
                            sim_row += row_sum;
                            const uint32_t newer_mask =
                                !diag ? 0xffffffffu
                                      : (e_self >= 31 ? 0u
                                                      : (e_self < 0 ? 0xffffffffu
                                                                    : (0xffffffffu << (e_self + 1))));
                            newer += __popc(hits & newer_mask);
                            if (!diag) {
                                const float cs = warp_column_sums_bits(r[h], lane);
                                if (cs != 0.f) atomicAdd(&s_sim[jb + lane], __float2int_rn(cs * kSimScale));
                            }
                        }
                    }
                  }
                }
                if (!ok) break;
                // row-side partials of this column group (newer capped so
                // that the groups' bytes cannot carry into the next row)
                if (valid_i) {
                    if (sim_row != 0.f) atomicAdd(&s_sim[i], __float2int_rn(sim_row * kSimScale));
                    if (newer != 0)
                        atomicAdd(&s_newer[i >> 2], (unsigned)min(newer, kNewerCap) << (8 * (i & 3)));
                }
            }
            if (!ok) break;
            mbar_arrive_warp(&inv_empty[ib]);
            ++kinv;
            // every contribution to this problem is in shared memory after this
            mbar_arrive_warp(epi_bar);
            ok = __all_sync(0xffffffffu, mbar_wait(epi_bar, kepi & 1, s_abort));
            ++kepi;
            if (!ok) break;
            if (kDot) {
                // sum_i of this problem comes from the dot warps
                const int sb = kprob & 1;
                ok = __all_sync(0xffffffffu, mbar_wait(&sum_ready[sb], (kprob >> 1) & 1, s_abort));
                if (!ok) break;
#pragma unroll
                for (int u = 0; u < kPrefetch; ++u) {
                    const int i = et + u * kEpiThreads;
                    pre_tot[u] = i < Cn ? prm.sum_s[p * prm.ld_ws + i] : 0.f;
                }
                mbar_arrive_warp(&sum_free[sb]);
            }
            ++kprob;
            // finalize this thread's rows, then clear exactly what it read
            auto finalize_row = [&](int i, float tot, float imp) {
                const float sim_i = (float)s_sim[i] * (1.0f / kSimScale);
                const int nw = (int)((s_newer[i >> 2] >> (8 * (i & 3))) & 0xffu);
                float rr = 0.f, z = INFINITY;
                if (i < Cn) {
                    rr = (tot - (nw < prm.beta ? sim_i : 0.f)) * inv_nm1;
                    z = prm.lambda * imp - (1.0f - prm.lambda) * rr;
                }
                if (prm.R) prm.R[p * prm.ld_out + i] = rr;
                prm.Z[p * prm.ld_out + i] = z;
                s_sim[i] = 0;
            };
#pragma unroll
            for (int u = 0; u < kPrefetch; ++u) {
                const int i = et + u * kEpiThreads;
                if (i < N) finalize_row(i, pre_tot[u], pre_imp[u]);
            }
            for (int i = et + kPrefetch * kEpiThreads; i < N; i += kEpiThreads) {
                const float tot = i < Cn ? prm.sum_s[p * prm.ld_ws + i] : 0.f;
                const float imp = i < Cn ? prm.I[p * prm.ld_out + i] : 0.f;
                finalize_row(i, tot, imp);
            }
            // a word of s_newer holds rows 4w..4w+3, finalized by four
            // neighbouring lanes of one warp; the first of them clears it once
            // all four have read it
            __syncwarp();
            for (int i = et; i < N; i += kEpiThreads)
                if ((i & 3) == 0) s_newer[i >> 2] = 0u;
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

template <int D, int MB, int W, bool kDot>
cudaError_t launch_t(const ScoreArgs& a, cudaStream_t s) {
    using C = Cfg<D, MB, W>;
    KeyMaps map, bmap;
    KeySource ks;
    if (!make_key_map(&map, a, D, kRows, &ks)) return cudaErrorInvalidValue;
    if (!make_key_map(&bmap, a, D, W * kRows, &ks))
        return cudaErrorInvalidValue;
    Params prm{a.P,      a.N,     a.n_obs,   a.beta, a.lambda, a.tau,    a.inv_norm,
               a.sum_s,  a.ld_ws, a.I,       a.R,    a.Z,      a.ld_out, a.status};
    prm.ks = ks;

    auto kern = gram_tc_kernel<D, MB, W, kDot>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmemBytes);
    if (e != cudaSuccess) return e;
    const int64_t sms = a.sms > 0 ? a.sms : sm_count();
    const int64_t grid = a.P < sms ? a.P : sms;
    kern<<<(unsigned)grid, kThreads + (kDot ? 32 * kDotWarps : 0), C::kSmemBytes, s>>>(map, bmap, prm, static_cast<const float*>(a.s_rows));
    return cudaGetLastError();
}

}  // namespace

bool gram_tc_shape_ok(const ScoreArgs& a) {
    return a.dtype == RKV_DTYPE_BF16 && (a.d == 64 || a.d == 128) && a.N >= 2 &&
           a.N <= kMaxBlocksLarge * kRows && a.P <= 0x7fffffff && (a.ld_ws % 4) == 0 &&
           a.beta >= 0 && a.beta <= kNewerCap;
}

bool gram_tc_supported(const ScoreArgs& a) { return gram_tc_shape_ok(a) && encode_fn() != nullptr; }

bool gram_tc_rows(const ScoreArgs& a) { return gram_tc_shape_ok(a) && a.N <= kMaxBlocksSmall * kRows; }

cudaError_t launch_gram_tc(const ScoreArgs& a, cudaStream_t s) {
    if (a.P == 0) return cudaSuccess;
    if (a.N <= kMaxBlocksSmall * kRows)
        return a.fused_stats
                   ? (a.d == 128 ? launch_t<128, kMaxBlocksSmall, 2, true>(a, s)
                                 : launch_t<64, kMaxBlocksSmall, 2, true>(a, s))
                   : (a.d == 128 ? launch_t<128, kMaxBlocksSmall, 2, false>(a, s)
                                 : launch_t<64, kMaxBlocksSmall, 2, false>(a, s));
    // longer rows: row pairs against streamed block pairs (k_gram_tc_pairs.cu)
    return launch_gram_tc_pairs(a, s);
}

}  // namespace rkv
