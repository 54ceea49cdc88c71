// k_gram_tc_pairs.cu -- thresholded key Gram on the sm_103a tensor cores for
// long rows (2048 < N <= 4352; the N <= 2048 kernel is in k_gram_tc.cu), with
// recency protection, R and Z computed in the epilogue.  The Gram itself never
// leaves the SM.
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
//   * The problem's keys are cut into T = ceil(N/128) blocks of 128 and the
//     blocks into T2 = ceil(T/2) pairs P_m = (2m, 2m+1).  Only the upper
//     triangle is multiplied: S is symmetric, so a pair found in block (I, J),
//     J > I, counts for row i directly and for row j through a warp
//     reduce-scatter of the sub-tile's columns and one shared-memory atomic per
//     column (only in sub-tiles that hold a similar pair).  newer_j never
//     changes there because i < j.
//   * A unit of MMA work is one row block against one block pair: a 128 x 256
//     fp32 accumulator from N = 256 instructions (128 when the pair's second
//     block lies past the problem).  The tensor core reads both operands from
//     shared memory for every instruction, so the wide N keeps the operand
//     bytes per flop down, and a commit and a barrier wait per unit are spread
//     over 1024 cycles of MMA.
//   * Schedule: row pair R holds P_R as the A operand (its two blocks are the
//     two row blocks a0 = 2R, a1 = 2R+1) and meets P_R itself (the diagonal
//     pair, no load), then P_{R+2}, ..., P_{T2-1} and last P_{R+1}; P_{R+1}
//     stays in shared memory as the next row pair's A, so every key block is
//     loaded about T/4 times per problem and no A operand is ever reloaded.
//     The lower-triangle block (a1, a0) of the diagonal pair is computed but
//     not used.
//   * Shared memory holds three pair stages (64 KB at d = 128): one is the A
//     pair, the other two take the streamed pairs in turn.  The stage of each
//     load follows from the schedule alone, so the producer and the MMA issuer
//     track it in step (Ring below) without a queue in shared memory.
//   * warp 0, one lane: TMA producer (cp.async.bulk.tensor, 3-D map
//     [P][N][d], boxes of 256 rows, 128B swizzle, rows past N zero-filled).
//     No multicast.
//   * warp 1: owns all 512 TMEM columns (two 128x256 fp32 accumulators); one
//     lane issues tcgen05.mma.cta_group::1.kind::f16 (bf16 x bf16 -> fp32,
//     M = 128, N = 256, K = 16 per instruction, exact products) and
//     tcgen05.commit.
//   * warps 2..17 (512 threads, four per scheduler for latency hiding): the
//     epilogue.  Warp w reads TMEM lanes 32*(w%4).. (one accumulator row per
//     thread) and one 32-column quarter of each of the unit's two column
//     blocks, and filters each 32x32 sub-tile -- the largest accumulator of
//     the row's 32 columns (returned by the TMEM load itself, tcgen05.ld.red
//     .max) times the largest inverse norm of the 32 columns -- skipping it
//     unless some S could exceed tau (the sub-tile holding the row's own
//     column always runs).  Both reads go through one 32-register buffer; a
//     sub-tile that needs the exact path is read again, and the accumulator
//     is handed back after the last read.  The exact path is branch-free: a
//     per-lane hit mask, row sums in registers, popc for the newer count.
//     Inverse norms are read from the workspace (L1-resident) and handed
//     between lanes by shuffle (the tensor core's operand reads keep the
//     shared-memory pipe busy); their per-chunk maxima sit in shared memory,
//     taken one problem ahead.
//   * Row-side partials (sum of above-tau S, count of newer similar tokens)
//     of the four column quarters meet in shared memory through atomics once
//     per row pair; the count is kept as one saturating byte per row (exact
//     for beta <= 63), so R and Z are written once per problem, with no
//     barrier per row block.
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

constexpr int kRows = 128;                 // rows (and columns) of one block
constexpr int kPairRows = 2 * kRows;       // rows of one block pair
constexpr int kChunkElems = 64;            // bf16 elements per 128-byte swizzle row
constexpr int kChunkBytes = kPairRows * 128;  // one [256 x 64] bf16 TMA box
constexpr int kMaxBlocks = 34;             // N <= 4352
constexpr int kEpiWarps = 16;
constexpr int kEpiThreads = 32 * kEpiWarps;
constexpr int kColGroups = kEpiWarps / 4;    // warps sharing one TMEM lane quarter
constexpr int kNewerCap = 255 / kColGroups;  // per-group cap of the newer count
constexpr int kThreads = 64 + kEpiThreads;   // producer warp, MMA warp, epilogue
constexpr uint32_t kTmemCols = 512;          // all of TMEM: two 128x256 accumulators
constexpr int kAccBufs = 2;
constexpr int kStages = 3;                   // pair stages: the A pair and two streamed

template <int D>
struct Cfg {
    static constexpr int KC = D / kChunkElems;  // swizzle chunks per row
    static constexpr int kStageBytes = KC * kChunkBytes;
    static constexpr int kMaxRows = kMaxBlocks * kRows;
    static constexpr size_t kSimOff = (size_t)kStages * kStageBytes;
    static constexpr size_t kNewerOff = kSimOff + sizeof(int) * kMaxRows;
    static constexpr size_t kInvMaxOff = kNewerOff + kMaxRows;  // one byte per row
    static constexpr size_t kBarOff = kInvMaxOff + 2 * sizeof(float) * kMaxBlocks * 4;
    static constexpr int kNumBars = 2 * kStages + 2 * kAccBufs + 2;
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

constexpr uint32_t kIdesc256 = idesc_bf16(kRows, kPairRows);
constexpr uint32_t kIdesc128 = idesc_bf16(kRows, kRows);

// Fixed-point scale of the shared-memory similarity sums (integer atomics are
// native in shared memory): a similarity is stored in units of 2^-18, so a row
// sum of up to 4352 similarities fits in 31 bits and each addition rounds by
// at most 2^-19.
constexpr float kSimScale = 262144.0f;

// Which pair stage each load of the schedule uses.  a holds the row pair's A
// operand; f and s take its streamed pairs in turn, f first (f was freed
// earlier: it held the previous row pair's second-to-last stream, s held the
// previous A).  The producer and the MMA issuer run the same sequence of
// calls, so they agree on every stage without exchanging it.
struct Ring {
    int a = 2, f = 0, s = 1;
    // the problem's first pair P_0 becomes the A operand of row pair 0
    RKV_DEV int start_problem() {
        const int st = f;
        f = s;
        s = a;
        a = st;
        return st;
    }
    RKV_DEV int stream(int k) const { return (k & 1) ? s : f; }
    // after a row pair that streamed n > 0 pairs: the last one is the next A
    RKV_DEV void end_row_pair(int n) {
        if (n <= 0) return;
        const int last = ((n - 1) & 1) ? s : f;
        const int other = ((n - 1) & 1) ? f : s;
        s = a;
        f = other;
        a = last;
    }
};

// The pair streamed k-th (of n) in row pair R: P_{R+2} .. P_{T2-1}, then P_{R+1}.
RKV_DEV int streamed_pair(int R, int k, int n) { return k < n - 1 ? R + 2 + k : R + 1; }

struct RowCtx {
    float inv_i;    // the row's inverse norm (0 past N)
    float thr;      // tau / inv_i: a raw accumulator above it is above tau
};

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

RKV_DEV void prefetch_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<uint64_t>(p)));
}

RKV_DEV float4 inv4(const float* inv, int j4, int ld) {
    // four inverse norms from j4 on (shared memory or the workspace); past the
    // row's pitch (the last chunk of a problem whose N is not a multiple of
    // 32) zeros, which no pair passes
    return j4 + 4 <= ld ? *reinterpret_cast<const float4*>(inv + j4) : make_float4(0.f, 0.f, 0.f, 0.f);
}

// Whether a sub-tile can hold a pair above tau (for the whole warp): the
// row's largest accumulator times the chunk's largest inverse norm against
// tau / inv_i; the sub-tile holding the row's own column always runs (S_ii >
// tau), and so does every sub-tile when tau <= 0.
RKV_DEV bool subtile_hot(float rmax, float im, const RowCtx& rc, bool diag, int cq, int q,
                         bool tau_pos) {
    // (rmax <= 0 never passes: thr > 0)
    const bool hot = !tau_pos || (diag && cq == q) || rmax * im > rc.thr;
    return __any_sync(0xffffffffu, hot);
}

// The exact path of a sub-tile that subtile_hot passed: r holds the raw
// accumulators k_i . k_j of columns jb .. jb+31 (overwritten).  Returns the
// row's above-tau similarity sum over the sub-tile and adds its count of newer
// similar tokens to *newer; for J > I the column side goes to s_sim through
// the warp's reduce-scatter.  Columns past N and the row's own column never
// count (for tau > 0 the zero-filled rows past N could not pass anyway).
RKV_DEV float subtile(uint32_t (&r)[32], const float* inv, int* s_sim,
                      const RowCtx& rc, bool diag, int cq, int q, int jb, int N, int lane,
                      int* newer) {
    const int nv = N - jb;  // columns of the chunk before N
    uint32_t allowed = nv >= 32 ? 0xffffffffu : (nv <= 0 ? 0u : (1u << nv) - 1u);
    if (diag && cq == q) allowed &= ~(1u << lane);  // the row's own column
    // the hits first: the filter's bound is loose, and most chunks it passes
    // hold no pair above tau.  Lane e holds the inverse norm of column jb + e
    // (one coalesced read) and hands it to the others by shuffle: the tensor
    // core's operand reads keep the shared-memory pipe busy, the shuffle
    // network is free.  r[e] becomes k_i . khat_j.
    const float iv_lane = lane < nv ? inv[jb + lane] : 0.f;
    uint32_t hits = 0;
#pragma unroll
    for (int e = 0; e < 32; ++e) {
        const float t = __uint_as_float(r[e]) * __shfl_sync(0xffffffffu, iv_lane, e);
        r[e] = __float_as_uint(t);
        hits |= (t > rc.thr) ? (1u << e) : 0u;
    }
    hits &= allowed;
    if (!__any_sync(0xffffffffu, hits != 0u)) return 0.f;
    float rs = 0.f;  // the row's hits before inv_i
#pragma unroll
    for (int e = 0; e < 32; ++e) {
        const float t = __uint_as_float(r[e]);
        const bool hit = (hits >> e) & 1u;
        rs += hit ? t : 0.f;
        // S_ij of the hits, in the registers of the raw values
        r[e] = __float_as_uint(hit ? t * rc.inv_i : 0.f);
    }
    if (!diag) {
        // column side: lane L adds column jb+L over the warp's rows
        const float cs = warp_column_sums_bits(r, lane);
        if (cs != 0.f) atomicAdd(&s_sim[jb + lane], __float2int_rn(cs * kSimScale));
        *newer += __popc(hits);  // every column is newer
    } else {
        // in a diagonal block the chunks right of the row's own hold newer
        // tokens, and in its own chunk the columns after the row
        const uint32_t nm = cq > q ? 0xffffffffu
                                   : (cq < q || lane == 31 ? 0u : (0xffffffffu << (lane + 1)));
        *newer += __popc(hits & nm);
    }
    return rs * rc.inv_i;
}

// ---------------------------------------------------------------- kernel --
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
gram_tc_pairs_kernel(const __grid_constant__ KeyMaps tmap, const Params prm) {
    using C = Cfg<D>;
    constexpr int kMaxRows = C::kMaxRows;
    constexpr int MB = kMaxBlocks;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    // pair stage t: KC chunks of [256 rows x 128 B]; block 2m at rows 0..127,
    // block 2m+1 at rows 128..255 of each chunk
    uint8_t* sP = smem;
    // above-tau similarity sums per row, fixed point (kSimScale units)
    int* s_sim = reinterpret_cast<int*>(smem + C::kSimOff);            // [kMaxRows]
    // newer-similar counts, one saturating byte per row, four rows per word
    unsigned int* s_newer = reinterpret_cast<unsigned int*>(smem + C::kNewerOff);
    float* s_invmax = reinterpret_cast<float*>(smem + C::kInvMaxOff);  // [2][MB*4]
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
    uint64_t* full = bars;
    uint64_t* empty = full + kStages;
    uint64_t* acc_full = empty + kStages;
    uint64_t* acc_empty = acc_full + kAccBufs;
    uint64_t* epi_bar = acc_empty + kAccBufs;
    uint64_t* drain_bar = epi_bar + 1;
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(drain_bar + 1);
    volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int N = prm.N;
    const int T = (N + kRows - 1) / kRows;
    const int T2 = (T + 1) / 2;  // block pairs (and row pairs) per problem

    if (threadIdx.x == 0) {
        for (int t = 0; t < kStages; ++t) {
            mbar_init(&full[t], 1);
            mbar_init(&empty[t], 1);
        }
        for (int t = 0; t < kAccBufs; ++t) {
            mbar_init(&acc_full[t], 1);
            mbar_init(&acc_empty[t], kEpiWarps);
        }
        mbar_init(epi_bar, kEpiWarps);
        mbar_init(drain_bar, 1);
        *s_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        prefetch_key_maps(&tmap);
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
            Ring ring;
            uint32_t use[kStages] = {0u, 0u, 0u};
            bool ok = true;
            auto load_pair = [&](int st, int64_t p, int m) {
                if (!(ok = mbar_wait(&empty[st], (use[st] & 1u) ^ 1u, s_abort))) return;
                mbar_arrive_expect_tx(&full[st], C::kStageBytes);
                load_key_rows(sP + st * C::kStageBytes, kChunkBytes, C::KC, &tmap, &full[st], p,
                              m * kPairRows, kPairRows, prm.ks);
                ++use[st];
            };
            for (int64_t p = blockIdx.x; ok && p < prm.P; p += gridDim.x) {
                load_pair(ring.start_problem(), p, 0);
                for (int R = 0; ok && R < T2; ++R) {
                    const int n = T2 - 1 - R;
                    for (int k = 0; ok && k < n; ++k) load_pair(ring.stream(k), p, streamed_pair(R, k, n));
                    ring.end_row_pair(n);
                }
            }
            if (!ok) {
                *s_abort = 1;
                set_error(prm.status, kDevErrTimeout, 1u);
            }
            // every copy issued has landed before the CTA may exit
            volatile int never = 0;
            for (int t = 0; t < kStages; ++t)
                if (use[t] > 0) mbar_wait(&full[t], (use[t] - 1u) & 1u, &never);
        }
    } else if (warp == 1) {
        // ----------------------------------------------------- MMA issuer --
        if (lane == 0) {
            Ring ring;
            uint32_t use[kStages] = {0u, 0u, 0u};
            uint32_t kacc = 0;
            bool ok = true;
            auto wait_full = [&](int st) {
                ok = mbar_wait(&full[st], use[st] & 1u, s_abort);
                ++use[st];
            };
            // one unit: row block (A at a_base) against the pair at b_base
            auto unit = [&](const uint8_t* a_base, const uint8_t* b_base, uint32_t idesc) {
                const int acc = kacc & 1;
                if (!(ok = mbar_wait(&acc_empty[acc], ((kacc >> 1) & 1u) ^ 1u, s_abort))) return;
                tc_fence_after();
                const uint32_t d_tmem = tmem + (uint32_t)(acc * kPairRows);
#pragma unroll
                for (int c = 0; c < C::KC; ++c) {
                    const uint64_t ad = sdesc_sw128(a_base + c * kChunkBytes);
                    const uint64_t bd = sdesc_sw128(b_base + c * kChunkBytes);
#pragma unroll
                    for (int k = 0; k < kChunkElems / 16; ++k)
                        mma_bf16(d_tmem, ad + 2 * k, bd + 2 * k, idesc, (c | k) != 0);
                }
                mma_commit(&acc_full[acc]);
                ++kacc;
            };
            for (int64_t p = blockIdx.x; ok && p < prm.P; p += gridDim.x) {
                const int st0 = ring.start_problem();
                wait_full(st0);
                for (int R = 0; ok && R < T2; ++R) {
                    const int n = T2 - 1 - R;
                    const bool has1 = 2 * R + 1 < T;
                    const uint8_t* A = sP + ring.a * C::kStageBytes;
                    // the diagonal pair: B is the A stage itself
                    unit(A, A, has1 ? kIdesc256 : kIdesc128);
                    if (ok && has1) unit(A + kRows * 128, A, kIdesc256);
                    for (int k = 0; ok && k < n; ++k) {
                        const int st = ring.stream(k);
                        wait_full(st);
                        if (!ok) break;
                        const int m = streamed_pair(R, k, n);
                        const uint32_t idesc = 2 * m + 1 < T ? kIdesc256 : kIdesc128;
                        const uint8_t* B = sP + st * C::kStageBytes;
                        unit(A, B, idesc);
                        if (ok) unit(A + kRows * 128, B, idesc);
                        // streamed pairs are free after their two units; the last
                        // one is the next row pair's A
                        if (ok && k < n - 1) mma_commit(&empty[st]);
                    }
                    if (!ok) break;
                    mma_commit(&empty[ring.a]);  // this row pair's A, after its last unit
                    ring.end_row_pair(n);
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
        const int et = threadIdx.x - 64;      // 0..511
        const int ew = warp - 2;              // epilogue warp 0..15
        const int q = warp & 3;               // TMEM lane quarter of this warp
        const int cg = ew >> 2;               // which column quarter of each block
        const int row = q * 32 + lane;        // accumulator row of this thread
        const uint32_t t_lane = tmem + ((uint32_t)(q * 32) << 16);
        const int Cn = N - prm.n_obs;
        const bool tau_pos = prm.tau > 0.f;
        const float inv_nm1 = 1.0f / (float)(N - 1);
        const int ld = (int)prm.ld_ws;
        uint32_t kacc = 0, kepi = 0;
        bool ok = true;
        for (int x = et; x < kMaxRows; x += kEpiThreads) s_sim[x] = 0;
        for (int x = et; x < kMaxRows / 4; x += kEpiThreads) s_newer[x] = 0u;
        // largest inverse norm of each 32-column chunk of a problem (inverse
        // norms at inv, pitch ldi) into buffer b: a warp per block of four
        // chunks, a float4 per lane, the maximum over each group of eight lanes
        auto chunk_maxima = [&](const float* inv, int ldi, int b) {
            for (int g = ew; g < T; g += kEpiWarps) {
                const int j = g * kRows + 4 * lane;
                const float4 v = inv4(inv, j, ldi);
                float m = j < N ? v.x : -INFINITY;
                m = fmaxf(m, j + 1 < N ? v.y : -INFINITY);
                m = fmaxf(m, j + 2 < N ? v.z : -INFINITY);
                m = fmaxf(m, j + 3 < N ? v.w : -INFINITY);
#pragma unroll
                for (int o = 4; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
                if ((lane & 7) == 0) s_invmax[b * MB * 4 + g * 4 + (lane >> 3)] = m;
            }
        };
        auto global_inv = [&](int p) { return prm.inv_norm + (int64_t)p * ld; };
        if (blockIdx.x < prm.P) chunk_maxima(global_inv(blockIdx.x), ld, 0);
        int ib = 0;
        for (int p = blockIdx.x; ok && p < prm.P; p += gridDim.x, ib ^= 1) {
            // the finalize inputs of this problem, on their way to L2
            {
                const int lines = (N + 31) / 32;  // 128-byte lines of one row
                if (et < lines)
                    prefetch_l2(prm.sum_s + (int64_t)p * ld + et * 32);
                else if (et < 2 * lines)
                    prefetch_l2(prm.I + (int64_t)p * prm.ld_out + (et - lines) * 32);
            }
            // inverse norms from the workspace (L1-resident); their chunk
            // maxima were taken one problem ahead
            const float* inv = global_inv(p);
            const float* invmax = s_invmax + ib * MB * 4;
            // this problem's chunk maxima are in shared memory, and the previous
            // problem's s_sim / s_newer entries are zero again, once every
            // epilogue warp is here
            mbar_arrive_warp(epi_bar);
            ok = __all_sync(0xffffffffu, mbar_wait(epi_bar, kepi & 1, s_abort));
            ++kepi;
            if (!ok) break;
            // the next problem's chunk maxima, into the other buffer
            if (p + gridDim.x < prm.P) chunk_maxima(global_inv(p + gridDim.x), ld, ib ^ 1);
            for (int R = 0; ok && R < T2; ++R) {
                const int a0 = 2 * R, a1 = 2 * R + 1;
                const int n = T2 - 1 - R;
                const int i0 = a0 * kRows + row, i1 = i0 + kRows;
                RowCtx rc0, rc1;
                rc0.inv_i = i0 < N ? inv[i0] : 0.f;
                rc1.inv_i = i1 < N ? inv[i1] : 0.f;
                rc0.thr = i0 < N ? prm.tau / rc0.inv_i : INFINITY;
                rc1.thr = i1 < N ? prm.tau / rc1.inv_i : INFINITY;
                float sim0 = 0.f, sim1 = 0.f;
                int newer0 = 0, newer1 = 0;
                // units of the row pair in MMA order: the diagonal pair (a0, then
                // a1 when it exists), then each streamed pair (a0, a1)
                const int nunits = (a1 < T ? 2 : 1) + 2 * n;
                for (int u = 0; ok && u < nunits; ++u) {
                    const int h = a1 < T ? (u & 1) : 0;
                    const int m = u < 2 ? R : streamed_pair(R, (u - 2) >> 1, n);
                    const int I = a0 + h;
                    const int J0 = 2 * m, J1 = 2 * m + 1;
                    // the warp's column quarter rotates with the blocks so that
                    // the hot sub-tiles next to the diagonal do not always land
                    // on the same warps
                    const int cq0 = (cg + I + J0) & 3, cq1 = (cq0 + 1) & 3;
                    const int acc = kacc & 1;
                    ok = __all_sync(0xffffffffu,
                                    mbar_wait(&acc_full[acc], (kacc >> 1) & 1u, s_abort));
                    if (!ok) break;
                    tc_fence_after();
                    ++kacc;
                    // the two sub-tiles' row maxima first, through one register
                    // buffer (the values of the second stay in r); a sub-tile that
                    // needs the exact path is read again, and the accumulator is
                    // handed back after the last read
                    uint32_t r[32];
                    float rmax0, rmax1;  // the row's largest accumulator of each chunk
                    const uint32_t tcol = t_lane + (uint32_t)(acc * kPairRows);
                    tmem_ld_32cols_max(tcol + (uint32_t)(cq0 * 32), r, rmax0);
                    tmem_ld_wait();
                    tmem_ld_32cols_max(tcol + (uint32_t)(kRows + cq1 * 32), r, rmax1);
                    tmem_ld_wait();
                    const RowCtx rc = h ? rc1 : rc0;
                    // (a1, a0) of the diagonal pair is below the diagonal: unused
                    const bool hot0 = J0 >= I && subtile_hot(rmax0, invmax[J0 * 4 + cq0], rc,
                                                             J0 == I, cq0, q, tau_pos);
                    const bool hot1 = J1 < T && subtile_hot(rmax1, invmax[J1 * 4 + cq1], rc,
                                                            J1 == I, cq1, q, tau_pos);
                    if (!hot0) {
                        tc_fence_before();
                        mbar_arrive_warp(&acc_empty[acc]);  // the accumulator is in registers now
                        if (!hot1) continue;
                    }
                    float rs = 0.f;
                    int nw = 0;
#pragma unroll 1
                    for (int pass = hot0 ? 0 : 1; pass < (hot1 ? 2 : 1); ++pass) {
                        if (hot0) {
                            // r holds the second sub-tile: read the one this pass needs
                            tmem_ld_32cols(tcol + (uint32_t)(pass * kRows + (pass ? cq1 : cq0) * 32), r);
                            tmem_ld_wait();
                            if (pass == (hot1 ? 1 : 0)) {
                                tc_fence_before();
                                mbar_arrive_warp(&acc_empty[acc]);
                            }
                        }
                        const int J = pass ? J1 : J0;
                        const int cq = pass ? cq1 : cq0;
                        rs += subtile(r, inv, s_sim, rc, J == I, cq, q, J * kRows + cq * 32, N,
                                      lane, &nw);
                    }
                    if (h) {
                        sim1 += rs;
                        newer1 += nw;
                    } else {
                        sim0 += rs;
                        newer0 += nw;
                    }
                }
                if (!ok) break;
                // row-side partials of this column quarter (newer capped so
                // that the quarters' bytes cannot carry into the next row)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int i = h ? i1 : i0;
                    const float sr = h ? sim1 : sim0;
                    const int nw = h ? newer1 : newer0;
                    if (i < N) {
                        if (sr != 0.f) atomicAdd(&s_sim[i], __float2int_rn(sr * kSimScale));
                        if (nw != 0)
                            atomicAdd(&s_newer[i >> 2], (unsigned)min(nw, kNewerCap) << (8 * (i & 3)));
                    }
                }
            }
            if (!ok) break;
            // every contribution to this problem is in shared memory after this
            mbar_arrive_warp(epi_bar);
            ok = __all_sync(0xffffffffu, mbar_wait(epi_bar, kepi & 1, s_abort));
            ++kepi;
            if (!ok) break;
            // finalize this thread's rows, four at a time (their inputs loaded
            // together), then clear exactly what it read
            for (int i0 = et; i0 < N; i0 += 4 * kEpiThreads) {
                float tot[4], imp[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int i = i0 + u * kEpiThreads;
                    tot[u] = i < Cn ? prm.sum_s[(int64_t)p * ld + i] : 0.f;
                    imp[u] = i < Cn ? prm.I[(int64_t)p * prm.ld_out + i] : 0.f;
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int i = i0 + u * kEpiThreads;
                    if (i >= N) break;
                    const float sim_i = (float)s_sim[i] * (1.0f / kSimScale);
                    const int nw = (int)((s_newer[i >> 2] >> (8 * (i & 3))) & 0xffu);
                    float rr = 0.f, z = INFINITY;
                    if (i < Cn) {
                        rr = (tot[u] - (nw < prm.beta ? sim_i : 0.f)) * inv_nm1;
                        z = prm.lambda * imp[u] - (1.0f - prm.lambda) * rr;
                    }
                    if (prm.R) prm.R[(int64_t)p * prm.ld_out + i] = rr;
                    prm.Z[(int64_t)p * prm.ld_out + i] = z;
                    s_sim[i] = 0;
                }
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

template <int D>
cudaError_t launch_t(const ScoreArgs& a, cudaStream_t s) {
    using C = Cfg<D>;
    static_assert(C::kSmemBytes <= 232448, "shared memory over the per-CTA limit");
    KeyMaps map;
    KeySource ks;
    if (!make_key_map(&map, a, D, kPairRows, &ks)) return cudaErrorInvalidValue;
    Params prm{a.P,      a.N,     a.n_obs,   a.beta, a.lambda, a.tau,    a.inv_norm,
               a.sum_s,  a.ld_ws, a.I,       a.R,    a.Z,      a.ld_out, a.status};
    prm.ks = ks;
    auto kern = gram_tc_pairs_kernel<D>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmemBytes);
    if (e != cudaSuccess) return e;
    const int64_t sms = a.sms > 0 ? a.sms : sm_count();
    const int64_t grid = a.P < sms ? a.P : sms;
    kern<<<(unsigned)grid, kThreads, C::kSmemBytes, s>>>(map, prm);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gram_tc_pairs(const ScoreArgs& a, cudaStream_t s) {
    if (a.P == 0) return cudaSuccess;
    return a.d == 128 ? launch_t<128>(a, s) : launch_t<64>(a, s);
}

}  // namespace rkv
