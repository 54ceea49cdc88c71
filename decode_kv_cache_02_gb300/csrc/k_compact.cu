// k_compact.cu -- top-k selection and compaction of the kept K/V rows, fused.
//
// R-KV review (yoonschallenge.tistory.com/1236), opening notes (the newest 8
// tokens always stay; the other tokens are scored and the best ones that fit
// the budget are kept), question 2, cause 3 (top-k over the scores, then the
// kept KV rows copied into the compacted cache) and cause 4 (re-layout of the
// KV tensor).  Ties in Z
// go to the larger (more recent) index; the kept candidates follow in
// ascending order, then the n_obs observation tokens.
//
// One CTA per problem does both steps, so the selection's latency hides behind
// the other CTAs' row copies and Z is read once:
//   select  the scores as order-preserving keys in shared memory; a histogram
//           of 256 buckets linear in the score between the problem's extremes
//           (bucket(z) never decreases with z, so every score in a higher
//           bucket is larger); only the bucket holding the k-th largest score
//           is ranked exactly (directly for up to 32 keys, else radix passes
//           over its compacted keys); a block scan in index order places each
//           kept index.
//   copy    by the TMA engine, through a ring of shared-memory stages: per
//           chunk of 32 output rows, each run of consecutive kept source rows
//           is one bulk load per tensor into the chunk's stage, and once the
//           stage is full one bulk store per tensor writes the chunk to its
//           contiguous output rows.  One warp keeps several chunks in flight
//           while the CTA's other warps have left, so a few SMs move the rows
//           at a rate that otherwise takes most of them.  In place, rows
//           before the first evicted token are skipped and the rest move in
//           ascending chunks: kept indices ascend and idx[r] >= r, so a chunk's
//           sources lie at or after its own rows and after every earlier
//           chunk's, and each chunk is stored only after its loads and those
//           of every earlier chunk have landed.
//   paged   the same chunked in-place order through the block table: kept V
//           rows move inside the pool, kept K rows come from the contiguous
//           copy the key statistics wrote (so K's reads never meet its
//           writes); every block id is checked before it is used.
#include "rkv_common.cuh"
#include "rkv_internal.h"
#include "rkv_paged.cuh"
#include "rkv_variant.cuh"
#include "tcgen05.cuh"
#include "../../include/rkv.h"

namespace rkv {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kCopyVecs = 8;  // vectors per thread per tensor in flight

RKV_DEV float from_orderable(uint32_t u) {
    return __uint_as_float((u & 0x80000000u) ? (u & 0x7fffffffu) : ~u);
}

// Exclusive scan of one int per thread over the block; returns the thread's
// prefix and the block total.
__device__ int block_scan(int v, int* s_warp, int* total) {
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
        if (lane < kWarps) s_warp[lane] = w;
    }
    __syncthreads();
    const int base = warp > 0 ? s_warp[warp - 1] : 0;
    *total = s_warp[kWarps - 1];
    __syncthreads();
    return base + x - v;
}

// The bin of the krem-th largest key in hist[0..255] (one warp): the digit,
// the rank left inside the bin and the bin's count, in every lane.
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

RKV_DEV int bucket_of(float z, float zmin, float scale) {
    return min(255, max(0, (int)((z - zmin) * scale)));
}

struct SelShared {
    uint32_t hist[256];
    float red[2][kWarps];
    int warp[kWarps];
    uint32_t m, uk, eq, need;
};

// The kk-th largest (kk >= 1) of the C keys: uk, and eq_cut such that the
// keys equal to uk of rank >= eq_cut among them (in index order) are in the
// top kk (ties go to the larger index).  zmin / zmax are this thread's bounds
// of the keys' finite float values; `list` (C entries) is scratch.  Every
// thread calls it; it ends with a barrier.
__device__ __forceinline__ void kth_largest(const uint32_t* keys, uint32_t* list, int C, int kk,
                                            float zmin, float zmax, SelShared& sh, uint32_t& uk_out,
                                            uint32_t& eq_cut_out) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int b = tid; b < 256; b += kThreads) sh.hist[b] = 0u;
    if (tid == 0) sh.m = 0u;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        zmin = fminf(zmin, __shfl_xor_sync(0xffffffffu, zmin, o));
        zmax = fmaxf(zmax, __shfl_xor_sync(0xffffffffu, zmax, o));
    }
    if (lane == 0) {
        sh.red[0][warp] = zmin;
        sh.red[1][warp] = zmax;
    }
    __syncthreads();
    zmin = sh.red[0][0];
    zmax = sh.red[1][0];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) {
        zmin = fminf(zmin, sh.red[0][w]);
        zmax = fmaxf(zmax, sh.red[1][w]);
    }
    const float range = zmax - zmin;
    const float scale = range > 0.f ? 255.5f / range : 0.f;
    for (int i = tid; i < C; i += kThreads)
        atomicAdd(&sh.hist[bucket_of(from_orderable(keys[i]), zmin, scale)], 1u);
    __syncthreads();
    uint32_t krem = (uint32_t)kk, bucket = 0, m = 0;
    if (warp == 0) find_bin(sh.hist, krem, bucket, m);
    if (tid == 0) sh.uk = bucket;
    __syncthreads();
    bucket = sh.uk;
    for (int i = tid; i < C; i += kThreads) {
        const uint32_t u = keys[i];
        if ((uint32_t)bucket_of(from_orderable(u), zmin, scale) == bucket) list[atomicAdd(&sh.m, 1u)] = u;
    }
    __syncthreads();
    if (warp == 0) {
        // the krem-th largest of the m keys in the bucket: uk, how many keys
        // equal it and how many of those are kept
        m = sh.m;
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
            // radix passes over the bucket's keys, from the highest bit where
            // they differ
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
            while (top > 0) {
                const int shf = top >= 8 ? top - 8 : 0;
                const uint32_t dm = top >= 8 ? 255u : ((1u << top) - 1u);
                const uint32_t pm = top == 32 ? 0u : ~((1u << top) - 1u);
                __syncwarp();
#pragma unroll
                for (int b = 0; b < 8; ++b) sh.hist[lane * 8 + b] = 0u;
                __syncwarp();
                for (uint32_t x = lane; x < m; x += 32) {
                    const uint32_t u = list[x];
                    if ((u & pm) == prefix) atomicAdd(&sh.hist[(u >> shf) & dm], 1u);
                }
                __syncwarp();
                uint32_t dg;
                find_bin(sh.hist, krem, dg, eq_count);
                prefix |= dg << shf;
                top = shf;
            }
            uk = prefix;
            need_eq = krem;
        }
        if (lane == 0) {
            sh.uk = uk;
            sh.eq = eq_count;
            sh.need = need_eq;
        }
    }
    __syncthreads();
    uk_out = sh.uk;
    eq_cut_out = sh.eq - sh.need;
}

// The top kk keys given their threshold (uk, eq_cut), in index order over
// contiguous ranges per thread with block scans.  kMark: keys outside the top
// kk become 0 (below every float's key); else: their indices, ascending,
// into out[0..kk).
template <bool kMark>
__device__ __forceinline__ void take_top(uint32_t* keys, int C, uint32_t uk, uint32_t eq_cut,
                                         int kk, int32_t* out, SelShared& sh) {
    const int tid = threadIdx.x;
    const int ipt = (C + kThreads - 1) / kThreads;
    const int lo = min(C, tid * ipt), hi = min(C, lo + ipt);
    int eq_before = 0;
    if (eq_cut > 0) {
        int n_eq = 0;
        for (int i = lo; i < hi; ++i) n_eq += (keys[i] == uk);
        int eq_total;
        eq_before = block_scan(n_eq, sh.warp, &eq_total);
    }
    if constexpr (kMark) {
        int e = eq_before;
        for (int i = lo; i < hi; ++i) {
            const uint32_t u = keys[i];
            bool in = false;
            if (u > uk) in = true;
            else if (u == uk) { in = (e >= (int)eq_cut); ++e; }
            if (!in) keys[i] = 0u;
        }
        __syncthreads();
    } else {
        int n_keep = 0;
        {
            int e = eq_before;
            for (int i = lo; i < hi; ++i) {
                const uint32_t u = keys[i];
                if (u > uk) ++n_keep;
                else if (u == uk) { n_keep += (e >= (int)eq_cut); ++e; }
            }
        }
        int keep_total;
        int pos = block_scan(n_keep, sh.warp, &keep_total);
        int e = eq_before;
        for (int i = lo; i < hi; ++i) {
            const uint32_t u = keys[i];
            bool keep = false;
            if (u > uk) keep = true;
            else if (u == uk) { keep = (e >= (int)eq_cut); ++e; }
            if (keep && pos < kk) out[pos++] = i;
        }
    }
}

// ------------------------------------------------------- bulk row copy --
constexpr int kChunkRows = 32;     // output rows per stage (one per lane)
constexpr int kMaxStages = 8;
constexpr size_t kStageTarget = 112 * 1024;  // shared memory per CTA with the stages

RKV_DEV void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(tc::smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(tc::smem_u32(bar))
        : "memory");
}
RKV_DEV void bulk_store(void* dst, const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(
                     reinterpret_cast<uint64_t>(dst)),
                 "r"(tc::smem_u32(src)), "r"(bytes)
                 : "memory");
}
RKV_DEV void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// every committed store group but the newest has read its shared memory
RKV_DEV void bulk_wait_read_but_one() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
RKV_DEV void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Output rows [r0, budget) of one problem from source rows sidx[r] (one warp).
// a / b: the two tensors (b may be null), rows of rb bytes, sources n_cap rows
// per problem; stages: S buffers of kChunkRows rows per tensor, full: their
// mbarriers (count 1, fresh).  Lane 0 issues and waits for every store.
RKV_DEV void copy_rows_bulk(const int32_t* sidx, int r0, int budget, int n_cap,
                            const uint8_t* a_src, const uint8_t* b_src, uint8_t* a_dst,
                            uint8_t* b_dst, int rb, uint8_t* stages, uint64_t* full, int S,
                            volatile int* abort_flag, DeviceStatus* st) {
    const int lane = threadIdx.x & 31;
    const int nch = (budget - r0 + kChunkRows - 1) / kChunkRows;
    const int tensors = b_src ? 2 : 1;
    const size_t tbytes = (size_t)kChunkRows * rb;  // one tensor's part of a stage
    auto stage = [&](int ch) { return stages + (size_t)(ch % S) * tensors * tbytes; };
    // loads of chunk ch: lane l holds row r0 + 32 ch + l
    auto issue = [&](int ch) {
        const int r = r0 + ch * kChunkRows + lane;
        const int src = r < budget ? sidx[r] : -1;
        const bool ok = src >= 0 && src < n_cap;
        if (r < budget && !ok) set_error(st, kDevErrIndex, (unsigned)r);
        const int prev = __shfl_up_sync(0xffffffffu, src, 1);
        const bool start = ok && (lane == 0 || prev != src - 1);
        const unsigned cont = __ballot_sync(0xffffffffu, ok && !start);
        const unsigned okm = __ballot_sync(0xffffffffu, ok);
        const unsigned after = lane < 31 ? cont >> (lane + 1) : 0u;
        const int len = __ffs(~after);  // this row and the run's rows after it
        uint64_t* bar = &full[ch % S];
        if (lane == 0) tc::mbar_arrive_expect_tx(bar, (uint32_t)(__popc(okm) * rb * tensors));
        __syncwarp();
        if (start) {
            uint8_t* d = stage(ch) + (size_t)lane * rb;
            bulk_load(d, a_src + (size_t)src * rb, (uint32_t)(len * rb), bar);
            if (b_src) bulk_load(d + tbytes, b_src + (size_t)src * rb, (uint32_t)(len * rb), bar);
        }
        return okm;
    };
    unsigned okm[kMaxStages];
    const int pre = nch < S ? nch : S;
    for (int ch = 0; ch < pre; ++ch) okm[ch] = issue(ch);
    bool ok = true;
    int waited = 0;    // chunks whose loads are known to have landed
    int issued = pre;  // chunks whose loads have been issued
    for (int ch = 0; ch < nch; ++ch) {
        const int sl = ch % S;
        if (lane == 0) {
            ok = tc::mbar_wait(&full[sl], (uint32_t)(ch / S) & 1u, abort_flag);
            if (!ok) {
                set_error(st, kDevErrTimeout, 0x300u);
                *abort_flag = 1;
            }
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
        waited = ch + 1;
        if (lane == 0) {
            const size_t o = (size_t)(r0 + ch * kChunkRows) * rb;
            const unsigned m = okm[sl];
            if (m == 0xffffffffu || (m & (m + 1u)) == 0u) {
                // the chunk's rows are a prefix of it (the last chunk may be short)
                const uint32_t n = (uint32_t)__popc(m) * (uint32_t)rb;
                if (n) {
                    bulk_store(a_dst + o, stage(ch), n);
                    if (b_src) bulk_store(b_dst + o, stage(ch) + tbytes, n);
                }
            } else {
                for (int l = 0; l < kChunkRows; ++l)
                    if (m >> l & 1u) {
                        bulk_store(a_dst + o + (size_t)l * rb, stage(ch) + (size_t)l * rb, rb);
                        if (b_src)
                            bulk_store(b_dst + o + (size_t)l * rb,
                                       stage(ch) + tbytes + (size_t)l * rb, rb);
                    }
            }
            bulk_commit();
        }
        // the stage of chunk ch - 1 takes chunk ch - 1 + S once its store has read it
        const int nxt = ch - 1 + S;
        if (ch >= 1 && nxt < nch) {
            if (lane == 0) bulk_wait_read_but_one();
            __syncwarp();
            okm[nxt % S] = issue(nxt);
            issued = nxt + 1;
        }
    }
    if (!ok && lane == 0) {
        // loads still in flight land before the shared memory is given up
        // (each wait bounded again)
        for (int ch = waited; ch < issued; ++ch) {
            const long long t0 = clock64();
            while (!tc::mbar_try_wait(&full[ch % S], (uint32_t)(ch / S) & 1u) &&
                   clock64() - t0 < tc::kWaitCycles) {
            }
        }
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
}

template <bool kPaged>
__global__ void __launch_bounds__(kThreads)
compact_kernel(const float* __restrict__ Z, int64_t ldz, int N, int n_obs, int budget,
               int32_t* __restrict__ idx, const uint4* a_src, const uint4* b_src, uint4* a_dst,
               uint4* b_dst, int n_cap, int out_cap, int vpr, int in_place, DeviceStatus* st,
               VariantIn var, PagedIn pg, int stages, uint32_t stage_off) {
    extern __shared__ uint32_t s_dyn[];
    const int C = N - n_obs, k = budget - n_obs;
    uint32_t* keys = s_dyn;                                         // [C]
    uint32_t* list = keys + C;                                      // [C]
    int32_t* sidx = reinterpret_cast<int32_t*>(list + C);           // [budget]
    __shared__ SelShared sh;
    float (*s_red)[kWarps] = sh.red;
    const int tid = threadIdx.x;
    const int64_t p = blockIdx.x;

    // ---------------------------------------------------------- select --
    float zmin = INFINITY, zmax = -INFINITY;
    if (var.I == nullptr) {
        for (int i = tid; i < C; i += kThreads) {
            const float z = Z[p * ldz + i];
            keys[i] = orderable(z);
            zmin = fminf(zmin, z);
            zmax = fmaxf(zmax, z);
        }
    } else {
        // scoring variant: Z from the base I and R rows, staged in the two
        // key arrays (I in `list`, R in `keys`, each entry of `keys` then
        // replaced by its own Z key)
        float* sI = reinterpret_cast<float*>(list);
        float* sR = reinterpret_cast<float*>(keys);
        float* sP = reinterpret_cast<float*>(sidx + budget);  // [C] with sentences
#pragma unroll 4
        for (int i = tid; i < C; i += kThreads) {
            sI[i] = var.I[p * var.ld + i];
            sR[i] = var.R[p * var.ld + i];
        }
        if (var.pen != nullptr) {
            // each candidate's sentence penalty, loads of several rows in flight
#pragma unroll 4
            for (int i = tid; i < C; i += kThreads) sP[i] = row_penalty(var, p, i);
        }
        __syncthreads();
        SoftmaxStats sm{0.f, 1.f};
        if (var.softmax) sm = softmax_stats<kThreads>(sR, C, s_red[0]);
        for (int i = tid; i < C; i += kThreads) {
            const float r = sR[i];
            const float z = __fsub_rn(variant_z(var.lambda, pooled_importance(sI, i, C, var.half),
                                                var.softmax ? softmax_term(r, sm) : r),
                                      var.pen != nullptr ? sP[i] : 0.f);
            keys[i] = orderable(z);
            zmin = fminf(zmin, z);
            zmax = fmaxf(zmax, z);
        }
        __syncthreads();  // `list` is reused for the bucket's keys below
    }
    if (var.sample) {
        // sampled selection: the pool of the top `pool` candidates by Z,
        // then the top k of Z / temperature + Gumbel noise within the pool
        uint32_t uk, eq_cut;
        if (var.pool < C) {
            kth_largest(keys, list, C, var.pool, zmin, zmax, sh, uk, eq_cut);
            take_top<true>(keys, C, uk, eq_cut, var.pool, nullptr, sh);
        }
        zmin = INFINITY;
        zmax = -INFINITY;
        const float* up = var.unif + p * var.ld_u;
        for (int i = tid; i < C; i += kThreads) {
            const uint32_t u = keys[i];
            if (u == 0u) continue;  // outside the pool
            const float g = -logf(-logf(up[i]));
            const float key = __fadd_rn(__fmul_rn(from_orderable(u), var.inv_temp), g);
            keys[i] = orderable(key);
            if (isfinite(key)) {
                zmin = fminf(zmin, key);
                zmax = fmaxf(zmax, key);
            }
        }
        __syncthreads();
    }
    {
        uint32_t uk, eq_cut;
        kth_largest(keys, list, C, k > 0 ? k : 1, zmin, zmax, sh, uk, eq_cut);
        if (k > 0) take_top<false>(keys, C, uk, eq_cut, k, sidx, sh);
    }
    for (int r = tid; r < n_obs; r += kThreads) sidx[k + r] = C + r;
    __syncthreads();
    int32_t* out = idx + p * (int64_t)budget;
    for (int r = tid; r < budget; r += kThreads) out[r] = sidx[r];
    if (var.seg != nullptr) {
        // the kept rows' sentence ids follow them (the cache-range mapping),
        // in place in ascending chunks: sidx[r] >= r, so a chunk's sources
        // lie at or after the chunk and are read before it is written
        int32_t* sg = var.seg + p * var.ld_seg;
        for (int c0 = 0; c0 < budget; c0 += kThreads) {
            const int r = c0 + tid;
            const int32_t v = r < budget ? sg[sidx[r]] : 0;
            __syncthreads();
            if (r < budget) sg[r] = v;
            __syncthreads();
        }
    }

    // ------------------------------------------------------------ copy --
    if constexpr (kPaged) {
        // a_src: contiguous K copy [P, N, vpr], or null when K moves inside
        // its pool like V; a_dst: K pool; b_dst: V pool
        int l = 0, h = budget;
        while (l < h) {
            const int mid = (l + h) >> 1;
            if (sidx[mid] == mid) l = mid + 1;
            else h = mid;
        }
        const int64_t kc_base = (int64_t)p * N * vpr;
        const int rows_per_chunk = kThreads * kCopyVecs / vpr;
        for (int c0 = l; c0 < budget; c0 += rows_per_chunk) {
            uint4 va[kCopyVecs], vb[kCopyVecs];
            int64_t dst[kCopyVecs];
#pragma unroll
            for (int t = 0; t < kCopyVecs; ++t) {
                const int e = t * kThreads + tid;
                const int r = c0 + e / vpr, v = e % vpr;
                dst[t] = -1;
                if (r < budget) {
                    const int s = sidx[r];
                    const int64_t dr = paged_phys_row(pg, p, r);
                    const int64_t sr = (s >= 0 && s < N) ? paged_phys_row(pg, p, s) : -1;
                    if (dr >= 0 && sr >= 0) {
                        dst[t] = dr * vpr + v;
                        va[t] = a_src ? a_src[kc_base + (int64_t)s * vpr + v] : a_dst[sr * vpr + v];
                        vb[t] = b_dst[sr * vpr + v];
                    } else if (v == 0) {
                        set_error(st, kDevErrIndex, (unsigned)r);
                    }
                }
            }
            __syncthreads();  // every source row of the chunk has been read
#pragma unroll
            for (int t = 0; t < kCopyVecs; ++t) {
                if (dst[t] >= 0) {
                    a_dst[dst[t]] = va[t];
                    b_dst[dst[t]] = vb[t];
                }
            }
            __syncthreads();
        }
        return;
    }
    const int64_t base = (int64_t)p * n_cap * vpr;
    if (stages > 0) {
        __shared__ uint64_t s_full[kMaxStages];
        __shared__ int s_abort;
        if (tid >= 32) return;  // one warp moves the rows
        int r0 = 0;
        if (in_place) {
            // first row r0 with sidx[r0] != r0 (sidx[r] == r holds exactly on a prefix)
            int l = 0, h = budget;
            while (l < h) {
                const int mid = (l + h) >> 1;
                if (sidx[mid] == mid) l = mid + 1;
                else h = mid;
            }
            r0 = l;
        }
        if (tid == 0) {
            for (int i = 0; i < stages; ++i) tc::mbar_init(&s_full[i], 1);
            s_abort = 0;
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        }
        __syncwarp();
        const int rb = vpr * 16;
        const int64_t ob = in_place ? base : (int64_t)p * out_cap * vpr;
        uint8_t* stage_mem = reinterpret_cast<uint8_t*>(s_dyn) + stage_off;
        if (r0 < budget)
            copy_rows_bulk(sidx, r0, budget, n_cap, reinterpret_cast<const uint8_t*>(a_src + base),
                           b_src ? reinterpret_cast<const uint8_t*>(b_src + base) : nullptr,
                           reinterpret_cast<uint8_t*>(a_dst + ob),
                           b_dst ? reinterpret_cast<uint8_t*>(b_dst + ob) : nullptr, rb, stage_mem,
                           s_full, stages, &s_abort, st);
        return;
    }
    if (!in_place) {
        const int64_t obase = (int64_t)p * out_cap * vpr;
        const int total = budget * vpr;
        for (int e0 = tid; e0 < total; e0 += kThreads * kCopyVecs) {
            uint4 va[kCopyVecs], vb[kCopyVecs];
            int dst[kCopyVecs];
#pragma unroll
            for (int t = 0; t < kCopyVecs; ++t) {
                const int e = e0 + t * kThreads;
                dst[t] = -1;
                if (e < total) {
                    const int r = e / vpr, v = e % vpr;
                    const int s = sidx[r];
                    if (s >= 0 && s < n_cap) {
                        dst[t] = r * vpr + v;
                        va[t] = __ldg(a_src + base + (int64_t)s * vpr + v);
                        if (b_src) vb[t] = __ldg(b_src + base + (int64_t)s * vpr + v);
                    } else if (st) {
                        set_error(st, kDevErrIndex, (unsigned)r);
                    }
                }
            }
#pragma unroll
            for (int t = 0; t < kCopyVecs; ++t) {
                if (dst[t] >= 0) {
                    a_dst[obase + dst[t]] = va[t];
                    if (b_dst) b_dst[obase + dst[t]] = vb[t];
                }
            }
        }
    } else {
        // first row r0 with sidx[r0] != r0 (sidx[r] == r holds exactly on a prefix)
        int l = 0, h = budget;
        while (l < h) {
            const int mid = (l + h) >> 1;
            if (sidx[mid] == mid) l = mid + 1;
            else h = mid;
        }
        const int rows_per_chunk = kThreads * kCopyVecs / vpr;
        for (int c0 = l; c0 < budget; c0 += rows_per_chunk) {
            uint4 va[kCopyVecs], vb[kCopyVecs];
            int dst[kCopyVecs];
#pragma unroll
            for (int t = 0; t < kCopyVecs; ++t) {
                const int e = t * kThreads + tid;  // vector within the chunk
                const int r = c0 + e / vpr, v = e % vpr;
                dst[t] = -1;
                if (r < budget) {
                    const int s = sidx[r];
                    if (s >= 0 && s < n_cap) {
                        dst[t] = r * vpr + v;
                        va[t] = a_dst[base + (int64_t)s * vpr + v];
                        if (b_dst) vb[t] = b_dst[base + (int64_t)s * vpr + v];
                    } else if (st) {
                        set_error(st, kDevErrIndex, (unsigned)r);
                    }
                }
            }
            __syncthreads();  // every source row of the chunk has been read
#pragma unroll
            for (int t = 0; t < kCopyVecs; ++t) {
                if (dst[t] >= 0) {
                    a_dst[base + dst[t]] = va[t];
                    if (b_dst) b_dst[base + dst[t]] = vb[t];
                }
            }
            __syncthreads();
        }
    }
}

}  // namespace

size_t compact_smem_bytes(int N, int n_obs, int budget, bool sentences) {
    const int C = N - n_obs;
    const size_t c = (size_t)(C > 0 ? C : 1);
    return sizeof(uint32_t) * 2 * c + sizeof(int32_t) * (size_t)budget +
           (sentences ? sizeof(float) * c : 0);
}

cudaError_t launch_compact(int64_t P, int N, const float* Z, int64_t ldz, int n_obs, int budget,
                           int32_t* idx, const void* src_a, const void* src_b, void* dst_a,
                           void* dst_b, int n_cap, int out_cap, int row_bytes, bool in_place,
                           DeviceStatus* st, cudaStream_t s, const VariantIn& var) {
    if (P == 0 || budget == 0) return cudaSuccess;
    const size_t sel = compact_smem_bytes(N, n_obs, budget, var.pen != nullptr);
    // the stages of the bulk copy after the selection's arrays, 128-byte aligned
    const size_t off = (sel + 127) / 128 * 128;
    const size_t stage_bytes = (size_t)kChunkRows * row_bytes * (src_b ? 2 : 1);
    int stages = off < kStageTarget ? (int)((kStageTarget - off) / stage_bytes) : 0;
    if (stages > kMaxStages) stages = kMaxStages;
    if (stages < 2) stages = 0;  // too little room: the register copy
    const size_t smem = stages ? off + stages * stage_bytes : sel;
    cudaError_t e = cudaFuncSetAttribute(compact_kernel<false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    compact_kernel<false><<<(unsigned)P, kThreads, smem, s>>>(
        Z, ldz, N, n_obs, budget, idx, static_cast<const uint4*>(src_a),
        static_cast<const uint4*>(src_b), static_cast<uint4*>(dst_a), static_cast<uint4*>(dst_b), n_cap,
        in_place ? n_cap : out_cap, row_bytes / 16, in_place ? 1 : 0, st, var, PagedIn{}, stages,
        (uint32_t)off);
    return cudaGetLastError();
}

cudaError_t launch_compact_paged(int64_t P, int N, const float* Z, int64_t ldz, int n_obs,
                                 int budget, int32_t* idx, const void* kc, void* k_pool,
                                 void* v_pool, const PagedIn& pg, int row_bytes, DeviceStatus* st,
                                 cudaStream_t s, const VariantIn& var) {
    if (P == 0 || budget == 0) return cudaSuccess;
    const size_t smem = compact_smem_bytes(N, n_obs, budget, var.pen != nullptr);
    cudaError_t e = cudaFuncSetAttribute(compact_kernel<true>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    compact_kernel<true><<<(unsigned)P, kThreads, smem, s>>>(
        Z, ldz, N, n_obs, budget, idx, static_cast<const uint4*>(kc), nullptr,
        static_cast<uint4*>(k_pool), static_cast<uint4*>(v_pool), N, N, row_bytes / 16, 1, st, var,
        pg, 0, 0u);
    return cudaGetLastError();
}

}  // namespace rkv
