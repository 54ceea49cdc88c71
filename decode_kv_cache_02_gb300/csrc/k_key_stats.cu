// k_key_stats.cu -- per-key norms and the plain similarity sums.
//
// R-KV review (yoonschallenge.tistory.com/1236), question 2, cause 3: "key
// vector normalisation" precedes the all-pairs cosine similarity.  Redundancy
// (summary-table row "redundancy") needs, for every key i,
//     sum_i = sum_{j != i} S_ij,   S_ij = khat_i . khat_j,  khat = k / max(|k|, eps).
// The unthresholded part of that sum is linear in the keys:
//     sum_i = khat_i . s - khat_i . khat_i,   s = sum_j khat_j,
// so it costs O(N d) per problem, not O(N^2 d).  The Gram kernels then only
// handle the thresholded part (pairs with S_ij > tau).
//
// One CTA of 256 threads per problem.  A row of d elements is split over
// L = d/8 lanes (16 bytes each, so a warp reads 32 x 16 contiguous bytes);
// every thread keeps several rows' loads in flight.  Pass 1 writes inv_norm
// and accumulates, per thread, the partial s of its 8 columns over its rows
// (no cross-lane traffic for s until one shared-memory reduction at the
// end); pass 2 re-reads the rows (from L2) and writes sum_i.  When the
// tensor-core importance kernel runs, only pass 1 is needed: it writes
// |khat_i|^2 into sum_i and s as bf16 rows (hi, lo) that the importance MMA
// multiplies with every key block anyway, which completes sum_i there.
//
// Paged input (key_stats_paged_kernel): rows are found through the block
// table; rows past N are neither read nor written.  When the tensor-core
// stages do not read the pool (small blocks, fp32), pass 1 also stores every
// row, bit for bit, into the contiguous copy Kc [P, N, d].
#include "rkv_common.cuh"
#include "rkv_internal.h"
#include "rkv_paged.cuh"
#include "../../include/rkv.h"

namespace rkv {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;  // rows in flight per thread
constexpr int kSRows = 16;  // rows of the s block handed to the importance MMA

// Sum over the L lanes that share a row (L = 8 or 16, aligned groups).  The
// mask names only those lanes: they always run the same number of row
// iterations, the two halves of a warp need not.
template <int L>
RKV_DEV float group_sum(float v) {
    const unsigned lane = threadIdx.x & 31u;
    const unsigned mask = ((1u << L) - 1u) << (lane & ~(unsigned)(L - 1));
#pragma unroll
    for (int o = L / 2; o > 0; o >>= 1) v += __shfl_xor_sync(mask, v, o);
    return v;
}

// 8 consecutive elements as raw 16-byte vectors (one for bf16, two for fp32)
template <typename T>
struct Raw8 {
    static constexpr int kVecs = (int)sizeof(T) * 8 / 16;
    uint4 u[kVecs];
    RKV_DEV void load(const T* p) {
#pragma unroll
        for (int t = 0; t < kVecs; ++t) u[t] = reinterpret_cast<const uint4*>(p)[t];
    }
    RKV_DEV void store(T* p) const {
#pragma unroll
        for (int t = 0; t < kVecs; ++t) reinterpret_cast<uint4*>(p)[t] = u[t];
    }
    RKV_DEV void to_float(float* o) const { load8(reinterpret_cast<const T*>(u), o); }
};

// Rows of one batch per thread in pass 1 of the contiguous kernel: kept packed
// until each is reduced, so eight bf16 rows (32 registers) stay in flight.
template <typename T>
constexpr int kRowsInFlight = sizeof(T) == 2 ? 8 : 4;

template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 4)
key_stats_kernel(const T* __restrict__ K, int n_cap, int N, float* __restrict__ inv_norm,
                 float* __restrict__ sum_s, int64_t ld, bool two_pass,
                 __nv_bfloat16* __restrict__ s_rows) {
    constexpr int L = D / 8;                 // lanes per row
    constexpr int RPI = kThreads / L;        // rows per iteration of the CTA
    __shared__ float s_part[RPI][D];
    __shared__ float s_vec[D];
    const int64_t p = blockIdx.x;
    const T* Kp = K + (size_t)p * n_cap * D;
    const int sub = threadIdx.x % L;         // which 8 columns
    const int r0 = threadIdx.x / L;          // first row of this thread
    const int col = sub * 8;

    float acc[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) acc[t] = 0.f;
    // ---- pass 1: norms and the partial sums of khat
    constexpr int KU = kRowsInFlight<T>;
    for (int base = r0; base < N; base += RPI * KU) {
        Raw8<T> raw[KU];
#pragma unroll
        for (int u = 0; u < KU; ++u) {
            const int i = base + u * RPI;
            if (i < N) raw[u].load(Kp + (size_t)i * D + col);
        }
#pragma unroll
        for (int u = 0; u < KU; ++u) {
            const int i = base + u * RPI;
            float v[8];
            if (i < N) {
                raw[u].to_float(v);
            } else {
#pragma unroll
                for (int t = 0; t < 8; ++t) v[t] = 0.f;
            }
            float n2 = 0.f;
#pragma unroll
            for (int t = 0; t < 8; ++t) n2 = fmaf(v[t], v[t], n2);
            n2 = group_sum<L>(n2);
            const float inv = 1.0f / fmaxf(sqrtf(n2), 1e-12f);
            if (i < N) {
                if (sub == 0) {
                    inv_norm[p * ld + i] = inv;
                    // |khat_i|^2, completed to sum_i by the importance kernel
                    if (!two_pass) sum_s[p * ld + i] = (n2 * inv) * inv;
                }
#pragma unroll
                for (int t = 0; t < 8; ++t) acc[t] = fmaf(v[t], inv, acc[t]);
            }
        }
    }
#pragma unroll
    for (int t = 0; t < 8; ++t) s_part[r0][col + t] = acc[t];
    __syncthreads();
    for (int c = threadIdx.x; c < D; c += kThreads) {
        float s = 0.f;
#pragma unroll 8
        for (int w = 0; w < RPI; ++w) s += s_part[w][c];
        s_vec[c] = s;
        if (!two_pass) {
            // s as two bf16 rows (s ~= hi + lo to 2^-16), then 14 zero rows:
            // extra B rows of the importance MMA, which then yields k_i . s
            __nv_bfloat16* sr = s_rows + (size_t)p * kSRows * D;
            const __nv_bfloat16 hi = __float2bfloat16_rn(s);
            sr[c] = hi;
            sr[D + c] = __float2bfloat16_rn(s - __bfloat162float(hi));
            for (int r = 2; r < kSRows; ++r) sr[r * D + c] = __float2bfloat16_rn(0.f);
        }
    }
    if (!two_pass) return;
    __syncthreads();
    float sv[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) sv[t] = s_vec[col + t];
    const T* Kp2 = Kp;
    // ---- pass 2: sum_i = khat_i . s - |khat_i|^2
    for (int base = r0; base < N; base += RPI * kUnroll) {
        float v[kUnroll][8];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int i = base + u * RPI;
            if (i < N) {
                load8(Kp2 + (size_t)i * D + col, v[u]);
            } else {
#pragma unroll
                for (int t = 0; t < 8; ++t) v[u][t] = 0.f;
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int i = base + u * RPI;
            float n2 = 0.f, ds = 0.f;
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                n2 = fmaf(v[u][t], v[u][t], n2);
                ds = fmaf(v[u][t], sv[t], ds);
            }
            n2 = group_sum<L>(n2);
            ds = group_sum<L>(ds);
            const float inv = 1.0f / fmaxf(sqrtf(n2), 1e-12f);
            if (i < N && sub == 0) sum_s[p * ld + i] = ds * inv - (n2 * inv) * inv;
        }
    }
}

// The same statistics of paged keys: rows through the block table (the
// sequence's ids staged in shared memory).  kMode 1 also stores every row into
// the contiguous copy Kc;
// kMode 2 reads in place.  Four CTAs per SM keep enough rows in flight, except
// for the copying fp32 variant, which would spill there.
template <typename T, int D, int kMode>
__global__ void __launch_bounds__(kThreads, (kMode == 1 && sizeof(T) == 4) ? 2 : 4)
key_stats_paged_kernel(const T* __restrict__ K, int n_cap, int N, float* __restrict__ inv_norm,
                 float* __restrict__ sum_s, int64_t ld, bool two_pass,
                 __nv_bfloat16* __restrict__ s_rows, PagedIn pg, T* __restrict__ Kc,
                 DeviceStatus* st) {
    constexpr int L = D / 8;                 // lanes per row
    constexpr int RPI = kThreads / L;        // rows per iteration of the CTA
    __shared__ float s_part[RPI][D];
    __shared__ float s_vec[D];
    constexpr bool kPaged = kMode != 0;
    const int64_t p = blockIdx.x;
    const T* Kp = K + (size_t)p * n_cap * D;
    T* Kcp = kMode == 1 ? Kc + (size_t)p * N * D : nullptr;
    // paged: the sequence's block ids in shared memory (-1 for an id outside
    // the pool), so that a row's address needs no global load
    extern __shared__ int32_t s_tab[];
    int64_t head_base = 0;
    if constexpr (kPaged) {
        const int nbk = (N + (1 << pg.log2bs) - 1) >> pg.log2bs;
        const int64_t sq = p / pg.H;
        head_base = p - sq * pg.H;
        for (int b = threadIdx.x; b < nbk; b += kThreads) {
            const int v = pg.table[sq * pg.max_blocks + b];
            s_tab[b] = (unsigned)v < (unsigned)pg.num_blocks ? v : -1;
        }
        __syncthreads();
    }
    auto phys_row = [&](int r) -> int64_t {  // paged row index in the pool, or -1
        const int blk = s_tab[r >> pg.log2bs];
        return blk < 0 ? -1
                       : (((int64_t)blk * pg.H + head_base) << pg.log2bs) |
                             (int64_t)(r & ((1 << pg.log2bs) - 1));
    };
    const int sub = threadIdx.x % L;         // which 8 columns
    const int r0 = threadIdx.x / L;          // first row of this thread
    const int col = sub * 8;

    float acc[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) acc[t] = 0.f;
    // ---- pass 1: norms and the partial sums of khat
    for (int base = r0; base < N; base += RPI * kUnroll) {
        float v[kUnroll][8];
        if constexpr (kMode == 1) {
            // rows through the table, each also stored into the contiguous copy
            Raw8<T> raw[kUnroll];
            bool ok[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int i = base + u * RPI;
                ok[u] = false;
                if (i < N) {
                    const int64_t pr = phys_row(i);
                    if (pr >= 0) {
                        raw[u].load(K + pr * D + col);
                        ok[u] = true;
                    } else if (sub == 0) {
                        set_error(st, kDevErrIndex, (unsigned)i);
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                if (ok[u]) {
                    raw[u].store(Kcp + (size_t)(base + u * RPI) * D + col);
                    raw[u].to_float(v[u]);
                } else {
#pragma unroll
                    for (int t = 0; t < 8; ++t) v[u][t] = 0.f;
                    if (base + u * RPI < N) {
                        Raw8<T> z{};
                        z.store(Kcp + (size_t)(base + u * RPI) * D + col);
                    }
                }
            }
        } else if constexpr (kMode == 2) {
            // paged rows read in place: every row's load issued before any is
            // used.  Direct reads take blocks of >= 128 rows, and the batch's
            // rows base + u*RPI lie in the 64-row window [base - r0, +64), so
            // in one block: one table lookup per batch.
            static_assert(RPI * kUnroll <= 128, "a batch must fit in one block");
            const int64_t pr0 = base < N ? phys_row(base) : -1;
            Raw8<T> raw[kUnroll];
            bool ok[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int i = base + u * RPI;
                ok[u] = false;
                if (i < N) {
                    if (pr0 >= 0) {
                        raw[u].load(K + (pr0 + u * RPI) * D + col);
                        ok[u] = true;
                    } else if (sub == 0) {
                        set_error(st, kDevErrIndex, (unsigned)i);
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                if (ok[u]) {
                    raw[u].to_float(v[u]);
                } else {
#pragma unroll
                    for (int t = 0; t < 8; ++t) v[u][t] = 0.f;
                }
            }
        } else {
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int i = base + u * RPI;
                if (i < N) {
                    load8(Kp + (size_t)i * D + col, v[u]);
                } else {
#pragma unroll
                    for (int t = 0; t < 8; ++t) v[u][t] = 0.f;
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int i = base + u * RPI;
            float n2 = 0.f;
#pragma unroll
            for (int t = 0; t < 8; ++t) n2 = fmaf(v[u][t], v[u][t], n2);
            n2 = group_sum<L>(n2);
            const float inv = 1.0f / fmaxf(sqrtf(n2), 1e-12f);
            if (i < N) {
                if (sub == 0) {
                    inv_norm[p * ld + i] = inv;
                    // |khat_i|^2, completed to sum_i by the importance kernel
                    if (!two_pass) sum_s[p * ld + i] = (n2 * inv) * inv;
                }
#pragma unroll
                for (int t = 0; t < 8; ++t) acc[t] = fmaf(v[u][t], inv, acc[t]);
            }
        }
    }
#pragma unroll
    for (int t = 0; t < 8; ++t) s_part[r0][col + t] = acc[t];
    __syncthreads();
    for (int c = threadIdx.x; c < D; c += kThreads) {
        float s = 0.f;
#pragma unroll 8
        for (int w = 0; w < RPI; ++w) s += s_part[w][c];
        s_vec[c] = s;
        if (!two_pass) {
            // s as two bf16 rows (s ~= hi + lo to 2^-16), then 14 zero rows:
            // extra B rows of the importance MMA, which then yields k_i . s
            __nv_bfloat16* sr = s_rows + (size_t)p * kSRows * D;
            const __nv_bfloat16 hi = __float2bfloat16_rn(s);
            sr[c] = hi;
            sr[D + c] = __float2bfloat16_rn(s - __bfloat162float(hi));
            for (int r = 2; r < kSRows; ++r) sr[r * D + c] = __float2bfloat16_rn(0.f);
        }
    }
    if (!two_pass) return;
    __syncthreads();
    float sv[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) sv[t] = s_vec[col + t];
    // the paged rows are re-read from the contiguous copy (written above by
    // this CTA; the barrier makes them visible)
    // (the paged two-pass case always has the contiguous copy: only the
    // CUDA-core importance, which reads contiguous keys, asks for pass 2)
    const T* Kp2 = kPaged ? Kcp : Kp;
    // ---- pass 2: sum_i = khat_i . s - |khat_i|^2
    for (int base = r0; base < N; base += RPI * kUnroll) {
        float v[kUnroll][8];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int i = base + u * RPI;
            if (i < N) {
                load8(Kp2 + (size_t)i * D + col, v[u]);
            } else {
#pragma unroll
                for (int t = 0; t < 8; ++t) v[u][t] = 0.f;
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int i = base + u * RPI;
            float n2 = 0.f, ds = 0.f;
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                n2 = fmaf(v[u][t], v[u][t], n2);
                ds = fmaf(v[u][t], sv[t], ds);
            }
            n2 = group_sum<L>(n2);
            ds = group_sum<L>(ds);
            const float inv = 1.0f / fmaxf(sqrtf(n2), 1e-12f);
            if (i < N && sub == 0) sum_s[p * ld + i] = ds * inv - (n2 * inv) * inv;
        }
    }
}

template <typename T, int D, int kMode>
cudaError_t launch_paged(const ScoreArgs& a, cudaStream_t s) {
    const size_t tab = sizeof(int32_t) * (size_t)((a.N + (1 << a.pg.log2bs) - 1) >> a.pg.log2bs);
    cudaError_t e = cudaFuncSetAttribute(key_stats_paged_kernel<T, D, kMode>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tab);
    if (e != cudaSuccess) return e;
    key_stats_paged_kernel<T, D, kMode><<<(unsigned)a.P, kThreads, tab, s>>>(
        static_cast<const T*>(a.K), a.n_cap, a.N, a.inv_norm, a.sum_s, a.ld_ws, a.stats_sum,
        static_cast<__nv_bfloat16*>(a.s_rows), a.pg, static_cast<T*>(a.Kc), a.status);
    return cudaGetLastError();
}

template <typename T, int D>
cudaError_t launch_t(const ScoreArgs& a, cudaStream_t s) {
    if (a.pg.table != nullptr) {
        // only bf16 pools are read in place by the tensor-core stages
        if constexpr (sizeof(T) == 2)
            if (a.Kc == nullptr) return launch_paged<T, D, 2>(a, s);
        return launch_paged<T, D, 1>(a, s);
    }
    key_stats_kernel<T, D><<<(unsigned)a.P, kThreads, 0, s>>>(
        static_cast<const T*>(a.K), a.n_cap, a.N, a.inv_norm, a.sum_s, a.ld_ws, a.stats_sum,
        static_cast<__nv_bfloat16*>(a.s_rows));
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_key_stats(const ScoreArgs& a, cudaStream_t s) {
    if (a.P == 0) return cudaSuccess;
    if (a.dtype == RKV_DTYPE_BF16)
        return a.d == 128 ? launch_t<__nv_bfloat16, 128>(a, s) : launch_t<__nv_bfloat16, 64>(a, s);
    return a.d == 128 ? launch_t<float, 128>(a, s) : launch_t<float, 64>(a, s);
}

}  // namespace rkv
