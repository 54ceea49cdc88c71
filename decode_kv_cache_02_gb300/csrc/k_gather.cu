// k_gather.cu -- copy the kept K/V rows into the compacted cache.
//
// R-KV review (yoonschallenge.tistory.com/1236), question 2, cause 3 (the
// kept KV rows are copied into the compacted cache) and cause 4 (pruning forces a re-layout
// of the KV tensor; allocating a new cache costs memory management).  The
// copy is byte-exact and can run in place, so no second cache is needed.
//
// Out of place: a grid-stride loop over 16-byte vectors of the destination,
// several vectors in flight per thread, coalesced along each row.
// In place: one CTA per problem.  Kept indices are strictly ascending and
// idx[r] >= r, so rows before the first evicted token are already where they
// belong and are skipped; from there the rows move in ascending chunks, each
// chunk read completely into registers before any of it is written, so no
// source row is overwritten before it is read.
#include "rkv_common.cuh"
#include "rkv_internal.h"
#include "../../include/rkv.h"

namespace rkv {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

__global__ void __launch_bounds__(kThreads)
gather_oop_kernel(const uint4* __restrict__ a, const uint4* __restrict__ b, uint4* __restrict__ da,
                  uint4* __restrict__ db, const int32_t* __restrict__ idx, int64_t P, int n_cap,
                  int out_cap, int budget, int vpr, int64_t total, DeviceStatus* st) {
    // element e -> (problem, kept row, vector)
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t e0 = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e0 < total;
         e0 += stride * kUnroll) {
        uint4 va[kUnroll], vb[kUnroll];
        int64_t dst[kUnroll];
#pragma unroll
        for (int t = 0; t < kUnroll; ++t) {
            const int64_t e = e0 + t * stride;
            dst[t] = -1;
            if (e < total) {
                const int v = (int)(e % vpr);
                const int64_t pr = e / vpr;  // p * budget + r
                const int64_t p = pr / budget;
                const int r = (int)(pr - p * budget);
                const int s = __ldg(idx + pr);
                if (s >= n_cap) set_error(st, kDevErrIndex, (unsigned)pr);
                if (s >= 0 && s < n_cap) {
                    const int64_t src = ((int64_t)p * n_cap + s) * vpr + v;
                    dst[t] = ((int64_t)p * out_cap + r) * vpr + v;
                    va[t] = __ldg(a + src);
                    if (b) vb[t] = __ldg(b + src);
                }
            }
        }
#pragma unroll
        for (int t = 0; t < kUnroll; ++t) {
            if (dst[t] >= 0) {
                da[dst[t]] = va[t];
                if (b) db[dst[t]] = vb[t];
            }
        }
    }
}

constexpr int kChunkVecs = 8;  // vectors per thread per tensor per chunk

__global__ void __launch_bounds__(kThreads)
gather_inplace_kernel(uint4* a, uint4* b, const int32_t* __restrict__ idx, int n_cap, int budget,
                      int vpr, DeviceStatus* st) {
    const int64_t p = blockIdx.x;
    const int32_t* ip = idx + p * (int64_t)budget;
    // first row r0 with idx[r0] != r0 (idx[r] == r holds exactly on a prefix)
    int lo = 0, hi = budget;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (ip[mid] == mid) lo = mid + 1;
        else hi = mid;
    }
    const int r0 = lo;
    uint4* ap = a + (int64_t)p * n_cap * vpr;
    uint4* bp = b ? b + (int64_t)p * n_cap * vpr : nullptr;
    const int rows_per_chunk = kThreads * kChunkVecs / vpr;
    for (int c0 = r0; c0 < budget; c0 += rows_per_chunk) {
        uint4 va[kChunkVecs], vb[kChunkVecs];
        int dst[kChunkVecs];
#pragma unroll
        for (int t = 0; t < kChunkVecs; ++t) {
            const int e = t * kThreads + threadIdx.x;  // vector within the chunk
            const int r = c0 + e / vpr, v = e % vpr;
            dst[t] = -1;
            if (r < budget) {
                const int s = ip[r];
                if (s >= n_cap) set_error(st, kDevErrIndex, (unsigned)r);
                if (s >= 0 && s < n_cap) {
                    dst[t] = r * vpr + v;
                    va[t] = ap[(int64_t)s * vpr + v];
                    if (bp) vb[t] = bp[(int64_t)s * vpr + v];
                }
            }
        }
        __syncthreads();  // every source row of the chunk has been read
#pragma unroll
        for (int t = 0; t < kChunkVecs; ++t) {
            if (dst[t] >= 0) {
                ap[dst[t]] = va[t];
                if (bp) bp[dst[t]] = vb[t];
            }
        }
        __syncthreads();
    }
}

}  // namespace

cudaError_t launch_gather(const void* src_a, const void* src_b, void* dst_a, void* dst_b,
                          const int32_t* idx, int64_t P, int n_cap, int out_cap, int budget,
                          int row_bytes, bool in_place, DeviceStatus* st, cudaStream_t s) {
    if (P == 0 || budget == 0) return cudaSuccess;
    const int vpr = row_bytes / 16;
    if (in_place) {
        gather_inplace_kernel<<<(unsigned)P, kThreads, 0, s>>>(
            static_cast<uint4*>(dst_a), static_cast<uint4*>(dst_b), idx, n_cap, budget, vpr, st);
    } else {
        const int64_t total = P * (int64_t)budget * vpr;
        int dev = 0, sms = 152;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        int64_t blocks = (total + (int64_t)kThreads * kUnroll - 1) / ((int64_t)kThreads * kUnroll);
        const int64_t cap = (int64_t)sms * 8;
        if (blocks > cap) blocks = cap;
        gather_oop_kernel<<<(unsigned)blocks, kThreads, 0, s>>>(
            static_cast<const uint4*>(src_a), static_cast<const uint4*>(src_b),
            static_cast<uint4*>(dst_a), static_cast<uint4*>(dst_b), idx, P, n_cap, out_cap, budget, vpr,
            total, st);
    }
    return cudaGetLastError();
}

}  // namespace rkv
