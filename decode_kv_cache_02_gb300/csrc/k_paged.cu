// k_paged.cu -- handing back the blocks a paged compaction emptied.
//
// R-KV review (yoonschallenge.tistory.com/1236), question 2, cause 4: in a
// block-structured (PagedAttention) cache, pruning that frees the old cache
// and allocates a compressed one costs memory management.  After the in-place
// compaction a sequence's kept rows occupy its first ceil(budget/bs) blocks;
// the blocks after them, up to the ceil(n_cached/bs) it held, are whole and
// unused.  This kernel lists their ids per sequence and clears the table
// entries, so the caller's block allocator can take them back.
#include "rkv_common.cuh"
#include "rkv_internal.h"

namespace rkv {
namespace {

__global__ void paged_release_kernel(int64_t S, int32_t* __restrict__ table, int max_blocks,
                                     int nb_keep, int n_free, int32_t* __restrict__ out_freed) {
    const int64_t total = S * n_free;
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t s = e / n_free;
        const int j = (int)(e - s * n_free);
        int32_t* t = table + s * max_blocks + nb_keep + j;
        out_freed[e] = *t;
        *t = -1;
    }
}

}  // namespace

cudaError_t launch_paged_release(int64_t S, int32_t* table, int max_blocks, int nb_keep,
                                 int nb_old, int32_t* out_freed, cudaStream_t s) {
    const int n_free = nb_old - nb_keep;
    if (S == 0 || n_free <= 0) return cudaSuccess;
    const int64_t total = S * n_free;
    const int threads = 256;
    const int64_t blocks = (total + threads - 1) / threads;
    paged_release_kernel<<<(unsigned)(blocks < 4096 ? blocks : 4096), threads, 0, s>>>(
        S, table, max_blocks, nb_keep, n_free, out_freed);
    return cudaGetLastError();
}

}  // namespace rkv
