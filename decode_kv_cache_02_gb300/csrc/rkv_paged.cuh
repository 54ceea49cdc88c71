// rkv_paged.cuh -- address translation of the paged KV pool.
#pragma once

#include "rkv_common.cuh"
#include "rkv_internal.h"

namespace rkv {

// Physical row of logical row r of problem p in the pool (in units of one
// row of d elements), or -1 when the table names no valid block.
RKV_DEV int64_t paged_phys_row(const PagedIn& pg, int64_t p, int r) {
    const int64_t s = p / pg.H;
    const int h = (int)(p - s * pg.H);
    const int blk = pg.table[s * pg.max_blocks + (r >> pg.log2bs)];
    if ((unsigned)blk >= (unsigned)pg.num_blocks) return -1;
    return (((int64_t)blk * pg.H + h) << pg.log2bs) | (int64_t)(r & ((1 << pg.log2bs) - 1));
}

}  // namespace rkv
