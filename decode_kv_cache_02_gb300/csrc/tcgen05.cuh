// tcgen05.cuh -- inline-PTX wrappers for the sm_103a tensor-core kernels:
// mbarriers (with bounded waits), TMA tensor loads, TMEM allocation, tcgen05
// MMA / commit / load, and shared-memory matrix descriptors.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "rkv_common.cuh"
#include "rkv_internal.h"

namespace rkv {
namespace tc {

// Upper bound on one mbarrier wait (~1 s at 2 GHz); a wait that runs out
// reports a device error instead of hanging.
constexpr long long kWaitCycles = 2000000000LL;

RKV_DEV uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
RKV_DEV void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}
RKV_DEV void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// One arrival for the whole (converged) warp, after every lane has reached
// this point: barriers counted in warps instead of threads take 32 times fewer
// shared-memory arrive operations.
RKV_DEV void mbar_arrive_warp(uint64_t* bar) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}
RKV_DEV void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
// One bounded poll: the thread may sleep in the hardware until the phase
// completes or the suspend hint (ns) runs out, instead of spinning.
constexpr uint32_t kSuspendHintNs = 200000;

RKV_DEV bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(kSuspendHintNs)
        : "memory");
    return ok != 0;
}
// Bounded wait for the phase with the given parity; false on timeout or when
// another role has already aborted.
RKV_DEV bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (*abort_flag) return false;
        if (clock64() - t0 > kWaitCycles) return false;
    }
    return true;
}
RKV_DEV void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
        : "memory");
}
// The same load with an L2 cache policy (createpolicy): how long the copied
// lines should stay in L2 relative to other traffic.
RKV_DEV void tma_load_3d_hint(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y, int z,
                              uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z),
        "l"(policy)
        : "memory");
}
// L2 policies for key streams read twice: the first read asks the lines to
// stay (evict_last), the second lets them go first (evict_first).
RKV_DEV uint64_t l2_policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
RKV_DEV uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// The tensor maps of a call's keys: `main` for every load but the last block
// of a paged sequence whose rows stop before the block's end, which goes
// through `tail` (the same pool, a row extent of KeySource::tail_rows).
struct KeyMaps {
    CUtensorMap main;
    CUtensorMap tail;
};

// TMA loads of key rows [r0, r0 + rows) of problem p into a 128-byte-swizzled
// K-major tile at dst (KC chunks of 64 columns, chunk_bytes apart).  From the
// contiguous map, one load per chunk; from a paged pool (ks.table set), one
// load per block of min(block size, 128) rows (sub-tiles start on 8-row, 1024-byte
// boundaries, which keeps the swizzle phase), blocks past the sequence and
// invalid ids at an outer coordinate past the pool, which reads as zeros, and
// the rows past N of the sequence's last block through the tail map, which
// reads them as zeros as well.
// policy != 0: every copy carries that L2 cache policy.  st != null: an
// invalid block id the sequence's table names is recorded there.
RKV_DEV void load_key_rows(uint8_t* dst, int chunk_bytes, int KC, const KeyMaps* maps,
                           uint64_t* bar, int64_t p, int r0, int rows, const KeySource& ks,
                           uint64_t policy = 0, DeviceStatus* st = nullptr) {
    if (ks.table == nullptr) {
        for (int c = 0; c < KC; ++c) {
            if (policy)
                tma_load_3d_hint(dst + c * chunk_bytes, &maps->main, bar, c * 64, r0, (int)p, policy);
            else
                tma_load_3d(dst + c * chunk_bytes, &maps->main, bar, c * 64, r0, (int)p);
        }
        return;
    }
    const int64_t s = p / ks.H;
    const int h = (int)(p - s * ks.H);
    const int32_t* row = ks.table + s * ks.max_blocks;
    const int box = ks.log2bs < 7 ? 1 << ks.log2bs : 128;  // rows per TMA box
    for (int t = 0; t < rows; t += box) {
        const int r = r0 + t;
        const int lb = r >> ks.log2bs;
        int z = ks.num_blocks * ks.H;
        if (lb < ks.nb) {
            const int blk = __ldg(row + lb);
            if ((unsigned)blk < (unsigned)ks.num_blocks) z = blk * ks.H + h;
            else if (st) set_error(st, kDevErrIndex, (unsigned)lb);
        }
        const int y = r & ((1 << ks.log2bs) - 1);
        const CUtensorMap* map = &maps->main + (lb == ks.nb - 1 && ks.tail_rows > 0 ? 1 : 0);
        for (int c = 0; c < KC; ++c) {
            if (policy)
                tma_load_3d_hint(dst + c * chunk_bytes + t * 128, map, bar, c * 64, y, z, policy);
            else
                tma_load_3d(dst + c * chunk_bytes + t * 128, map, bar, c * 64, y, z);
        }
    }
}
// Eight bf16 of a 128-byte-swizzled K-major tile: 16-byte unit u of row r
// sits at unit u ^ (r mod 8) of the row (the TMA 128-byte swizzle).
RKV_DEV uint4 swizzled_unit(const uint8_t* tile, int r, int u) {
    return *reinterpret_cast<const uint4*>(tile + r * 128 + ((u ^ (r & 7)) << 4));
}

// the two bf16 of a 32-bit word as a packed fp32 pair (low element first)
RKV_DEV unsigned long long bf16x2_to_f32x2(uint32_t w) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(w << 16), "r"(w & 0xffff0000u));
    return r;
}

// acc.xy += a.xy * b.xy on packed fp32 pairs
RKV_DEV void fma_f32x2(unsigned long long& acc, unsigned long long a, unsigned long long b) {
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(a), "l"(b));
}

RKV_DEV float f32x2_sum(unsigned long long v) {
    return __uint_as_float((uint32_t)v) + __uint_as_float((uint32_t)(v >> 32));
}

// k . s over the D elements of row r of a key block (KC swizzled chunks of
// 64), s in fp32; four packed accumulators keep the FMA chains short
// (chunks of 128 rows x 128 bytes, kChunkBytes apart)
template <int KC>
RKV_DEV float row_dot(const uint8_t* blk, int r, const float* s32) {
    constexpr int kChunkBytes = 128 * 128;
    unsigned long long acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
    for (int c = 0; c < KC; ++c) {
        const uint8_t* tile = blk + c * kChunkBytes;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const uint4 k = swizzled_unit(tile, r, u);
            const ulonglong2 s01 = *reinterpret_cast<const ulonglong2*>(s32 + c * 64 + u * 8);
            const ulonglong2 s23 = *reinterpret_cast<const ulonglong2*>(s32 + c * 64 + u * 8 + 4);
            fma_f32x2(acc[0], bf16x2_to_f32x2(k.x), s01.x);
            fma_f32x2(acc[1], bf16x2_to_f32x2(k.y), s01.y);
            fma_f32x2(acc[2], bf16x2_to_f32x2(k.z), s23.x);
            fma_f32x2(acc[3], bf16x2_to_f32x2(k.w), s23.y);
        }
    }
    return (f32x2_sum(acc[0]) + f32x2_sum(acc[1])) + (f32x2_sum(acc[2]) + f32x2_sum(acc[3]));
}

// The same dot product one 64-column chunk at a time, for kernels whose
// other warps leave little register room.
template <int KC>
RKV_DEV float row_dot_lean(const uint8_t* blk, int r, const float* s32) {
    constexpr int kChunkBytes = 128 * 128;
    unsigned long long acc[2] = {0ull, 0ull};
#pragma unroll 1
    for (int c = 0; c < KC; ++c) {
        const uint8_t* tile = blk + c * kChunkBytes;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const uint4 k = swizzled_unit(tile, r, u);
            const ulonglong2 s01 = *reinterpret_cast<const ulonglong2*>(s32 + c * 64 + u * 8);
            const ulonglong2 s23 = *reinterpret_cast<const ulonglong2*>(s32 + c * 64 + u * 8 + 4);
            fma_f32x2(acc[0], bf16x2_to_f32x2(k.x), s01.x);
            fma_f32x2(acc[1], bf16x2_to_f32x2(k.y), s01.y);
            fma_f32x2(acc[0], bf16x2_to_f32x2(k.z), s23.x);
            fma_f32x2(acc[1], bf16x2_to_f32x2(k.w), s23.y);
        }
    }
    return f32x2_sum(acc[0]) + f32x2_sum(acc[1]);
}

RKV_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
RKV_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
RKV_DEV void tmem_alloc(uint32_t* dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst)),
                 "r"(ncols)
                 : "memory");
}
RKV_DEV void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
RKV_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
RKV_DEV void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                      uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
RKV_DEV void mma_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}
RKV_DEV void tmem_ld_32cols(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, "
        "[%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
}
// The same load that also returns, per lane, the maximum of the 32 values
// (tcgen05.ld.red with .max, an sm_103a form): the reduction comes with the
// load instead of a tree of max instructions over the registers.
RKV_DEV void tmem_ld_32cols_max(uint32_t taddr, uint32_t (&r)[32], float& m) {
    asm volatile(
        "tcgen05.ld.red.sync.aligned.32x32b.x32.max.f32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, "
        "%32, [%33];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31]), "=f"(m)
        : "r"(taddr));
}
RKV_DEV void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor of a K-major tile written by TMA with the
// 128-byte swizzle: 8-row groups 1024 bytes apart (stride byte offset), rows
// of 128 bytes.  The tile base must be 1024-byte aligned; advancing the start
// address by 32 bytes selects the next 16-element K slice.
RKV_DEV uint64_t sdesc_sw128(const void* p) {
    const uint64_t a = smem_u32(p);
    uint64_t d = (a >> 4) & 0x3FFFull;   // start address
    d |= 1ull << 16;                      // leading byte offset (unused here)
    d |= (uint64_t)(1024 >> 4) << 32;     // stride byte offset
    d |= 1ull << 46;                      // descriptor version
    d |= 2ull << 61;                      // 128-byte swizzle
    return d;
}

// Instruction descriptor of tcgen05.mma kind::f16: D fp32, A and B bf16,
// both K-major, shape M x N.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

// Smallest power of two >= n, at least 32 (a legal TMEM allocation).
__host__ __device__ constexpr uint32_t tmem_cols(uint32_t n) {
    uint32_t c = 32;
    while (c < n) c <<= 1;
    return c;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled from the driver (no link-time dependency on libcuda).
EncodeTiledFn encode_fn();

// 3-D bf16 tensor map [outer][rows][inner] with a box of 64 inner elements
// (128 bytes, 128-byte swizzle) x box_rows x 1; rows >= `rows` read as zero.
bool make_map_3d_bf16(CUtensorMap* map, const void* base, int inner, int rows,
                      int64_t outer, int64_t row_stride_elems, int64_t outer_stride_elems,
                      int box_rows);

int sm_count();
// The tensor maps of a call's keys: the contiguous [P][N][D] map with boxes of
// box_rows rows (ks: no table), or, for paged keys read directly, the pool map
// [H * num_blocks][block size][D] with boxes of min(block size, 128) rows, its
// copy with a row extent of the last block's rows before N, and ks filled from
// the call's table.
bool make_key_map(KeyMaps* maps, const ScoreArgs& a, int D, int box_rows, KeySource* ks);
// One prefetch of each of a call's key maps.
RKV_DEV void prefetch_key_maps(const KeyMaps* maps) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&maps->main)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&maps->tail)) : "memory");
}

}  // namespace tc
}  // namespace rkv
