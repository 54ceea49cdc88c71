// tcgen05_host.cu -- host helpers of the tensor-core kernels: the driver's
// tensor-map encoder (looked up at run time) and the SM count.
#include <mutex>

#include "tcgen05.cuh"

namespace rkv {
namespace tc {

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

bool make_map_3d_bf16(CUtensorMap* map, const void* base, int inner, int rows, int64_t outer,
                      int64_t row_stride_elems, int64_t outer_stride_elems, int box_rows) {
    EncodeTiledFn enc = encode_fn();
    if (!enc || rows < 1 || outer < 1) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)rows, (cuuint64_t)outer};
    const cuuint64_t strides[2] = {(cuuint64_t)row_stride_elems * 2,
                                   (cuuint64_t)outer_stride_elems * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_key_map(KeyMaps* maps, const ScoreArgs& a, int D, int box_rows, KeySource* ks) {
    *ks = KeySource{};
    if (!a.paged_direct) {
        if (!make_map_3d_bf16(&maps->main, a.K, D, a.N, a.P, D, (int64_t)a.n_cap * D, box_rows))
            return false;
        maps->tail = maps->main;  // not used without a table
        return true;
    }
    const int bs = 1 << a.pg.log2bs;
    ks->table = a.pg.table;
    ks->max_blocks = a.pg.max_blocks;
    ks->log2bs = a.pg.log2bs;
    ks->H = a.pg.H;
    ks->nb = (a.N + bs - 1) / bs;
    ks->num_blocks = a.pg.num_blocks;
    const int rem = a.N - (ks->nb - 1) * bs;  // rows of the last block before N
    ks->tail_rows = rem < bs ? rem : 0;
    const int64_t outer = (int64_t)a.pg.H * a.pg.num_blocks;
    const int box = bs < 128 ? bs : 128;
    if (!make_map_3d_bf16(&maps->main, a.K, D, bs, outer, D, (int64_t)bs * D, box))
        return false;
    if (ks->tail_rows == 0) {
        maps->tail = maps->main;
        return true;
    }
    return make_map_3d_bf16(&maps->tail, a.K, D, ks->tail_rows, outer, D, (int64_t)bs * D, box);
}

int sm_count() {
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        n = 148;
    return n;
}

}  // namespace tc
}  // namespace rkv
