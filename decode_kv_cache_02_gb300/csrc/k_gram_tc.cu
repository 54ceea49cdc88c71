// k_gram_tc.cu -- tensor-core (tcgen05) thresholded key Gram; see below.
#include "rkv_common.cuh"
#include "rkv_internal.h"
#include "../../include/rkv.h"

namespace rkv {

bool gram_tc_supported(const ScoreArgs& a) {
    (void)a;
    return false;
}

cudaError_t launch_gram_tc(const ScoreArgs& a, cudaStream_t s) {
    (void)a;
    (void)s;
    return cudaErrorNotSupported;
}

}  // namespace rkv
