// rkv_internal.h -- launchers shared between the C-ABI layer and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/rkv.h"

namespace rkv {

struct DeviceStatus;

// A paged pool [num_blocks, H, 1 << log2bs, d]: logical row r of problem
// p = s * H + h lives in block table[s * max_blocks + (r >> log2bs)], head h,
// row r & (bs - 1).  table == nullptr: the contiguous layout.
struct PagedIn {
    const int32_t* table = nullptr;
    int max_blocks = 0;
    int log2bs = 0;
    int H = 1;
    int num_blocks = 0;
};

// Where the tensor-core kernels' TMA loads find the key rows: with table ==
// nullptr the contiguous map (outer coordinate = problem); otherwise a map of
// the paged pool (rows = the rows of one block, outer = block * H + head) read
// one block (or, for blocks over 128 rows, 128 rows) at a time through the
// table, blocks past the sequence's nb blocks (and invalid ids) read as zero.
// The sequence's last block is read through a second map of the pool whose
// row extent is tail_rows, so its rows past N read as zero too and the pool's
// unfilled space is never touched.
struct KeySource {
    const int32_t* table = nullptr;
    int max_blocks = 0;
    int log2bs = 0;
    int H = 1;
    int nb = 0;          // blocks holding the problem's N rows
    int num_blocks = 0;
    int tail_rows = 0;   // rows of the last block before N (0: the block is full)
};

// Everything the scoring kernels of one call need.
struct ScoreArgs {
    const void* K;       // [P, n_cap, d]
    const void* Q;       // [P, G, n_obs, d]
    int64_t P;
    int G, d, n_cap, N, n_obs, beta;
    int dtype;           // RKV_DTYPE_*
    float lambda, tau;
    // workspace rows (stride ld_ws floats per problem)
    float* inv_norm;     // 1 / max(|k_i|, eps)
    float* sum_s;        // sum_{j != i} S_ij
    void* s_rows;        // [P, 16, d] bf16: s = sum_j khat_j as (hi, lo, 0...)
    bool stats_sum;      // key stats write sum_s (else importance completes it)
    int64_t ld_ws;
    // outputs (stride ld_out floats per problem); R may be null
    float* I;
    float* R;
    float* Z;
    int64_t ld_out;
    DeviceStatus* status;
    // paged input: key stats read K through pg and write the contiguous
    // copy Kc [P, N, d], which the later stages read instead
    PagedIn pg;
    void* Kc = nullptr;
    // paged keys read directly by the tensor-core stages (K is then the pool)
    bool paged_direct = false;
    // the key statistics come from the resident importance kernel (inv_i,
    // |khat_i|^2, s in fp32 at s_rows) and the Gram completes sum_i; no
    // separate statistics pass
    bool fused_stats = false;
    // SMs the persistent kernels size their grid to (0: the whole device);
    // the SM count of the partition they are launched on
    int sms = 0;
};

// One SM partition of the device with a stream of its own (rkv_lanes.cu).
struct Lane {
    void* ctx = nullptr;  // the partition's CUcontext
    cudaStream_t stream = nullptr;
    int sms = 0;
    int id = 0;  // 1: tensor lane, 2: hbm lane (0 is the caller's stream)
};
// tensor: the Gram's partition; hbm: the importance and compaction's.
struct Lanes {
    Lane tensor, hbm;
};
// The split of the current device with about tensor_sms SMs on the tensor
// lane (whole groups of the split, 4 SMs here), created on first use and kept; nullptr when the
// driver offers no SM partitions.
const Lanes* lanes_for_current_device(int tensor_sms);
// Makes a lane's context current for the scope: kernels launched and events
// created meanwhile belong to the lane (lane == nullptr: no change).
class LaneScope {
public:
    explicit LaneScope(const Lane* lane);
    ~LaneScope();
    LaneScope(const LaneScope&) = delete;
    LaneScope& operator=(const LaneScope&) = delete;

private:
    bool pushed_;
};

cudaError_t launch_key_stats(const ScoreArgs& a, cudaStream_t s);
cudaError_t launch_importance(const ScoreArgs& a, cudaStream_t s);
// *_shape_ok: the sizes and parameters a tensor-core kernel takes;
// *_supported: that, and the driver's tensor-map entry point is present.
bool importance_tc_shape_ok(const ScoreArgs& a);
bool importance_tc_supported(const ScoreArgs& a);
// the importance kernel that keeps a problem's logits in TMEM takes this shape
bool importance_tc_resident(const ScoreArgs& a);
cudaError_t launch_importance_tc(const ScoreArgs& a, cudaStream_t s);
cudaError_t launch_gram_simt(const ScoreArgs& a, cudaStream_t s);
bool gram_tc_shape_ok(const ScoreArgs& a);
bool gram_tc_supported(const ScoreArgs& a);
// the one-row-block Gram (N <= 2048), which can complete sum_i itself
bool gram_tc_rows(const ScoreArgs& a);
cudaError_t launch_gram_tc(const ScoreArgs& a, cudaStream_t s);
// the tensor-core Gram for 2048 < N <= 4352 (launch_gram_tc dispatches to it)
cudaError_t launch_gram_tc_pairs(const ScoreArgs& a, cudaStream_t s);

cudaError_t launch_select(int64_t P, int N, const float* Z, int64_t ldz, int n_obs,
                          int budget, int32_t* idx, DeviceStatus* st, cudaStream_t s);

// Copies kept rows of up to two tensors (b may be null): sources hold n_cap
// rows per problem, destinations out_cap (= n_cap in place).  row_bytes is a
// multiple of 16; in_place means dst == src for both tensors.
cudaError_t launch_gather(const void* src_a, const void* src_b, void* dst_a, void* dst_b,
                          const int32_t* idx, int64_t P, int n_cap, int out_cap, int budget,
                          int row_bytes, bool in_place, DeviceStatus* st, cudaStream_t s);

// idx rows = 0..n-1 then -1 (nothing evicted).
cudaError_t launch_identity_idx(int64_t P, int n, int budget, int32_t* idx, cudaStream_t s);
// A scoring variant applied inside the fused select + gather: Z is computed
// from the base I and R rows (stride ld) instead of read.  I == nullptr: read Z.
struct VariantIn {
    const float* I = nullptr;
    const float* R = nullptr;
    int64_t ld = 0;
    float lambda = 0.f;
    int softmax = 0;
    int half = 0;  // (pool window - 1) / 2
    // sentence-level penalty: Z_i -= pen[s, seg[p, i]] for 0 <= seg < count[s],
    // s = (p / heads) % num_seqs; seg rows are compacted with the kept rows
    const float* pen = nullptr;  // [num_seqs, max_sent]
    const int32_t* count = nullptr;
    int32_t* seg = nullptr;  // [P, ld_seg]
    int64_t ld_seg = 0;
    int64_t num_seqs = 1;
    int heads = 1;
    int max_sent = 0;
    // sampled selection: pool of the top `pool` candidates by Z, then the top
    // k of Z * inv_temp - log(-log(u)) within it (u: unif rows, stride ld_u)
    bool sample = false;
    int pool = 0;
    float inv_temp = 1.f;
    const float* unif = nullptr;
    int64_t ld_u = 0;
};

// Sentence penalties pen[s, a] = max_{b > a, cos(a, b) > tau} cos(a, b) from
// reps [S, max_sent, hidden] (fp32) and count [S].
cudaError_t launch_sentence_penalty(int64_t S, int max_sent, int hidden, const float* reps,
                                    const int32_t* count, float tau, float* pen, cudaStream_t s);
// Sentence representations: the mean hidden state of each sentence's tokens.
cudaError_t launch_sentence_reps(const void* hidden, int dtype, const int32_t* token_seg,
                                 int64_t S, int T, int hidden_dim, int max_sent, float* reps,
                                 cudaStream_t s);

// select + gather fused (one CTA per problem); dynamic shared memory it needs
size_t compact_smem_bytes(int N, int n_obs, int budget, bool sentences = false);
cudaError_t launch_compact(int64_t P, int N, const float* Z, int64_t ldz, int n_obs, int budget,
                           int32_t* idx, const void* src_a, const void* src_b, void* dst_a,
                           void* dst_b, int n_cap, int out_cap, int row_bytes, bool in_place,
                           DeviceStatus* st, cudaStream_t s, const VariantIn& var = VariantIn{});
// The same on a paged pool, in place: kept K rows come from the contiguous
// copy kc [P, N, d], kept V rows move inside v_pool; both land in the pool
// rows of logical positions 0..budget-1.
cudaError_t launch_compact_paged(int64_t P, int N, const float* Z, int64_t ldz, int n_obs,
                                 int budget, int32_t* idx, const void* kc, void* k_pool,
                                 void* v_pool, const PagedIn& pg, int row_bytes, DeviceStatus* st,
                                 cudaStream_t s, const VariantIn& var = VariantIn{});
// Hands back each sequence's blocks past the kept ones: out_freed[s, j] =
// table[s, nb_keep + j], then that entry = -1, for j < nb_old - nb_keep.
cudaError_t launch_paged_release(int64_t S, int32_t* table, int max_blocks, int nb_keep,
                                 int nb_old, int32_t* out_freed, cudaStream_t s);

// Variant scores (redundancy softmax, importance pooling window, sentence
// penalty) from the base I and R rows of v: Z, and I', R' when I_out / R_out
// are given (stride ld_out).
cudaError_t launch_variant(int64_t P, int N, int n_obs, const VariantIn& v, float* Z,
                           float* I_out, float* R_out, int64_t ld_out, cudaStream_t s);

// One bounded wait that nothing completes (the failure path of every wait):
// records kDevErrTimeout in st after the wait limit (~1 s).
cudaError_t launch_wait_timeout(DeviceStatus* st, cudaStream_t s);

// rkv_compress_ex; with clear_status the workspace's device error word is
// cleared (enqueued) once the arguments have passed every check; with lanes
// the step may take the two-partition schedule (rkv_set_overlap), whose first
// use creates the partitions' contexts.
int compress_call(const rkv_desc* desc, const void* K, const void* V, const void* Q_obs,
                  int n_cached, int budget, int n_obs, float lambda, int beta, float tau,
                  const rkv_variant* variant, void* out_K, void* out_V, int32_t* out_idx,
                  void* workspace, size_t workspace_bytes, void* stream, bool clear_status,
                  bool lanes);

}  // namespace rkv
