/*
 * rkv.h -- C ABI of librkv, the GB300 (sm_103a) implementation of R-KV's
 * decode-time KV-cache compression step.
 *
 * The operation (R-KV review, yoonschallenge.tistory.com/1236):
 *   - opening notes and summary-table row "Decoding-time compression
 *     scheme": the fixed cache B_budget and the buffer B_buffer of newly
 *     generated tokens are merged (here: rows 0..budget-1 followed by the
 *     buffer rows, n_cached rows in all); the newest n_obs (8) observation
 *     tokens are always kept; every other token is scored and only the top
 *     ones are kept, so that exactly `budget` rows remain.
 *   - row "importance": I_i is the softmax attention the n_obs observation
 *     queries give key i (mean over the queries, scale 1/sqrt(d), causal among
 *     the observation tokens), max-pooled over the G query heads that share
 *     the KV head.
 *   - row "redundancy": R_i is the mean cosine similarity of key i to the
 *     other n_cached-1 keys of the same KV head; a similar pair is one with
 *     cosine > tau; token i is protected (its above-tau similarities are
 *     dropped from its sum) when fewer than beta newer tokens are similar to
 *     it, i.e. the beta most recent tokens of a similar group are protected.
 *   - row "final selection criterion": Z_i = lambda*I_i - (1-lambda)*R_i
 *     (lambda = 0.1 on the page); ties go to the newer token.
 *   - question 2, cause 3: the kept K/V rows are copied into the new cache.
 *
 * One "problem" is one (layer, sequence, KV head).  All P problems of a call
 * share n_cached, budget and the parameters and are processed by one launch
 * per kernel.
 *
 * Layouts (every array contiguous, row-major; element type `dtype`):
 *   K, V                 [P, n_capacity, head_dim]; problem p starts at
 *                        element p*n_capacity*head_dim.  head_dim*elem_size
 *                        must be a multiple of 16 bytes and every base pointer
 *                        16-byte aligned.
 *   out_K, out_V         [P, out_capacity, head_dim] (out_capacity = 0 in the
 *                        descriptor means n_capacity): an out-of-place call
 *                        may write the kept rows into buffers of just
 *                        `budget` rows per problem.
 *   Q_obs                [P, G, n_obs, head_dim]: query q of query head g of
 *                        problem p.  Query head g of the G that share the KV
 *                        head of problem p.
 *   out_idx              [P, budget] int32.
 *   out_I, out_R, out_Z  [P, n_cached] float.
 *
 * Ownership and execution: every pointer is device memory owned by the
 * caller.  The calls never allocate or free device memory and never
 * synchronise: they check their arguments on the host, enqueue kernels on
 * `stream` (a cudaStream_t, or NULL for the legacy default stream) and return.
 * Results are valid in stream order.  Scratch memory is the caller's
 * `workspace` of at least rkv_workspace_size() bytes, 256-byte aligned; one
 * workspace must not be used by two calls that may overlap on the GPU.
 *
 * Errors: each call returns RKV_OK or an RKV_ERR_* code and enqueues nothing
 * on error.  Errors raised on the device (a bounded wait that timed out, an
 * index found out of range) are recorded in the workspace and read by
 * rkv_get_device_status().  Not thread-safe only where stated.
 */
#ifndef RKV_H
#define RKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
    RKV_OK = 0,
    RKV_ERR_INVALID_ARG = 1, /* a size, count or pointer is invalid */
    RKV_ERR_UNSUPPORTED = 2, /* dtype / head_dim / group size not supported */
    RKV_ERR_WORKSPACE = 3,   /* workspace missing, misaligned or too small */
    RKV_ERR_ALIAS = 4,       /* outputs partially overlap inputs */
    RKV_ERR_CUDA = 5,        /* a CUDA runtime call or launch failed */
    RKV_ERR_DEVICE = 6,      /* a kernel recorded an error (see status) */
    RKV_ERR_TOO_LARGE = 7    /* request exceeds rkv_compress_noalloc's scratch */
};

enum { RKV_DTYPE_BF16 = 0, RKV_DTYPE_FP32 = 1 };

/* Shape of one call's problems. */
typedef struct {
    int64_t num_problems; /* P = layers * sequences * kv_heads (>= 0)        */
    int32_t gqa_group;    /* G, query heads per KV head, 1..16               */
    int32_t head_dim;     /* d, 64 or 128                                    */
    int32_t n_capacity;   /* rows allocated per problem in K and V           */
    int32_t dtype;        /* RKV_DTYPE_BF16 or RKV_DTYPE_FP32 (K, V, Q, out) */
    int32_t out_capacity; /* rows per problem in out_K/out_V (and rkv_gather's
                             dst); 0 = n_capacity.  Must be >= budget, and 0 or
                             n_capacity for in-place compaction.             */
} rkv_desc;

/* Largest n_cached accepted by rkv_compress / rkv_score. */
#define RKV_MAX_TOKENS 32768

/* Bytes of workspace rkv_compress / rkv_score need for `desc` and n_cached
 * tokens with n_obs observation tokens.  0 if the arguments are invalid. */
size_t rkv_workspace_size(const rkv_desc* desc, int n_cached, int n_obs);

/* One compression round (the whole step above) for all P problems.
 *   n_cached   rows in use per problem (merged cache + buffer), <= n_capacity
 *   budget     rows kept per problem, n_obs <= budget <= n_capacity and
 *              budget <= out_capacity
 *   n_obs      observation tokens (the newest n_obs rows), >= 1
 *   lambda, beta, tau   the parameters of Z, protection and similarity
 *   out_K/out_V  receive the kept rows in ascending original position in
 *              their rows 0..budget-1; rows >= budget are not touched.  They
 *              may be K/V themselves (in-place compaction) but must not
 *              overlap them otherwise (RKV_ERR_ALIAS).
 *   out_idx    [P, budget]: kept original row indices, strictly ascending;
 *              the last n_obs are n_cached-n_obs .. n_cached-1.
 * n_cached <= budget evicts nothing: out_idx = 0..n_cached-1 then -1, and the
 * rows are copied only when the outputs are not the inputs. */
int rkv_compress(const rkv_desc* desc, const void* K, const void* V, const void* Q_obs,
                 int n_cached, int budget, int n_obs, float lambda, int beta, float tau,
                 void* out_K, void* out_V, int32_t* out_idx,
                 void* workspace, size_t workspace_bytes, void* stream);

/* The scores alone (for tests and analysis): out_I, out_R, out_Z
 * [P, n_cached].  Observation tokens get R = 0 and Z = +inf. */
int rkv_score(const rkv_desc* desc, const void* K, const void* Q_obs, int n_cached,
              int n_obs, float lambda, int beta, float tau,
              float* out_I, float* out_R, float* out_Z,
              void* workspace, size_t workspace_bytes, void* stream);

/* Variants of the scoring (all off: the step above).
 *   redundancy_softmax  the R-KV review, question 2, cause 3, lists a softmax
 *                       of the redundancy among the operations of a
 *                       compression round.  1: the candidates' redundancy
 *                       becomes R'_i = exp(R_i) / sum_{j<C} exp(R_j) (R_i as
 *                       above, C = n_cached - n_obs candidates), so it sums
 *                       to 1 over the candidates; 0: R as above.
 *   pool_window         w, odd, 1..RKV_MAX_POOL_WINDOW.  A SnapKV-style
 *                       pooling of the importance over positions (SnapKV is
 *                       the attention-only method the review compares
 *                       against): I'_i = max of I_j over the candidates j
 *                       with |j - i| <= (w-1)/2 (the window is cut at the
 *                       candidates' ends).  1: no pooling.
 *   sentences           a sentence-level penalty (below), or NULL.
 *   schedule            a recent window and sampled selection (below), or
 *                       NULL.  With a schedule the L newest rows take the
 *                       place of the observation tokens in everything that
 *                       follows (they are not candidates; Z = +inf, R = 0).
 * Z_i = lambda*I'_i - (1-lambda)*R'_i - pen_i; observation tokens keep their
 * I, get R = 0 and Z = +inf as before.  A NULL variant is all off. */
/* Sentence-level redundancy (the SkipKV review, yoonschallenge.tistory.com/
 * 1230, summary-table rows "Method 1: Sentence-level KV Storage Skipping",
 * "Final eviction score" and "Cache Range Monitoring").  A sentence is
 * represented by the mean of its tokens' last-layer hidden states
 * (rkv_sentence_reps computes it); when the cosine similarity of sentence a
 * and a later sentence b of the same sequence exceeds tau, a is the
 * redundant one.  Its penalty is pen_a = max of cos(a, b) over the later b
 * with cos(a, b) > tau (0 if none), and every cached row of sentence a has
 * pen_a subtracted from its Z, so redundant earlier sentences go first while
 * the budget still decides how many rows stay.  The sentence of each cached
 * row is tracked in seg_id, which the compression compacts along with the
 * rows (the cache-range mapping the review describes).
 *   reps      [num_seqs, max_sentences, hidden_dim] fp32 (rows >= count[s]
 *             ignored)
 *   count     [num_seqs] sentences in use per sequence (device memory)
 *   seg_id    [P, ld_seg] int32: sentence of cached row i of problem p, or
 *             -1 (ids outside 0..count-1 count as none).  Problem p belongs
 *             to sequence (p / heads) % num_seqs (problems ordered layer,
 *             sequence, head).  After rkv_compress_ex / rkv_paged_compress
 *             entries 0..budget-1 hold the kept rows' sentences.
 *   penalty   [num_seqs, max_sentences] fp32, written: pen_a per sentence.
 * All pointers are device memory owned by the caller. */
typedef struct {
    const float* reps;
    const int32_t* count;
    int32_t* seg_id;
    float* penalty;
    int64_t num_seqs;      /* >= 1 */
    int32_t heads;         /* >= 1 */
    int32_t max_sentences; /* 1 .. RKV_MAX_SENTENCES */
    int32_t hidden_dim;    /* 4 .. RKV_MAX_HIDDEN, a multiple of 4 */
    int32_t ld_seg;        /* row stride of seg_id, >= n_cached */
    float tau;             /* sentence-similarity threshold */
} rkv_sentences;
#define RKV_MAX_SENTENCES 65536
#define RKV_MAX_HIDDEN 16384

/* ForesightKV-style schedule and selection (the ForesightKV summary page,
 * gist.science/ko/paper/2602.03203, section "Dynamic eviction process"):
 * when the cache holds B + L rows the newest L are kept and the rest are
 * compressed to B - L by the scores; the decision takes the top K and then
 * samples (multinomial sampling) to add randomness.  The R-KV score Z stands
 * in for the page's learned scorer.  Here:
 *   - the newest L = recent_window rows (n_obs <= L <= budget) are kept like
 *     the observation tokens (which still supply the importance queries);
 *     the other C = n_cached - L rows are the candidates, k = budget - L of
 *     them are kept;
 *   - the pool is the top pool_size candidates by Z (ties to the newer);
 *   - k of the pool are drawn without replacement with probabilities
 *     proportional to exp(Z_i / temperature): exactly the k largest
 *     Z_i / temperature + g_i over the pool, g_i = -log(-log(u_i)) (Gumbel
 *     noise) from the caller's uniforms u [P, ld_uniforms] in [0, 1), so a
 *     seeded generator on the caller's side makes the draw reproducible.
 * pool_size == k is the deterministic top-k (uniforms may be NULL). */
typedef struct {
    int32_t recent_window;  /* L */
    int32_t pool_size;      /* K, k <= K <= C */
    float temperature;      /* > 0 */
    int32_t ld_uniforms;    /* >= C when uniforms are given */
    const float* uniforms;  /* [P, ld_uniforms]; needed when K > k */
} rkv_schedule;

typedef struct {
    int32_t redundancy_softmax;       /* 0 or 1 */
    int32_t pool_window;              /* odd, 1 .. RKV_MAX_POOL_WINDOW */
    const rkv_sentences* sentences;   /* NULL: no sentence-level penalty */
    const rkv_schedule* schedule;     /* NULL: keep the n_obs newest, top-k */
} rkv_variant;
#define RKV_MAX_POOL_WINDOW 255

/* Sentence representations: out_reps[s, a, :] = mean of hidden[s, t, :] over
 * the tokens t with token_seg[s, t] == a (zeros for a sentence without
 * tokens).  hidden [num_seqs, T, hidden_dim] (dtype bf16 or fp32), token_seg
 * [num_seqs, T] int32 (-1: no sentence; ids >= max_sentences ignored),
 * out_reps [num_seqs, max_sentences, hidden_dim] fp32. */
int rkv_sentence_reps(const void* hidden, const int32_t* token_seg, int64_t num_seqs, int T,
                      int hidden_dim, int dtype, int max_sentences, float* out_reps,
                      void* stream);

/* The penalties alone: writes sent->penalty from reps, count and tau. */
int rkv_sentence_penalty(const rkv_sentences* sent, void* stream);

/* rkv_compress / rkv_score with a variant (invalid variant fields:
 * RKV_ERR_INVALID_ARG).  rkv_score_ex's out_I and out_R are the I' and R'
 * that enter Z. */
int rkv_compress_ex(const rkv_desc* desc, const void* K, const void* V, const void* Q_obs,
                    int n_cached, int budget, int n_obs, float lambda, int beta, float tau,
                    const rkv_variant* variant, void* out_K, void* out_V, int32_t* out_idx,
                    void* workspace, size_t workspace_bytes, void* stream);
int rkv_score_ex(const rkv_desc* desc, const void* K, const void* Q_obs, int n_cached,
                 int n_obs, float lambda, int beta, float tau, const rkv_variant* variant,
                 float* out_I, float* out_R, float* out_Z,
                 void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------- paged --
 * The step on a paged KV cache.  The review (question 2, cause 4) names the
 * clash between pruning and a block-structured (PagedAttention) cache as a
 * main limitation: pruning re-lays the KV tensor out, and freeing the old
 * cache to allocate a compressed one costs memory management.  Here a
 * sequence's rows live in fixed-size blocks of a shared pool, compaction runs
 * in place inside the sequence's own blocks, and the blocks it empties are
 * handed back whole.
 *
 * Layout: K_pool, V_pool [num_blocks, num_kv_heads, block_size, head_dim]:
 * one (block, head) is a contiguous block_size x head_dim tile.  Sequence s
 * (one row of block_table [num_seqs, max_blocks_per_seq], int32) holds its
 * logical row r of head h at block block_table[s][r / block_size], row
 * r % block_size.  Problem p = s * num_kv_heads + h; Q_obs is
 * [P, G, n_obs, head_dim] and out_idx [P, budget] as for rkv_compress.
 * The entries 0 .. ceil(n_cached / block_size) - 1 of every table row must be
 * distinct valid block ids, not shared between sequences; entries outside
 * 0..num_blocks-1 are recorded as a device error and their rows skipped.
 *
 * Effect: for every problem the kept rows (out_idx) move to logical rows
 * 0..budget-1 of the same sequence and head, in place; rows past budget in
 * the last kept block are left as they were.  The blocks past the kept ones,
 * entries ceil(budget/bs) .. ceil(n_cached/bs) - 1 of each row, are no longer
 * used: their ids are written to out_freed [num_seqs, n_free] (n_free =
 * rkv_paged_freed_per_seq()) and the table entries are set to -1.  Rows after
 * n_cached in each sequence's last block (space it has not filled yet) are
 * neither read nor written, and blocks not named by the first
 * ceil(n_cached/bs) entries of any row are not touched. */
typedef struct {
    int64_t num_seqs;           /* S, rows of the block table (>= 0)         */
    int32_t num_kv_heads;       /* H, heads per block; P = S * H problems     */
    int32_t gqa_group;          /* G, query heads per KV head, 1..16          */
    int32_t head_dim;           /* d, 64 or 128                               */
    int32_t block_size;         /* rows per block, a power of two, 1..1024    */
    int32_t num_blocks;         /* blocks in each pool (>= 1)                 */
    int32_t max_blocks_per_seq; /* row stride of block_table (>= 1)           */
    int32_t dtype;              /* RKV_DTYPE_BF16 or RKV_DTYPE_FP32           */
} rkv_paged_desc;

/* Workspace bytes rkv_paged_compress needs for these arguments (0 if they
 * are invalid).  bf16 pools with blocks of at least 128 rows are read in
 * place by the tensor-core stages when the call's shapes fit them (n_cached
 * <= 4352, gqa_group * n_obs a multiple of 8 up to 128, beta <= 63): then the
 * size equals rkv_workspace_size() of the same problems.  Otherwise (blocks
 * under 128 rows, fp32 pools, the CUDA-core paths) it adds one contiguous
 * copy of the P problems' keys [P, n_cached, head_dim], which the key
 * statistics write for the later stages. */
size_t rkv_paged_workspace_size(const rkv_paged_desc* desc, int n_cached, int n_obs,
                                int beta);

/* Blocks freed per sequence: ceil(n_cached/bs) - ceil(budget/bs), or 0 when
 * n_cached <= budget; -1 if the arguments are invalid. */
int rkv_paged_freed_per_seq(const rkv_paged_desc* desc, int n_cached, int budget);

/* One compression round on the paged cache (see above).  n_cached <= budget:
 * out_idx is the identity and nothing moves or is freed.  Problems whose
 * scores, keys and kept indices exceed the fused selection kernel's shared
 * memory (8*(n_cached-n_obs) + 4*budget > 160 KB) return RKV_ERR_UNSUPPORTED. */
int rkv_paged_compress(const rkv_paged_desc* desc, void* K_pool, void* V_pool,
                       const void* Q_obs, int32_t* block_table, int n_cached, int budget,
                       int n_obs, float lambda, int beta, float tau,
                       const rkv_variant* variant, int32_t* out_idx, int32_t* out_freed,
                       void* workspace, size_t workspace_bytes, void* stream);

/* The selection alone: for scores Z [P, n] (fp32), out_idx [P, budget] as
 * rkv_compress would produce it (top budget-n_obs of the candidates
 * 0..n-n_obs-1 by Z, ties to the larger index, then the n_obs observation
 * tokens, ascending).  Requires n_obs <= budget < n <= RKV_MAX_TOKENS. */
int rkv_select(int64_t num_problems, int n, const float* Z, int n_obs, int budget,
               int32_t* out_idx, void* stream);

/* The copy alone: dst[p, r, :] = src[p, idx[p, r], :] for r < budget where
 * idx >= 0; src laid out as K in `desc`, dst as out_K (out_capacity rows per
 * problem); idx rows strictly ascending.  dst may equal src (in place, with
 * out_capacity 0 or n_capacity) but must not overlap it otherwise. */
int rkv_gather(const rkv_desc* desc, const void* src, const int32_t* idx, int budget,
               void* dst, void* stream);

/* Clears the device error word at the start of `workspace` (enqueued on
 * `stream`).  Call once on a fresh workspace before its first use, unless the
 * workspace was allocated zero-filled. */
int rkv_workspace_init(void* workspace, void* stream);

/* Synchronises `stream`, returns the first error a kernel recorded in
 * `workspace` since the last call (RKV_OK if none) and clears it. */
int rkv_get_device_status(void* workspace, void* stream);

/* rkv_compress without a caller workspace.  The pages have no counterpart:
 * this is a deployment convenience for callers that may not allocate device
 * memory while they run (an engine plugin or custom op whose host framework
 * owns all device memory, a process whose memory is reserved up front for the
 * KV cache).  Same arguments, results and stream semantics as rkv_compress;
 * the scratch is a static array of RKV_NOALLOC_SCRATCH_BYTES inside the
 * library, held by every GPU that loads it until exit.  Requests whose
 * rkv_workspace_size() exceeds it return RKV_ERR_TOO_LARGE before anything is
 * enqueued (16 MiB holds the scratch of about 700 thousand token slots, e.g.
 * one Llama-8B layer at batch 64 with N = 1152, or 195 problems of 4096).
 * Never allocates or frees device memory.
 * Every call looks up the array's device address on the current device
 * (cudaGetSymbolAddress, a host-side lookup).  The first lookup on a device
 * may load the library's device code there; make the first call on each
 * device before any stream capture: if the lookup fails (for instance because
 * a capture forbids loading code), the call returns RKV_ERR_CUDA and enqueues
 * nothing.  All calls share the array.  Once a call's arguments pass their
 * checks it clears the array's device error word (enqueued on `stream` before
 * its kernels); a rejected call enqueues nothing.  Calls that may overlap on
 * the GPU race on the array and must be serialised by the caller. */
#define RKV_NOALLOC_SCRATCH_BYTES (16u << 20)
int rkv_compress_noalloc(const rkv_desc* desc, const void* K, const void* V, const void* Q_obs,
                         int n_cached, int budget, int n_obs, float lambda, int beta, float tau,
                         void* out_K, void* out_V, int32_t* out_idx, void* stream);

/* rkv_get_device_status for rkv_compress_noalloc's static scratch on the
 * current device: synchronises `stream`, returns RKV_ERR_DEVICE if a kernel
 * recorded an error there since the last read (and clears it), RKV_OK
 * otherwise. */
int rkv_noalloc_device_status(void* stream);

/* rkv_selftest_wait_timeout on the static scratch of the current device (the
 * error word that rkv_noalloc_device_status reads). */
int rkv_noalloc_selftest_wait_timeout(void* stream);

/* Self-test of the failure path: enqueues one bounded wait that nothing
 * completes (the primitive every wait of the kernels uses).  After its limit
 * (about a second) it records a timeout in `workspace`, which
 * rkv_get_device_status() then reports as RKV_ERR_DEVICE; the context stays
 * usable.  Nothing hangs and nothing traps. */
int rkv_selftest_wait_timeout(void* workspace, void* stream);

/* Human-readable name of an RKV_* code. */
const char* rkv_strerror(int code);

/* Step schedule of rkv_compress / rkv_compress_ex / rkv_paged_compress
 * (process-wide).  A call whose keys are bf16 rows with N <= 2048 (contiguous,
 * or a paged pool of blocks of 128 rows or more, grouped by whole sequences),
 * that passes no variant, whose selection fits the fused compaction and whose
 * stream is not being captured into a graph can run on two SM partitions of
 * the device (driver green contexts, created at the first such call and
 * kept): the problems are cut into `groups` equal groups; importance and Gram
 * of each group run on the tensor partition (about tensor_sms SMs), and each
 * group's selection and row copy run on the other SMs while the tensor
 * partition scores the next group (the last group's on the whole device).
 * It needs at least
 * 2 * groups * tensor_sms problems.  Results are bit for bit those of one
 * launch per stage over the whole device.
 *   mode RKV_SCHEDULE_ONE_LAUNCH: always one launch per stage;
 *   mode RKV_SCHEDULE_AUTO (default): grouped where a cost model of the
 *     kernels' measured per-problem times predicts a gain (the Llama-8B-shaped
 *     step: yes; a few thousand problems or long rows compacted in place: no;
 *     paged pools: never);
 *   mode RKV_SCHEDULE_GROUPED: grouped wherever the call is eligible.
 * Defaults: groups = 8, tensor_sms = 0 (112 of every 152 SMs).  Calls that
 * take the grouped schedule share the partitions' streams and run one after
 * another whatever stream they were given; where the driver offers no
 * partitions the one-launch schedule runs, and so it does under a profiler or
 * other tool injected into the process (CUDA_INJECTION64_PATH, or the
 * variables Nsight Compute sets: ncu cannot profile launches in a green
 * context).
 * rkv_compress_noalloc always takes the one-launch schedule.  Returns
 * RKV_ERR_INVALID_ARG for an unknown mode, groups outside 2..32 or
 * 0 < tensor_sms < 8. */
enum {
    RKV_SCHEDULE_ONE_LAUNCH = 0,
    RKV_SCHEDULE_AUTO = 1,
    RKV_SCHEDULE_GROUPED = 2
};
int rkv_set_overlap(int mode, int groups, int tensor_sms);

/* Launch trace (not thread-safe).  While enabled, each launch of the library
 * is preceded and followed, on its own stream, by a one-thread kernel that
 * stores the device's global nanosecond timer, so launches on the two SM
 * partitions of the grouped step (rkv_set_overlap) are placed on one clock.
 * Enabling clears the trace; up to 8192 launches are kept.  rkv_trace_read
 * synchronises the device, writes per launch (in enqueue order, up to
 * max_records) the kernel (index of rkv_kernel_name), the lane (0: the
 * caller's stream, 1: the tensor partition, 2: the other partition) and the
 * start and end stamps in ns, clears the trace and returns the number of
 * records written (a negative RKV_* code on a CUDA error).  Any output
 * pointer may be null. */
int rkv_trace_enable(int on);
int rkv_trace_read(int* kernel, int* lane, uint64_t* start_ns, uint64_t* end_ns,
                   int max_records);

/* Per-kernel timing (not thread-safe).  While enabled, each launch of the
 * library is bracketed by CUDA events on its stream.  rkv_timing_read waits for
 * the events, writes per-kernel totals (milliseconds) and launch counts for up
 * to `max_kernels` kernels in the order of rkv_kernel_name(), returns the
 * number of kernel kinds, and with reset != 0 clears the totals. */
int rkv_timing_enable(int on);
int rkv_timing_read(double* total_ms, int64_t* launches, int max_kernels, int reset);
const char* rkv_kernel_name(int kernel);

#ifdef __cplusplus
}
#endif
#endif /* RKV_H */
