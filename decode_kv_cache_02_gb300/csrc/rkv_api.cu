// rkv_api.cu -- the C ABI of librkv (declared in include/rkv.h): argument
// checks, workspace layout, per-kernel timing and the launch sequence.
//
// One compression round (R-KV review, yoonschallenge.tistory.com/1236,
// question 2, cause 3, in the page's order):
//   key statistics (norms, plain similarity sums)      k_key_stats.cu
//   attention importance                                k_importance_tc.cu / k_importance.cu
//   thresholded Gram -> redundancy, protection, R, Z    k_gram_tc.cu / k_gram_simt.cu
//   top-k selection                                     k_select.cu
//   copy of the kept K/V rows                           k_gather.cu
// Each stage is one launch over all problems of the call; the calls never
// allocate, free or synchronise.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <array>
#include <map>
#include <mutex>
#include <vector>

#include "../../include/rkv.h"
#include "rkv_common.cuh"
#include "rkv_internal.h"

namespace {

using rkv::DeviceStatus;
using rkv::ScoreArgs;

enum KernelId {
    kKeyStats = 0,
    kImportance,
    kImportanceTc,
    kGramTc,
    kGramSimt,
    kSelect,
    kGather,
    kIdentity,
    kCompact,
    kVariant,
    kKeyStatsPaged,
    kCompactPaged,
    kPagedRelease,
    kSentencePenalty,
    kSentenceReps,
    kNumKernels
};
const char* const kKernelNames[kNumKernels] = {
    "key_stats", "importance", "importance_tc", "gram_tc", "gram_simt", "select", "gather",
    "identity_idx", "compact", "variant", "key_stats_paged", "compact_paged", "paged_release",
    "sentence_penalty", "sentence_reps"};

// ---------------------------------------------------------------- timing --
// Events belong to the context they were created in, and a stream records
// only its own context's events: each pool is kept per context (nullptr: the
// caller's), the one current while the launch is enqueued.
struct TimedLaunch {
    int kernel;
    cudaEvent_t start, stop;
    const void* ctx;
};
bool g_timing = false;
std::vector<TimedLaunch> g_pending;
double g_total_ms[kNumKernels];
int64_t g_launches[kNumKernels];
std::map<const void*, std::vector<cudaEvent_t>> g_event_pool;

cudaEvent_t take_event(const void* ctx) {
    std::vector<cudaEvent_t>& pool = g_event_pool[ctx];
    if (!pool.empty()) {
        cudaEvent_t e = pool.back();
        pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
}

// ---------------------------------------------------------------- tracing --
// A trace stamps the device's global nanosecond timer before and after each
// launch, on the launch's own stream, with a one-thread kernel: unlike events,
// the stamps of launches in different contexts (the SM partitions) share one
// clock, so a trace shows which launches ran at the same time.
constexpr int kTraceMax = 16384;
__device__ unsigned long long g_trace_ns[kTraceMax];

__global__ void trace_stamp_kernel(int slot) {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    g_trace_ns[slot] = t;
}

struct TraceRecord {
    int kernel, lane, slot;  // stamps at slot (start) and slot + 1 (end)
};
bool g_trace = false;
std::vector<TraceRecord> g_trace_recs;
int g_trace_slots = 0;

// Runs `launch` with events around it when timing is on (and stamps when a
// trace is on); lane names the SM partition whose context is current
// meanwhile (nullptr: the caller's context and stream).
template <typename F>
cudaError_t timed(int kernel, cudaStream_t s, F&& launch, const rkv::Lane* lane = nullptr) {
    const bool stamp = g_trace && g_trace_slots + 2 <= kTraceMax;
    const int slot = g_trace_slots;
    if (stamp) {
        trace_stamp_kernel<<<1, 1, 0, s>>>(slot);
        g_trace_slots += 2;
        g_trace_recs.push_back(TraceRecord{kernel, lane ? lane->id : 0, slot});
    }
    cudaError_t e;
    if (!g_timing) {
        e = launch();
    } else {
        const void* ctx = lane ? lane->ctx : nullptr;
        TimedLaunch t{kernel, take_event(ctx), take_event(ctx), ctx};
        cudaEventRecord(t.start, s);
        e = launch();
        cudaEventRecord(t.stop, s);
        g_pending.push_back(t);
    }
    if (stamp) trace_stamp_kernel<<<1, 1, 0, s>>>(slot + 1);
    return e;
}

// ------------------------------------------------------------ workspace --
constexpr size_t kAlign = 256;
// the fused select + gather keeps a problem's scores, bucket keys and kept
// indices in shared memory; larger problems take the separate kernels
constexpr size_t kCompactSmemMax = 160 * 1024;
// paged pools with blocks of at least 128 rows are read directly by the
// tensor-core stages (one TMA box per 128-row tile); smaller blocks split a
// tile into boxes too small to keep the producers ahead (64-row blocks made
// the Gram ~25% slower), and take the contiguous key copy instead
constexpr int kDirectLog2Block = 7;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct Workspace {
    DeviceStatus* status;
    float* inv_norm;
    float* sum_s;
    float* I;
    float* R;
    float* Z;
    void* s_rows;
    void* Kc;  // paged calls: contiguous copy of the keys [P, N, d]
    int64_t ld;
    size_t bytes;
};

int64_t row_pitch(int n) { return ((int64_t)n + 3) / 4 * 4; }

// Carves the workspace; with base == nullptr only computes the size.  kc_bytes
// (paged calls) appends the contiguous key copy.
Workspace carve(void* base, int64_t P, int n, size_t kc_bytes = 0) {
    Workspace w{};
    w.ld = row_pitch(n);
    const size_t arr = align_up(sizeof(float) * (size_t)P * (size_t)w.ld);
    char* b = static_cast<char*>(base);
    size_t off = 0;
    w.status = reinterpret_cast<DeviceStatus*>(b + off);
    off += kAlign;
    w.inv_norm = reinterpret_cast<float*>(b + off);
    off += arr;
    w.sum_s = reinterpret_cast<float*>(b + off);
    off += arr;
    w.I = reinterpret_cast<float*>(b + off);
    off += arr;
    w.R = reinterpret_cast<float*>(b + off);
    off += arr;
    w.Z = reinterpret_cast<float*>(b + off);
    off += arr;
    w.s_rows = b + off;
    off += align_up(2 * (size_t)P * 16 * 128);
    w.Kc = kc_bytes ? b + off : nullptr;
    off += align_up(kc_bytes);
    w.bytes = off;
    return w;
}

// ------------------------------------------------------------- checking --
size_t elem_size(int dtype) { return dtype == RKV_DTYPE_BF16 ? 2 : 4; }

int check_desc(const rkv_desc* d) {
    if (!d) return RKV_ERR_INVALID_ARG;
    if (d->num_problems < 0 || d->n_capacity < 1 || d->out_capacity < 0) return RKV_ERR_INVALID_ARG;
    if (d->num_problems > (int64_t)1 << 31) return RKV_ERR_INVALID_ARG;
    if (d->dtype != RKV_DTYPE_BF16 && d->dtype != RKV_DTYPE_FP32) return RKV_ERR_UNSUPPORTED;
    if (d->head_dim != 64 && d->head_dim != 128) return RKV_ERR_UNSUPPORTED;
    if (d->gqa_group < 1 || d->gqa_group > 16) return RKV_ERR_UNSUPPORTED;
    return RKV_OK;
}

// Rows per problem of the outputs of rkv_compress / rkv_gather.
int out_cap(const rkv_desc* d) { return d->out_capacity > 0 ? d->out_capacity : d->n_capacity; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// [a, a+na) and [b, b+nb) overlap without being the same range
bool partial_overlap(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    if (x == y) return false;
    return x < y + nb && y < x + na;
}

// What a variant asks for: zvar = Z formed from I and R (softmax, pooling,
// sentences); sched = a recent window / sampled selection.
struct VarFlags {
    bool zvar = false;
    bool sched = false;
    bool any() const { return zvar || sched; }
};

// A variant's fields (sizes that depend on the call: check_variant_sizes).
int check_variant(const rkv_variant* v, VarFlags* f) {
    *f = VarFlags{};
    if (!v) return RKV_OK;
    if (v->redundancy_softmax != 0 && v->redundancy_softmax != 1) return RKV_ERR_INVALID_ARG;
    if (v->pool_window < 1 || v->pool_window > RKV_MAX_POOL_WINDOW || (v->pool_window & 1) == 0)
        return RKV_ERR_INVALID_ARG;
    if (const rkv_sentences* t = v->sentences) {
        if (!t->reps || !t->count || !t->seg_id || !t->penalty || !aligned16(t->reps))
            return RKV_ERR_INVALID_ARG;
        if (t->num_seqs < 1 || t->heads < 1 || t->max_sentences < 1 ||
            t->max_sentences > RKV_MAX_SENTENCES || t->hidden_dim < 4 ||
            t->hidden_dim > RKV_MAX_HIDDEN || (t->hidden_dim & 3) != 0 || t->ld_seg < 1)
            return RKV_ERR_INVALID_ARG;
        if (t->num_seqs * (int64_t)t->max_sentences >= ((int64_t)1 << 31)) return RKV_ERR_INVALID_ARG;
    }
    if (const rkv_schedule* c = v->schedule) {
        if (c->recent_window < 1 || c->pool_size < 0 || c->ld_uniforms < 0 ||
            !(c->temperature > 0.f) || !(c->temperature < INFINITY))
            return RKV_ERR_INVALID_ARG;
    }
    f->zvar = v->redundancy_softmax != 0 || v->pool_window > 1 || v->sentences != nullptr;
    f->sched = v->schedule != nullptr;
    return RKV_OK;
}

// Rows that are always kept: the schedule's window, else the observation tokens.
int tail_rows(const rkv_variant* v, int n_obs) {
    return (v && v->schedule) ? v->schedule->recent_window : n_obs;
}

// Whether the call samples (a pool larger than the number kept).
bool samples(const rkv_variant* v, int n_cached, int budget) {
    if (!v || !v->schedule || n_cached <= budget) return false;
    return v->schedule->pool_size > budget - v->schedule->recent_window;
}

// The variant's sizes against the call: sentence rows cover the cached rows;
// the window holds the observation tokens and leaves candidates; with a budget
// (budget > 0), k <= pool <= C and uniforms for a sampled pool.
int check_variant_sizes(const rkv_variant* v, int n_cached, int n_obs, int budget) {
    if (!v) return RKV_OK;
    if (v->sentences && v->sentences->ld_seg < n_cached) return RKV_ERR_INVALID_ARG;
    if (const rkv_schedule* c = v->schedule) {
        const int L = c->recent_window;
        if (L < n_obs || L >= n_cached) return RKV_ERR_INVALID_ARG;
        if (budget > 0) {
            if (L > budget) return RKV_ERR_INVALID_ARG;
            const int k = budget - L, C = n_cached - L;
            if (c->pool_size < k || c->pool_size > C) return RKV_ERR_INVALID_ARG;
            if (c->pool_size > k && (!c->uniforms || c->ld_uniforms < C)) return RKV_ERR_INVALID_ARG;
        }
    }
    return RKV_OK;
}

int check_scores(const rkv_desc* d, const void* K, const void* Q, int n_cached, int n_obs,
                 void* ws, size_t ws_bytes) {
    int rc = check_desc(d);
    if (rc) return rc;
    if (n_cached < 2 || n_cached > d->n_capacity || n_cached > RKV_MAX_TOKENS)
        return RKV_ERR_INVALID_ARG;
    if (n_obs < 1 || n_obs >= n_cached) return RKV_ERR_INVALID_ARG;
    if (d->gqa_group * n_obs > 128) return RKV_ERR_UNSUPPORTED;
    if (d->num_problems > 0 && (!K || !Q || !aligned16(K) || !aligned16(Q)))
        return RKV_ERR_INVALID_ARG;
    if (!ws || (reinterpret_cast<uintptr_t>(ws) % kAlign) != 0) return RKV_ERR_WORKSPACE;
    if (ws_bytes < carve(nullptr, d->num_problems, n_cached).bytes) return RKV_ERR_WORKSPACE;
    return RKV_OK;
}

// Runs the four scoring stages; I/R/Z land in the given rows.  With a paged
// K (pg), the key statistics read through the block table and write the
// contiguous copy w.Kc, which the later stages read.
ScoreArgs score_args(const rkv_desc* d, const void* K, const void* Q, int n_cached, int n_obs,
                     float lambda, int beta, float tau, float* I, float* R, float* Z,
                     int64_t ld_out, const Workspace& w) {
    // I, R, Z as defined on the page (R may be null: not stored)
    ScoreArgs a{};
    a.K = K;
    a.Q = Q;
    a.P = d->num_problems;
    a.G = d->gqa_group;
    a.d = d->head_dim;
    a.n_cap = d->n_capacity;
    a.N = n_cached;
    a.n_obs = n_obs;
    a.beta = beta;
    a.dtype = d->dtype;
    a.lambda = lambda;
    a.tau = tau;
    a.inv_norm = w.inv_norm;
    a.sum_s = w.sum_s;
    a.s_rows = w.s_rows;
    a.ld_ws = w.ld;
    a.I = I;
    a.R = R;
    a.Z = Z;
    a.ld_out = ld_out;
    a.status = w.status;
    return a;
}

// Whether the importance kernel takes the key statistics and the Gram
// completes sum_i (contiguous keys, or a paged pool the tensor-core stages
// read in place, whose rows fit the resident importance kernel and the
// one-row-block Gram): no pass over K is spent on them.
bool stats_fused(const ScoreArgs& b) {
    return (!b.pg.table || b.paged_direct) && rkv::gram_tc_supported(b) &&
           rkv::importance_tc_supported(b) && rkv::importance_tc_resident(b) &&
           rkv::gram_tc_rows(b);
}

int run_scores(const rkv_desc* d, const void* K, const void* Q, int n_cached, int n_obs,
               float lambda, int beta, float tau, float* I, float* R, float* Z, int64_t ld_out,
               const Workspace& w, cudaStream_t s, const rkv::PagedIn* pg = nullptr,
               bool direct = false) {
    ScoreArgs a = score_args(d, K, Q, n_cached, n_obs, lambda, beta, tau, I, R, Z, ld_out, w);
    ScoreArgs b = a;  // what the stages after the key statistics read
    if (pg) {
        a.pg = *pg;
        // direct: the tensor-core stages read the pool straight through the
        // table (paged_reads_pool); otherwise the key statistics write a
        // contiguous copy for them
        if (direct) {
            b.pg = *pg;
            b.paged_direct = true;
        } else {
            a.Kc = w.Kc;
            b.K = w.Kc;
            b.n_cap = n_cached;
        }
    }
    const bool gram_tc = rkv::gram_tc_supported(b);
    const bool imp_tc = rkv::importance_tc_supported(b);
    a.stats_sum = b.stats_sum = !imp_tc;  // the tensor-core importance completes sum_i itself
    // paged pools read in place (blocks of 128 rows or more) as well: the
    // importance kernel's loads check the table's ids then
    b.fused_stats = (!pg || direct) && stats_fused(b);
    cudaError_t e = b.fused_stats ? cudaSuccess
                                  : timed(pg ? kKeyStatsPaged : kKeyStats, s,
                                          [&] { return rkv::launch_key_stats(a, s); });
    if (e == cudaSuccess) {
        if (imp_tc)
            e = timed(kImportanceTc, s, [&] { return rkv::launch_importance_tc(b, s); });
        else
            e = timed(kImportance, s, [&] { return rkv::launch_importance(b, s); });
    }
    if (e == cudaSuccess) {
        if (gram_tc)
            e = timed(kGramTc, s, [&] { return rkv::launch_gram_tc(b, s); });
        else
            e = timed(kGramSimt, s, [&] { return rkv::launch_gram_simt(b, s); });
    }
    return e == cudaSuccess ? RKV_OK : RKV_ERR_CUDA;
}

// ---------------------------------------------------------------- overlap --
// The step on two SM partitions of the device (rkv_lanes.cu).  The importance
// and the Gram are bound by their SMs (the importance's time grows in
// proportion as the SMs it gets shrink, the Gram's with the tensor pipes it
// loses), while the compaction, spread over the whole device, is bound by
// HBM, and on a few SMs moves ~65 GB/s per SM.  So the problems are cut into
// groups, the tensor lane (most SMs) runs importance and Gram group after
// group, and the hbm lane (the rest) compacts each group once its Gram is
// done, while the tensor lane goes on with the next.  The last group's
// compaction takes the whole device.  Groups only shift the base pointers:
// every kernel sees a smaller call of the same shape.
// Eight groups with 112 of GB300's 152 SMs on the tensor lane measured best
// on the Llama-shaped step (6.54 ms against 6.85 for one launch per stage;
// 6-9 groups within 0.06 ms; 108 SMs 6.71, 116 SMs 6.9).  tensor_sms 0: the
// same share of the device's SMs.
int g_overlap_mode = RKV_SCHEDULE_AUTO;
int g_overlap_groups = 8;
int g_overlap_tensor_sms = 0;
std::mutex g_overlap_mu;  // one call at a time enqueues on the shared lanes
bool g_lanes_refused = false;  // a partition refused the first launch of a call

int overlap_tensor_sms() {
    if (g_overlap_tensor_sms > 0) return g_overlap_tensor_sms;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    return sms * 112 / 152 / 4 * 4;
}
constexpr int kMaxGroups = 32;

struct LaneEvents {
    cudaEvent_t ev[kMaxGroups + 2] = {};
    bool made = false;
};

// Per-group events of one lane, created in the lane's context.
bool lane_events(const rkv::Lane* lane, LaneEvents* le) {
    if (le->made) return true;
    rkv::LaneScope scope(lane);
    for (auto& e : le->ev)
        if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return false;
    le->made = true;
    return true;
}

ScoreArgs group_args(const ScoreArgs& b, int64_t p0, int64_t n) {
    ScoreArgs c = b;
    const int64_t es = 2;  // the fused path is bf16 only
    if (b.pg.table)  // a paged pool: the group's sequences' rows of the table (p0 % H == 0)
        c.pg.table = b.pg.table + (p0 / b.pg.H) * b.pg.max_blocks;
    else
        c.K = static_cast<const char*>(b.K) + p0 * b.n_cap * b.d * es;
    c.Q = static_cast<const char*>(b.Q) + p0 * b.G * b.n_obs * b.d * es;
    c.P = n;
    c.inv_norm += p0 * b.ld_ws;
    c.sum_s += p0 * b.ld_ws;
    c.s_rows = static_cast<char*>(b.s_rows) + p0 * 32 * b.d;  // 16 bf16 rows of d per problem
    c.I += p0 * b.ld_out;
    c.Z += p0 * b.ld_out;
    if (c.R) c.R += p0 * b.ld_out;
    return c;
}

struct CompactCall {
    int n_cached, tail, budget, n_cap, ocap, row_bytes;
    bool in_place;
    const void *K, *V;
    void *out_K, *out_V;
    int32_t* out_idx;
    // a paged pool (K, V the pools, compacted in place through g.pg)
    bool paged = false;
};

cudaError_t compact_group(const ScoreArgs& g, int64_t p0, const CompactCall& c, cudaStream_t s) {
    const int64_t rb = c.row_bytes;
    if (c.paged)
        return rkv::launch_compact_paged(g.P, c.n_cached, g.Z, g.ld_out, c.tail, c.budget,
                                         c.out_idx + p0 * c.budget, nullptr, c.out_K, c.out_V,
                                         g.pg, c.row_bytes, g.status, s);
    return rkv::launch_compact(g.P, c.n_cached, g.Z, g.ld_out, c.tail, c.budget,
                               c.out_idx + p0 * c.budget,
                               static_cast<const char*>(c.K) + p0 * c.n_cap * rb,
                               static_cast<const char*>(c.V) + p0 * c.n_cap * rb,
                               static_cast<char*>(c.out_K) + p0 * c.ocap * rb,
                               static_cast<char*>(c.out_V) + p0 * c.ocap * rb, c.n_cap, c.ocap,
                               c.row_bytes, c.in_place, g.status, s);
}

// Whether the grouped schedule is expected to beat one launch per stage.
// Per-problem device times measured on GB300 with one launch per stage over
// the whole device (the Llama-8B shape): importance 4.9e-4 ns per key element
// (N d), Gram 1.14e-6 ns per N^2 d, compaction 2.9e-4 ns per byte of kept
// rows (both tensors; in place an upper bound).  Grouping stretches
// importance and Gram by the device's SMs over the tensor partition's and
// hides the compaction of every group but the last; each group costs ~28 us
// of launch ramp and tail, and the step ends with about 1.3 groups'
// compaction.  Llama-8B step (16,384 problems, N = 1152): +0.31 ms predicted,
// +0.31 measured; the decode stream's rounds (8,192 problems, N = 1766, in
// place): -0.2 ms predicted, -0.4 measured, so they keep one launch per stage.
bool grouped_pays(const ScoreArgs& b, const CompactCall& cc, int tensor_sms, int groups) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        sms <= tensor_sms)
        return false;
    const double nd = (double)b.N * b.d;
    const double t_score = 4.9e-4 * nd + 1.14e-6 * nd * b.N;          // ns a problem
    const double t_compact = 2.9e-4 * (double)cc.budget * cc.row_bytes * 2;
    const double stretch = (double)sms / tensor_sms - 1.0;
    const double gain_ns = (double)b.P * (t_compact - stretch * t_score) - groups * 28e3 -
                           1.3 * t_compact * (double)b.P / groups;
    return gain_ns > 0.0;
}

// Returns -1 when the step does not take this schedule (the caller runs the
// serial one), else an RKV_* code.
int run_overlapped(const ScoreArgs& base, const CompactCall& cc, cudaStream_t s) {
    if (g_overlap_mode == RKV_SCHEDULE_ONE_LAUNCH || g_lanes_refused) return -1;
    const int tensor_sms = overlap_tensor_sms();
    // at least a few waves of the tensor lane per group, or nothing to gain
    if (tensor_sms < 8 || base.P < 2 * (int64_t)g_overlap_groups * tensor_sms) return -1;
    // automatic: the cost model's call; never for paged pools, whose
    // compaction (a register copy through the table, in place) is too slow on
    // the small partition (the 128-row-block paged round: 9.5 ms grouped
    // against 7.1 ms one launch per stage)
    if (g_overlap_mode == RKV_SCHEDULE_AUTO &&
        (cc.paged || !grouped_pays(base, cc, tensor_sms, g_overlap_groups)))
        return -1;
    ScoreArgs b = base;
    if (!stats_fused(b)) return -1;
    b.fused_stats = true;
    // under a profiler or other injected tool (ncu cannot profile launches in
    // a green context) and on a stream being captured into a graph (the
    // lanes' streams belong to other contexts) the one-launch schedule runs
    if (getenv("CUDA_INJECTION64_PATH") || getenv("NV_NSIGHT_INJECTION_TRANSPORT_TYPE") ||
        getenv("NV_COMPUTE_PROFILER_PERFWORKS_DIR"))
        return -1;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone)
        return -1;
    std::lock_guard<std::mutex> lock(g_overlap_mu);
    const rkv::Lanes* L = rkv::lanes_for_current_device(tensor_sms);
    if (!L) return -1;
    const rkv::Lane* T = &L->tensor;
    const rkv::Lane* H = &L->hbm;
    // Group bounds: equal groups of whole waves of the tensor lane's
    // persistent CTAs, the last one the remainder.  Each group costs the
    // tensor lane a launch ramp and a tail of its two kernels (~28 us
    // measured on the Llama-shaped step), and the step ends with the hbm
    // lane's compaction of the second-to-last group and the whole device's of
    // the last, so a handful of groups is the balance.
    // (paged: whole sequences, so that a group is a block of the table's rows)
    const int64_t wave = T->sms;
    const int64_t unit = b.pg.table ? b.pg.H : 1;
    int64_t per = (b.P + g_overlap_groups - 1) / g_overlap_groups;
    per = (per + wave - 1) / wave * wave;
    per = (per + unit - 1) / unit * unit;
    int64_t bounds[kMaxGroups + 1];
    int G = 0;
    bounds[0] = 0;
    while (G < kMaxGroups - 1 && bounds[G] + per < b.P) {
        bounds[G + 1] = bounds[G] + per;
        ++G;
    }
    bounds[++G] = b.P;
    if (G < 2) return -1;
    static std::map<const rkv::Lanes*, std::array<LaneEvents, 3>> events;  // per split and device
    LaneEvents& ev_t = events[L][0];
    LaneEvents& ev_h = events[L][1];
    LaneEvents& ev_s = events[L][2];
    if (!lane_events(T, &ev_t) || !lane_events(H, &ev_h) || !lane_events(nullptr, &ev_s))
        return RKV_ERR_CUDA;
    auto first = [&](int c) { return bounds[c]; };
    auto group = [&](int c) { return group_args(b, bounds[c], bounds[c + 1] - bounds[c]); };
    // ev_s[0]: the call's start on the caller's stream; ev_t[c]: the Gram of
    // group c done; ev_h[0]: the hbm lane's last compaction done
    cudaError_t e = cudaEventRecord(ev_s.ev[0], s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(T->stream, ev_s.ev[0], 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(H->stream, ev_s.ev[0], 0);
    for (int c = 0; c < G && e == cudaSuccess; ++c) {
        ScoreArgs g = group(c);
        g.sms = T->sms;
        {
            rkv::LaneScope scope(T);
            e = timed(kImportanceTc, T->stream,
                      [&] { return rkv::launch_importance_tc(g, T->stream); }, T);
            if (c == 0 && e != cudaSuccess) {
                // the partition refused the call's first launch (its error is
                // cleared by the launcher): nothing of the call has run, so
                // one launch per stage takes this call and every later one
                g_lanes_refused = true;
                return -1;
            }
            if (e == cudaSuccess)
                e = timed(kGramTc, T->stream, [&] { return rkv::launch_gram_tc(g, T->stream); },
                          T);
            if (e == cudaSuccess) e = cudaEventRecord(ev_t.ev[c], T->stream);
        }
        if (e != cudaSuccess || c + 1 == G) break;
        e = cudaStreamWaitEvent(H->stream, ev_t.ev[c], 0);
        if (e == cudaSuccess) {
            rkv::LaneScope scope(H);
            e = timed(cc.paged ? kCompactPaged : kCompact, H->stream,
                      [&] { return compact_group(g, first(c), cc, H->stream); },
                      H);
        }
    }
    if (e == cudaSuccess) {
        rkv::LaneScope scope(H);
        e = cudaEventRecord(ev_h.ev[0], H->stream);
    }
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, ev_t.ev[G - 1], 0);
    if (e == cudaSuccess) {
        const ScoreArgs g = group(G - 1);
        e = timed(cc.paged ? kCompactPaged : kCompact, s,
                  [&] { return compact_group(g, first(G - 1), cc, s); });
    }
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, ev_h.ev[0], 0);
    if (e != cudaSuccess) {
        // whatever was enqueued on the lanes still runs before the caller's
        // stream goes on (best effort: the call reports the error either way)
        {
            rkv::LaneScope scope(T);
            cudaEventRecord(ev_t.ev[kMaxGroups + 1], T->stream);
        }
        {
            rkv::LaneScope scope(H);
            cudaEventRecord(ev_h.ev[kMaxGroups + 1], H->stream);
        }
        cudaStreamWaitEvent(s, ev_t.ev[kMaxGroups + 1], 0);
        cudaStreamWaitEvent(s, ev_h.ev[kMaxGroups + 1], 0);
    }
    return e == cudaSuccess ? RKV_OK : RKV_ERR_CUDA;
}

// The device-side form of a variant: with zvar Z is formed from the base I
// and R rows of w; a sampled schedule adds the pool and the uniforms.
rkv::VariantIn variant_in(const rkv_variant& v, const VarFlags& f, float lambda,
                          const Workspace& w, bool sample) {
    rkv::VariantIn vin;
    if (sample) {
        const rkv_schedule* c = v.schedule;
        vin.sample = true;
        vin.pool = c->pool_size;
        vin.inv_temp = 1.0f / c->temperature;
        vin.unif = c->uniforms;
        vin.ld_u = c->ld_uniforms;
    }
    if (!f.zvar) return vin;
    vin.I = w.I;
    vin.R = w.R;
    vin.ld = w.ld;
    vin.lambda = lambda;
    vin.softmax = v.redundancy_softmax;
    vin.half = (v.pool_window - 1) / 2;
    if (const rkv_sentences* t = v.sentences) {
        vin.pen = t->penalty;
        vin.count = t->count;
        vin.seg = t->seg_id;
        vin.ld_seg = t->ld_seg;
        vin.num_seqs = t->num_seqs;
        vin.heads = t->heads;
        vin.max_sent = t->max_sentences;
    }
    return vin;
}

// The sentence penalties a variant needs, before anything reads them.
cudaError_t launch_penalty(const rkv_variant* v, cudaStream_t s) {
    if (!v || !v->sentences) return cudaSuccess;
    const rkv_sentences* t = v->sentences;
    return timed(kSentencePenalty, s, [&] {
        return rkv::launch_sentence_penalty(t->num_seqs, t->max_sentences, t->hidden_dim, t->reps,
                                            t->count, t->tau, t->penalty, s);
    });
}

// The scores with a variant: the base scores into the workspace, then I', R'
// and Z into the given rows (I_out, R_out may be null).
int run_scores_variant(const rkv_desc* d, const void* K, const void* Q, int n_cached, int n_obs,
                       float lambda, int beta, float tau, const rkv_variant& v, float* I_out,
                       float* R_out, float* Z, int64_t ld_out, const Workspace& w,
                       cudaStream_t s) {
    if (launch_penalty(&v, s) != cudaSuccess) return RKV_ERR_CUDA;
    int rc = run_scores(d, K, Q, n_cached, n_obs, lambda, beta, tau, w.I, w.R, w.Z, w.ld, w, s);
    if (rc) return rc;
    VarFlags f;
    f.zvar = true;  // the variant kernel always forms Z from I and R
    const rkv::VariantIn vin = variant_in(v, f, lambda, w, false);
    const int tail = tail_rows(&v, n_obs);
    cudaError_t e = timed(kVariant, s, [&] {
        return rkv::launch_variant(d->num_problems, n_cached, tail, vin, Z, I_out, R_out, ld_out,
                                   s);
    });
    return e == cudaSuccess ? RKV_OK : RKV_ERR_CUDA;
}

}  // namespace

extern "C" {

size_t rkv_workspace_size(const rkv_desc* desc, int n_cached, int n_obs) {
    if (check_desc(desc) != RKV_OK || n_cached < 1 || n_cached > RKV_MAX_TOKENS || n_obs < 0)
        return 0;
    return carve(nullptr, desc->num_problems, n_cached).bytes;
}

int rkv_score_ex(const rkv_desc* desc, const void* K, const void* Q_obs, int n_cached,
                 int n_obs, float lambda, int beta, float tau, const rkv_variant* variant,
                 float* out_I, float* out_R, float* out_Z, void* workspace,
                 size_t workspace_bytes, void* stream) {
    VarFlags vf;
    int rc = check_variant(variant, &vf);
    if (rc) return rc;
    rc = check_scores(desc, K, Q_obs, n_cached, n_obs, workspace, workspace_bytes);
    if (rc) return rc;
    if (beta < 0) return RKV_ERR_INVALID_ARG;
    if (desc->num_problems == 0) return RKV_OK;
    if (!out_I || !out_R || !out_Z) return RKV_ERR_INVALID_ARG;
    if (check_variant_sizes(variant, n_cached, n_obs, 0)) return RKV_ERR_INVALID_ARG;
    const Workspace w = carve(workspace, desc->num_problems, n_cached);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (vf.zvar || tail_rows(variant, n_obs) > n_obs)
        return run_scores_variant(desc, K, Q_obs, n_cached, n_obs, lambda, beta, tau, *variant,
                                  out_I, out_R, out_Z, n_cached, w, s);
    return run_scores(desc, K, Q_obs, n_cached, n_obs, lambda, beta, tau, out_I, out_R, out_Z,
                      n_cached, w, s);
}

int rkv_score(const rkv_desc* desc, const void* K, const void* Q_obs, int n_cached, int n_obs,
              float lambda, int beta, float tau, float* out_I, float* out_R, float* out_Z,
              void* workspace, size_t workspace_bytes, void* stream) {
    return rkv_score_ex(desc, K, Q_obs, n_cached, n_obs, lambda, beta, tau, nullptr, out_I, out_R,
                        out_Z, workspace, workspace_bytes, stream);
}

int rkv_compress(const rkv_desc* desc, const void* K, const void* V, const void* Q_obs,
                 int n_cached, int budget, int n_obs, float lambda, int beta, float tau,
                 void* out_K, void* out_V, int32_t* out_idx, void* workspace,
                 size_t workspace_bytes, void* stream) {
    return rkv_compress_ex(desc, K, V, Q_obs, n_cached, budget, n_obs, lambda, beta, tau, nullptr,
                           out_K, out_V, out_idx, workspace, workspace_bytes, stream);
}

int rkv_compress_ex(const rkv_desc* desc, const void* K, const void* V, const void* Q_obs,
                    int n_cached, int budget, int n_obs, float lambda, int beta, float tau,
                    const rkv_variant* variant, void* out_K, void* out_V, int32_t* out_idx,
                    void* workspace, size_t workspace_bytes, void* stream) {
    return rkv::compress_call(desc, K, V, Q_obs, n_cached, budget, n_obs, lambda, beta, tau,
                              variant, out_K, out_V, out_idx, workspace, workspace_bytes, stream,
                              false, true);
}

}  // extern "C"

namespace rkv {

// The body of rkv_compress_ex.  clear_status: once every argument check has
// passed, the device error word at the start of the workspace is cleared
// (enqueued before the first kernel), so a call that is rejected enqueues
// nothing at all.
int compress_call(const rkv_desc* desc, const void* K, const void* V, const void* Q_obs,
                  int n_cached, int budget, int n_obs, float lambda, int beta, float tau,
                  const rkv_variant* variant, void* out_K, void* out_V, int32_t* out_idx,
                  void* workspace, size_t workspace_bytes, void* stream, bool clear_status,
                  bool lanes) {
    VarFlags vf;
    int rc = check_variant(variant, &vf);
    if (rc) return rc;
    rc = check_desc(desc);
    if (rc) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t P = desc->num_problems;
    const int ocap = out_cap(desc);
    if (n_cached < 1 || n_cached > desc->n_capacity || budget < 1 || budget > desc->n_capacity ||
        budget > ocap || n_obs < 1 || n_obs > budget || beta < 0)
        return RKV_ERR_INVALID_ARG;
    const size_t es = elem_size(desc->dtype);
    const size_t bytes = (size_t)P * desc->n_capacity * desc->head_dim * es;
    const size_t obytes = (size_t)P * ocap * desc->head_dim * es;
    if (P > 0) {
        if (!K || !V || !out_K || !out_V || !out_idx || !Q_obs) return RKV_ERR_INVALID_ARG;
        if (!aligned16(K) || !aligned16(V) || !aligned16(out_K) || !aligned16(out_V) ||
            !aligned16(Q_obs))
            return RKV_ERR_INVALID_ARG;
        if (partial_overlap(out_K, obytes, K, bytes) || partial_overlap(out_V, obytes, V, bytes) ||
            partial_overlap(out_K, obytes, V, bytes) || partial_overlap(out_V, obytes, K, bytes) ||
            partial_overlap(out_K, obytes, out_V, obytes) ||
            (out_K == V) || (out_V == K) || (out_K == out_V && P > 0))
            return RKV_ERR_ALIAS;
    }
    const bool in_place = (out_K == K) && (out_V == V);
    if (!in_place && (out_K == K || out_V == V)) return RKV_ERR_ALIAS;  // mixed modes
    if (in_place && ocap != desc->n_capacity) return RKV_ERR_INVALID_ARG;
    const int row_bytes = desc->head_dim * (int)es;
    if (n_cached <= budget) {
        // nothing to evict
        if (!workspace || (reinterpret_cast<uintptr_t>(workspace) % kAlign) != 0 ||
            workspace_bytes < kAlign)
            return RKV_ERR_WORKSPACE;
        if (P == 0) return RKV_OK;
        if (clear_status && cudaMemsetAsync(workspace, 0, sizeof(DeviceStatus), s) != cudaSuccess)
            return RKV_ERR_CUDA;
        cudaError_t e = timed(kIdentity, s, [&] {
            return rkv::launch_identity_idx(P, n_cached, budget, out_idx, s);
        });
        if (e == cudaSuccess && !in_place) {
            e = timed(kGather, s, [&] {
                return rkv::launch_gather(K, V, out_K, out_V, out_idx, P, desc->n_capacity, ocap,
                                          budget, row_bytes, false,
                                          reinterpret_cast<DeviceStatus*>(workspace), s);
            });
        }
        return e == cudaSuccess ? RKV_OK : RKV_ERR_CUDA;
    }
    rc = check_scores(desc, K, Q_obs, n_cached, n_obs, workspace, workspace_bytes);
    if (rc) return rc;
    if (P == 0) return RKV_OK;
    if (check_variant_sizes(variant, n_cached, n_obs, budget)) return RKV_ERR_INVALID_ARG;
    const Workspace w = carve(workspace, P, n_cached);
    const int tail = tail_rows(variant, n_obs);
    const bool sample = samples(variant, n_cached, budget);
    const bool fused = rkv::compact_smem_bytes(n_cached, tail, budget,
                                               vf.zvar && variant->sentences) <= kCompactSmemMax;
    if (sample && !fused) return RKV_ERR_UNSUPPORTED;
    if (clear_status && cudaMemsetAsync(w.status, 0, sizeof(DeviceStatus), s) != cudaSuccess)
        return RKV_ERR_CUDA;
    if (lanes && fused && !vf.any()) {
        // the two-partition schedule, where the step takes it
        const ScoreArgs a = score_args(desc, K, Q_obs, n_cached, n_obs, lambda, beta, tau, w.I,
                                       nullptr, w.Z, w.ld, w);
        const CompactCall cc{n_cached, tail, budget, desc->n_capacity, ocap, row_bytes, in_place,
                             K, V, out_K, out_V, out_idx};
        rc = run_overlapped(a, cc, s);
        if (rc >= 0) return rc;
    }
    if (!fused && (vf.zvar || tail > n_obs)) {
        rc = run_scores_variant(desc, K, Q_obs, n_cached, n_obs, lambda, beta, tau, *variant,
                                nullptr, nullptr, w.Z, w.ld, w, s);
    } else {
        if (vf.zvar && launch_penalty(variant, s) != cudaSuccess) return RKV_ERR_CUDA;
        rc = run_scores(desc, K, Q_obs, n_cached, n_obs, lambda, beta, tau, w.I,
                        vf.zvar ? w.R : nullptr, w.Z, w.ld, w, s);
    }
    if (rc) return rc;
    cudaError_t e;
    if (fused) {
        // selection and compaction in one pass per problem (a variant's Z is
        // formed there from I and R; a schedule's window is the kept tail)
        rkv::VariantIn vin;
        if (vf.any()) vin = variant_in(*variant, vf, lambda, w, sample);
        e = timed(kCompact, s, [&] {
            return rkv::launch_compact(P, n_cached, w.Z, w.ld, tail, budget, out_idx, K, V, out_K,
                                       out_V, desc->n_capacity, ocap, row_bytes, in_place, w.status, s,
                                       vin);
        });
    } else {
        e = timed(kSelect, s, [&] {
            return rkv::launch_select(P, n_cached, w.Z, w.ld, tail, budget, out_idx, w.status, s);
        });
        if (e == cudaSuccess)
            e = timed(kGather, s, [&] {
                return rkv::launch_gather(K, V, out_K, out_V, out_idx, P, desc->n_capacity, ocap,
                                          budget, row_bytes, in_place, w.status, s);
            });
    }
    return e == cudaSuccess ? RKV_OK : RKV_ERR_CUDA;
}

}  // namespace rkv

// ---------------------------------------------------------------- paged --

namespace {

int log2_exact(int x) {
    int l = 0;
    while ((1 << l) < x) ++l;
    return (1 << l) == x ? l : -1;
}

int blocks_for(int rows, int bs) { return (rows + bs - 1) / bs; }

// The contiguous descriptor of the same problems (capacity = the pool's rows
// per sequence, only used for sizes) after the paged descriptor's checks.
int check_paged_desc(const rkv_paged_desc* d, rkv_desc* flat) {
    if (!d) return RKV_ERR_INVALID_ARG;
    if (d->num_seqs < 0 || d->num_kv_heads < 1 || d->num_blocks < 1 ||
        d->max_blocks_per_seq < 1)
        return RKV_ERR_INVALID_ARG;
    if (d->block_size < 1 || d->block_size > 1024 || log2_exact(d->block_size) < 0)
        return RKV_ERR_INVALID_ARG;
    if (d->num_seqs * (int64_t)d->num_kv_heads > ((int64_t)1 << 31)) return RKV_ERR_INVALID_ARG;
    if ((int64_t)d->num_blocks * d->num_kv_heads * d->block_size > ((int64_t)1 << 40))
        return RKV_ERR_INVALID_ARG;
    flat->num_problems = d->num_seqs * d->num_kv_heads;
    flat->gqa_group = d->gqa_group;
    flat->head_dim = d->head_dim;
    const int64_t cap = (int64_t)d->max_blocks_per_seq * d->block_size;
    flat->n_capacity = (int32_t)(cap < RKV_MAX_TOKENS ? cap : RKV_MAX_TOKENS);
    flat->dtype = d->dtype;
    return check_desc(flat);
}

size_t kc_bytes_for(const rkv_desc& flat, int n_cached) {
    return (size_t)flat.num_problems * n_cached * flat.head_dim * elem_size(flat.dtype);
}

// Whether the tensor-core stages read a paged pool straight through the
// table (no contiguous key copy): bf16 pools with blocks of at least 128 rows
// whose shapes the tensor-core importance and Gram take.  Smaller blocks split
// a tile into boxes too small to keep the producers ahead (64-row blocks made
// the Gram ~25% slower); they, fp32 pools and the CUDA-core paths read the
// copy.
bool paged_reads_pool(const rkv_paged_desc* d, const rkv_desc& flat, int n_cached, int n_obs,
                      int beta) {
    if (flat.dtype != RKV_DTYPE_BF16 || log2_exact(d->block_size) < kDirectLog2Block) return false;
    if ((int64_t)d->num_kv_heads * d->num_blocks >= ((int64_t)1 << 31)) return false;
    ScoreArgs b{};
    b.P = flat.num_problems;
    b.G = flat.gqa_group;
    b.d = flat.head_dim;
    b.N = n_cached;
    b.n_obs = n_obs;
    b.beta = beta;
    b.dtype = flat.dtype;
    b.ld_ws = row_pitch(n_cached);
    return rkv::gram_tc_shape_ok(b) && rkv::importance_tc_shape_ok(b);
}

// The contiguous key copy a paged call needs (0 when the pool is read directly).
size_t paged_kc_bytes(const rkv_paged_desc* d, const rkv_desc& flat, int n_cached, int n_obs,
                      int beta) {
    return paged_reads_pool(d, flat, n_cached, n_obs, beta) ? 0 : kc_bytes_for(flat, n_cached);
}

}  // namespace

extern "C" {

size_t rkv_paged_workspace_size(const rkv_paged_desc* desc, int n_cached, int n_obs,
                                int beta) {
    rkv_desc flat{};
    if (check_paged_desc(desc, &flat) != RKV_OK || n_cached < 1 || n_cached > flat.n_capacity ||
        n_obs < 0 || beta < 0)
        return 0;
    return carve(nullptr, flat.num_problems, n_cached,
                 paged_kc_bytes(desc, flat, n_cached, n_obs, beta))
        .bytes;
}

int rkv_paged_freed_per_seq(const rkv_paged_desc* desc, int n_cached, int budget) {
    rkv_desc flat{};
    if (check_paged_desc(desc, &flat) != RKV_OK || n_cached < 1 || budget < 1 ||
        n_cached > flat.n_capacity || budget > flat.n_capacity)
        return -1;
    if (n_cached <= budget) return 0;
    return blocks_for(n_cached, desc->block_size) - blocks_for(budget, desc->block_size);
}

int rkv_paged_compress(const rkv_paged_desc* desc, void* K_pool, void* V_pool,
                       const void* Q_obs, int32_t* block_table, int n_cached, int budget,
                       int n_obs, float lambda, int beta, float tau,
                       const rkv_variant* variant, int32_t* out_idx, int32_t* out_freed,
                       void* workspace, size_t workspace_bytes, void* stream) {
    VarFlags vf;
    int rc = check_variant(variant, &vf);
    if (rc) return rc;
    rkv_desc flat{};
    rc = check_paged_desc(desc, &flat);
    if (rc) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t P = flat.num_problems;
    if (n_cached < 1 || n_cached > flat.n_capacity || budget < 1 || budget > flat.n_capacity ||
        n_obs < 1 || n_obs > budget || beta < 0)
        return RKV_ERR_INVALID_ARG;
    const size_t es = elem_size(flat.dtype);
    const size_t pool_bytes =
        (size_t)desc->num_blocks * desc->num_kv_heads * desc->block_size * desc->head_dim * es;
    const int n_free = n_cached <= budget ? 0
                                          : blocks_for(n_cached, desc->block_size) -
                                                blocks_for(budget, desc->block_size);
    if (P > 0) {
        if (!K_pool || !V_pool || !Q_obs || !block_table || !out_idx) return RKV_ERR_INVALID_ARG;
        if (n_free > 0 && !out_freed) return RKV_ERR_INVALID_ARG;
        if (!aligned16(K_pool) || !aligned16(V_pool) || !aligned16(Q_obs))
            return RKV_ERR_INVALID_ARG;
        if (K_pool == V_pool || partial_overlap(K_pool, pool_bytes, V_pool, pool_bytes))
            return RKV_ERR_ALIAS;
    }
    if (n_cached <= budget) {
        // nothing to evict: the rows stay where they are
        if (P == 0) return RKV_OK;
        cudaError_t e = timed(kIdentity, s, [&] {
            return rkv::launch_identity_idx(P, n_cached, budget, out_idx, s);
        });
        return e == cudaSuccess ? RKV_OK : RKV_ERR_CUDA;
    }
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) % kAlign) != 0) return RKV_ERR_WORKSPACE;
    if (n_cached < 2 || n_obs >= n_cached) return RKV_ERR_INVALID_ARG;
    if (flat.gqa_group * n_obs > 128) return RKV_ERR_UNSUPPORTED;
    const int tail = tail_rows(variant, n_obs);
    if (rkv::compact_smem_bytes(n_cached, tail, budget, vf.zvar && variant->sentences) >
        kCompactSmemMax)
        return RKV_ERR_UNSUPPORTED;
    const bool direct = paged_reads_pool(desc, flat, n_cached, n_obs, beta);
    const size_t kc = direct ? 0 : kc_bytes_for(flat, n_cached);
    {
        // the in-place read needs the tensor-core stages (the driver's
        // tensor-map entry point); nothing else reads the pool directly
        ScoreArgs b{};
        b.P = P; b.G = flat.gqa_group; b.d = flat.head_dim; b.N = n_cached; b.n_obs = n_obs;
        b.beta = beta; b.dtype = flat.dtype; b.ld_ws = row_pitch(n_cached);
        if (direct && !(rkv::gram_tc_supported(b) && rkv::importance_tc_supported(b)))
            return RKV_ERR_CUDA;
    }
    if (workspace_bytes < carve(nullptr, P, n_cached, kc).bytes) return RKV_ERR_WORKSPACE;
    if (check_variant_sizes(variant, n_cached, n_obs, budget)) return RKV_ERR_INVALID_ARG;
    if (P == 0) return RKV_OK;
    const Workspace w = carve(workspace, P, n_cached, kc);
    rkv::PagedIn pg;
    pg.table = block_table;
    pg.max_blocks = desc->max_blocks_per_seq;
    pg.log2bs = log2_exact(desc->block_size);
    pg.H = desc->num_kv_heads;
    pg.num_blocks = desc->num_blocks;
    const int row_bytes = desc->head_dim * (int)es;
    if (direct && !vf.any()) {
        // the two-partition schedule, where the round takes it (pools read in
        // place; the kept rows move inside their blocks, group by group)
        ScoreArgs a = score_args(&flat, K_pool, Q_obs, n_cached, n_obs, lambda, beta, tau, w.I,
                                 nullptr, w.Z, w.ld, w);
        a.pg = pg;
        a.paged_direct = true;
        CompactCall cc{n_cached, tail, budget, flat.n_capacity, flat.n_capacity, row_bytes, true,
                       K_pool, V_pool, K_pool, V_pool, out_idx};
        cc.paged = true;
        rc = run_overlapped(a, cc, s);
        if (rc > 0) return rc;
        if (rc == RKV_OK) {
            cudaError_t e = cudaSuccess;
            if (n_free > 0)
                e = timed(kPagedRelease, s, [&] {
                    return rkv::launch_paged_release(desc->num_seqs, block_table,
                                                     desc->max_blocks_per_seq,
                                                     blocks_for(budget, desc->block_size),
                                                     blocks_for(n_cached, desc->block_size),
                                                     out_freed, s);
                });
            return e == cudaSuccess ? RKV_OK : RKV_ERR_CUDA;
        }
    }
    if (vf.zvar && launch_penalty(variant, s) != cudaSuccess) return RKV_ERR_CUDA;
    rc = run_scores(&flat, K_pool, Q_obs, n_cached, n_obs, lambda, beta, tau, w.I,
                    vf.zvar ? w.R : nullptr, w.Z, w.ld, w, s, &pg, direct);
    if (rc) return rc;
    rkv::VariantIn vin;
    if (vf.any()) vin = variant_in(*variant, vf, lambda, w, samples(variant, n_cached, budget));
    cudaError_t e = timed(kCompactPaged, s, [&] {
        return rkv::launch_compact_paged(P, n_cached, w.Z, w.ld, tail, budget, out_idx,
                                         direct ? nullptr : w.Kc,
                                         K_pool, V_pool, pg, row_bytes, w.status, s, vin);
    });
    if (e == cudaSuccess && n_free > 0)
        e = timed(kPagedRelease, s, [&] {
            return rkv::launch_paged_release(desc->num_seqs, block_table, desc->max_blocks_per_seq,
                                             blocks_for(budget, desc->block_size),
                                             blocks_for(n_cached, desc->block_size), out_freed, s);
        });
    return e == cudaSuccess ? RKV_OK : RKV_ERR_CUDA;
}

int rkv_sentence_penalty(const rkv_sentences* sent, void* stream) {
    if (!sent) return RKV_ERR_INVALID_ARG;
    rkv_variant v{0, 1, sent, nullptr};
    VarFlags f;
    int rc = check_variant(&v, &f);
    if (rc) return rc;
    return launch_penalty(&v, static_cast<cudaStream_t>(stream)) == cudaSuccess ? RKV_OK
                                                                               : RKV_ERR_CUDA;
}

int rkv_sentence_reps(const void* hidden, const int32_t* token_seg, int64_t num_seqs, int T,
                      int hidden_dim, int dtype, int max_sentences, float* out_reps,
                      void* stream) {
    if (num_seqs < 0 || T < 0 || hidden_dim < 4 || hidden_dim > RKV_MAX_HIDDEN ||
        (hidden_dim & 3) != 0 || max_sentences < 1 || max_sentences > RKV_MAX_SENTENCES)
        return RKV_ERR_INVALID_ARG;
    if (dtype != RKV_DTYPE_BF16 && dtype != RKV_DTYPE_FP32) return RKV_ERR_UNSUPPORTED;
    const int64_t chunks = (hidden_dim / 4 + 255) / 256;
    if (num_seqs * chunks >= ((int64_t)1 << 31)) return RKV_ERR_INVALID_ARG;
    if (num_seqs == 0) return RKV_OK;
    if (!out_reps || !aligned16(out_reps) || (T > 0 && (!hidden || !token_seg || !aligned16(hidden))))
        return RKV_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = timed(kSentenceReps, s, [&] {
        return rkv::launch_sentence_reps(hidden, dtype, token_seg, num_seqs, T, hidden_dim,
                                         max_sentences, out_reps, s);
    });
    return e == cudaSuccess ? RKV_OK : RKV_ERR_CUDA;
}

int rkv_select(int64_t num_problems, int n, const float* Z, int n_obs, int budget,
               int32_t* out_idx, void* stream) {
    if (num_problems < 0 || n_obs < 0 || n_obs > budget || budget >= n || n > RKV_MAX_TOKENS ||
        budget < 1)
        return RKV_ERR_INVALID_ARG;
    if (num_problems == 0) return RKV_OK;
    if (!Z || !out_idx) return RKV_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = timed(kSelect, s, [&] {
        return rkv::launch_select(num_problems, n, Z, n, n_obs, budget, out_idx, nullptr, s);
    });
    return e == cudaSuccess ? RKV_OK : RKV_ERR_CUDA;
}

int rkv_gather(const rkv_desc* desc, const void* src, const int32_t* idx, int budget, void* dst,
               void* stream) {
    int rc = check_desc(desc);
    if (rc) return rc;
    const int ocap = out_cap(desc);
    if (budget < 1 || budget > desc->n_capacity || budget > ocap) return RKV_ERR_INVALID_ARG;
    if (desc->num_problems == 0) return RKV_OK;
    if (!src || !dst || !idx || !aligned16(src) || !aligned16(dst)) return RKV_ERR_INVALID_ARG;
    if (src == dst && ocap != desc->n_capacity) return RKV_ERR_INVALID_ARG;
    const size_t es = elem_size(desc->dtype);
    const size_t bytes = (size_t)desc->num_problems * desc->n_capacity * desc->head_dim * es;
    const size_t obytes = (size_t)desc->num_problems * ocap * desc->head_dim * es;
    if (partial_overlap(src, bytes, dst, obytes)) return RKV_ERR_ALIAS;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = timed(kGather, s, [&] {
        return rkv::launch_gather(src, nullptr, dst, nullptr, idx, desc->num_problems,
                                  desc->n_capacity, ocap, budget, desc->head_dim * (int)es,
                                  src == dst, nullptr, s);
    });
    return e == cudaSuccess ? RKV_OK : RKV_ERR_CUDA;
}

int rkv_selftest_wait_timeout(void* workspace, void* stream) {
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) % kAlign) != 0)
        return RKV_ERR_WORKSPACE;
    return rkv::launch_wait_timeout(reinterpret_cast<DeviceStatus*>(workspace),
                                    static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? RKV_OK
               : RKV_ERR_CUDA;
}

int rkv_workspace_init(void* workspace, void* stream) {
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) % kAlign) != 0)
        return RKV_ERR_WORKSPACE;
    return cudaMemsetAsync(workspace, 0, sizeof(DeviceStatus), static_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? RKV_OK
               : RKV_ERR_CUDA;
}

int rkv_get_device_status(void* workspace, void* stream) {
    if (!workspace) return RKV_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    DeviceStatus h{};
    if (cudaStreamSynchronize(s) != cudaSuccess) return RKV_ERR_CUDA;
    if (cudaMemcpy(&h, workspace, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess)
        return RKV_ERR_CUDA;
    if (h.code != 0) {
        const DeviceStatus zero{};
        if (cudaMemcpy(workspace, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
            return RKV_ERR_CUDA;
        return RKV_ERR_DEVICE;
    }
    return RKV_OK;
}

const char* rkv_strerror(int code) {
    switch (code) {
        case RKV_OK: return "ok";
        case RKV_ERR_INVALID_ARG: return "invalid argument";
        case RKV_ERR_UNSUPPORTED: return "unsupported dtype, head_dim or group size";
        case RKV_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        case RKV_ERR_ALIAS: return "outputs partially overlap inputs";
        case RKV_ERR_CUDA: return "CUDA launch or runtime error";
        case RKV_ERR_DEVICE: return "a kernel recorded an error";
        case RKV_ERR_TOO_LARGE: return "request exceeds the static scratch of rkv_compress_noalloc";
        default: return "unknown error code";
    }
}

int rkv_set_overlap(int mode, int groups, int tensor_sms) {
    if (mode < RKV_SCHEDULE_ONE_LAUNCH || mode > RKV_SCHEDULE_GROUPED || groups < 2 ||
        groups > kMaxGroups || (tensor_sms != 0 && tensor_sms < 8))
        return RKV_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_overlap_mu);
    g_overlap_mode = mode;
    g_overlap_groups = groups;
    g_overlap_tensor_sms = tensor_sms;
    return RKV_OK;
}

int rkv_trace_enable(int on) {
    g_trace = on != 0;
    if (g_trace) {
        g_trace_recs.clear();
        g_trace_slots = 0;
    }
    return RKV_OK;
}

int rkv_trace_read(int* kernel, int* lane, uint64_t* start_ns, uint64_t* end_ns, int max_records) {
    if (cudaDeviceSynchronize() != cudaSuccess) return -RKV_ERR_CUDA;
    const int n = (int)g_trace_recs.size() < max_records ? (int)g_trace_recs.size() : max_records;
    std::vector<unsigned long long> ns((size_t)g_trace_slots + 1);
    if (g_trace_slots > 0 &&
        cudaMemcpyFromSymbol(ns.data(), g_trace_ns, sizeof(unsigned long long) * g_trace_slots) !=
            cudaSuccess)
        return -RKV_ERR_CUDA;
    for (int i = 0; i < n; ++i) {
        const TraceRecord& r = g_trace_recs[i];
        if (kernel) kernel[i] = r.kernel;
        if (lane) lane[i] = r.lane;
        if (start_ns) start_ns[i] = ns[r.slot];
        if (end_ns) end_ns[i] = ns[r.slot + 1];
    }
    g_trace_recs.clear();
    g_trace_slots = 0;
    return n;
}

int rkv_timing_enable(int on) {
    g_timing = on != 0;
    return RKV_OK;
}

int rkv_timing_read(double* total_ms, int64_t* launches, int max_kernels, int reset) {
    for (TimedLaunch& t : g_pending) {
        if (cudaEventSynchronize(t.stop) != cudaSuccess) return -RKV_ERR_CUDA;
        float ms = 0.f;
        cudaEventElapsedTime(&ms, t.start, t.stop);
        g_total_ms[t.kernel] += ms;
        g_launches[t.kernel] += 1;
        g_event_pool[t.ctx].push_back(t.start);
        g_event_pool[t.ctx].push_back(t.stop);
    }
    g_pending.clear();
    for (int k = 0; k < kNumKernels && k < max_kernels; ++k) {
        if (total_ms) total_ms[k] = g_total_ms[k];
        if (launches) launches[k] = g_launches[k];
    }
    if (reset) {
        memset(g_total_ms, 0, sizeof(g_total_ms));
        memset(g_launches, 0, sizeof(g_launches));
    }
    return kNumKernels;
}

const char* rkv_kernel_name(int kernel) {
    if (kernel < 0 || kernel >= kNumKernels) return nullptr;
    return kKernelNames[kernel];
}

}  // extern "C"
