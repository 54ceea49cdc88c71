"""Thin ctypes binding of librkv (include/rkv.h), one function per C entry
point with the same name.

The binding only checks tensor metadata, allocates outputs the caller did not
pass, and forwards raw device pointers plus the current CUDA stream to the
library; every step of the computation runs in librkv's kernels.  There is no
fallback: if ``librkv.so`` is missing the import of a function raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "librkv.so")

RKV_OK = 0
RKV_DTYPE_BF16 = 0
RKV_DTYPE_FP32 = 1
RKV_MAX_TOKENS = 32768

EXPORTED = [
    "rkv_workspace_size", "rkv_compress", "rkv_score", "rkv_select", "rkv_gather",
    "rkv_workspace_init", "rkv_get_device_status", "rkv_strerror", "rkv_timing_enable",
    "rkv_timing_read", "rkv_kernel_name", "rkv_compress_noalloc", "rkv_compress_ex",
    "rkv_score_ex", "rkv_paged_workspace_size", "rkv_paged_freed_per_seq", "rkv_paged_compress",
    "rkv_sentence_reps", "rkv_sentence_penalty", "rkv_selftest_wait_timeout",
    "rkv_noalloc_device_status", "rkv_noalloc_selftest_wait_timeout", "rkv_set_overlap",
    "rkv_trace_enable", "rkv_trace_read",
]
RKV_MAX_POOL_WINDOW = 255
RKV_ERR_DEVICE = 6
RKV_ERR_TOO_LARGE = 7


class RkvError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {strerror(code)} (code {code})")


class _Desc(ctypes.Structure):
    _fields_ = [("num_problems", ctypes.c_int64), ("gqa_group", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("n_capacity", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("out_capacity", ctypes.c_int32)]


class _Sentences(ctypes.Structure):
    _fields_ = [("reps", ctypes.c_void_p), ("count", ctypes.c_void_p),
                ("seg_id", ctypes.c_void_p), ("penalty", ctypes.c_void_p),
                ("num_seqs", ctypes.c_int64), ("heads", ctypes.c_int32),
                ("max_sentences", ctypes.c_int32), ("hidden_dim", ctypes.c_int32),
                ("ld_seg", ctypes.c_int32), ("tau", ctypes.c_float)]


class _Schedule(ctypes.Structure):
    _fields_ = [("recent_window", ctypes.c_int32), ("pool_size", ctypes.c_int32),
                ("temperature", ctypes.c_float), ("ld_uniforms", ctypes.c_int32),
                ("uniforms", ctypes.c_void_p)]


class _Variant(ctypes.Structure):
    _fields_ = [("redundancy_softmax", ctypes.c_int32), ("pool_window", ctypes.c_int32),
                ("sentences", ctypes.POINTER(_Sentences)),
                ("schedule", ctypes.POINTER(_Schedule))]


class Schedule:
    """ForesightKV-style schedule (rkv_schedule in include/rkv.h): keep the
    newest recent_window rows, pool the top pool_size candidates by Z, draw
    budget - recent_window of them without replacement with probabilities
    proportional to exp(Z / temperature), using uniforms [P, >= C] fp32 in
    [0, 1) (from a seeded generator).  pool_size = budget - recent_window:
    deterministic top-k (uniforms may be None)."""

    def __init__(self, recent_window: int, pool_size: int, temperature: float = 1.0,
                 uniforms=None):
        if uniforms is not None:
            _cuda(uniforms, "uniforms")
            if uniforms.dtype != torch.float32 or uniforms.dim() != 2:
                raise ValueError("uniforms must be fp32 [P, >= C]")
        self.recent_window, self.pool_size = int(recent_window), int(pool_size)
        self.temperature, self.uniforms = float(temperature), uniforms

    def _c(self) -> _Schedule:
        u = self.uniforms
        return _Schedule(self.recent_window, self.pool_size, self.temperature,
                         u.shape[1] if u is not None else 0,
                         u.data_ptr() if u is not None else None)


class Sentences:
    """Sentence-level penalty inputs (rkv_sentences in include/rkv.h):
    reps [S, max_sentences, hidden] fp32, count [S] int32, seg_id [P, ld_seg]
    int32 (the sentence of each cached row; compacted in place by the
    compression), heads (problem p belongs to sequence (p // heads) % S),
    tau.  penalty [S, max_sentences] fp32 receives the sentence penalties."""

    def __init__(self, reps, count, seg_id, heads: int, tau: float, penalty=None):
        for t, n in ((reps, "reps"), (count, "count"), (seg_id, "seg_id")):
            _cuda(t, n)
        if reps.dtype != torch.float32 or reps.dim() != 3:
            raise ValueError("reps must be fp32 [S, max_sentences, hidden]")
        if count.dtype != torch.int32 or seg_id.dtype != torch.int32 or seg_id.dim() != 2:
            raise ValueError("count, seg_id must be int32 ([S], [P, ld_seg])")
        self.reps, self.count, self.seg_id = reps, count, seg_id
        self.heads, self.tau = int(heads), float(tau)
        self.penalty = penalty if penalty is not None else torch.empty(
            reps.shape[:2], dtype=torch.float32, device=reps.device)

    def _c(self) -> _Sentences:
        S, M, Dh = self.reps.shape
        return _Sentences(self.reps.data_ptr(), self.count.data_ptr(), self.seg_id.data_ptr(),
                          self.penalty.data_ptr(), S, self.heads, M, Dh, self.seg_id.shape[1],
                          self.tau)


def _variant(redundancy_softmax: bool, pool_window: int, sentences, schedule=None):
    """The C variant struct (and the structs it points to, which the caller
    keeps alive for the call)."""
    sc = sentences._c() if sentences is not None else None
    sh = schedule._c() if schedule is not None else None
    v = _Variant(1 if redundancy_softmax else 0, int(pool_window),
                 ctypes.pointer(sc) if sc is not None else None,
                 ctypes.pointer(sh) if sh is not None else None)
    return v, (sc, sh)


class _PagedDesc(ctypes.Structure):
    _fields_ = [("num_seqs", ctypes.c_int64), ("num_kv_heads", ctypes.c_int32),
                ("gqa_group", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("num_blocks", ctypes.c_int32),
                ("max_blocks_per_seq", ctypes.c_int32), ("dtype", ctypes.c_int32)]


_lock = threading.Lock()
_lib = None


def load(path: str | None = None):
    """Loads librkv.so (built by ``decode_kv_cache_02_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(
                f"librkv.so not found at {p}; build it with "
                "`python -m decode_kv_cache_02_gb300.build` (no fallback exists)")
        lib = ctypes.CDLL(p)
        vp, sz, i32, i64, f32 = (ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int,
                                 ctypes.c_int64, ctypes.c_float)
        dp = ctypes.POINTER(_Desc)
        lib.rkv_workspace_size.argtypes = [dp, i32, i32]
        lib.rkv_workspace_size.restype = sz
        lib.rkv_compress.argtypes = [dp, vp, vp, vp, i32, i32, i32, f32, i32, f32, vp, vp, vp,
                                     vp, sz, vp]
        lib.rkv_compress.restype = i32
        lib.rkv_score.argtypes = [dp, vp, vp, i32, i32, f32, i32, f32, vp, vp, vp, vp, sz, vp]
        lib.rkv_score.restype = i32
        vr = ctypes.POINTER(_Variant)
        lib.rkv_compress_ex.argtypes = [dp, vp, vp, vp, i32, i32, i32, f32, i32, f32, vr, vp, vp,
                                        vp, vp, sz, vp]
        lib.rkv_compress_ex.restype = i32
        lib.rkv_score_ex.argtypes = [dp, vp, vp, i32, i32, f32, i32, f32, vr, vp, vp, vp, vp, sz,
                                     vp]
        lib.rkv_score_ex.restype = i32
        pdp = ctypes.POINTER(_PagedDesc)
        lib.rkv_paged_workspace_size.argtypes = [pdp, i32, i32, i32]
        lib.rkv_paged_workspace_size.restype = sz
        lib.rkv_paged_freed_per_seq.argtypes = [pdp, i32, i32]
        lib.rkv_paged_freed_per_seq.restype = i32
        lib.rkv_paged_compress.argtypes = [pdp, vp, vp, vp, vp, i32, i32, i32, f32, i32, f32, vr,
                                           vp, vp, vp, sz, vp]
        lib.rkv_paged_compress.restype = i32
        lib.rkv_sentence_reps.argtypes = [vp, vp, i64, i32, i32, i32, i32, vp, vp]
        lib.rkv_sentence_reps.restype = i32
        lib.rkv_sentence_penalty.argtypes = [ctypes.POINTER(_Sentences), vp]
        lib.rkv_sentence_penalty.restype = i32
        lib.rkv_selftest_wait_timeout.argtypes = [vp, vp]
        lib.rkv_selftest_wait_timeout.restype = i32
        lib.rkv_noalloc_device_status.argtypes = [vp]
        lib.rkv_noalloc_device_status.restype = i32
        lib.rkv_noalloc_selftest_wait_timeout.argtypes = [vp]
        lib.rkv_noalloc_selftest_wait_timeout.restype = i32
        lib.rkv_select.argtypes = [i64, i32, vp, i32, i32, vp, vp]
        lib.rkv_select.restype = i32
        lib.rkv_gather.argtypes = [dp, vp, vp, i32, vp, vp]
        lib.rkv_gather.restype = i32
        lib.rkv_workspace_init.argtypes = [vp, vp]
        lib.rkv_workspace_init.restype = i32
        lib.rkv_get_device_status.argtypes = [vp, vp]
        lib.rkv_get_device_status.restype = i32
        lib.rkv_strerror.argtypes = [i32]
        lib.rkv_strerror.restype = ctypes.c_char_p
        lib.rkv_set_overlap.argtypes = [i32, i32, i32]
        lib.rkv_set_overlap.restype = i32
        lib.rkv_trace_enable.argtypes = [i32]
        lib.rkv_trace_enable.restype = i32
        lib.rkv_trace_read.argtypes = [vp, vp, vp, vp, i32]
        lib.rkv_trace_read.restype = i32
        lib.rkv_timing_enable.argtypes = [i32]
        lib.rkv_timing_enable.restype = i32
        lib.rkv_timing_read.argtypes = [ctypes.POINTER(ctypes.c_double),
                                        ctypes.POINTER(ctypes.c_int64), i32, i32]
        lib.rkv_timing_read.restype = i32
        lib.rkv_compress_noalloc.argtypes = [dp, vp, vp, vp, i32, i32, i32, f32, i32, f32, vp,
                                             vp, vp, vp]
        lib.rkv_compress_noalloc.restype = i32
        lib.rkv_kernel_name.argtypes = [i32]
        lib.rkv_kernel_name.restype = ctypes.c_char_p
        _lib = lib
        return lib


def strerror(code: int) -> str:
    return load().rkv_strerror(int(code)).decode()


def _check(rc: int, where: str):
    if rc != RKV_OK:
        raise RkvError(rc, where)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return RKV_DTYPE_BF16
    if t.dtype == torch.float32:
        return RKV_DTYPE_FP32
    raise TypeError(f"unsupported dtype {t.dtype} (bf16 or fp32)")


def _cuda(t: torch.Tensor, name: str):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _stream_ptr(stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def make_desc(K: torch.Tensor, gqa_group: int, out=None) -> _Desc:
    """Descriptor of a K (or V) tensor [P, n_capacity, head_dim], with the
    outputs' rows per problem taken from `out` [P, out_capacity, head_dim]."""
    if K.dim() != 3:
        raise ValueError("K must be [P, n_capacity, head_dim]")
    P, n_cap, d = K.shape
    out_cap = 0 if out is None or out.dim() != 3 or out.shape[1] == n_cap else out.shape[1]
    return _Desc(P, int(gqa_group), d, n_cap, _dtype_code(K), out_cap)


def rkv_workspace_size(K: torch.Tensor, gqa_group: int, n_cached: int, n_obs: int) -> int:
    desc = make_desc(K, gqa_group)
    return int(load().rkv_workspace_size(ctypes.byref(desc), int(n_cached), int(n_obs)))


def alloc_workspace(K: torch.Tensor, gqa_group: int, n_cached: int, n_obs: int) -> torch.Tensor:
    """A zero-filled uint8 device tensor of rkv_workspace_size() bytes."""
    n = rkv_workspace_size(K, gqa_group, n_cached, n_obs)
    if n == 0:
        raise ValueError("invalid workspace request")
    return torch.zeros(n, dtype=torch.uint8, device=K.device)


def _compress_args(K, V, Q_obs, n_cached, budget, n_obs, out_K, out_V, out_idx, workspace):
    for t, n in ((K, "K"), (V, "V"), (Q_obs, "Q_obs")):
        _cuda(t, n)
    if V.shape != K.shape or V.dtype != K.dtype or Q_obs.dtype != K.dtype:
        raise ValueError("K, V, Q_obs must share shape/dtype")
    if Q_obs.dim() != 4 or Q_obs.shape[0] != K.shape[0] or Q_obs.shape[2] != n_obs \
            or Q_obs.shape[3] != K.shape[2]:
        raise ValueError("Q_obs must be [P, G, n_obs, d]")
    G = Q_obs.shape[1]
    if out_K is None:
        out_K = torch.empty_like(K)
    if out_V is None:
        out_V = torch.empty_like(V)
    if out_idx is None:
        out_idx = torch.empty((K.shape[0], budget), dtype=torch.int32, device=K.device)
    if workspace is None:
        workspace = alloc_workspace(K, G, max(n_cached, 1), n_obs)
    for t, n in ((out_K, "out_K"), (out_V, "out_V"), (out_idx, "out_idx")):
        _cuda(t, n)
    # outputs hold n_capacity rows per problem, or any count >= budget
    if out_K.dim() != 3 or out_V.shape != out_K.shape or out_K.shape[0] != K.shape[0] \
            or out_K.shape[2] != K.shape[2] or out_K.shape[1] < budget \
            or out_K.dtype != K.dtype or out_V.dtype != K.dtype \
            or out_idx.shape != (K.shape[0], budget) or out_idx.dtype != torch.int32:
        raise ValueError("output shapes")
    desc = make_desc(K, G, out_K)
    return desc, out_K, out_V, out_idx, workspace


def rkv_compress(K, V, Q_obs, n_cached: int, budget: int, n_obs: int = 8, lam: float = 0.1,
                 beta: int = 2, tau: float = 0.9, out_K=None, out_V=None, out_idx=None,
                 workspace=None, stream=None):
    """One compression round of every problem in K/V [P, n_cap, d] with
    Q_obs [P, G, n_obs, d].  Returns (out_K, out_V, out_idx); pass
    out_K=K, out_V=V to compact in place."""
    desc, out_K, out_V, out_idx, workspace = _compress_args(
        K, V, Q_obs, n_cached, budget, n_obs, out_K, out_V, out_idx, workspace)
    rc = load().rkv_compress(ctypes.byref(desc), K.data_ptr(), V.data_ptr(), Q_obs.data_ptr(),
                             int(n_cached), int(budget), int(n_obs), float(lam), int(beta),
                             float(tau), out_K.data_ptr(), out_V.data_ptr(), out_idx.data_ptr(),
                             workspace.data_ptr(), workspace.numel(), _stream_ptr(stream))
    _check(rc, "rkv_compress")
    return out_K, out_V, out_idx


def rkv_compress_ex(K, V, Q_obs, n_cached: int, budget: int, n_obs: int = 8, lam: float = 0.1,
                    beta: int = 2, tau: float = 0.9, redundancy_softmax: bool = False,
                    pool_window: int = 1, sentences: Sentences | None = None,
                    schedule: Schedule | None = None, out_K=None, out_V=None, out_idx=None,
                    workspace=None, stream=None):
    """rkv_compress with a scoring variant: redundancy_softmax turns R into a
    softmax over the candidates, pool_window (odd) max-pools I over that many
    neighbouring positions, sentences adds the sentence-level penalty (and
    compacts sentences.seg_id with the rows), schedule keeps a recent window
    and samples the kept candidates."""
    desc, out_K, out_V, out_idx, workspace = _compress_args(
        K, V, Q_obs, n_cached, budget, n_obs, out_K, out_V, out_idx, workspace)
    var, _keep = _variant(redundancy_softmax, pool_window, sentences, schedule)
    rc = load().rkv_compress_ex(ctypes.byref(desc), K.data_ptr(), V.data_ptr(), Q_obs.data_ptr(),
                                int(n_cached), int(budget), int(n_obs), float(lam), int(beta),
                                float(tau), ctypes.byref(var), out_K.data_ptr(), out_V.data_ptr(),
                                out_idx.data_ptr(), workspace.data_ptr(), workspace.numel(),
                                _stream_ptr(stream))
    _check(rc, "rkv_compress_ex")
    return out_K, out_V, out_idx


def rkv_compress_noalloc(K, V, Q_obs, n_cached: int, budget: int, n_obs: int = 8,
                         lam: float = 0.1, beta: int = 2, tau: float = 0.9, out_K=None,
                         out_V=None, out_idx=None, stream=None):
    """rkv_compress with the library's static scratch instead of a workspace,
    for callers that may not allocate device memory while they run (pass
    preallocated out_K / out_V / out_idx to allocate nothing at all).  Calls
    that may overlap on the GPU share the scratch and must be serialised."""
    for t, n in ((K, "K"), (V, "V"), (Q_obs, "Q_obs")):
        _cuda(t, n)
    if V.shape != K.shape or V.dtype != K.dtype or Q_obs.dtype != K.dtype or Q_obs.dim() != 4:
        raise ValueError("K, V, Q_obs must share shape/dtype; Q_obs is [P, G, n_obs, d]")
    if out_K is None:
        out_K = torch.empty_like(K)
    if out_V is None:
        out_V = torch.empty_like(V)
    if out_idx is None:
        out_idx = torch.empty((K.shape[0], budget), dtype=torch.int32, device=K.device)
    if out_V.shape != out_K.shape:
        raise ValueError("out_K and out_V must have the same shape")
    desc = make_desc(K, Q_obs.shape[1], out_K)
    rc = load().rkv_compress_noalloc(ctypes.byref(desc), K.data_ptr(), V.data_ptr(),
                                     Q_obs.data_ptr(), int(n_cached), int(budget), int(n_obs),
                                     float(lam), int(beta), float(tau), out_K.data_ptr(),
                                     out_V.data_ptr(), out_idx.data_ptr(), _stream_ptr(stream))
    _check(rc, "rkv_compress_noalloc")
    return out_K, out_V, out_idx


def _score(K, Q_obs, n_cached, n_obs, lam, beta, tau, variant, workspace, stream, _keep=None):
    _cuda(K, "K")
    _cuda(Q_obs, "Q_obs")
    G = Q_obs.shape[1]
    desc = make_desc(K, G)
    P = K.shape[0]
    I = torch.empty((P, n_cached), dtype=torch.float32, device=K.device)
    R = torch.empty_like(I)
    Z = torch.empty_like(I)
    if workspace is None:
        workspace = alloc_workspace(K, G, n_cached, n_obs)
    args = (int(n_cached), int(n_obs), float(lam), int(beta), float(tau))
    outs = (I.data_ptr(), R.data_ptr(), Z.data_ptr(), workspace.data_ptr(), workspace.numel(),
            _stream_ptr(stream))
    if variant is None:
        rc = load().rkv_score(ctypes.byref(desc), K.data_ptr(), Q_obs.data_ptr(), *args, *outs)
        _check(rc, "rkv_score")
    else:
        rc = load().rkv_score_ex(ctypes.byref(desc), K.data_ptr(), Q_obs.data_ptr(), *args,
                                 ctypes.byref(variant), *outs)
        _check(rc, "rkv_score_ex")
    return I, R, Z


def rkv_score(K, Q_obs, n_cached: int, n_obs: int = 8, lam: float = 0.1, beta: int = 2,
              tau: float = 0.9, workspace=None, stream=None):
    """(I, R, Z), each fp32 [P, n_cached]."""
    return _score(K, Q_obs, n_cached, n_obs, lam, beta, tau, None, workspace, stream)


def rkv_score_ex(K, Q_obs, n_cached: int, n_obs: int = 8, lam: float = 0.1, beta: int = 2,
                 tau: float = 0.9, redundancy_softmax: bool = False, pool_window: int = 1,
                 sentences: Sentences | None = None, schedule: Schedule | None = None,
                 workspace=None, stream=None):
    """(I', R', Z), each fp32 [P, n_cached], for a scoring variant (see
    rkv_compress_ex); I' and R' are the terms that enter Z."""
    var, keep = _variant(redundancy_softmax, pool_window, sentences, schedule)
    return _score(K, Q_obs, n_cached, n_obs, lam, beta, tau, var, workspace, stream, keep)


def rkv_select(Z, n_obs: int, budget: int, out_idx=None, stream=None):
    """idx [P, budget] of the kept tokens for fp32 scores Z [P, n]."""
    _cuda(Z, "Z")
    if Z.dtype != torch.float32 or Z.dim() != 2:
        raise ValueError("Z must be fp32 [P, n]")
    P, n = Z.shape
    if out_idx is None:
        out_idx = torch.empty((P, budget), dtype=torch.int32, device=Z.device)
    rc = load().rkv_select(P, n, Z.data_ptr(), int(n_obs), int(budget), out_idx.data_ptr(),
                           _stream_ptr(stream))
    _check(rc, "rkv_select")
    return out_idx


def rkv_gather(src, idx, budget: int, dst=None, stream=None):
    """dst[p, r] = src[p, idx[p, r]] for r < budget (dst=src: in place)."""
    _cuda(src, "src")
    _cuda(idx, "idx")
    if idx.dtype != torch.int32 or idx.shape != (src.shape[0], budget):
        raise ValueError("idx must be int32 [P, budget]")
    if dst is None:
        dst = torch.empty_like(src)
    _cuda(dst, "dst")
    if dst.dim() != 3 or dst.shape[0] != src.shape[0] or dst.shape[2] != src.shape[2] \
            or dst.shape[1] < budget or dst.dtype != src.dtype:
        raise ValueError("dst must be [P, >= budget, d] of src's dtype")
    desc = make_desc(src, 1, dst)
    rc = load().rkv_gather(ctypes.byref(desc), src.data_ptr(), idx.data_ptr(), int(budget),
                           dst.data_ptr(), _stream_ptr(stream))
    _check(rc, "rkv_gather")
    return dst


def rkv_workspace_init(workspace, stream=None):
    _check(load().rkv_workspace_init(workspace.data_ptr(), _stream_ptr(stream)),
           "rkv_workspace_init")


def rkv_get_device_status(workspace, stream=None) -> int:
    """Synchronises the stream; returns RKV_OK or the device error code."""
    return int(load().rkv_get_device_status(workspace.data_ptr(), _stream_ptr(stream)))


RKV_SCHEDULE_ONE_LAUNCH, RKV_SCHEDULE_AUTO, RKV_SCHEDULE_GROUPED = 0, 1, 2
DEFAULT_OVERLAP = (RKV_SCHEDULE_AUTO, 8, 0)  # the library's default step schedule


def rkv_set_overlap(mode: int, groups: int = 8, tensor_sms: int = 0):
    """Step schedule of rkv_compress: RKV_SCHEDULE_ONE_LAUNCH, _AUTO (grouped
    where the cost model predicts a gain) or _GROUPED (wherever eligible):
    groups of problems scored on about tensor_sms SMs (0: 112 of every 152)
    while the previous group is compacted on the rest."""
    _check(load().rkv_set_overlap(int(mode), int(groups), int(tensor_sms)), "rkv_set_overlap")


def rkv_trace_enable(on: bool = True):
    load().rkv_trace_enable(1 if on else 0)


def rkv_trace_read(max_records: int = 8192) -> list:
    """[(kernel name, lane, start ns, end ns)] of the traced launches in
    enqueue order (lane 0: the caller's stream, 1: the tensor partition, 2:
    the other partition); clears the trace."""
    lib = load()
    n = int(max_records)
    k = (ctypes.c_int * n)()
    ln = (ctypes.c_int * n)()
    t0 = (ctypes.c_uint64 * n)()
    t1 = (ctypes.c_uint64 * n)()
    m = lib.rkv_trace_read(k, ln, t0, t1, n)
    if m < 0:
        raise RkvError(-m, "rkv_trace_read")
    return [(lib.rkv_kernel_name(k[i]).decode(), ln[i], t0[i], t1[i]) for i in range(m)]


def rkv_timing_enable(on: bool = True):
    load().rkv_timing_enable(1 if on else 0)


def rkv_timing_read(reset: bool = True) -> dict:
    """{kernel name: (total ms, launches)} of the timed launches so far."""
    lib = load()
    n = 16
    ms = (ctypes.c_double * n)()
    cnt = (ctypes.c_int64 * n)()
    k = lib.rkv_timing_read(ms, cnt, n, 1 if reset else 0)
    if k < 0:
        raise RkvError(-k, "rkv_timing_read")
    return {lib.rkv_kernel_name(i).decode(): (ms[i], cnt[i]) for i in range(min(k, n))}


# ------------------------------------------------------------------ paged --

def make_paged_desc(K_pool: torch.Tensor, block_table: torch.Tensor, gqa_group: int) -> _PagedDesc:
    """Descriptor of a pool [num_blocks, H, block_size, d] and a block table
    [num_seqs, max_blocks_per_seq] (int32)."""
    if K_pool.dim() != 4:
        raise ValueError("K_pool must be [num_blocks, H, block_size, head_dim]")
    if block_table.dim() != 2 or block_table.dtype != torch.int32:
        raise ValueError("block_table must be int32 [num_seqs, max_blocks_per_seq]")
    nb, H, bs, d = K_pool.shape
    S, mb = block_table.shape
    return _PagedDesc(S, H, int(gqa_group), d, bs, nb, mb, _dtype_code(K_pool))


def rkv_paged_workspace_size(K_pool, block_table, gqa_group: int, n_cached: int,
                             n_obs: int, beta: int = 2) -> int:
    """Workspace bytes of rkv_paged_compress for these arguments (no
    contiguous key copy when the tensor-core stages read the pool in place)."""
    desc = make_paged_desc(K_pool, block_table, gqa_group)
    return int(load().rkv_paged_workspace_size(ctypes.byref(desc), int(n_cached), int(n_obs),
                                               int(beta)))


def rkv_paged_freed_per_seq(K_pool, block_table, n_cached: int, budget: int) -> int:
    desc = make_paged_desc(K_pool, block_table, 1)
    n = int(load().rkv_paged_freed_per_seq(ctypes.byref(desc), int(n_cached), int(budget)))
    if n < 0:
        raise ValueError("invalid paged request")
    return n


def rkv_paged_compress(K_pool, V_pool, Q_obs, block_table, n_cached: int, budget: int,
                       n_obs: int = 8, lam: float = 0.1, beta: int = 2, tau: float = 0.9,
                       redundancy_softmax: bool = False, pool_window: int = 1,
                       sentences: Sentences | None = None, schedule: Schedule | None = None,
                       out_idx=None, out_freed=None, workspace=None, stream=None):
    """One compression round of a paged cache, in place: K_pool, V_pool
    [num_blocks, H, block_size, d], Q_obs [S*H, G, n_obs, d], block_table
    [S, max_blocks] int32 (entries of freed blocks become -1).  Returns
    (out_idx [S*H, budget], out_freed [S, n_free])."""
    for t, n in ((K_pool, "K_pool"), (V_pool, "V_pool"), (Q_obs, "Q_obs"),
                 (block_table, "block_table")):
        _cuda(t, n)
    if V_pool.shape != K_pool.shape or V_pool.dtype != K_pool.dtype or Q_obs.dtype != K_pool.dtype:
        raise ValueError("K_pool, V_pool, Q_obs must share shape/dtype")
    G = Q_obs.shape[1]
    desc = make_paged_desc(K_pool, block_table, G)
    P = desc.num_seqs * desc.num_kv_heads
    if Q_obs.dim() != 4 or Q_obs.shape[0] != P or Q_obs.shape[2] != n_obs \
            or Q_obs.shape[3] != K_pool.shape[3]:
        raise ValueError("Q_obs must be [num_seqs * H, G, n_obs, d]")
    n_free = rkv_paged_freed_per_seq(K_pool, block_table, n_cached, budget)
    if out_idx is None:
        out_idx = torch.empty((P, budget), dtype=torch.int32, device=K_pool.device)
    if out_freed is None:
        out_freed = torch.empty((desc.num_seqs, n_free), dtype=torch.int32, device=K_pool.device)
    if workspace is None:
        n = rkv_paged_workspace_size(K_pool, block_table, G, max(n_cached, 1), n_obs, beta)
        if n == 0:
            raise ValueError("invalid workspace request")
        workspace = torch.zeros(n, dtype=torch.uint8, device=K_pool.device)
    _cuda(out_idx, "out_idx")
    _cuda(out_freed, "out_freed")
    if out_idx.shape != (P, budget) or out_idx.dtype != torch.int32 \
            or out_freed.shape != (desc.num_seqs, n_free) or out_freed.dtype != torch.int32:
        raise ValueError("output shapes")
    var, _keep = _variant(redundancy_softmax, pool_window, sentences, schedule)
    rc = load().rkv_paged_compress(
        ctypes.byref(desc), K_pool.data_ptr(), V_pool.data_ptr(), Q_obs.data_ptr(),
        block_table.data_ptr(), int(n_cached), int(budget), int(n_obs), float(lam), int(beta),
        float(tau), ctypes.byref(var), out_idx.data_ptr(), out_freed.data_ptr(),
        workspace.data_ptr(), workspace.numel(), _stream_ptr(stream))
    _check(rc, "rkv_paged_compress")
    return out_idx, out_freed


# -------------------------------------------------------------- sentences --

def rkv_sentence_reps(hidden, token_seg, max_sentences: int, out_reps=None, stream=None):
    """Mean hidden state of each sentence: hidden [S, T, Dh] (bf16/fp32),
    token_seg [S, T] int32 (-1: none; a sentence's tokens consecutive) ->
    reps [S, max_sentences, Dh] fp32."""
    _cuda(hidden, "hidden")
    _cuda(token_seg, "token_seg")
    S, T, Dh = hidden.shape
    if token_seg.shape != (S, T) or token_seg.dtype != torch.int32:
        raise ValueError("token_seg must be int32 [S, T]")
    if out_reps is None:
        out_reps = torch.empty((S, max_sentences, Dh), dtype=torch.float32, device=hidden.device)
    rc = load().rkv_sentence_reps(hidden.data_ptr(), token_seg.data_ptr(), S, T, Dh,
                                  _dtype_code(hidden), int(max_sentences), out_reps.data_ptr(),
                                  _stream_ptr(stream))
    _check(rc, "rkv_sentence_reps")
    return out_reps


def rkv_sentence_penalty(sentences: Sentences, stream=None):
    """Writes and returns sentences.penalty [S, max_sentences]."""
    sc = sentences._c()
    _check(load().rkv_sentence_penalty(ctypes.byref(sc), _stream_ptr(stream)),
           "rkv_sentence_penalty")
    return sentences.penalty


def rkv_selftest_wait_timeout(workspace, stream=None):
    """Enqueues one bounded wait that nothing completes; afterwards
    rkv_get_device_status(workspace) reports RKV_ERR_DEVICE."""
    _check(load().rkv_selftest_wait_timeout(workspace.data_ptr(), _stream_ptr(stream)),
           "rkv_selftest_wait_timeout")


def rkv_noalloc_device_status(stream=None) -> int:
    """Synchronises the stream; returns RKV_OK or the device error code
    recorded in rkv_compress_noalloc's static scratch (and clears it)."""
    return int(load().rkv_noalloc_device_status(_stream_ptr(stream)))


def rkv_noalloc_selftest_wait_timeout(stream=None):
    """rkv_selftest_wait_timeout on rkv_compress_noalloc's static scratch."""
    _check(load().rkv_noalloc_selftest_wait_timeout(_stream_ptr(stream)),
           "rkv_noalloc_selftest_wait_timeout")
