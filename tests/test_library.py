"""Host-side checks of the C-ABI library (no GPU needed): it builds, loads and
exports every function include/rkv.h declares; sizes and argument errors are
answered on the host without touching the device."""
import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from decode_kv_cache_02_gb300 import build, rkv
    build.build()
    return rkv.load()


def _declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(rkv_\w+)\s*\(", src))
    return names


def test_exports_every_declared_symbol(lib):
    declared = _declared_functions()
    assert "rkv_compress" in declared and "rkv_score" in declared
    for name in declared:
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"
    from decode_kv_cache_02_gb300 import rkv
    assert set(rkv.EXPORTED) >= declared


def test_strerror(lib):
    from decode_kv_cache_02_gb300 import rkv
    assert rkv.strerror(0) == "ok"
    assert "workspace" in rkv.strerror(3)
    assert rkv.strerror(999) == "unknown error code"


def _desc(P=4, G=4, d=128, n_cap=1152, dtype=0, out_cap=0):
    from decode_kv_cache_02_gb300 import rkv
    return rkv._Desc(P, G, d, n_cap, dtype, out_cap)


def test_workspace_size(lib):
    d = _desc()
    n = lib.rkv_workspace_size(ctypes.byref(d), 1152, 8)
    # status block + five fp32 [P, N] arrays (inverse norms, similarity sums,
    # I, R, Z) + the [P, 16, 128] bf16 s rows, each rounded to 256 bytes
    assert n == 256 + 5 * ((4 * 1152 * 4 + 255) // 256 * 256) + (2 * 4 * 16 * 128 + 255) // 256 * 256
    assert lib.rkv_workspace_size(None, 1152, 8) == 0
    bad = _desc(d=96)
    assert lib.rkv_workspace_size(ctypes.byref(bad), 1152, 8) == 0


def test_argument_errors_need_no_device(lib):
    from decode_kv_cache_02_gb300 import rkv
    d = _desc()
    fake = 1 << 20  # never dereferenced: every call below fails its checks first
    ws = 1 << 24
    call = lambda **kw: lib.rkv_compress(
        ctypes.byref(kw.get("desc", d)), kw.get("K", fake), fake + 2 ** 30, fake + 2 ** 31,
        kw.get("n", 1152), kw.get("budget", 1024), kw.get("n_obs", 8), 0.1, kw.get("beta", 2),
        0.9, kw.get("oK", fake + 2 ** 32), kw.get("oV", fake + 2 ** 33), fake + 2 ** 34,
        kw.get("ws", ws), kw.get("ws_bytes", 1), None)
    assert lib.rkv_compress(None, 0, 0, 0, 1, 1, 1, 0.1, 2, 0.9, 0, 0, 0, 0, 0, None) == 1
    assert call(n_obs=0) == 1                      # no observation token
    assert call(n_obs=2000) == 1                   # n_obs > budget
    assert call(n=2000) == 1                       # n_cached > capacity
    assert call(beta=-1) == 1
    assert call(K=fake + 2) == 1                   # misaligned
    assert call(desc=_desc(d=80)) == 2             # unsupported head_dim
    assert call(desc=_desc(dtype=7)) == 2
    assert call(ws_bytes=10) == 3                  # workspace too small
    assert call(ws=ws + 16, ws_bytes=1 << 40) == 3  # workspace misaligned
    assert call(oK=fake + 4096, ws_bytes=1 << 40) == 4  # partial overlap with K
    assert lib.rkv_select(1, 100, fake, 8, 100, fake, None) == 1   # budget >= n
    assert lib.rkv_select(1, 100, fake, 9, 8, fake, None) == 1     # n_obs > budget
    assert lib.rkv_gather(ctypes.byref(d), fake, fake, 0, fake, None) == 1
    # outputs of out_capacity rows per problem
    assert call(desc=_desc(out_cap=-1)) == 1
    assert call(desc=_desc(out_cap=1000)) == 1     # budget > out_capacity
    assert call(desc=_desc(out_cap=1024), oK=fake, oV=fake + 2 ** 30, ws_bytes=1 << 40) == 1
    #   (in place needs out_capacity = n_capacity)
    assert call(desc=_desc(out_cap=1024), oK=fake + 2 ** 30 - 4 * 1024 * 256 + 256,
                ws_bytes=1 << 40) == 4           # out_K's 1024-row problems run into V
    assert call(desc=_desc(out_cap=1024), ws_bytes=10) == 3  # valid, reaches the workspace check
    assert lib.rkv_gather(ctypes.byref(_desc(out_cap=100)), fake, fake, 200, fake + 2 ** 30,
                          None) == 1             # budget > out_capacity
    assert lib.rkv_gather(ctypes.byref(_desc(out_cap=1024)), fake, fake, 200, fake,
                          None) == 1             # in place with another row count


def test_variant_argument_errors(lib):
    """rkv_compress_ex / rkv_score_ex reject an invalid variant before
    anything else (nothing is dereferenced or enqueued)."""
    from decode_kv_cache_02_gb300 import rkv
    d = _desc()
    fake = 1 << 20
    for soft, win in ((2, 1), (-1, 1), (0, 0), (0, 2), (1, 8), (0, rkv.RKV_MAX_POOL_WINDOW + 2),
                      (0, -3)):
        v = rkv._Variant(soft, win)
        rc = lib.rkv_compress_ex(ctypes.byref(d), fake, fake + 2 ** 30, fake + 2 ** 31, 1152,
                                 1024, 8, 0.1, 2, 0.9, ctypes.byref(v), fake + 2 ** 32,
                                 fake + 2 ** 33, fake + 2 ** 34, fake + 2 ** 35, 1 << 40, None)
        assert rc == 1, (soft, win)
        rc = lib.rkv_score_ex(ctypes.byref(d), fake, fake + 2 ** 31, 1152, 8, 0.1, 2, 0.9,
                              ctypes.byref(v), fake + 2 ** 32, fake + 2 ** 33, fake + 2 ** 34,
                              fake + 2 ** 35, 1 << 40, None)
        assert rc == 1, (soft, win)
    # a valid variant still meets the ordinary checks (workspace too small)
    v = rkv._Variant(1, rkv.RKV_MAX_POOL_WINDOW)
    assert lib.rkv_compress_ex(ctypes.byref(d), fake, fake + 2 ** 30, fake + 2 ** 31, 1152, 1024,
                               8, 0.1, 2, 0.9, ctypes.byref(v), fake + 2 ** 32, fake + 2 ** 33,
                               fake + 2 ** 34, fake + 2 ** 35, 10, None) == 3


def test_paged_sizes_and_argument_errors(lib):
    """Paged descriptor checks, freed-block counts and workspace sizes are
    answered on the host; invalid calls enqueue nothing."""
    from decode_kv_cache_02_gb300 import rkv
    D = lambda **kw: rkv._PagedDesc(kw.get("S", 4), kw.get("H", 8), kw.get("G", 4),
                                    kw.get("d", 128), kw.get("bs", 16), kw.get("nb", 400),
                                    kw.get("mb", 80), kw.get("dtype", 0))
    d = D()
    assert lib.rkv_paged_freed_per_seq(ctypes.byref(d), 1152, 1024) == 72 - 64
    assert lib.rkv_paged_freed_per_seq(ctypes.byref(d), 1000, 1024) == 0
    assert lib.rkv_paged_freed_per_seq(ctypes.byref(d), 1153, 1024) == 73 - 64
    assert lib.rkv_paged_freed_per_seq(ctypes.byref(D(bs=12)), 1152, 1024) == -1  # not 2^k
    assert lib.rkv_paged_freed_per_seq(ctypes.byref(D(mb=10)), 1152, 1024) == -1  # > capacity
    flat = lib.rkv_workspace_size(ctypes.byref(_desc(P=32, n_cap=1152)), 1152, 8)
    copy = (32 * 1152 * 128 * 2 + 255) // 256 * 256  # contiguous keys [P, N, d] bf16
    # blocks under 128 rows: the key statistics write a contiguous copy
    assert lib.rkv_paged_workspace_size(ctypes.byref(d), 1152, 8, 2) == flat + copy
    # bf16 blocks of 128 rows or more are read in place by the tensor-core
    # stages: exactly the contiguous call's workspace
    for bs in (128, 256, 1024):
        big = D(bs=bs, mb=(1152 + bs - 1) // bs, nb=4 * ((1152 + bs - 1) // bs))
        assert lib.rkv_paged_workspace_size(ctypes.byref(big), 1152, 8, 2) == flat
        assert lib.rkv_paged_workspace_size(ctypes.byref(big), 1152, 8, 63) == flat
        # beta past the tensor-core Gram's cap and fp32 pools take the copy
        assert lib.rkv_paged_workspace_size(ctypes.byref(big), 1152, 8, 64) == flat + copy
        big32 = D(bs=bs, mb=(1152 + bs - 1) // bs, nb=4 * ((1152 + bs - 1) // bs), dtype=1)
        flat32 = lib.rkv_workspace_size(ctypes.byref(_desc(P=32, n_cap=1152, dtype=1)), 1152, 8)
        assert lib.rkv_paged_workspace_size(ctypes.byref(big32), 1152, 8, 2) == \
            flat32 + 2 * copy
    assert lib.rkv_paged_workspace_size(ctypes.byref(D(bs=0)), 1152, 8, 2) == 0
    assert lib.rkv_paged_workspace_size(ctypes.byref(d), 1152, 8, -1) == 0
    fake = 1 << 20
    v = rkv._Variant(0, 1)
    call = lambda desc, n=1152, budget=1024, K=fake, V=fake + 2 ** 36, ws_bytes=1 << 40: \
        lib.rkv_paged_compress(ctypes.byref(desc), K, V, fake + 2 ** 37, fake + 2 ** 38, n,
                               budget, 8, 0.1, 2, 0.9, ctypes.byref(v), fake + 2 ** 39,
                               fake + 2 ** 40, fake + 2 ** 41, ws_bytes, None)
    assert call(D(bs=3)) == 1                      # block size not a power of two
    assert call(D(bs=2048)) == 1                   # block size too large
    assert call(D(mb=70)) == 1                     # n_cached beyond the table's rows
    assert call(D(d=80)) == 2                      # unsupported head_dim
    assert call(D(), K=fake + 8) == 1              # misaligned pool
    assert call(D(), V=fake) == 4                  # K and V pools are the same memory
    assert call(D(), ws_bytes=10) == 3             # workspace too small
    assert call(D(mb=2000), n=30000, budget=2048) == 2  # beyond the fused kernel's shared memory


def test_sentence_argument_errors(lib):
    """Invalid sentence descriptors are refused on the host."""
    from decode_kv_cache_02_gb300 import rkv
    fake = 1 << 20
    S_ = lambda **kw: rkv._Sentences(kw.get("reps", fake), fake + 2 ** 30, fake + 2 ** 31,
                                     fake + 2 ** 32, kw.get("S", 2), kw.get("heads", 8),
                                     kw.get("M", 40), kw.get("Dh", 4096), kw.get("ld", 1152),
                                     0.9)
    for kw in ({"S": 0}, {"heads": 0}, {"M": 0}, {"M": 70000}, {"Dh": 4098}, {"Dh": 0},
               {"Dh": 20000}, {"reps": fake + 4}, {"reps": 0}):
        assert lib.rkv_sentence_penalty(ctypes.byref(S_(**kw)), None) == 1, kw
    d = _desc(P=16)
    v = rkv._Variant(0, 1, ctypes.pointer(S_(ld=1000)))  # seg rows shorter than n_cached
    rc = lib.rkv_compress_ex(ctypes.byref(d), fake, fake + 2 ** 30, fake + 2 ** 31, 1152, 1024,
                             8, 0.1, 2, 0.9, ctypes.byref(v), fake + 2 ** 32, fake + 2 ** 33,
                             fake + 2 ** 34, fake + 2 ** 35, 1 << 40, None)
    assert rc == 1
    assert lib.rkv_sentence_reps(fake, fake, 2, 10, 4098, 0, 8, fake, None) == 1
    assert lib.rkv_sentence_reps(fake, fake, 2, 10, 4096, 5, 8, fake, None) == 2


def test_schedule_argument_errors(lib):
    """Schedule checks: window, pool bounds, uniforms for a sampled pool,
    temperature."""
    from decode_kv_cache_02_gb300 import rkv
    d = _desc(P=16)
    fake = 1 << 20

    def call(L=128, K=896, T=1.0, u=fake + 2 ** 36, ld=1024, n_obs=8):
        sch = rkv._Schedule(L, K, T, ld, u)
        v = rkv._Variant(0, 1, None, ctypes.pointer(sch))
        return lib.rkv_compress_ex(ctypes.byref(d), fake, fake + 2 ** 30, fake + 2 ** 31, 1152,
                                   1024, n_obs, 0.1, 2, 0.9, ctypes.byref(v), fake + 2 ** 32,
                                   fake + 2 ** 33, fake + 2 ** 34, fake + 2 ** 35, 1 << 40, None)
    assert call(L=4) == 1            # window smaller than the observation tokens
    assert call(L=1100) == 1         # window larger than the budget
    assert call(K=800) == 1          # pool smaller than the number kept
    assert call(K=1100) == 1         # pool larger than the candidates
    assert call(K=900, u=None) == 1  # sampled pool without uniforms
    assert call(K=900, ld=100) == 1  # uniform rows shorter than the candidates
    assert call(T=0.0) == 1 and call(T=float("inf")) == 1


def test_overlap_setting(lib):
    """The step schedule setting checks its range and touches no device."""
    assert lib.rkv_set_overlap(1, 33, 104) == 1  # more groups than the schedule keeps events for
    assert lib.rkv_set_overlap(1, 1, 104) == 1   # one group is not a grouped schedule
    assert lib.rkv_set_overlap(2, 4, 4) == 1     # fewer SMs than one partition group
    assert lib.rkv_set_overlap(3, 8, 0) == 1     # no such mode
    assert lib.rkv_set_overlap(0, 8, 104) == 0   # one launch per stage
    assert lib.rkv_set_overlap(1, 8, 0) == 0     # the default


def test_trace_without_a_device(lib):
    """The launch trace switches on and off on the host; reading it needs the
    device and reports a CUDA error where there is none."""
    assert lib.rkv_trace_enable(1) == 0
    assert lib.rkv_trace_enable(0) == 0
    if not __import__("torch").cuda.is_available():
        assert lib.rkv_trace_read(None, None, None, None, 0) == -5  # -RKV_ERR_CUDA


def test_binding_rejects_cpu_tensors(lib):
    from decode_kv_cache_02_gb300 import rkv
    K = torch.zeros(1, 16, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        rkv.rkv_compress(K, K.clone(), torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16), 16, 12)


def test_product_path_does_not_touch_oracle():
    """The product package never imports the oracle."""
    pkg = os.path.join(ROOT, "decode_kv_cache_02_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                src = open(os.path.join(dirpath, fn)).read()
                assert "import oracle" not in src and "rkv_oracle" not in src, fn
