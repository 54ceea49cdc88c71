"""rkv_compress_noalloc, the entry point for callers that may not allocate
device memory while they run (an inference engine's plugin or custom op whose
framework owns all device memory, a process whose memory is reserved up front
for the KV cache).  It must give the same kept tokens and rows as
rkv_compress, call after call, while using only the library's static scratch,
allocate nothing, and report device-side errors through
rkv_noalloc_device_status.

This file is named so that pytest collects it last."""
import numpy as np
import pytest
import torch

from decode_kv_cache_02_gb300 import rkv, workloads as wl
from tests import parity

pytestmark = pytest.mark.gpu


def _noalloc(K, V, Q, w, out_K, out_V, out_idx):
    rkv.rkv_compress_noalloc(K, V, Q, w.n_cached, w.budget, w.n_obs, w.lam, w.beta, w.tau,
                             out_K=out_K, out_V=out_V, out_idx=out_idx)


def test_noalloc_matches_workspace_entry_point(cuda_ok):
    w = wl.BY_NAME["llama8b_layer"]
    K, V, Q = wl.make_inputs(w, device="cuda")
    ref_K, ref_V, ref_idx = rkv.rkv_compress(K, V, Q, w.n_cached, w.budget, w.n_obs, w.lam,
                                             w.beta, w.tau)
    _, _, Z = rkv.rkv_score(K, Q, w.n_cached, w.n_obs, w.lam, w.beta, w.tau)
    out_K, out_V = torch.empty_like(K), torch.empty_like(V)
    out_idx = torch.empty_like(ref_idx)
    C, k = w.n_cached - w.n_obs, w.budget - w.n_obs
    z = Z.double().cpu().numpy()
    for call in range(2):  # the scratch keeps the previous call's contents
        out_K.zero_()
        out_idx.fill_(-7)
        _noalloc(K, V, Q, w, out_K, out_V, out_idx)
        torch.cuda.synchronize()
        gi, ri = out_idx.cpu().numpy(), ref_idx.cpu().numpy()
        parity.check_idx_valid(gi, w.n_cached, w.budget, w.n_obs)
        for p in range(w.problems):
            zk = np.sort(z[p, :C])[::-1][k - 1]
            diff = set(gi[p, :k].tolist()) ^ set(ri[p, :k].tolist())
            assert all(abs(z[p, i] - zk) <= parity.KEPT_BAND for i in diff), (call, p, diff)
        rows = torch.gather(K, 1, out_idx.long()[:, :, None].expand(-1, -1, K.shape[2]))
        assert torch.equal(out_K[:, : w.budget], rows)
        rows = torch.gather(V, 1, out_idx.long()[:, :, None].expand(-1, -1, V.shape[2]))
        assert torch.equal(out_V[:, : w.budget], rows)
        assert rkv.rkv_noalloc_device_status() == rkv.RKV_OK


def test_noalloc_allocates_nothing(cuda_ok):
    # with the outputs preallocated and one call made (which may load the
    # library's device code), a further call changes neither torch's
    # allocator nor the device's free memory
    w = wl.BY_NAME["llama8b_layer"]
    K, V, Q = wl.make_inputs(w, device="cuda")
    out_K, out_V = torch.empty_like(K), torch.empty_like(V)
    out_idx = torch.empty((w.problems, w.budget), dtype=torch.int32, device="cuda")
    _noalloc(K, V, Q, w, out_K, out_V, out_idx)
    torch.cuda.synchronize()
    torch_before = torch.cuda.memory_allocated()
    free_before = torch.cuda.mem_get_info()[0]
    _noalloc(K, V, Q, w, out_K, out_V, out_idx)
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() == torch_before
    assert torch.cuda.mem_get_info()[0] == free_before


def test_noalloc_reports_device_errors(cuda_ok):
    # a bounded wait that runs out records its error in the static scratch;
    # the accessor reports it once, clears it, and the next call still works
    assert rkv.rkv_noalloc_device_status() == rkv.RKV_OK
    rkv.rkv_noalloc_selftest_wait_timeout()
    assert rkv.rkv_noalloc_device_status() == rkv.RKV_ERR_DEVICE
    assert rkv.rkv_noalloc_device_status() == rkv.RKV_OK
    w = wl.BY_NAME["llama8b_layer"]
    K, V, Q = wl.make_inputs(w, device="cuda", problems=2)
    ref_K, _, ref_idx = rkv.rkv_compress(K, V, Q, w.n_cached, w.budget, w.n_obs, w.lam,
                                         w.beta, w.tau)
    out_K, out_V = torch.empty_like(K), torch.empty_like(V)
    out_idx = torch.empty_like(ref_idx)
    _noalloc(K, V, Q, w, out_K, out_V, out_idx)
    assert rkv.rkv_noalloc_device_status() == rkv.RKV_OK
    assert torch.equal(out_idx, ref_idx)
    assert torch.equal(out_K[:, : w.budget], ref_K[:, : w.budget])


def test_noalloc_rejects_oversize_request(cuda_ok):
    # 600 problems x 4224 tokens needs ~40 MB of scratch, more than the array
    K = torch.zeros(600, 4224, 64, dtype=torch.bfloat16, device="cuda")
    Q = torch.zeros(600, 1, 8, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(rkv.RkvError) as e:
        rkv.rkv_compress_noalloc(K, K, Q, 4224, 4096, 8, out_K=K, out_V=K)
    assert e.value.code == rkv.RKV_ERR_TOO_LARGE
