"""GPU parity of the paged round (rkv_paged_compress) against the oracle's
paged round: kept sets, the pools after the in-place compaction (byte for
byte, including every row that must stay untouched), the block table and the
freed block ids."""
import numpy as np
import pytest
import torch

import oracle
from decode_kv_cache_02_gb300 import rkv, workloads as wl
from tests import parity

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _raw(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu()
    return (t.view(torch.int16) if t.dtype == torch.bfloat16 else t).numpy()


def _make_paged(w, bs, extra=5, seed=0, tail_garbage=True):
    """The workload's logical K, V, Q scattered into pools through a shuffled
    block table.  Rows past N in the last block hold large values, unused
    blocks a sentinel, and the table's entries past the blocks in use ids
    that do not exist (none of these may be read)."""
    K, V, Q = wl.make_inputs(w, device=DEV)
    S, H = w.layers * w.batch, w.kv_heads
    N, d = w.n_cached, w.head_dim
    nb = -(-N // bs)
    num_blocks = S * nb + extra
    g = torch.Generator().manual_seed(seed)
    perm = torch.randperm(num_blocks, generator=g)
    mb = nb + 2
    table = torch.full((S, mb), 1 << 30, dtype=torch.int32)
    table[:, :nb] = perm[:S * nb].reshape(S, nb).to(torch.int32)
    K_pool = torch.full((num_blocks, H, bs, d), -7.5, dtype=K.dtype, device=DEV)
    V_pool = torch.full_like(K_pool, 3.25)
    Kl = K[:, :N].reshape(S, H, N, d)
    Vl = V[:, :N].reshape(S, H, N, d)
    pad = nb * bs - N
    if pad:
        fill = 1e4 if tail_garbage else 0.0
        Kl = torch.cat([Kl, torch.full((S, H, pad, d), fill, dtype=K.dtype, device=DEV)], 2)
        Vl = torch.cat([Vl, torch.full((S, H, pad, d), fill, dtype=K.dtype, device=DEV)], 2)
    blocks = table[:, :nb].long().to(DEV)
    K_pool[blocks] = Kl.reshape(S, H, nb, bs, d).permute(0, 2, 1, 3, 4)
    V_pool[blocks] = Vl.reshape(S, H, nb, bs, d).permute(0, 2, 1, 3, 4)
    return K_pool, V_pool, Q, table.to(DEV)


def _paged_check(w, bs, problems=None, softmax=False, window=1, **kw):
    K_pool, V_pool, Q, table = _make_paged(w, bs, **kw)
    K0, V0, T0 = _raw(K_pool), _raw(V_pool), table.cpu().numpy()
    ws_bytes = rkv.rkv_paged_workspace_size(K_pool, table, w.gqa, w.n_cached, w.n_obs,
                                           w.beta)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=DEV)
    idx, freed = rkv.rkv_paged_compress(K_pool, V_pool, Q, table, w.n_cached, w.budget, w.n_obs,
                                        w.lam, w.beta, w.tau, redundancy_softmax=softmax,
                                        pool_window=window, workspace=ws)
    assert rkv.rkv_get_device_status(ws) == 0
    gi = idx.cpu().numpy()
    P = gi.shape[0]
    problems = list(range(P)) if problems is None else problems
    if w.n_cached <= w.budget:
        assert np.all(gi[:, :w.n_cached] == np.arange(w.n_cached))
        np.testing.assert_array_equal(_raw(K_pool), K0)
        np.testing.assert_array_equal(table.cpu().numpy(), T0)
        return
    parity.check_idx_valid(gi, w.n_cached, w.budget, w.n_obs)
    exp = oracle.paged_compress(K0, V0, Q.cpu(), T0, w.n_cached, w.budget, w.n_obs, w.lam,
                                w.beta, w.tau, idx_used=gi, redundancy_softmax=softmax,
                                pool_window=window)
    sc = exp["scores"]
    sub = {k: sc[k][problems] for k in ("Z", "border")}
    band = parity.scaled_band(sub, w.n_cached - w.n_obs) if softmax else parity.KEPT_BAND
    bad, excused = parity.kept_mismatches(gi[problems], sub, w.budget, w.n_obs, band=band)
    assert bad == 0, f"{bad} kept-set mismatches outside the tie band ({excused} excused)"
    np.testing.assert_array_equal(_raw(K_pool), exp["K_pool"])
    np.testing.assert_array_equal(_raw(V_pool), exp["V_pool"])
    np.testing.assert_array_equal(table.cpu().numpy(), exp["table"])
    np.testing.assert_array_equal(freed.cpu().numpy(), exp["freed"])
    return excused


def test_paged_llama_shapes_block16():
    """Llama-shaped problems (d = 128, G = 4, bf16), ragged N, 16-row blocks."""
    w = wl.BY_NAME["llama8b_layer"].scaled(n_cached=301, budget=200, layers=1, batch=3,
                                           kv_heads=2)
    _paged_check(w, 16)


def test_paged_full_row_block16():
    """A whole Llama row (N = 1152 -> 1024) for 2 sequences x 8 heads: eight
    16-row blocks freed per sequence."""
    w = wl.BY_NAME["llama8b_layer"].scaled(layers=1, batch=2, kv_heads=8)
    _paged_check(w, 16, problems=[0, 5, 9, 15])


@pytest.mark.parametrize("bs", [1, 64, 128, 1024])
def test_paged_block_sizes(bs):
    """One row per block up to one block per sequence (nothing freed)."""
    w = wl.BY_NAME["llama8b_layer"].scaled(n_cached=301, budget=200, layers=1, batch=2,
                                           kv_heads=2, head_dim=64)
    _paged_check(w, bs)


def test_paged_long_rows_block256():
    """Rows past 2048 (the long-row Gram) read in place from 256-row blocks,
    the last one partly filled (N = 2500: 196 of its rows before N; the rest
    hold large values that no stage may read)."""
    w = wl.BY_NAME["llama8b_layer"].scaled(n_cached=2500, budget=2200, layers=1, batch=2,
                                           kv_heads=2)
    _paged_check(w, 256)


def test_paged_fp32_cuda_core_path():
    """fp32 keys take the CUDA-core importance and Gram on the contiguous copy."""
    w = wl.BY_NAME["tiny"].scaled(batch=2)
    _paged_check(w, 32)


def test_paged_with_variant():
    w = wl.BY_NAME["llama8b_layer"].scaled(n_cached=640, budget=512, layers=1, batch=2,
                                           kv_heads=2)
    _paged_check(w, 64, softmax=True, window=5)


def test_paged_identity_when_not_over_budget():
    w = wl.BY_NAME["llama8b_layer"].scaled(n_cached=1000, budget=1024, layers=1, batch=2,
                                           kv_heads=2)
    _paged_check(w, 16)


@pytest.mark.parametrize("bs,d,n,budget,blk", [(16, 64, 301, 200, 3), (128, 128, 600, 300, 3)])
def test_paged_bad_block_id_is_reported(bs, d, n, budget, blk):
    """A table entry naming no block is caught by the kernels' own checks:
    its rows are skipped and the device status reports it.  Blocks of 128
    rows take the path whose importance kernel reads the pool in place with
    the key statistics folded in (no separate statistics pass); the id is in
    a block past the budget, which only the scoring reads."""
    w = wl.BY_NAME["llama8b_layer"].scaled(n_cached=n, budget=budget, layers=1, batch=2,
                                           kv_heads=2, head_dim=d)
    K_pool, V_pool, Q, table = _make_paged(w, bs)
    table[1, blk] = K_pool.shape[0] + 11
    ws_bytes = rkv.rkv_paged_workspace_size(K_pool, table, w.gqa, w.n_cached, w.n_obs,
                                           w.beta)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=DEV)
    rkv.rkv_paged_compress(K_pool, V_pool, Q, table, w.n_cached, w.budget, w.n_obs,
                           workspace=ws)
    assert rkv.rkv_get_device_status(ws) == rkv.RKV_ERR_DEVICE
    assert rkv.rkv_get_device_status(ws) == 0  # read and cleared


def test_paged_grouped_schedule_matches_one_launch():
    """The grouped step schedule on a pool read in place (blocks of 128 rows):
    groups of whole sequences scored on one SM partition while the previous
    group's kept rows move inside their blocks on the other.  Pools, table,
    kept indices and freed blocks must equal those of one launch per stage,
    and the oracle's on a few sequences."""
    w = wl.BY_NAME["llama8b_layer"].scaled(layers=1, batch=160, kv_heads=8)  # 1,280 problems
    results = []
    for mode in (rkv.RKV_SCHEDULE_ONE_LAUNCH, rkv.RKV_SCHEDULE_GROUPED):
        K_pool, V_pool, Q, table = _make_paged(w, 128)
        ws_bytes = rkv.rkv_paged_workspace_size(K_pool, table, w.gqa, w.n_cached, w.n_obs,
                                               w.beta)
        ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=DEV)
        rkv.rkv_set_overlap(mode, 3, 104)
        try:
            rkv.rkv_timing_read(reset=True)
            rkv.rkv_timing_enable(True)
            idx, freed = rkv.rkv_paged_compress(K_pool, V_pool, Q, table, w.n_cached, w.budget,
                                                w.n_obs, w.lam, w.beta, w.tau, workspace=ws)
            rkv.rkv_timing_enable(False)
            torch.cuda.synchronize()
            launches = rkv.rkv_timing_read(reset=True)
        finally:
            rkv.rkv_set_overlap(*rkv.DEFAULT_OVERLAP)
        assert rkv.rkv_get_device_status(ws) == 0
        if mode == rkv.RKV_SCHEDULE_GROUPED and launches["gram_tc"][1] == 1:
            pytest.skip("the driver offers no SM partitions: one launch per stage ran")
        results.append((_raw(K_pool), _raw(V_pool), table.cpu().numpy(), idx.cpu().numpy(),
                        freed.cpu().numpy()))
    assert launches["gram_tc"][1] == launches["compact_paged"][1] == 3
    for a, b in zip(results[0], results[1]):
        np.testing.assert_array_equal(a, b)
