"""GPU parity of the ForesightKV-style schedule (ForesightKV summary page,
gist.science/ko/paper/2602.03203, section "Dynamic eviction process"): a
recent window kept like the observation tokens, and the kept candidates drawn
from a pool of the top-K by multinomial sampling without replacement (Gumbel
keys from the caller's uniforms), against the oracle on the same uniforms."""
import numpy as np
import pytest
import torch

import oracle
from decode_kv_cache_02_gb300 import rkv, workloads as wl
from tests import parity

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _uniforms(P, C, seed=5):
    g = torch.Generator(device=DEV).manual_seed(seed)
    return torch.rand((P, C), generator=g, device=DEV)


def _run(w, L, pool_extra, T=0.05, seed=5, softmax=False, window=1, in_place=False):
    K, V, Q = wl.make_inputs(w, device=DEV)
    P, N = K.shape[0], w.n_cached
    C, k = N - L, w.budget - L
    u = _uniforms(P, C, seed) if pool_extra > 0 else None
    sch = rkv.Schedule(L, k + pool_extra, T, u)
    src_K, src_V = (K.clone(), V.clone()) if in_place else (K, V)
    oK, oV, idx = rkv.rkv_compress_ex(K, V, Q, N, w.budget, w.n_obs, w.lam, w.beta, w.tau,
                                      redundancy_softmax=softmax, pool_window=window,
                                      schedule=sch,
                                      **({"out_K": K, "out_V": V} if in_place else {}))
    torch.cuda.synchronize()
    gi = idx.cpu().numpy()
    parity.check_idx_valid(gi, N, w.budget, L)
    ref = oracle.compress(src_K.cpu(), Q.cpu(), N, w.budget, w.n_obs, w.lam, w.beta, w.tau,
                          redundancy_softmax=softmax, pool_window=window, recent_window=L,
                          pool_size=k + pool_extra, temperature=T,
                          uniforms=u.cpu().numpy() if u is not None else None)
    sc = ref["scores"]
    if pool_extra > 0:
        bad, excused = parity.sampled_mismatches(gi, sc, sc["sampled"], w.budget, L, T)
    else:
        band = parity.scaled_band(sc, C) if softmax else parity.KEPT_BAND
        bad, excused = parity.kept_mismatches(gi, sc, w.budget, L, band=band)
    assert bad == 0, f"{bad} kept-set mismatches outside the tie band ({excused} excused)"
    parity.check_gathered(oK, src_K, idx, w.budget)
    parity.check_gathered(oV, src_V, idx, w.budget)
    return gi, u, (K, V, Q, sch)


def test_recent_window_top_k(cuda_ok):
    """ForesightKV's schedule on the Llama shape: N = B + L with L = 128, the
    128 newest kept, the rest compressed to B - L by the R-KV score."""
    w = wl.BY_NAME["llama8b_layer"].scaled(kv_heads=2)
    _run(w, 128, 0)


def test_sampled_selection(cuda_ok):
    """Top-K pool then multinomial sampling: parity with the oracle on the
    same uniforms; the same uniforms give the same rows, others do not."""
    w = wl.BY_NAME["llama8b_layer"].scaled(kv_heads=2)
    gi, u, (K, V, Q, sch) = _run(w, 128, 100)
    again = rkv.rkv_compress_ex(K, V, Q, w.n_cached, w.budget, w.n_obs, w.lam, w.beta, w.tau,
                                schedule=sch)[2].cpu().numpy()
    np.testing.assert_array_equal(again, gi)
    other = rkv.Schedule(128, sch.pool_size, sch.temperature,
                         _uniforms(u.shape[0], u.shape[1], seed=6))
    diff = rkv.rkv_compress_ex(K, V, Q, w.n_cached, w.budget, w.n_obs, w.lam, w.beta, w.tau,
                               schedule=other)[2].cpu().numpy()
    assert (diff != gi).any()


def test_sampled_with_variants_in_place(cuda_ok):
    w = wl.BY_NAME["llama8b_layer"].scaled(n_cached=640, budget=512, kv_heads=2)
    _run(w, 32, 100, T=0.02, softmax=False, window=5, in_place=True)


def test_sampled_fp32_and_small_window(cuda_ok):
    """fp32 (CUDA-core scoring), window = n_obs, pool = every candidate."""
    w = wl.BY_NAME["tiny"].scaled(batch=2)
    C, k = w.n_cached - w.n_obs, w.budget - w.n_obs
    _run(w, w.n_obs, C - k, T=0.1)


def test_scores_with_window(cuda_ok):
    """rkv_score_ex with a window: the window's rows are not candidates."""
    w = wl.BY_NAME["llama8b_layer"].scaled(n_cached=640, budget=512, kv_heads=1)
    K, V, Q = wl.make_inputs(w, device=DEV)
    I, R, Z = rkv.rkv_score_ex(K, Q, w.n_cached, w.n_obs, w.lam, w.beta, w.tau,
                               schedule=rkv.Schedule(64, 448))
    I0, R0, Z0 = rkv.rkv_score(K, Q, w.n_cached, w.n_obs, w.lam, w.beta, w.tau)
    C = w.n_cached - 64
    # the same terms; the variant kernel rounds lambda*I - (1-lambda)*R without
    # a fused multiply-add, the Gram's epilogue may contract it
    torch.testing.assert_close(Z[:, :C], Z0[:, :C], rtol=1e-6, atol=1e-7)
    assert torch.isinf(Z[:, C:]).all() and (R[:, C:] == 0).all()


def test_paged_sampled(cuda_ok):
    from tests.test_gpu_paged import _make_paged, _raw
    w = wl.BY_NAME["llama8b_layer"].scaled(n_cached=301, budget=200, layers=1, batch=3,
                                           kv_heads=2)
    L, extra, T = 32, 40, 0.05
    K_pool, V_pool, Q, table = _make_paged(w, 16)
    K0, V0, T0 = _raw(K_pool), _raw(V_pool), table.cpu().numpy()
    P, C, k = 6, w.n_cached - L, w.budget - L
    u = _uniforms(P, C)
    idx, freed = rkv.rkv_paged_compress(K_pool, V_pool, Q, table, w.n_cached, w.budget, w.n_obs,
                                        w.lam, w.beta, w.tau,
                                        schedule=rkv.Schedule(L, k + extra, T, u))
    gi = idx.cpu().numpy()
    exp = oracle.paged_compress(K0, V0, Q.cpu(), T0, w.n_cached, w.budget, w.n_obs, w.lam,
                                w.beta, w.tau, idx_used=gi, recent_window=L,
                                pool_size=k + extra, temperature=T, uniforms=u.cpu().numpy())
    sc = exp["scores"]
    bad, _ = parity.sampled_mismatches(gi, sc, sc["sampled"], w.budget, L, T)
    assert bad == 0
    np.testing.assert_array_equal(_raw(K_pool), exp["K_pool"])
    np.testing.assert_array_equal(_raw(V_pool), exp["V_pool"])
    np.testing.assert_array_equal(freed.cpu().numpy(), exp["freed"])
