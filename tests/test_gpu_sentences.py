"""GPU parity of the sentence-level penalty (SkipKV review,
yoonschallenge.tistory.com/1230, rows "Method 1", "Final eviction score" and
"Cache Range Monitoring") against the oracle: sentence representations,
penalties, the step's scores and kept set with the penalty, and the sentence
ids compacted with the kept rows."""
import numpy as np
import pytest
import torch

import oracle
from decode_kv_cache_02_gb300 import rkv, workloads as wl
from tests import parity

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _sentences(w, hidden_dim=256, seed=11):
    S = w.batch
    si = wl.make_sentences(S, w.kv_heads, w.layers, w.n_cached, hidden_dim, device=DEV,
                           seed=seed)
    reps = rkv.rkv_sentence_reps(si.hidden, si.token_seg, si.max_sentences)
    sent = rkv.Sentences(reps, si.count, si.seg_id.clone(), si.heads, wl.SENT_TAU)
    return si, sent


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_sentence_reps(cuda_ok, dtype):
    si = wl.make_sentences(3, 1, 1, 301, 136, device=DEV, dtype=dtype)
    reps = rkv.rkv_sentence_reps(si.hidden, si.token_seg, si.max_sentences + 2)
    ref = oracle.sentence_reps(si.hidden.cpu(), si.token_seg.cpu(), si.max_sentences + 2)
    np.testing.assert_allclose(reps.cpu().numpy(), ref, rtol=0, atol=1e-5)


def test_sentence_penalty(cuda_ok):
    w = wl.BY_NAME["llama8b_layer"].scaled(n_cached=1152, layers=1, batch=4, kv_heads=2)
    si, sent = _sentences(w, hidden_dim=wl.HIDDEN_LLAMA8B)
    pen = rkv.rkv_sentence_penalty(sent).cpu().numpy()
    ref, border = oracle.sentence_penalty(sent.reps.cpu(), si.count.cpu(), wl.SENT_TAU)
    ok = ~border
    np.testing.assert_allclose(pen[ok], ref[ok], rtol=0, atol=1e-5)
    assert np.count_nonzero(ref) > 0  # the inputs do contain redundant sentences


def _check(w, softmax=False, window=1, in_place=False, hidden_dim=256):
    si, sent = _sentences(w, hidden_dim)
    K, V, Q = wl.make_inputs(w, device=DEV)
    C = w.n_cached - w.n_obs
    seg0 = sent.seg_id.clone()
    I, R, Z = rkv.rkv_score_ex(K, Q, w.n_cached, w.n_obs, w.lam, w.beta, w.tau,
                               redundancy_softmax=softmax, pool_window=window, sentences=sent)
    pen, pborder = oracle.sentence_penalty(sent.reps.cpu(), si.count.cpu(), wl.SENT_TAU)
    rp = oracle.row_penalties(pen, si.count.cpu(), seg0.cpu(), si.heads, w.n_cached)
    problems = list(range(K.shape[0]))
    base = oracle.score(K[:, :w.n_cached].cpu(), Q.cpu(), w.n_obs, w.lam, w.beta, w.tau)
    sc = oracle.variant(base, w.n_obs, w.lam, softmax, window, row_penalty=rp)
    # rows of a sentence whose threshold decision is borderline join the tie band
    rb = oracle.row_penalties(pborder.astype(np.float64), si.count.cpu(), seg0.cpu(), si.heads,
                              w.n_cached) > 0
    sc["border"] = sc["border"] | rb
    sub = {"I": I, "R": R, "Z": Z}
    err = (parity.scaled_score_errors(sub, sc, C) if softmax
           else parity.score_errors(sub, sc, C))
    assert max(err.values()) <= parity.SCORE_ATOL, err
    src_K, src_V = (K.clone(), V.clone()) if in_place else (K, V)
    oK, oV, idx = rkv.rkv_compress_ex(K, V, Q, w.n_cached, w.budget, w.n_obs, w.lam, w.beta,
                                      w.tau, redundancy_softmax=softmax, pool_window=window,
                                      sentences=sent,
                                      **({"out_K": K, "out_V": V} if in_place else {}))
    torch.cuda.synchronize()
    gi = idx.cpu().numpy()
    parity.check_idx_valid(gi, w.n_cached, w.budget, w.n_obs)
    np.testing.assert_array_equal(gi, rkv.rkv_select(Z, w.n_obs, w.budget).cpu().numpy())
    band = parity.scaled_band(sc, C) if softmax else parity.KEPT_BAND
    bad, excused = parity.kept_mismatches(gi, sc, w.budget, w.n_obs, band=band)
    assert bad == 0, f"{bad} kept-set mismatches outside the tie band ({excused} excused)"
    parity.check_gathered(oK, src_K, idx, w.budget, problems)
    parity.check_gathered(oV, src_V, idx, w.budget, problems)
    # the sentence ids followed the kept rows; rows past the budget untouched
    s0 = seg0.cpu().numpy()
    s1 = sent.seg_id.cpu().numpy()
    np.testing.assert_array_equal(s1[:, :w.budget], np.take_along_axis(s0, gi, axis=1))
    np.testing.assert_array_equal(s1[:, w.budget:], s0[:, w.budget:])
    # the penalty does what the SkipKV review says: rows of redundant sentences go first
    pen_rows = rp[:, :C] > 0
    kept = np.zeros((gi.shape[0], C), dtype=bool)
    np.put_along_axis(kept, gi[:, :w.budget - w.n_obs], True, axis=1)
    assert kept[pen_rows].mean() < kept[~pen_rows].mean()
    return excused


def test_step_with_sentences(cuda_ok):
    w = wl.BY_NAME["llama8b_layer"].scaled(layers=2, batch=2, kv_heads=2)
    _check(w)


def test_step_with_sentences_and_variants(cuda_ok):
    w = wl.BY_NAME["llama8b_layer"].scaled(n_cached=640, budget=512, layers=1, batch=2,
                                           kv_heads=2)
    _check(w, softmax=True, window=5, in_place=True)


def test_step_with_sentences_fp32(cuda_ok):
    _check(wl.BY_NAME["tiny"].scaled(batch=2), hidden_dim=64)


def test_paged_step_with_sentences(cuda_ok):
    """The paged round compacts the sentence ids the same way."""
    from tests.test_gpu_paged import _make_paged, _raw
    w = wl.BY_NAME["llama8b_layer"].scaled(n_cached=301, budget=200, layers=1, batch=3,
                                           kv_heads=2)
    si, sent = _sentences(w)
    seg0 = sent.seg_id.clone()
    K_pool, V_pool, Q, table = _make_paged(w, 16)
    K0, V0, T0 = _raw(K_pool), _raw(V_pool), table.cpu().numpy()
    idx, freed = rkv.rkv_paged_compress(K_pool, V_pool, Q, table, w.n_cached, w.budget, w.n_obs,
                                        w.lam, w.beta, w.tau, sentences=sent)
    gi = idx.cpu().numpy()
    pen, pborder = oracle.sentence_penalty(sent.reps.cpu(), si.count.cpu(), wl.SENT_TAU)
    rp = oracle.row_penalties(pen, si.count.cpu(), seg0.cpu(), si.heads, w.n_cached)
    exp = oracle.paged_compress(K0, V0, Q.cpu(), T0, w.n_cached, w.budget, w.n_obs, w.lam,
                                w.beta, w.tau, idx_used=gi, row_penalty=rp)
    sc = exp["scores"]
    bad, _ = parity.kept_mismatches(gi, sc, w.budget, w.n_obs)
    assert bad == 0
    np.testing.assert_array_equal(_raw(K_pool), exp["K_pool"])
    np.testing.assert_array_equal(_raw(V_pool), exp["V_pool"])
    np.testing.assert_array_equal(freed.cpu().numpy(), exp["freed"])
    np.testing.assert_array_equal(sent.seg_id.cpu().numpy()[:, :w.budget],
                                  np.take_along_axis(seg0.cpu().numpy(), gi, axis=1))
