"""The sustained decode stream at its full size: batch 32 x 32 layers x 8 KV
heads = 8,192 problems, 16,384 generated tokens per sequence appended 128 at a
time, compressed in place back to the budget of 1,638 rows whenever the cache
holds more (R-KV review, yoonschallenge.tistory.com/1236, summary-table row
"Decoding-time compression scheme": a buffer of 128 new tokens, compression
every 128 tokens).  That is 116 compression rounds, each one rkv_compress call
over all 8,192 problems in place -- the configuration the benchmark times.

Every round, a seeded sample of 16 (layer, sequence, head) problems is checked
against the oracle run on that round's own input state: the scores of
rkv_score within 2e-3, the kept set of the in-place call within the tie band,
and the compacted rows byte for byte against the pre-round rows at the kept
indices.  The oracle runs on a host thread while the GPU carries on with the
next rounds."""
import concurrent.futures as cf

import numpy as np
import pytest
import torch

import oracle
from decode_kv_cache_02_gb300 import rkv, workloads as wl
from tests import parity

pytestmark = pytest.mark.gpu

SAMPLE = 16


def _check_round(sample, n, w, Ks, Qs, K_after, idx, gpu_scores):
    """The oracle's verdict on one round (run on a host thread)."""
    C = n - w.n_obs
    sc = oracle.score(Ks[:, :n], Qs, w.n_obs, w.lam, w.beta, w.tau)
    err = parity.score_errors(gpu_scores, sc, C)
    assert max(err.values()) <= parity.SCORE_ATOL, (n, err)
    parity.check_observation_scores(gpu_scores, C)
    parity.check_idx_valid(idx, n, w.budget, w.n_obs)
    bad, excused = parity.kept_mismatches(idx, sc, w.budget, w.n_obs)
    assert bad == 0, (n, bad, excused)
    # in place: the first `budget` rows now hold the pre-round rows at idx
    raw = Ks.view(torch.int16).numpy()
    exp = oracle.gather(raw, idx)
    np.testing.assert_array_equal(K_after.view(torch.int16).numpy()[:, : w.budget],
                                  exp[:, : w.budget])
    return excused


def test_stream_full_size_every_round(cuda_ok):
    w = wl.BY_NAME["stream"]
    P, dev = w.problems, "cuda"
    sample = torch.tensor(sorted(np.random.default_rng(5).choice(P, SAMPLE, replace=False)))
    sample_d = sample.to(dev)
    src = wl.StreamSource(w, device=dev)
    cap = w.budget + w.buffer
    K = torch.zeros(P, cap, w.head_dim, dtype=w.torch_dtype, device=dev)
    V = torch.zeros_like(K)
    idx = torch.empty((P, w.budget), dtype=torch.int32, device=dev)
    ws = rkv.alloc_workspace(K, w.gqa, cap, w.n_obs)
    n, rounds = 0, 0
    pending = []
    with cf.ThreadPoolExecutor(max_workers=1) as pool:
        while src.t < w.gen_tokens:
            kc, vc = src.next_chunk()
            K[:, n:n + w.buffer] = kc
            V[:, n:n + w.buffer] = vc
            n += w.buffer
            if n <= w.budget:
                continue
            Q = src.queries(K[:, n - 1])
            Ks = K[sample_d].cpu()
            Qs = Q[sample_d].cpu()
            I, R, Z = rkv.rkv_score(K[sample_d].contiguous(), Q[sample_d].contiguous(), n,
                                    w.n_obs, w.lam, w.beta, w.tau)
            rkv.rkv_compress(K, V, Q, n, w.budget, w.n_obs, w.lam, w.beta, w.tau, out_K=K,
                             out_V=V, out_idx=idx, workspace=ws)
            gpu = {"I": I.cpu(), "R": R.cpu(), "Z": Z.cpu()}
            pending.append(pool.submit(_check_round, sample, n, w, Ks, Qs, K[sample_d].cpu(),
                                       idx[sample_d].cpu().numpy(), gpu))
            rounds += 1
            n = w.budget
        torch.cuda.synchronize()
        assert rkv.rkv_get_device_status(ws) == 0
        for f in pending:
            f.result()
    # 16,384 tokens, first compression when the cache first exceeds 1,638
    # rows (at 1,664), then every 128 tokens
    assert rounds == (w.gen_tokens - 1664) // w.buffer + 1 == 116
