"""GPU parity: librkv (through its C ABI) against the fp64 oracle on seeded
synthetic inputs of every workload shape, plus edge cases."""
import numpy as np
import pytest
import torch

import oracle
from decode_kv_cache_02_gb300 import rkv, workloads as wl
from tests import parity

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _run_scores(K, Q, w, n=None, **kw):
    n = w.n_cached if n is None else n
    I, R, Z = rkv.rkv_score(K, Q, n, w.n_obs, kw.get("lam", w.lam), kw.get("beta", w.beta),
                            kw.get("tau", w.tau))
    return {"I": I, "R": R, "Z": Z}


def _oracle_scores(K, Q, w, problems, n=None, **kw):
    n = w.n_cached if n is None else n
    return oracle.score(K[problems, :n].cpu(), Q[problems].cpu(), w.n_obs,
                        kw.get("lam", w.lam), kw.get("beta", w.beta), kw.get("tau", w.tau))


def _full_check(w, K, V, Q, problems, in_place=False):
    C, k = w.n_cached - w.n_obs, w.budget - w.n_obs
    gpu = _run_scores(K, Q, w)
    sc = _oracle_scores(K, Q, w, problems)
    sub = {kk: v[problems] for kk, v in gpu.items()}
    err = parity.score_errors(sub, sc, C)
    assert max(err.values()) <= parity.SCORE_ATOL, err
    parity.check_observation_scores(sub, C)
    if in_place:
        K0, V0 = K.clone(), V.clone()
        oK, oV, idx = rkv.rkv_compress(K, V, Q, w.n_cached, w.budget, w.n_obs, w.lam, w.beta,
                                       w.tau, out_K=K, out_V=V)
        src_K, src_V = K0, V0
    else:
        oK, oV, idx = rkv.rkv_compress(K, V, Q, w.n_cached, w.budget, w.n_obs, w.lam, w.beta,
                                       w.tau)
        src_K, src_V = K, V
    torch.cuda.synchronize()
    gi = idx.cpu().numpy()
    parity.check_idx_valid(gi, w.n_cached, w.budget, w.n_obs)
    bad, excused = parity.kept_mismatches(gi[problems], sc, w.budget, w.n_obs)
    assert bad == 0, f"{bad} kept-set mismatches outside the tie band ({excused} excused)"
    parity.check_gathered(oK, src_K, idx, w.budget, problems)
    parity.check_gathered(oV, src_V, idx, w.budget, problems)
    # every problem: gathered rows equal the source rows (device-side property)
    rows = torch.gather(src_K[:, : w.n_cached], 1,
                        idx.long()[:, :, None].expand(-1, -1, K.shape[2]))
    assert torch.equal(oK[:, : w.budget], rows)
    return err, excused


@pytest.mark.parametrize("in_place", [False, True])
def test_tiny_workload_full(cuda_ok, in_place):
    w = wl.BY_NAME["tiny"]
    K, V, Q = wl.make_inputs(w, device=DEV)
    _full_check(w, K, V, Q, list(range(w.problems)), in_place=in_place)


@pytest.mark.parametrize("in_place", [False, True])
def test_llama_layer_full(cuda_ok, in_place):
    w = wl.BY_NAME["llama8b_layer"]
    K, V, Q = wl.make_inputs(w, device=DEV)
    _full_check(w, K, V, Q, list(range(w.problems)), in_place=in_place)


def test_llama_full_step_sampled(cuda_ok):
    """The 32-layer x 64-sequence x 8-head step in the bench's launch
    configuration (all 16,384 problems in one call), oracle on 256 sampled
    problems, the copy checked on every problem."""
    w = wl.BY_NAME["llama8b_full"]
    K, V, Q = wl.make_inputs(w, device=DEV)
    problems = sorted(np.random.default_rng(0).choice(w.problems, 256, replace=False).tolist())
    _full_check(w, K, V, Q, problems)


def test_qwen_large_budget_sampled(cuda_ok):
    """The 48-layer x 16-sequence x 8-head Qwen-14B step (N = 4224 -> 4096,
    G = 5) in one call, oracle on 256 sampled problems."""
    w = wl.BY_NAME["qwen14b"]
    K, V, Q = wl.make_inputs(w, device=DEV)
    problems = sorted(np.random.default_rng(1).choice(w.problems, 256, replace=False).tolist())
    _full_check(w, K, V, Q, problems)


def test_ragged_and_capacity(cuda_ok):
    """N not a multiple of any tile, spare capacity rows (NaN-filled, never
    read), G = 5, head_dim 64 and 128, bf16 and fp32."""
    for d, dt, G, N, budget in ((128, "bf16", 5, 301, 200), (64, "bf16", 3, 129, 100),
                                (64, "fp32", 2, 77, 40), (128, "fp32", 4, 190, 131)):
        w = wl.BY_NAME["llama8b_layer"].scaled(head_dim=d, dtype=dt, gqa=G, n_cached=N,
                                               budget=budget, layers=1, batch=1, kv_heads=3)
        K, V, Q = wl.make_inputs(w, device=DEV, n_cap=N + 37)
        _full_check(w, K, V, Q, list(range(w.problems)))


@pytest.mark.parametrize("n_cached,budget", [(13000, 12000), (14000, 13000)])
def test_long_context_selection_paths(cuda_ok, n_cached, budget):
    """Long contexts on both sides of the fused select + gather's shared-memory
    limit (scores, sort keys and kept indices of one problem): the first size
    runs the fused kernel with ~150 KB of shared memory, the second the
    separate select and gather kernels (and, with a scoring variant, the
    separate variant kernel)."""
    w = wl.BY_NAME["llama8b_layer"].scaled(head_dim=64, n_cached=n_cached, budget=budget,
                                           layers=1, batch=1, kv_heads=1)
    K, V, Q = wl.make_inputs(w, device=DEV)
    _full_check(w, K, V, Q, [0])
    _variant_check(w, K, V, Q, [0], True, 5)


@pytest.mark.parametrize("n_cached,budget", [(1152, 1024), (14000, 13000), (900, 1024)])
def test_outputs_of_budget_rows(cuda_ok, n_cached, budget):
    """Outputs of just `budget` rows per problem (out_capacity = budget) get
    the same kept rows, bit for bit, as outputs of the inputs' capacity: the
    fused select + gather, the separate select and gather (long rows), the
    copy when nothing is evicted, rkv_compress_noalloc and rkv_gather."""
    w = wl.BY_NAME["llama8b_layer"].scaled(n_cached=n_cached, budget=budget, layers=1,
                                           batch=1, kv_heads=3 if n_cached > 2000 else 16)
    K, V, Q = wl.make_inputs(w, device=DEV, n_cap=max(n_cached, budget) + 40)
    args = (w.n_cached, w.budget, w.n_obs, w.lam, w.beta, w.tau)
    oK, oV, idx = rkv.rkv_compress(K, V, Q, *args)
    P, d = K.shape[0], K.shape[2]
    cK = torch.full((P, w.budget, d), 7.0, dtype=K.dtype, device=DEV)
    cV = torch.full_like(cK, 7.0)
    _, _, idx2 = rkv.rkv_compress(K, V, Q, *args, out_K=cK, out_V=cV)
    torch.cuda.synchronize()
    assert torch.equal(idx, idx2)
    kept = min(w.n_cached, w.budget)
    assert torch.equal(cK[:, :kept], oK[:, :kept]) and torch.equal(cV[:, :kept], oV[:, :kept])
    if kept < w.budget:  # rows past the kept ones are not touched
        assert bool((cK[:, kept:] == 7.0).all()) and bool((cV[:, kept:] == 7.0).all())
    if w.n_cached > w.budget:
        nK = torch.empty_like(cK)
        nV = torch.empty_like(cV)
        rkv.rkv_compress_noalloc(K, V, Q, *args, out_K=nK, out_V=nV)
        g = rkv.rkv_gather(V, idx, w.budget, dst=torch.empty_like(cV))
        torch.cuda.synchronize()
        assert torch.equal(nK, cK) and torch.equal(nV, cV)
        assert torch.equal(g, cV)
        # a scoring variant (Z formed in the select + gather, or the separate
        # variant kernel for long rows) writes the same rows either way
        vK, vV, vi = rkv.rkv_compress_ex(K, V, Q, *args, redundancy_softmax=True, pool_window=5)
        bK = torch.empty_like(cK)
        bV = torch.empty_like(cV)
        _, _, vi2 = rkv.rkv_compress_ex(K, V, Q, *args, redundancy_softmax=True, pool_window=5,
                                        out_K=bK, out_V=bV)
        torch.cuda.synchronize()
        assert torch.equal(vi, vi2)
        assert torch.equal(bK, vK[:, :w.budget]) and torch.equal(bV, vV[:, :w.budget])


def _variant_check(w, K, V, Q, problems, softmax, window, in_place=False):
    """Variant scores through rkv_score_ex and the kept set and rows through
    rkv_compress_ex, against the oracle's base scores plus its variant."""
    C = w.n_cached - w.n_obs
    I, R, Z = rkv.rkv_score_ex(K, Q, w.n_cached, w.n_obs, w.lam, w.beta, w.tau,
                               redundancy_softmax=softmax, pool_window=window)
    base = _oracle_scores(K, Q, w, problems)
    sc = oracle.variant(base, w.n_obs, w.lam, softmax, window)
    sub = {"I": I[problems], "R": R[problems], "Z": Z[problems]}
    err = parity.scaled_score_errors(sub, sc, C)
    assert max(err.values()) <= parity.SCORE_ATOL, err
    parity.check_observation_scores(sub, C)
    src_K, src_V = (K.clone(), V.clone()) if in_place else (K, V)
    oK, oV, idx = rkv.rkv_compress_ex(K, V, Q, w.n_cached, w.budget, w.n_obs, w.lam, w.beta,
                                      w.tau, redundancy_softmax=softmax, pool_window=window,
                                      **({"out_K": K, "out_V": V} if in_place else {}))
    torch.cuda.synchronize()
    gi = idx.cpu().numpy()
    parity.check_idx_valid(gi, w.n_cached, w.budget, w.n_obs)
    # the step forms Z inside its selection kernel with the same arithmetic as
    # rkv_score_ex: the same Z bit for bit, so the same kept set everywhere
    np.testing.assert_array_equal(gi, rkv.rkv_select(Z, w.n_obs, w.budget).cpu().numpy())
    bad, excused = parity.kept_mismatches(gi[problems], sc, w.budget, w.n_obs,
                                          band=parity.scaled_band(sc, C))
    assert bad == 0, f"{bad} kept-set mismatches outside the tie band ({excused} excused)"
    parity.check_gathered(oK, src_K, idx, w.budget, problems)
    parity.check_gathered(oV, src_V, idx, w.budget, problems)
    return err, excused


@pytest.mark.parametrize("softmax,window", [(True, 1), (False, 7), (True, 7), (True, 255)])
def test_scoring_variants_llama_layer(cuda_ok, softmax, window):
    """Redundancy softmax and importance pooling window on Llama-shaped
    problems (tensor-core scoring path)."""
    w = wl.BY_NAME["llama8b_layer"].scaled(kv_heads=2)
    K, V, Q = wl.make_inputs(w, device=DEV)
    _variant_check(w, K, V, Q, list(range(w.problems)), softmax, window)


def test_scoring_variants_other_paths(cuda_ok):
    """The variants after the CUDA-core scoring (fp32; beta above the
    tensor-core path's cap), after the two-pass importance (long rows), and
    with in-place compaction."""
    tiny = wl.BY_NAME["tiny"]
    K, V, Q = wl.make_inputs(tiny, device=DEV)
    _variant_check(tiny, K, V, Q, list(range(tiny.problems)), True, 5)
    w = wl.BY_NAME["llama8b_layer"].scaled(n_cached=640, budget=512, kv_heads=1, beta=64)
    K, V, Q = wl.make_inputs(w, device=DEV)
    _variant_check(w, K, V, Q, list(range(w.problems)), True, 3, in_place=True)
    q = wl.BY_NAME["qwen14b"].scaled(layers=1, batch=1, kv_heads=2)
    K, V, Q = wl.make_inputs(q, device=DEV)
    _variant_check(q, K, V, Q, [0, 1], True, 9)


def test_parameter_sweep(cuda_ok):
    """lambda, beta and tau swept one at a time around the page's setting
    (beta 64 takes the CUDA-core Gram, tau <= 0 the all-pairs branch), with
    and without the variants."""
    base = wl.BY_NAME["llama8b_layer"].scaled(n_cached=640, budget=512, kv_heads=2)
    K, V, Q = wl.make_inputs(base, device=DEV)
    for lam in (0.0, 0.05, 0.3, 0.7, 1.0):
        _full_check(base.scaled(lam=lam), K, V, Q, [0, 1])
    for beta in (0, 1, 3, 8, 63, 64):
        _full_check(base.scaled(beta=beta), K, V, Q, [0, 1])
    for tau in (-0.2, 0.0, 0.3, 0.6, 0.95):
        _full_check(base.scaled(tau=tau), K, V, Q, [0, 1])
    for lam, beta, tau in ((0.0, 2, 0.9), (0.5, 8, 0.6), (1.0, 1, 0.3)):
        _variant_check(base.scaled(lam=lam, beta=beta, tau=tau), K, V, Q, [0, 1], True, 7)


def test_parameter_variants(cuda_ok):
    """lambda in {0, 1}, beta in {0, 1, 5}, tau in {0.5, 0.99}."""
    base = wl.BY_NAME["llama8b_layer"].scaled(n_cached=640, budget=512, kv_heads=2)
    K, V, Q = wl.make_inputs(base, device=DEV)
    for lam, beta, tau in ((0.0, 2, 0.9), (1.0, 2, 0.9), (0.1, 0, 0.9), (0.1, 1, 0.5),
                           (0.1, 5, 0.99)):
        w = base.scaled(lam=lam, beta=beta, tau=tau)
        _full_check(w, K, V, Q, [0, 1])


def test_identity_when_not_over_budget(cuda_ok):
    w = wl.BY_NAME["llama8b_layer"].scaled(kv_heads=2)
    K, V, Q = wl.make_inputs(w, device=DEV)
    for n in (w.budget, 500):
        oK, oV, idx = rkv.rkv_compress(K, V, Q, n, w.budget, w.n_obs)
        torch.cuda.synchronize()
        gi = idx.cpu().numpy()
        assert np.all(gi[:, :n] == np.arange(n)) and np.all(gi[:, n:] == -1)
        assert torch.equal(oK[:, :n], K[:, :n]) and torch.equal(oV[:, :n], V[:, :n])


def test_select_bit_exact_with_ties(cuda_ok):
    """Selection alone on fp32 scores with many exact ties: bit-exact against
    the oracle's selection of the same values."""
    for P, n, n_obs, budget, levels in ((64, 1152, 8, 1024, 7), (16, 4224, 8, 4096, 0),
                                        (33, 97, 8, 64, 3), (8, 300, 1, 2, 0), (5, 50, 8, 8, 0)):
        Z = wl.random_scores(P, n, device=DEV, seed=n, tie_levels=levels)
        idx = rkv.rkv_select(Z, n_obs, budget)
        torch.cuda.synchronize()
        ref = oracle.select(Z.cpu().double().numpy(), n_obs, budget)
        np.testing.assert_array_equal(idx.cpu().numpy(), ref)


def test_gather_bit_exact(cuda_ok):
    for dt in (torch.bfloat16, torch.float32):
        P, n_cap, d, budget = 7, 700, 128, 512
        g = torch.Generator(device=DEV).manual_seed(3)
        src = torch.randn(P, n_cap, d, generator=g, device=DEV).to(dt)
        idx = wl.random_indices(P, 650, budget, device=DEV)
        out = rkv.rkv_gather(src, idx, budget)
        torch.cuda.synchronize()
        parity.check_gathered(out, src, idx, budget)
        inplace = src.clone()
        rkv.rkv_gather(inplace, idx, budget, dst=inplace)
        torch.cuda.synchronize()
        parity.check_gathered(inplace, src, idx, budget)
        assert torch.equal(inplace[:, budget:], src[:, budget:])  # rows past budget untouched


def test_device_status_clean(cuda_ok):
    w = wl.BY_NAME["tiny"]
    K, V, Q = wl.make_inputs(w, device=DEV)
    ws = rkv.alloc_workspace(K, w.gqa, w.n_cached, w.n_obs)
    rkv.rkv_compress(K, V, Q, w.n_cached, w.budget, w.n_obs, workspace=ws)
    assert rkv.rkv_get_device_status(ws) == 0


def test_bounded_wait_runs_out_and_is_reported(cuda_ok):
    """A bounded wait that nothing completes ends with a recorded timeout
    (no hang, no trap); the status is read once and cleared, and the context
    still runs a compression round correctly afterwards."""
    w = wl.BY_NAME["tiny"]
    K, V, Q = wl.make_inputs(w, device=DEV)
    ws = rkv.alloc_workspace(K, w.gqa, w.n_cached, w.n_obs)
    rkv.rkv_selftest_wait_timeout(ws)
    assert rkv.rkv_get_device_status(ws) == rkv.RKV_ERR_DEVICE
    assert rkv.rkv_get_device_status(ws) == 0
    _full_check(w, K, V, Q, list(range(w.problems)))


def test_stream_rounds(cuda_ok):
    """Sustained decode stream (batch x layers x heads scaled down to 64
    problems, 40 rounds): the cache is compacted in place each round, and each
    round's scores and kept set are checked against the oracle run on that
    round's own input state."""
    w = wl.BY_NAME["stream"]
    P, rounds = 64, 40
    src = wl.StreamSource(w, device=DEV, problems=P)
    cap = w.budget + w.buffer
    K = torch.zeros(P, cap, w.head_dim, dtype=w.torch_dtype, device=DEV)
    V = torch.zeros_like(K)
    n = 0
    checked = 0
    for r in range(rounds):
        kc, vc = src.next_chunk()
        K[:, n:n + w.buffer] = kc
        V[:, n:n + w.buffer] = vc
        n += w.buffer
        if n <= w.budget:
            continue
        Q = src.queries(K[:, n - 1])
        ww = w.scaled(n_cached=n)
        if r % 4 == 0:
            _full_check(ww, K.clone(), V.clone(), Q, list(range(0, P, 8)))
            checked += 1
        rkv.rkv_compress(K, V, Q, n, w.budget, w.n_obs, w.lam, w.beta, w.tau, out_K=K, out_V=V)
        n = w.budget
    torch.cuda.synchronize()
    assert checked >= 5
