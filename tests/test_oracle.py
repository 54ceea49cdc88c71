"""Pins of the fp64 oracle against facts that do not come from the oracle.

Each test names the passage of the R-KV review page
(yoonschallenge.tistory.com/1236) it checks and the mistake it would catch.
The pages print no worked example (no score of any concrete input), so the
pins are closed forms, brute force over subsets, reductions to library
routines (numpy matmul, torch softmax / topk) and invariants.
"""
import itertools
import math

import numpy as np
import pytest
import torch

import oracle
from decode_kv_cache_02_gb300 import workloads as wl


def _basis(N, d):
    K = np.zeros((N, d))
    for i in range(N):
        K[i, i % d] = 1.0
    return K


# ---------------------------------------------------------------- cosine --

def test_cosine_equals_normalised_matmul():
    """Redundancy row: cosine similarity of key vectors.  numpy's matmul of
    row-normalised keys is an independent route (catches a missing norm, a
    transposed operand or a wrong index)."""
    rng = np.random.default_rng(0)
    K = rng.standard_normal((37, 19)) * rng.uniform(0.1, 5.0, size=(37, 1))
    Kn = K / np.linalg.norm(K, axis=1, keepdims=True)
    np.testing.assert_allclose(oracle.cosine(K), Kn @ Kn.T, rtol=0, atol=1e-13)


def test_cosine_zero_key_is_zero():
    K = np.zeros((4, 3))
    K[1] = [1.0, 2.0, 3.0]
    K[2] = [-1.0, 0.5, 0.0]
    S = oracle.cosine(K)
    assert np.all(S[0] == 0.0) and np.all(S[:, 0] == 0.0)


# ------------------------------------------------------------- attention --

@pytest.mark.parametrize("N,d,G,n_obs", [(23, 16, 3, 8), (9, 4, 1, 1), (40, 64, 5, 8)])
def test_attention_equals_torch_softmax(N, d, G, n_obs):
    """Importance row: softmax attention of the observation queries.  Each
    query row equals torch's fp64 softmax over its causal prefix of keys with
    scale 1/sqrt(d) (catches a wrong scale, mask offset or normaliser)."""
    g = torch.Generator().manual_seed(N * 100 + d)
    K = torch.randn(N, d, generator=g, dtype=torch.float64)
    Q = torch.randn(G, n_obs, d, generator=g, dtype=torch.float64) * 2.0
    p = oracle.attention(K.numpy(), Q.numpy())
    for h in range(G):
        for q in range(n_obs):
            last = N - n_obs + q
            ref = torch.softmax(Q[h, q] @ K[: last + 1].T / math.sqrt(d), dim=0)
            np.testing.assert_allclose(p[h, q, : last + 1], ref.numpy(), rtol=1e-12, atol=1e-15)
            assert np.all(p[h, q, last + 1:] == 0.0)


def test_importance_zero_queries_closed_form():
    """Q = 0: every observation query attends uniformly to its causal prefix,
    so I_i = (1/n_obs) * sum_q [i <= N-n_obs+q] / (N-n_obs+q+1) (catches a
    mean taken over the wrong axis or a shifted mask)."""
    N, d, G, n_obs = 30, 8, 4, 8
    rng = np.random.default_rng(1)
    K = rng.standard_normal((1, N, d))
    Q = np.zeros((1, G, n_obs, d))
    sc = oracle.score(K, Q, n_obs, 0.1, 2, 0.9)
    expect = np.zeros(N)
    for q in range(n_obs):
        last = N - n_obs + q
        expect[: last + 1] += 1.0 / (last + 1)
    expect /= n_obs
    np.testing.assert_allclose(sc["I"][0], expect, rtol=1e-13, atol=0)


def test_importance_gqa_max_pool():
    """Importance row: under GQA the heads sharing one KV head are max-pooled.
    With one head of queries set to zero (uniform attention) and the others
    copies of one query set, I is the elementwise max of the two single-head
    importances (catches a mean or sum over heads)."""
    N, d, n_obs = 25, 16, 8
    rng = np.random.default_rng(2)
    K = rng.standard_normal((1, N, d))
    Qa = rng.standard_normal((1, 1, n_obs, d)) * 3.0
    Qz = np.zeros((1, 1, n_obs, d))
    Ia = oracle.score(K, Qa, n_obs, 0.1, 2, 0.9)["I"][0]
    Iz = oracle.score(K, Qz, n_obs, 0.1, 2, 0.9)["I"][0]
    Q3 = np.concatenate([Qa, Qz, Qa], axis=1)
    I3 = oracle.score(K, Q3, n_obs, 0.1, 2, 0.9)["I"][0]
    np.testing.assert_allclose(I3, np.maximum(Ia, Iz), rtol=1e-14, atol=0)
    assert np.any(Ia > Iz) and np.any(Iz > Ia)


# ------------------------------------------------------------- redundancy --

def test_identical_keys_give_R_one():
    """Closed form: all keys identical -> every cosine is 1; each candidate
    has at least n_obs >= beta similar newer tokens, so none is protected and
    R = (N-1)/(N-1) = 1 exactly (catches self-similarity counted, a wrong
    denominator, or protection applied to every token)."""
    N, d = 50, 32
    rng = np.random.default_rng(3)
    k = rng.standard_normal(d)
    K = np.tile(k, (1, N, 1)) * rng.uniform(0.5, 2.0, size=(1, N, 1))  # scaled copies
    Q = rng.standard_normal((1, 4, 8, d))
    sc = oracle.score(K, Q, 8, 0.1, 2, 0.9)
    C = N - 8
    np.testing.assert_allclose(sc["R"][0, :C], 1.0, rtol=0, atol=1e-13)
    np.testing.assert_allclose(sc["sum"][0], N - 1, rtol=0, atol=1e-11)


def test_orthonormal_keys_give_R_zero():
    N, d = 20, 24
    K = _basis(N, d)[None]
    Q = np.random.default_rng(4).standard_normal((1, 2, 8, d))
    sc = oracle.score(K, Q, 8, 0.1, 2, 0.9)
    assert np.all(sc["R"][0] == 0.0) and np.all(sc["sum"][0] == 0.0)


def _triple_case(beta, tau=0.9, N=16):
    """Orthonormal keys (in N+1 dims) except positions a=2 < b=5 < c=9,
    which are scaled copies of one key: S is 1 inside the triple, 0 elsewhere."""
    K = np.zeros((N, N + 1))
    K[:, :N] = np.eye(N)
    K[5] = 2.5 * K[2]
    K[9] = 0.3 * K[2]
    Q = np.zeros((1, 1, 4, N + 1))
    return oracle.score(K[None], Q, 4, 0.0, beta, tau)


@pytest.mark.parametrize("beta,expect", [
    (0, (2, 2, 2)),   # nobody protected
    (1, (2, 2, 0)),   # only the newest copy (no similar token newer than it)
    (2, (2, 0, 0)),   # the two newest copies
    (3, (0, 0, 0)),   # all three
])
def test_recency_protection_triple(beta, expect):
    """Redundancy row: among similar tokens the beta most recent are
    protected.  A triple of copies at a < b < c with beta = 0..3 gives these
    closed forms (R in units of 1/(N-1)); catches 'older' counted instead of
    'newer', an off-by-one in the beta comparison, and a missing
    normalisation (the copies are scaled by 2.5 and 0.3)."""
    N = 16
    sc = _triple_case(beta)
    a, b, c = 2, 5, 9
    np.testing.assert_allclose(
        [sc["R"][0, a], sc["R"][0, b], sc["R"][0, c]],
        np.array(expect) / (N - 1), rtol=0, atol=1e-15)
    assert list(sc["newer"][0, [a, b, c]]) == [2, 1, 0]
    others = [i for i in range(N - 4) if i not in (a, b, c)]
    assert np.all(sc["R"][0, others] == 0.0)


def test_similarity_threshold_is_strict():
    """S exactly equal to tau is not 'similar' (reading of the threshold as a
    strict inequality): with tau = 1 the triple's cosines of exactly 1 protect
    nothing, with tau just below 1 they do."""
    N = 16
    strict = _triple_case(beta=1, tau=1.0)
    assert list(strict["newer"][0, [2, 5, 9]]) == [0, 0, 0]
    np.testing.assert_allclose(strict["R"][0, [2, 5, 9]], 2 / (N - 1), atol=1e-15)
    below = _triple_case(beta=1, tau=1.0 - 1e-9)
    assert list(below["newer"][0, [2, 5, 9]]) == [2, 1, 0]


def test_negative_similarity_lowers_R():
    """A key and its negation have cosine -1: redundancy is a signed mean, and
    -1 is never above tau (catches an absolute value)."""
    N = 12
    K = np.zeros((1, N, N))
    K[0, :, :] = np.eye(N)
    K[0, 6] = -K[0, 3]
    sc = oracle.score(K, np.zeros((1, 1, 4, N)), 4, 0.1, 2, 0.9)
    np.testing.assert_allclose(sc["R"][0, 3], -1 / (N - 1), atol=1e-15)
    np.testing.assert_allclose(sc["R"][0, 6], -1 / (N - 1), atol=1e-15)
    assert sc["newer"][0, 3] == 0


def test_combined_score_extremes():
    """Final selection criterion: Z rises with importance and falls with
    redundancy.  lambda = 1 gives Z = I, lambda = 0 gives Z = -R; the
    observation tokens carry +inf (always kept)."""
    P, N, d, n_obs = 3, 40, 16, 8
    rng = np.random.default_rng(5)
    K = rng.standard_normal((P, N, d))
    Q = rng.standard_normal((P, 2, n_obs, d))
    s1 = oracle.score(K, Q, n_obs, 1.0, 2, 0.5)
    s0 = oracle.score(K, Q, n_obs, 0.0, 2, 0.5)
    C = N - n_obs
    np.testing.assert_array_equal(s1["Z"][:, :C], s1["I"][:, :C])
    np.testing.assert_array_equal(s0["Z"][:, :C], -s0["R"][:, :C])
    assert np.all(np.isinf(s1["Z"][:, C:]))


# -------------------------------------------------------------- selection --

def _key_order_ok(Z, kept, C):
    """Every kept candidate beats every evicted one on (Z, index)."""
    ev = [i for i in range(C) if i not in kept]
    if not ev or not kept:
        return True
    worst_kept = min((Z[i], i) for i in kept)
    best_evicted = max((Z[i], i) for i in ev)
    return worst_kept > best_evicted


@pytest.mark.parametrize("seed", range(6))
def test_selection_brute_force(seed):
    """Top-k row (the best tokens that fit the budget are kept): for tiny problems,
    enumerate every k-subset of candidates; the oracle's kept set has the
    largest total score, and ties are broken toward larger indices."""
    rng = np.random.default_rng(100 + seed)
    N, d, n_obs, budget = 12, 4, 3, 8
    K = rng.standard_normal((1, N, d))
    Q = rng.standard_normal((1, 2, n_obs, d))
    sc = oracle.score(K, Q, n_obs, 0.1, 1, 0.6)
    Z = sc["Z"][0]
    if seed % 2:  # quantise to create exact ties
        Z = np.round(Z * 20) / 20
        Z[N - n_obs:] = np.inf
    idx = oracle.select(Z[None], n_obs, budget)[0]
    C, k = N - n_obs, budget - n_obs
    kept = [int(i) for i in idx[:k]]
    best = max(sum(Z[list(s)]) for s in itertools.combinations(range(C), k))
    assert abs(sum(Z[kept]) - best) < 1e-12
    assert _key_order_ok(Z, set(kept), C)
    assert list(idx[k:]) == list(range(C, N))
    assert all(idx[r] < idx[r + 1] for r in range(budget - 1))


def test_selection_all_ties_keeps_newest():
    """Equal scores everywhere: the tie rule keeps the most recent candidates."""
    Z = np.zeros((1, 20))
    Z[0, 15:] = np.inf
    idx = oracle.select(Z, 5, 9)[0]
    assert list(idx) == [11, 12, 13, 14, 15, 16, 17, 18, 19]


def test_lambda_one_is_attention_topk():
    """lambda = 1 reduces to attention-only eviction (the SnapKV-style
    baseline the page compares against): the kept candidates are torch.topk of
    the importance."""
    w = wl.WORKLOADS[0]
    K, V, Q = wl.make_inputs(w)
    sc = oracle.score(K, Q, w.n_obs, 1.0, w.beta, w.tau)
    idx = oracle.select(sc["Z"], w.n_obs, w.budget)
    C, k = w.n_cached - w.n_obs, w.budget - w.n_obs
    for p in range(w.problems):
        top = torch.topk(torch.from_numpy(sc["I"][p, :C]), k).indices
        assert set(top.tolist()) == set(idx[p, :k].tolist())


def test_lambda_zero_is_bottom_redundancy():
    w = wl.WORKLOADS[0]
    K, V, Q = wl.make_inputs(w)
    sc = oracle.score(K, Q, w.n_obs, 0.0, w.beta, w.tau)
    idx = oracle.select(sc["Z"], w.n_obs, w.budget)
    C, k = w.n_cached - w.n_obs, w.budget - w.n_obs
    for p in range(w.problems):
        low = np.argsort(sc["R"][p, :C], kind="stable")[:k]
        assert set(low.tolist()) == set(idx[p, :k].tolist())


@pytest.mark.parametrize("copies,beta", [(2, 1), (3, 2)])
def test_duplicate_earlier_copy_goes_first(copies, beta):
    """Redundancy row + recency protection: with equal importance (Q = 0, so
    every candidate gets the same attention) and a key repeated `copies` times,
    evicting one token removes the earliest copy; the newer copies are
    protected."""
    rng = np.random.default_rng(7)
    N, d, n_obs = 24, 512, 4
    K = rng.standard_normal((1, N, d))
    pos = [3, 8, 14][:copies]
    for p_ in pos[1:]:
        K[0, p_] = K[0, pos[0]] * (1.0 + 0.1 * p_) + 1e-3 * rng.standard_normal(d)
    Q = np.zeros((1, 2, n_obs, d))
    sc = oracle.score(K, Q, n_obs, 0.1, beta, 0.9)
    idx = oracle.select(sc["Z"], n_obs, N - 1)[0]
    evicted = sorted(set(range(N)) - set(idx.tolist()))
    assert evicted == [pos[0]]


# --------------------------------------------------------------- variants --
# Question 2, cause 3 of the review lists a softmax of the redundancy; the
# summary table's comparison method SnapKV pools its importance over
# positions.  Readings R10 / R11 of the oracle; off by default.

def _sc(I, R):
    return {"I": np.asarray(I, dtype=np.float64), "R": np.asarray(R, dtype=np.float64)}


@pytest.mark.parametrize("w", [3, 7, 31])
def test_variant_pooling_equals_maximum_filter(w):
    """I' = max of I over the window, cut at the candidates' ends:
    scipy.ndimage.maximum_filter1d with edge replication is the same window
    maximum (catches an off-by-one half width or a window reaching into the
    observation tokens)."""
    from scipy.ndimage import maximum_filter1d
    wk = wl.WORKLOADS[0]
    K, V, Q = wl.make_inputs(wk)
    sc = oracle.score(K, Q, wk.n_obs, wk.lam, wk.beta, wk.tau)
    C = wk.n_cached - wk.n_obs
    out = oracle.variant(sc, wk.n_obs, wk.lam, pool_window=w)
    ref = maximum_filter1d(sc["I"][:, :C], size=w, axis=1, mode="nearest")
    np.testing.assert_array_equal(out["I"][:, :C], ref)
    np.testing.assert_array_equal(out["I"][:, C:], sc["I"][:, C:])
    np.testing.assert_array_equal(out["R"], sc["R"])
    np.testing.assert_allclose(out["Z"][:, :C], wk.lam * ref - (1 - wk.lam) * sc["R"][:, :C],
                               rtol=0, atol=1e-15)


def test_variant_pooling_spike_closed_form():
    """A single spike spreads to exactly the (w-1)/2 neighbours on each side
    inside the candidates; a spike on an observation token spreads nowhere."""
    N, n_obs, w = 20, 4, 5
    C = N - n_obs
    for s_ in (0, 7, C - 1, C + 1):
        I = np.zeros((1, N))
        I[0, s_] = 1.0
        out = oracle.variant(_sc(I, np.zeros((1, N))), n_obs, 1.0, pool_window=w)
        exp = np.zeros(N)
        if s_ < C:
            exp[max(0, s_ - 2):min(C, s_ + 3)] = 1.0
        else:
            exp[s_] = 1.0
        np.testing.assert_array_equal(out["I"][0], exp)


def test_variant_softmax_equals_scipy():
    """R' = softmax of R over the C candidates only (scipy.special.softmax
    of the candidates' row); observation tokens R = 0, Z = +inf."""
    from scipy.special import softmax
    wk = wl.WORKLOADS[0]
    K, V, Q = wl.make_inputs(wk)
    sc = oracle.score(K, Q, wk.n_obs, wk.lam, wk.beta, wk.tau)
    C = wk.n_cached - wk.n_obs
    out = oracle.variant(sc, wk.n_obs, wk.lam, redundancy_softmax=True)
    ref = softmax(sc["R"][:, :C], axis=1)
    np.testing.assert_allclose(out["R"][:, :C], ref, rtol=1e-13, atol=0)
    np.testing.assert_allclose(out["R"][:, :C].sum(axis=1), 1.0, rtol=0, atol=1e-13)
    assert np.all(out["R"][:, C:] == 0) and np.all(np.isposinf(out["Z"][:, C:]))
    np.testing.assert_array_equal(out["I"], sc["I"])


def test_variant_softmax_closed_form():
    """R_j = ln c_j gives R'_j = c_j / sum c exactly (up to rounding)."""
    c = np.array([1.0, 2.0, 3.0, 4.0, 10.0])
    N, n_obs = 7, 2
    R = np.zeros((1, N))
    R[0, :5] = np.log(c)
    out = oracle.variant(_sc(np.zeros((1, N)), R), n_obs, 0.0, redundancy_softmax=True)
    np.testing.assert_allclose(out["R"][0, :5], c / c.sum(), rtol=1e-14, atol=0)
    np.testing.assert_allclose(out["Z"][0, :5], -c / c.sum(), rtol=1e-14, atol=0)


def test_variant_identical_keys_uniform_redundancy():
    """All keys identical: R = 1 everywhere, so the softmax is 1/C."""
    P, N, d, n_obs = 2, 30, 8, 4
    K = np.tile(np.random.default_rng(3).standard_normal(d), (P, N, 1))
    Q = np.random.default_rng(4).standard_normal((P, 2, n_obs, d))
    sc = oracle.score(K, Q, n_obs, 0.1, 2, 0.9)
    out = oracle.variant(sc, n_obs, 0.1, redundancy_softmax=True)
    np.testing.assert_allclose(out["R"][:, :N - n_obs], 1.0 / (N - n_obs), rtol=1e-14, atol=0)


def test_variant_off_is_identity_and_softmax_keeps_redundancy_order():
    """Window 1 without softmax changes nothing; the softmax is monotone, so
    with lambda = 0 (redundancy only) the kept set does not change."""
    wk = wl.WORKLOADS[0]
    K, V, Q = wl.make_inputs(wk)
    sc = oracle.score(K, Q, wk.n_obs, 0.0, wk.beta, wk.tau)
    same = oracle.variant(sc, wk.n_obs, 0.0)
    for k_ in ("I", "R", "Z"):
        np.testing.assert_array_equal(same[k_], sc[k_])
    soft = oracle.variant(sc, wk.n_obs, 0.0, redundancy_softmax=True)
    np.testing.assert_array_equal(oracle.select(soft["Z"], wk.n_obs, wk.budget),
                                  oracle.select(sc["Z"], wk.n_obs, wk.budget))
    res = oracle.compress(K, Q, wk.n_cached, wk.budget, wk.n_obs, 0.0, wk.beta, wk.tau,
                          redundancy_softmax=True)
    np.testing.assert_array_equal(res["idx"], oracle.select(sc["Z"], wk.n_obs, wk.budget))


# ------------------------------------------------------------------ paged --
# Question 2, cause 4 of the review: the paged round is the plain round read
# and written through a block table, with the emptied blocks handed back.

def _paged_case(S=3, H=2, bs=8, N=45, budget=30, d=16, extra=5, seed=0):
    rng = np.random.default_rng(seed)
    nb = -(-N // bs)
    num_blocks = S * nb + extra
    perm = rng.permutation(num_blocks)
    table = perm[:S * nb].reshape(S, nb).astype(np.int32)
    K_pool = rng.standard_normal((num_blocks, H, bs, d)).astype(np.float32)
    V_pool = rng.standard_normal((num_blocks, H, bs, d)).astype(np.float32)
    Q = rng.standard_normal((S * H, 2, 4, d))
    return K_pool, V_pool, Q, table, perm


def test_paged_rows_follow_the_table():
    """With the table naming consecutive blocks, the logical rows are the
    pool with the head and block axes swapped (a torch permute, not the
    oracle's loop)."""
    S, H, bs, nb, d = 2, 3, 4, 5, 6
    pool = np.random.default_rng(1).standard_normal((S * nb, H, bs, d))
    table = np.arange(S * nb, dtype=np.int32).reshape(S, nb)
    ref = torch.from_numpy(pool).reshape(S, nb, H, bs, d).permute(0, 2, 1, 3, 4)
    ref = ref.reshape(S * H, nb * bs, d).numpy()
    np.testing.assert_array_equal(oracle.paged_rows(pool, table, nb * bs), ref)
    np.testing.assert_array_equal(oracle.paged_rows(pool, table, 7), ref[:, :7])


def test_paged_round_equals_contiguous_round():
    """Kept sets equal the contiguous round on the same logical rows; every
    kept row lands at its logical position; blocks no table names, rows past
    the budget in the last kept block and the freed blocks' data are left as
    they were; the freed ids are the table's tail, ceil(N/bs) - ceil(B/bs)
    per sequence, and their entries become -1."""
    K_pool, V_pool, Q, table, perm = _paged_case()
    S, H, bs, N, B, n_obs = 3, 2, 8, 45, 30, 4
    out = oracle.paged_compress(K_pool, V_pool, Q, table, N, B, n_obs, 0.1, 2, 0.6)
    K_log = oracle.paged_rows(K_pool, table, N)
    V_log = oracle.paged_rows(V_pool, table, N)
    ref = oracle.compress(K_log, Q, N, B, n_obs, 0.1, 2, 0.6)
    np.testing.assert_array_equal(out["idx"], ref["idx"])
    new_K = oracle.paged_rows(out["K_pool"], table, B)
    new_V = oracle.paged_rows(out["V_pool"], table, B)
    np.testing.assert_array_equal(new_K, oracle.gather(K_log, ref["idx"])[:, :B])
    np.testing.assert_array_equal(new_V, oracle.gather(V_log, ref["idx"])[:, :B])
    nb_keep, nb_old = -(-B // bs), -(-N // bs)
    assert out["freed"].shape == (S, nb_old - nb_keep) == (S, 2)
    np.testing.assert_array_equal(out["freed"], table[:, nb_keep:nb_old])
    assert np.all(out["table"][:, nb_keep:nb_old] == -1)
    np.testing.assert_array_equal(out["table"][:, :nb_keep], table[:, :nb_keep])
    untouched = sorted(set(range(K_pool.shape[0])) - set(table[:, :nb_keep].ravel().tolist()))
    # the unfilled space after N in the old last block is among them
    assert set(table[:, nb_old - 1].tolist()) <= set(untouched)
    np.testing.assert_array_equal(out["K_pool"][untouched], K_pool[untouched])
    np.testing.assert_array_equal(out["V_pool"][untouched], V_pool[untouched])
    last = table[:, nb_keep - 1]
    np.testing.assert_array_equal(out["K_pool"][last, :, B % bs:], K_pool[last, :, B % bs:])


def test_paged_round_ignores_physical_placement():
    """Renumbering the physical blocks (pool and table together) changes
    nothing but the placement."""
    K_pool, V_pool, Q, table, _ = _paged_case(seed=2)
    N, B, n_obs = 45, 30, 4
    a = oracle.paged_compress(K_pool, V_pool, Q, table, N, B, n_obs, 0.1, 2, 0.6)
    ren = np.random.default_rng(3).permutation(K_pool.shape[0])
    K2, V2 = np.empty_like(K_pool), np.empty_like(V_pool)
    K2[ren], V2[ren] = K_pool, V_pool
    b = oracle.paged_compress(K2, V2, Q, ren[table].astype(np.int32), N, B, n_obs, 0.1, 2, 0.6)
    np.testing.assert_array_equal(a["idx"], b["idx"])
    np.testing.assert_array_equal(b["K_pool"][ren], a["K_pool"])
    np.testing.assert_array_equal(b["V_pool"][ren], a["V_pool"])
    np.testing.assert_array_equal(b["freed"], ren[a["freed"]])


def test_paged_round_identity_when_not_over_budget():
    K_pool, V_pool, Q, table, _ = _paged_case(N=45, budget=48)
    out = oracle.paged_compress(K_pool, V_pool, Q, table, 45, 48, 4, 0.1, 2, 0.6)
    np.testing.assert_array_equal(out["K_pool"], K_pool)
    np.testing.assert_array_equal(out["table"], table)
    assert out["freed"].shape[1] == 0


# -------------------------------------------------------------- sentences --
# SkipKV review (yoonschallenge.tistory.com/1230), rows "Method 1" and "Final
# eviction score": readings R12-R14 of the oracle.

def test_sentence_reps_equal_index_add_mean():
    """The mean hidden state per sentence equals torch's index_add divided
    by the token counts (catches a wrong divisor or a shifted run)."""
    si = wl.make_sentences(2, 1, 1, 97, 12, dtype=torch.float32)
    reps = oracle.sentence_reps(si.hidden, si.token_seg, si.max_sentences)
    for s_ in range(2):
        seg = si.token_seg[s_].long()
        tot = torch.zeros(si.max_sentences, 12, dtype=torch.float64).index_add_(
            0, seg, si.hidden[s_].double())
        cnt = torch.bincount(seg, minlength=si.max_sentences).double().clamp(min=1)[:, None]
        np.testing.assert_allclose(reps[s_], (tot / cnt).numpy(), rtol=0, atol=1e-12)


def test_sentence_penalty_equals_normalised_matmul():
    """pen[a] = the largest cosine above tau with a later sentence: a masked
    upper-triangular max of numpy's normalised matmul."""
    rng = np.random.default_rng(5)
    reps = rng.standard_normal((2, 9, 16))
    reps[0, 2] = reps[0, 6] * 1.5 + 0.05 * rng.standard_normal(16)
    reps[1, 0] = reps[1, 8] * 0.5 + 0.05 * rng.standard_normal(16)
    count = np.array([9, 9])
    pen, _ = oracle.sentence_penalty(reps, count, 0.3)
    for s_ in range(2):
        X = reps[s_] / np.linalg.norm(reps[s_], axis=1, keepdims=True)
        C = X @ X.T
        up = np.triu(np.ones((9, 9), dtype=bool), 1) & (C > 0.3)
        ref = np.where(up.any(axis=1), np.where(up, C, -np.inf).max(axis=1), 0.0)
        np.testing.assert_allclose(pen[s_], ref, rtol=0, atol=1e-13)
    assert pen[0, 2] > 0.99 and pen[1, 0] > 0.99


def test_sentence_penalty_closed_forms():
    """Only the earlier of two equal sentences is penalised (by exactly 1);
    of three copies the first two; the threshold is strict (cos = 3/5 at
    tau = 0.6 gives nothing); the penalty is the similarity itself, also
    below zero when tau is; sentences past count and zero vectors give 0."""
    e = np.eye(4)
    reps = np.stack([e[0], e[1], 2 * e[0], 3 * e[0] + 4 * e[2], e[3], 3 * e[1]])[None]
    pen, _ = oracle.sentence_penalty(reps, np.array([6]), 0.9)
    np.testing.assert_allclose(pen[0], [1, 1, 0, 0, 0, 0], rtol=0, atol=1e-15)
    pen, _ = oracle.sentence_penalty(reps[:, [0, 3]], np.array([2]), 0.6)
    assert pen[0, 0] == 0.0
    pen, _ = oracle.sentence_penalty(reps[:, [0, 3]], np.array([2]), 0.5999)
    assert pen[0, 0] == 0.6
    neg = np.stack([e[0], -e[0] + np.sqrt(15) * e[1]])[None]  # cos = -1/4
    pen, _ = oracle.sentence_penalty(neg, np.array([2]), -0.5)
    assert abs(pen[0, 0] + 0.25) < 1e-15
    pen, _ = oracle.sentence_penalty(reps, np.array([2]), 0.9)   # sentence 2 not counted
    assert np.all(pen == 0)
    zero = np.zeros((1, 2, 4))
    assert np.all(oracle.sentence_penalty(zero, np.array([2]), -1.0)[0] == 0)


def test_row_penalties_follow_the_sentence_ids():
    pen = np.array([[0.5, 0.0, 0.9], [0.7, 0.2, 0.0]])
    count = np.array([3, 2])
    seg = np.array([[0, 0, 2, -1, 5], [0, 1, 2, 1, 0]] * 2)  # P = 4, heads = 1, 2 layers
    out = oracle.row_penalties(pen, count, seg, 1, 5)
    np.testing.assert_array_equal(out[0], [0.5, 0.5, 0.9, 0, 0])
    np.testing.assert_array_equal(out[1], [0.7, 0.2, 0, 0.2, 0.7])  # id 2 >= count 2
    np.testing.assert_array_equal(out[2], out[0])


def test_redundant_earlier_sentence_goes_first():
    """SkipKV's point: with equal importance and a sentence repeated later,
    evicting that many tokens removes the earlier copy's rows."""
    rng = np.random.default_rng(8)
    N, d, n_obs = 40, 32, 4
    K = rng.standard_normal((1, N, d))
    Q = np.zeros((1, 2, n_obs, d))
    seg = np.repeat(np.arange(5), 8)[None]  # five sentences of 8 rows
    reps = rng.standard_normal((1, 5, 24))
    reps[0, 3] = reps[0, 1] + 0.01 * rng.standard_normal(24)
    pen, _ = oracle.sentence_penalty(reps, np.array([5]), 0.9)
    assert pen[0, 1] > 0.99 and np.count_nonzero(pen) == 1
    rp = oracle.row_penalties(pen, np.array([5]), seg, 1, N)
    res = oracle.compress(K, Q, N, N - 8, n_obs, 0.1, 2, 0.9, row_penalty=rp)
    evicted = sorted(set(range(N)) - set(res["idx"][0].tolist()))
    assert evicted == list(range(8, 16))


# --------------------------------------------------------------- schedule --
# ForesightKV summary page (gist.science/ko/paper/2602.03203), section
# "Dynamic eviction process": readings R15-R16 of the oracle.

def test_gumbel_top_k_is_multinomial_without_replacement():
    """The sampled selection draws k of the pool with probabilities
    proportional to exp(Z / T), one after another without replacement: the
    frequencies of the kept pairs over 40,000 seeded draws match the exact
    probabilities of sequential sampling (enumerated by hand, not via the
    Gumbel route) within a chi-square bound."""
    Z = np.array([[0.3, -0.2, 0.9, 0.1, 0.5, np.inf]])  # last row: the window
    T, draws = 0.5, 40000
    w = np.exp(Z[0, :5] / T)
    pr = w / w.sum()
    exact = {}
    for a, b in itertools.permutations(range(5), 2):
        key = tuple(sorted((a, b)))
        exact[key] = exact.get(key, 0.0) + pr[a] * pr[b] / (1 - pr[a])
    u = np.random.default_rng(21).random((draws, 5))
    counts = {}
    for t in range(draws):
        sel = oracle.schedule_select(Z, 1, 3, 5, T, u[t:t + 1])
        key = tuple(sel["idx"][0, :2].tolist())
        counts[key] = counts.get(key, 0) + 1
    chi2 = sum((counts.get(key, 0) - draws * p_) ** 2 / (draws * p_) for key, p_ in exact.items())
    assert chi2 < 35.0, chi2  # 9 degrees of freedom: p ~ 1e-4
    assert abs(sum(exact.values()) - 1.0) < 1e-12


def test_schedule_pool_window_and_limits():
    """Only pool members are ever kept; the window is always kept; a pool of
    exactly k is the plain top-k; a tiny temperature gives the top-k of Z."""
    rng = np.random.default_rng(4)
    P, N, L, B = 6, 60, 10, 30
    Z = rng.standard_normal((P, N))
    u = rng.random((P, N))
    k, C = B - L, N - L
    s1 = oracle.schedule_select(Z, L, B, k + 12, 1.0, u)
    for p in range(P):
        kept = s1["idx"][p, :k]
        assert s1["pool"][p, kept].all()
        assert s1["pool"][p].sum() == k + 12
        assert list(s1["idx"][p, k:]) == list(range(C, N))
    np.testing.assert_array_equal(oracle.schedule_select(Z, L, B, k)["idx"],
                                  oracle.select(Z, L, B))
    np.testing.assert_array_equal(oracle.schedule_select(Z, L, B, C, 1e-9, u)["idx"],
                                  oracle.select(Z, L, B))


def test_compress_with_recent_window():
    """With a window L > n_obs the L newest rows are kept and the importance
    still comes from the n_obs observation queries (scores equal the plain
    scores on the candidates)."""
    w = wl.WORKLOADS[0]
    K, V, Q = wl.make_inputs(w)
    L = 16
    res = oracle.compress(K, Q, w.n_cached, w.budget, w.n_obs, w.lam, w.beta, w.tau,
                          recent_window=L)
    base = oracle.score(K[:, :w.n_cached], Q, w.n_obs, w.lam, w.beta, w.tau)
    C = w.n_cached - L
    np.testing.assert_array_equal(res["scores"]["Z"][:, :C], base["Z"][:, :C])
    assert np.all(np.isposinf(res["scores"]["Z"][:, C:]))
    np.testing.assert_array_equal(res["idx"], oracle.select(base["Z"], L, w.budget))


# ------------------------------------------------------------- invariants --

def test_compress_invariants_tiny_and_identity():
    """Scheme row: exactly `budget` tokens stay, the newest n_obs always stay,
    indices are ascending; with n_cached <= budget nothing is evicted."""
    w = wl.WORKLOADS[0]
    K, V, Q = wl.make_inputs(w, n_cap=w.n_cached + 5)
    res = oracle.compress(K, Q, w.n_cached, w.budget, w.n_obs, w.lam, w.beta, w.tau)
    idx = res["idx"]
    assert idx.shape == (w.problems, w.budget)
    assert np.all(np.diff(idx, axis=1) > 0)
    assert np.all(idx[:, -w.n_obs:] == np.arange(w.n_cached - w.n_obs, w.n_cached))
    ident = oracle.compress(K, Q, 50, w.budget, w.n_obs, w.lam, w.beta, w.tau)["idx"]
    assert np.all(ident[:, :50] == np.arange(50)) and np.all(ident[:, 50:] == -1)


def test_gather_copies_bytes():
    rng = np.random.default_rng(9)
    src = rng.standard_normal((2, 10, 6)).astype(np.float32)
    idx = np.array([[0, 3, 4, 9], [1, 2, 7, 8]], dtype=np.int32)
    out = oracle.gather(src, idx)
    for p in range(2):
        np.testing.assert_array_equal(out[p, :4], src[p, idx[p]])
        assert np.all(out[p, 4:] == 0)


def test_page_parameters_fixture():
    """The page's printed defaults (buffer 128, 8 observation tokens,
    lambda = 0.1) are the ones every workload uses."""
    import json
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "rkv_page_parameters.json")
    fx = json.load(open(path))
    for w in wl.WORKLOADS:
        assert w.n_obs == fx["n_obs"]["value"]
        assert w.lam == fx["lambda"]["value"]
        if w.keys == "ar1":
            assert w.n_cached - w.budget == fx["buffer"]["value"] or w.name == "stream"
    assert wl.BY_NAME["stream"].buffer == fx["buffer"]["value"]
