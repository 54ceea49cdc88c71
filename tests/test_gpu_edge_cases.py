"""GPU parity on the method's own edge cases, through the C ABI, against the
fp64 oracle and against closed forms the definitions fix (R-KV review,
yoonschallenge.tistory.com/1236, summary-table rows "importance",
"redundancy" and "final selection criterion"):

- keys that all point the same way (scaled by powers of two, so the bf16
  values are exact): every cosine is 1, every candidate has more than beta
  newer similar tokens, so R = 1, and every Gram sub-tile holds pairs
  above tau;
- groups of exact copies of orthogonal keys with Q = 0: every S is 0 or 1, I
  is the same for every candidate, R is (m-1)/(N-1) for the unprotected
  members of a group of m and 0 for the beta newest, Z ties exactly inside a
  group, ties go to the newer token, so the earliest copy of the largest
  group is the one evicted first -- and the kept set must equal the
  oracle's exactly;
- a zero-norm key: its norm is clamped, so all its similarities are 0;
- Q = 0: uniform causal attention, I_i = (1/n_obs) sum_q [i <= N-n_obs+q] /
  (N-n_obs+q+1);
- lambda = 1: the kept candidates are the top k of I.

Each runs on the tensor-core path at N = 1152 (the resident importance) and
N = 4224 (the two-pass importance, 34-block Gram), and on the fp32 CUDA-core
path."""
import numpy as np
import pytest
import torch

import oracle
from decode_kv_cache_02_gb300 import rkv, workloads as wl
from tests import parity

pytestmark = pytest.mark.gpu

DEV = "cuda"

# (dtype, head_dim, n_cached, problems): tensor-core paths at the Llama-8B
# and Qwen-14B lengths, and the fp32 path
SHAPES = [("bf16", 128, 1152, 3), ("bf16", 128, 4224, 2), ("fp32", 64, 320, 3)]
IDS = ["bf16-1152", "bf16-4224", "fp32-320"]


def _dt(name):
    return {"bf16": torch.bfloat16, "fp32": torch.float32}[name]


def _pow2_scales(P, N, g):
    """Per-row scales 2^e, e in -2..2: exact in bf16 and fp32."""
    return 2.0 ** torch.randint(-2, 3, (P, N, 1), generator=g).double()


def _run(K, Q, n, budget, n_obs=8, lam=0.1, beta=2, tau=0.9):
    """GPU scores and step (out of place) for inputs given on the host."""
    Kd, Qd = K.to(DEV), Q.to(DEV)
    Vd = torch.randn(K.shape, generator=torch.Generator().manual_seed(9)).to(K.dtype).to(DEV)
    I, R, Z = rkv.rkv_score(Kd, Qd, n, n_obs, lam, beta, tau)
    oK, oV, idx = rkv.rkv_compress(Kd, Vd, Qd, n, budget, n_obs, lam, beta, tau)
    torch.cuda.synchronize()
    gpu = {"I": I.cpu(), "R": R.cpu(), "Z": Z.cpu()}
    return gpu, idx.cpu().numpy(), (Kd, Vd, oK, oV, idx)


def _parity(gpu, idx, K, Q, n, budget, n_obs=8, lam=0.1, beta=2, tau=0.9, moved=None):
    """Scores within 2e-3 of the oracle, kept set within the tie band, rows
    byte-exact; returns the oracle's scores."""
    C = n - n_obs
    sc = oracle.score(K, Q, n_obs, lam, beta, tau)
    err = parity.score_errors(gpu, sc, C)
    assert max(err.values()) <= parity.SCORE_ATOL, err
    parity.check_observation_scores(gpu, C)
    parity.check_idx_valid(idx, n, budget, n_obs)
    bad, excused = parity.kept_mismatches(idx, sc, budget, n_obs)
    assert bad == 0, f"{bad} kept-set mismatches outside the tie band ({excused} excused)"
    if moved is not None:
        Kd, Vd, oK, oV, didx = moved
        parity.check_gathered(oK, Kd, didx, budget)
        parity.check_gathered(oV, Vd, didx, budget)
    return sc


@pytest.mark.parametrize("dt,d,N,P", SHAPES, ids=IDS)
def test_identical_keys_give_redundancy_one(cuda_ok, dt, d, N, P):
    g = torch.Generator().manual_seed(N + d)
    u = torch.randn(P, 1, d, generator=g).to(_dt(dt)).double()
    K = (u * _pow2_scales(P, N, g)).to(_dt(dt))  # exact: same direction bit for bit
    Q = torch.randn(P, 4, 8, d, generator=g).to(_dt(dt))
    budget = N - 64
    gpu, idx, moved = _run(K, Q, N, budget)
    sc = _parity(gpu, idx, K, Q, N, budget, moved=moved)
    C = N - 8
    # the closed form, in the oracle (fp64: sqrt(x)^2 may differ from x by an ulp)
    assert np.abs(sc["R"][:, :C] - 1.0).max() < 1e-12
    assert np.abs(gpu["R"][:, :C].double().numpy() - 1.0).max() <= parity.SCORE_ATOL


def _groups(P, N, d, g, big=1):
    """Keys that are exact copies of the d standard basis directions (scaled
    by powers of two), N/d per direction except one group of N/d + big and
    one of N/d - big, at seeded random positions.  Returns the keys and the
    group of every row."""
    m = N // d
    assert m * d == N
    sizes = [m] * d
    sizes[0] += big
    sizes[1] -= big
    grp = torch.cat([torch.full((s,), j) for j, s in enumerate(sizes)])
    K = torch.zeros(P, N, d, dtype=torch.float64)
    gid = torch.empty(P, N, dtype=torch.long)
    for p in range(P):
        perm = grp[torch.randperm(N, generator=g)]
        gid[p] = perm
        K[p, torch.arange(N), perm] = 1.0
    return K * _pow2_scales(P, N, g), gid


@pytest.mark.parametrize("dt,d,N,P", SHAPES, ids=IDS)
@pytest.mark.parametrize("beta", [1, 2])
def test_duplicate_copies_earliest_goes_first(cuda_ok, dt, d, N, P, beta):
    g = torch.Generator().manual_seed(7 * N + beta)
    Kd, gid = _groups(P, N, d, g)
    K = Kd.to(_dt(dt))
    Q = torch.zeros(P, 4, 8, d, dtype=_dt(dt))
    n_obs, C = 8, N - 8
    for budget in (N - 1, N - 40):
        gpu, idx, moved = _run(K, Q, N, budget, beta=beta)
        sc = _parity(gpu, idx, K, Q, N, budget, beta=beta, moved=moved)
        # closed form: R = (m-1)/(N-1) for the unprotected members of a group
        # of m (at least beta newer copies), 0 for the beta newest
        for p in range(P):
            ids = gid[p].numpy()
            for i in range(C):
                members = np.flatnonzero(ids == ids[i])
                newer = int((members > i).sum())
                want = 0.0 if newer < beta else (len(members) - 1) / (N - 1)
                assert abs(sc["R"][p, i] - want) < 1e-12
        # every S is 0 or 1 and every candidate has the same I, so the GPU's
        # Z ties exactly where the oracle's does: the kept sets are equal
        np.testing.assert_array_equal(idx, oracle.select(sc["Z"], n_obs, budget))
        if budget == N - 1:
            # the one evicted token is the earliest unprotected copy of the
            # largest group (group 0)
            for p in range(P):
                gone = sorted(set(range(N)) - set(idx[p].tolist()))
                first = int(np.flatnonzero(gid[p].numpy() == 0)[0])
                assert gone == [first], (p, gone, first)


@pytest.mark.parametrize("dt,d,N,P", SHAPES, ids=IDS)
@pytest.mark.parametrize("tau", [0.9, -0.2])
def test_zero_norm_key(cuda_ok, dt, d, N, P, tau):
    w = wl.BY_NAME["llama8b_layer"].scaled(head_dim=d, dtype=dt, n_cached=N, budget=N - 100,
                                           layers=1, batch=1, kv_heads=P)
    K, _, Q = wl.make_inputs(w, device="cpu")
    zero_rows = [(0, 3), (0, N // 2), (P - 1, N - 20), (P - 1, 0)]
    for p, i in zero_rows:
        K[p, i] = 0
    gpu, idx, moved = _run(K, Q, N, w.budget, tau=tau)
    sc = _parity(gpu, idx, K, Q, N, w.budget, tau=tau, moved=moved)
    for p, i in zero_rows:
        # no similarity with anything: R is 0 (tau > 0), or every other key
        # counts as similar with S = 0 (tau < 0)
        assert sc["R"][p, i] == 0.0
        assert abs(float(gpu["R"][p, i])) <= parity.SCORE_ATOL


@pytest.mark.parametrize("dt,d,N,P", SHAPES, ids=IDS)
def test_zero_queries_give_uniform_importance(cuda_ok, dt, d, N, P):
    w = wl.BY_NAME["llama8b_layer"].scaled(head_dim=d, dtype=dt, n_cached=N, budget=N - 100,
                                           layers=1, batch=1, kv_heads=P)
    K, _, Q = wl.make_inputs(w, device="cpu")
    Q = torch.zeros_like(Q)
    gpu, idx, moved = _run(K, Q, N, w.budget)
    _parity(gpu, idx, K, Q, N, w.budget, moved=moved)
    n_obs = 8
    q = np.arange(n_obs)
    i = np.arange(N)[:, None]
    closed = ((i <= N - n_obs + q) / (N - n_obs + q + 1.0)).mean(axis=1)
    err = np.abs(gpu["I"].double().numpy() - closed[None, :]).max()
    assert err <= 1e-6, err


@pytest.mark.parametrize("dt,d,N,P", SHAPES, ids=IDS)
def test_lambda_one_keeps_attention_top_k(cuda_ok, dt, d, N, P):
    w = wl.BY_NAME["llama8b_layer"].scaled(head_dim=d, dtype=dt, n_cached=N, budget=N - 200,
                                           layers=1, batch=1, kv_heads=P, lam=1.0)
    K, _, Q = wl.make_inputs(w, device="cpu")
    gpu, idx, moved = _run(K, Q, N, w.budget, lam=1.0)
    sc = _parity(gpu, idx, K, Q, N, w.budget, lam=1.0, moved=moved)
    C, k = N - 8, w.budget - 8
    I_gpu = gpu["I"].double().numpy()
    for p in range(P):
        # the GPU's kept candidates are the top k of its own I (Z = I), and of
        # the oracle's I up to the tie band
        kept = set(idx[p, :k].tolist())
        order = np.lexsort((-np.arange(C), -I_gpu[p, :C]))  # I desc, index desc
        assert kept == set(order[:k].tolist())
        ik = np.sort(sc["I"][p, :C])[::-1][k - 1]
        top = set(np.argsort(-sc["I"][p, :C], kind="stable")[:k].tolist())
        assert all(abs(sc["I"][p, i] - ik) <= parity.KEPT_BAND for i in kept ^ top)
