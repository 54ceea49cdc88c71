"""The two-partition step schedule (rkv_set_overlap): importance and Gram of
one group of problems on the tensor partition while the previous group is
compacted on the other SMs.  It must give exactly what the one-launch-per-
stage schedule gives (every kept index and every kept byte), in place and out
of place, with a short last group, and agree with the oracle on sampled
problems of every group."""
import numpy as np
import pytest
import torch

import oracle
from decode_kv_cache_02_gb300 import rkv, workloads as wl
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture
def serial_after():
    yield
    rkv.rkv_set_overlap(*rkv.DEFAULT_OVERLAP)


def _compress(K, V, Q, w, in_place):
    if in_place:
        K, V = K.clone(), V.clone()
        return rkv.rkv_compress(K, V, Q, w.n_cached, w.budget, w.n_obs, w.lam, w.beta, w.tau,
                                out_K=K, out_V=V)
    return rkv.rkv_compress(K, V, Q, w.n_cached, w.budget, w.n_obs, w.lam, w.beta, w.tau)


@pytest.mark.parametrize("groups,tensor_sms,in_place",
                         [(4, 104, False), (3, 120, True), (8, 96, False)])
def test_overlap_matches_one_launch_schedule(cuda_ok, serial_after, groups, tensor_sms,
                                             in_place):
    w = wl.BY_NAME["llama8b_full"]
    P = 2600  # groups of whole waves of the tensor partition, the last one short
    K, V, Q = wl.make_inputs(w, device="cuda", problems=P)
    b = w.budget
    rkv.rkv_set_overlap(rkv.RKV_SCHEDULE_ONE_LAUNCH, 8, tensor_sms)
    rK, rV, ridx = _compress(K, V, Q, w, in_place)
    rkv.rkv_set_overlap(rkv.RKV_SCHEDULE_GROUPED, groups, tensor_sms)
    for call in range(2):  # the partitions and their events are reused by the second call
        rkv.rkv_timing_read(reset=True)
        rkv.rkv_timing_enable(True)
        oK, oV, idx = _compress(K, V, Q, w, in_place)
        rkv.rkv_timing_enable(False)
        torch.cuda.synchronize()
        launches = rkv.rkv_timing_read(reset=True)
        if launches["gram_tc"][1] == 1:
            pytest.skip("the driver offers no SM partitions: one launch per stage ran")
        # one Gram and one importance launch per group, a compaction per group
        assert launches["gram_tc"][1] == launches["importance_tc"][1] == launches["compact"][1]
        assert 2 <= launches["gram_tc"][1] <= groups
        assert torch.equal(idx, ridx)
        assert torch.equal(oK[:, :b].view(torch.int16), rK[:, :b].view(torch.int16))
        assert torch.equal(oV[:, :b].view(torch.int16), rV[:, :b].view(torch.int16))
    # the oracle on problems spread over every group
    problems = sorted(np.random.default_rng(groups).choice(P, 24, replace=False).tolist())
    sc = oracle.score(K[problems, :w.n_cached].cpu(), Q[problems].cpu(), w.n_obs, w.lam, w.beta,
                      w.tau)
    gi = idx.cpu().numpy()
    parity.check_idx_valid(gi, w.n_cached, b, w.n_obs)
    bad, excused = parity.kept_mismatches(gi[problems], sc, b, w.n_obs)
    assert bad == 0, f"{bad} kept-set mismatches outside the tie band ({excused} excused)"
    parity.check_gathered(oK, K, idx, b, problems)
    parity.check_gathered(oV, V, idx, b, problems)


def test_partitions_run_at_the_same_time(cuda_ok, serial_after):
    """The launch trace (one global timer for both partitions) shows the
    groups' compactions running while the tensor partition scores the next
    group, and every launch of the call on its lane."""
    w = wl.BY_NAME["llama8b_full"]
    K, V, Q = wl.make_inputs(w, device="cuda", problems=4096)
    rkv.rkv_set_overlap(rkv.RKV_SCHEDULE_GROUPED, 8, 0)
    _compress(K, V, Q, w, False)  # partitions created, kernels loaded
    torch.cuda.synchronize()
    rkv.rkv_trace_enable(True)
    _compress(K, V, Q, w, False)
    recs = rkv.rkv_trace_read()
    rkv.rkv_trace_enable(False)
    if not any(lane for _, lane, _, _ in recs):
        pytest.skip("the driver offers no SM partitions: one launch per stage ran")
    lanes = {}
    for name, lane, a, b in recs:
        assert b > a
        lanes.setdefault(lane, []).append((name, a, b))
    assert {n for n, _, _ in lanes[1]} == {"importance_tc", "gram_tc"}
    assert {n for n, _, _ in lanes[2]} == {"compact"}
    assert [n for n, _, _ in lanes[0]] == ["compact"]  # the last group, whole device
    G = len([1 for n, _, _ in lanes[1] if n == "gram_tc"])
    assert len(lanes[2]) == G - 1
    # each group's compaction starts after its Gram ends, and at least one
    # compaction overlaps a later group's scoring
    grams = [(a, b) for n, a, b in lanes[1] if n == "gram_tc"]
    comps = [(a, b) for _, a, b in lanes[2]]
    assert all(c[0] >= g[1] for g, c in zip(grams, comps))
    scoring = [(a, b) for _, a, b in lanes[1]]
    overlap = sum(max(0, min(b, d) - max(a, c)) for a, b in scoring for c, d in comps)
    assert overlap > 0
