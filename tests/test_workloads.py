"""The synthetic workload generator: shapes, determinism and the statistics
the recipe promises (AR(1) neighbour similarity, re-emitted segments)."""
import math

import torch

from decode_kv_cache_02_gb300 import workloads as wl


def test_shapes_and_determinism():
    w = wl.BY_NAME["llama8b_layer"]
    K, V, Q = wl.make_inputs(w, n_cap=w.n_cached + 3)
    assert K.shape == (8, w.n_cached + 3, 128) and K.dtype == torch.bfloat16
    assert Q.shape == (8, 4, 8, 128)
    assert torch.isnan(K[:, w.n_cached:].float()).all()
    K2, V2, Q2 = wl.make_inputs(w, n_cap=w.n_cached + 3)
    assert torch.equal(K[:, :w.n_cached], K2[:, :w.n_cached]) and torch.equal(Q, Q2)


def test_ar1_neighbour_similarity_and_repeats():
    w = wl.BY_NAME["llama8b_layer"].scaled(kv_heads=16, copy_noise=0.0)
    K, _, _ = wl.make_inputs(w)
    k = K.float()
    kn = k / k.norm(dim=-1, keepdim=True)
    adj = (kn[:, 1:] * kn[:, :-1]).sum(-1)
    # stationary AR(1): neighbour cosine close to rho
    assert abs(adj.mean().item() - wl.RHO) < 0.03
    # with zero copy noise, re-emitted segments are exact copies of earlier ones
    segs = k.view(k.shape[0], -1, wl.SEGMENT, k.shape[-1])
    S = segs.shape[1]
    copies = 0
    for s in range(1, S):
        eq = (segs[:, s:s + 1] == segs[:, :s]).all(-1).all(-1).any(-1)
        copies += int(eq.sum())
    frac = copies / (k.shape[0] * (S - 1))
    assert abs(frac - w.repeat_prob) < 0.08


def test_walk_closed_form_equals_recurrence():
    # the chunked closed form of the walk against the recurrence applied token
    # by token, across several chunks and a ragged tail
    g = torch.Generator().manual_seed(5)
    e = torch.randn(3, 2 * wl.WALK_CHUNK + 37, 16, generator=g, dtype=torch.float64)
    ref = e.clone()
    c = math.sqrt(1.0 - wl.RHO ** 2)
    for t in range(1, ref.shape[1]):
        ref[:, t] = wl.RHO * ref[:, t - 1] + c * ref[:, t]
    got = wl._ar1_walk_(e.float().clone())
    assert torch.allclose(got.double(), ref, atol=1e-5, rtol=0)


def test_tiny_has_noisy_copies():
    w = wl.BY_NAME["tiny"]
    K, _, _ = wl.make_inputs(w)
    diff = (K[:, 40:48] - K[:, 10:18]).float()
    assert diff.abs().max() < 0.1 and diff.abs().max() > 0


def test_stream_source_history_and_walk():
    w = wl.BY_NAME["stream"].scaled(gen_tokens=512)
    s = wl.StreamSource(w, problems=4)
    ks = [s.next_chunk()[0] for _ in range(4)]
    full = torch.cat(ks, 1).float()
    assert torch.equal(full.to(w.torch_dtype), s.history)
    kn = full / full.norm(dim=-1, keepdim=True)
    adj = (kn[:, 1:] * kn[:, :-1]).sum(-1)
    assert adj.mean().item() > 0.75


def test_random_indices_ascending():
    idx = wl.random_indices(5, 300, 200)
    assert idx.dtype == torch.int32 and (idx[:, 1:] > idx[:, :-1]).all()
    assert int(idx.max()) < 300
