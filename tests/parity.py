"""Comparison helpers for the GPU-vs-oracle parity tests.

Tolerances (the target fixed for this method): scores I, R, Z within 2e-3
absolute; kept sets identical except tokens whose oracle score lies within
2e-3 of the k-th largest oracle score, or whose protection/similarity depends
on a threshold-borderline pair (|S_ij - tau| < 1e-5); gathered rows
bit-exact for the GPU's own indices.  Scoring variants (the redundancy
softmax puts R near 1/C) take the same 2e-3 scaled by each problem's scale
min(1, max_i |X*_i|): tighter than the absolute bound where the values are
small, and never looser than it (a sentence penalty can push |Z*| past 1).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

SCORE_ATOL = 2e-3
KEPT_BAND = 2e-3


def score_errors(gpu: dict, sc: dict, C: int) -> dict:
    """Max abs error of I, R, Z over the candidates (and I over all)."""
    out = {}
    for name in ("I", "R", "Z"):
        g = gpu[name].detach().cpu().double().numpy()
        hi = g.shape[1] if name == "I" else C
        out[name] = float(np.abs(g[:, :hi] - sc[name][:, :hi]).max())
    return out


def scaled_score_errors(gpu: dict, sc: dict, C: int) -> dict:
    """Max over problems of the error of I, R, Z over the candidates relative
    to the problem's scale min(1, max_i |X*_i|) (for scoring variants whose
    values are ~1/C, where an absolute 2e-3 would compare nothing; capped at
    1 so the bound is never looser than the absolute one)."""
    out = {}
    for name in ("I", "R", "Z"):
        g = gpu[name].detach().cpu().double().numpy()[:, :C]
        ref = sc[name][:, :C]
        scale = np.clip(np.abs(ref).max(axis=1), 1e-300, 1.0)
        out[name] = float((np.abs(g - ref).max(axis=1) / scale).max())
    return out


def scaled_band(sc: dict, C: int, rel: float = KEPT_BAND) -> np.ndarray:
    """Per-problem tie band rel * min(1, max_i |Z*_i|) over the candidates."""
    return rel * np.minimum(np.abs(sc["Z"][:, :C]).max(axis=1), 1.0)


def check_observation_scores(gpu: dict, C: int):
    R = gpu["R"].detach().cpu().numpy()
    Z = gpu["Z"].detach().cpu().numpy()
    assert np.all(R[:, C:] == 0.0)
    assert np.all(np.isposinf(Z[:, C:]))


def check_idx_valid(idx: np.ndarray, N: int, budget: int, n_obs: int):
    assert idx.shape[1] == budget
    assert np.all(np.diff(idx, axis=1) > 0), "indices not strictly ascending"
    assert np.all(idx[:, -n_obs:] == np.arange(N - n_obs, N)), "observation tokens missing"
    assert np.all(idx[:, : budget - n_obs] < N - n_obs) and np.all(idx >= 0)


def kept_mismatches(idx_gpu: np.ndarray, sc: dict, budget: int, n_obs: int,
                    band=KEPT_BAND) -> tuple[int, int]:
    """(unexcused, excused) counts of tokens kept by one side only; `band` is
    one number or one per problem."""
    P, N = sc["Z"].shape
    C, k = N - n_obs, budget - n_obs
    ref = oracle.select(sc["Z"], n_obs, budget)
    bad = ok = 0
    for p in range(P):
        z = sc["Z"][p, :C]
        zk = np.sort(z)[::-1][k - 1]
        diff = set(idx_gpu[p, :k].tolist()) ^ set(ref[p, :k].tolist())
        b = band[p] if np.ndim(band) else band
        for i in diff:
            if abs(z[i] - zk) <= b or sc["border"][p, i]:
                ok += 1
            else:
                bad += 1
    return bad, ok


def check_gathered(out: torch.Tensor, src: torch.Tensor, idx: torch.Tensor, budget: int,
                   problems=None):
    """out rows 0..budget-1 equal src rows idx, byte for byte (the oracle's
    byte copy on sampled problems)."""
    ps = list(range(src.shape[0])) if problems is None else list(problems)
    s = src[ps].cpu()
    raw = s.view(torch.int16) if s.dtype == torch.bfloat16 else s.view(torch.int32)
    exp = oracle.gather(raw.numpy(), idx[ps].cpu().numpy())
    o = out[ps].cpu()
    got = (o.view(torch.int16) if o.dtype == torch.bfloat16 else o.view(torch.int32)).numpy()
    np.testing.assert_array_equal(got[:, :budget], exp[:, :budget])


def sampled_mismatches(idx_gpu: np.ndarray, sc: dict, sel: dict, budget: int, n_tail: int,
                       temperature: float, band: float = KEPT_BAND) -> tuple[int, int]:
    """(unexcused, excused) kept-set differences of a sampled selection
    (oracle ``schedule_select`` result ``sel``, same uniforms).  Excused: a
    token whose Z is within ``band`` of the pool's last Z (pool membership can
    flip), whose sampling key is within band / temperature (+ 1e-5 for the
    noise's fp32 rounding) of the k-th key, or a threshold-borderline token."""
    k = budget - n_tail
    bad = ok = 0
    for p in range(idx_gpu.shape[0]):
        diff = set(idx_gpu[p, :k].tolist()) ^ set(sel["idx"][p, :k].tolist())
        for i in diff:
            near_pool = abs(sc["Z"][p, i] - sel["z_pool"][p]) <= band
            near_cut = abs(sel["keys"][p, i] - sel["key_k"][p]) <= band / temperature + 1e-5
            if near_pool or near_cut or sc["border"][p, i]:
                ok += 1
            else:
                bad += 1
    return bad, ok
