"""Seeded synthetic workloads for the compression step.

This module draws random tensors and holds the workload shapes; it contains
none of the method's arithmetic (no similarity, softmax, score or selection),
so the tests, the benchmark and the oracle side may all take their inputs from
it.

Shapes and parameters follow the R-KV review page
(yoonschallenge.tistory.com/1236): summary-table row "Decoding-time
compression scheme" (buffer of 128 generated tokens, 8 observation tokens) and
row "final selection criterion" (lambda = 0.1).  The pages evaluate on
reasoning traces of DeepSeek-R1-Distill models (MATH-500, AIME 2024); neither
the models nor the traces are available here, so the synthetic keys below
stand in for them: an AR(1) random walk (neighbouring keys are similar, as in
a smooth hidden-state trajectory) in which a fraction of 64-token segments is
re-emitted as noisy copies of earlier segments (the repeated reflection loops
the page describes in its summary-table row "key observation").

Layouts: K, V ``[P, n_cap, d]``, Q_obs ``[P, G, n_obs, d]``, one problem per
(layer, sequence, KV head), problems ordered layer-major then sequence then
head; query head ``g`` of problem ``p`` is query head ``h*G + g`` of the model,
where ``h`` is the KV head of ``p``.
"""
from __future__ import annotations

import dataclasses
import math

import torch

SEGMENT = 64  # tokens per re-emittable segment
RHO = 0.9     # AR(1) coefficient of the key walk


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    layers: int
    batch: int
    kv_heads: int
    gqa: int              # query heads per KV head (G)
    head_dim: int         # d
    dtype: str            # "bf16" or "fp32"
    n_cached: int         # N: merged cache length when the step runs
    budget: int           # rows kept per problem
    n_obs: int = 8
    lam: float = 0.1
    beta: int = 2
    tau: float = 0.9
    keys: str = "ar1"     # "ar1" (repeated-segment walk) or "gauss_dup"
    repeat_prob: float = 0.3
    copy_noise: float = 0.05
    seed: int = 1234
    # stream simulation only
    gen_tokens: int = 0   # tokens generated per sequence
    buffer: int = 128     # tokens generated between two compression rounds

    @property
    def problems(self) -> int:
        return self.layers * self.batch * self.kv_heads

    @property
    def torch_dtype(self) -> torch.dtype:
        return {"bf16": torch.bfloat16, "fp32": torch.float32}[self.dtype]

    def scaled(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads, in order: tiny, Llama-8B layer, Llama-8B full step,
# Qwen-14B large budget, sustained decode stream.
WORKLOADS = [
    Workload("tiny", layers=1, batch=1, kv_heads=2, gqa=4, head_dim=64, dtype="fp32",
             n_cached=96, budget=64, keys="gauss_dup", copy_noise=0.01, seed=1234),
    Workload("llama8b_layer", layers=1, batch=1, kv_heads=8, gqa=4, head_dim=128,
             dtype="bf16", n_cached=1152, budget=1024, seed=1235),
    Workload("llama8b_full", layers=32, batch=64, kv_heads=8, gqa=4, head_dim=128,
             dtype="bf16", n_cached=1152, budget=1024, seed=1236),
    Workload("qwen14b", layers=48, batch=16, kv_heads=8, gqa=5, head_dim=128,
             dtype="bf16", n_cached=4224, budget=4096, seed=1237),
    Workload("stream", layers=32, batch=32, kv_heads=8, gqa=4, head_dim=128,
             dtype="bf16", n_cached=1766, budget=1638, repeat_prob=0.4,
             gen_tokens=16384, buffer=128, seed=1238),
]
BY_NAME = {w.name: w for w in WORKLOADS}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


WALK_CHUNK = 128  # tokens per batched step of the walk


def _walk_matrices(n: int, device):
    """For the walk over n tokens after a known value x: the tokens are
    x_u = RHO^(u+1) * x + c * sum_{v <= u} RHO^(u-v) * e_v (u = 0..n-1, c =
    sqrt(1 - RHO^2)); returns the lower-triangular [n, n] matrix of the
    innovations' weights and the [n] weights of x (fp32)."""
    c = math.sqrt(1.0 - RHO * RHO)
    u = torch.arange(n, dtype=torch.float64)
    lag = u[:, None] - u[None, :]
    L = torch.where(lag >= 0, c * RHO ** lag.clamp(min=0), torch.zeros((), dtype=torch.float64))
    return L.float().to(device), (RHO ** (u + 1)).float().to(device)


def _ar1_walk_(k: torch.Tensor) -> torch.Tensor:
    """In place: k[:, 0] stays, k[:, t] = rho*k[:, t-1] + sqrt(1-rho^2)*k[:, t]
    (the incoming values are the innovations).  Stationary variance 1.
    Evaluated WALK_CHUNK tokens at a time in closed form (one batched matmul
    per chunk) rather than token by token."""
    T = k.shape[1]
    if T < 2:
        return k
    L, pw = _walk_matrices(min(WALK_CHUNK, T - 1), k.device)
    t0 = 1
    while t0 < T:
        n = min(WALK_CHUNK, T - t0)
        k[:, t0:t0 + n] = torch.matmul(L[:n, :n], k[:, t0:t0 + n]) + pw[:n, None] * k[:, t0 - 1:t0]
        t0 += n
    return k


def _reemit_segments_(k: torch.Tensor, first_seg: int, n_seg: int, prob: float,
                      noise: float, g: torch.Generator, history: torch.Tensor | None = None):
    """In place, for segments s = first_seg .. first_seg+n_seg-1 of k (positions
    relative to ``history`` when given): with probability ``prob`` replace the
    segment by a copy of a uniformly chosen earlier segment plus N(0, noise^2)
    noise.  Segments are processed in order, so a copy may copy a copy."""
    P, _, d = k.shape
    src_buf = k if history is None else history
    off = 0 if history is None else first_seg * SEGMENT
    ar = torch.arange(SEGMENT, device=k.device)
    for s in range(first_seg, first_seg + n_seg):
        if s == 0:
            continue
        hit = torch.rand(P, generator=g, device=k.device) < prob
        src = torch.floor(torch.rand(P, generator=g, device=k.device) * s).long().clamp_(max=s - 1)
        rows = (src[:, None] * SEGMENT + ar[None, :])  # [P, SEGMENT] into src_buf
        copy = torch.gather(src_buf, 1, rows[:, :, None].expand(P, SEGMENT, d)).float()
        copy += noise * torch.randn(P, SEGMENT, d, generator=g, device=k.device)
        lo = s * SEGMENT - off
        seg = k[:, lo:lo + SEGMENT]
        seg.copy_(torch.where(hit[:, None, None], copy.to(seg.dtype), seg))
        if history is not None:
            history[:, s * SEGMENT:(s + 1) * SEGMENT].copy_(seg.to(history.dtype))


def make_inputs(w: Workload, device="cpu", n_cap: int | None = None,
                problems: int | None = None, seed: int | None = None):
    """K, V [P, n_cap, d] and Q_obs [P, G, n_obs, d] in the workload's dtype.

    Rows n_cached..n_cap-1 (spare capacity) are filled with NaN so that any
    read past n_cached shows up.  ``problems`` overrides P (for scaled-down
    copies of a workload)."""
    P = w.problems if problems is None else problems
    N, d, G = w.n_cached, w.head_dim, w.gqa
    n_cap = N if n_cap is None else n_cap
    assert n_cap >= N
    g = _gen(w.seed if seed is None else seed, device)
    dt = w.torch_dtype
    if w.keys == "gauss_dup":
        # K, V, Q ~ N(0, 1); tokens 40..47 are noisy copies of tokens 10..17
        k = torch.randn(P, N, d, generator=g, device=device)
        v = torch.randn(P, N, d, generator=g, device=device)
        q = torch.randn(P, G, w.n_obs, d, generator=g, device=device)
        if N >= 48:
            k[:, 40:48] = k[:, 10:18] + w.copy_noise * torch.randn(
                P, 8, d, generator=g, device=device)
    else:
        k = torch.randn(P, N, d, generator=g, device=device)
        _ar1_walk_(k)
        _reemit_segments_(k, 0, N // SEGMENT, w.repeat_prob, w.copy_noise, g)
        v = torch.randn(P, N, d, generator=g, device=device)
        q = observation_queries(k[:, N - 1], G, w.n_obs, g)
    K = torch.full((P, n_cap, d), float("nan"), dtype=dt, device=device)
    V = torch.full((P, n_cap, d), float("nan"), dtype=dt, device=device)
    K[:, :N] = k.to(dt)
    V[:, :N] = v.to(dt)
    return K, V, q.to(dt).contiguous()


def observation_queries(k_last: torch.Tensor, G: int, n_obs: int,
                        g: torch.Generator) -> torch.Tensor:
    """Q_obs [P, G, n_obs, d]: for each query head an independent continuation
    of the AR(1) walk for n_obs steps from the last cached key."""
    P, d = k_last.shape
    L, pw = _walk_matrices(n_obs, k_last.device)
    e = torch.randn(P, G, n_obs, d, generator=g, device=k_last.device)
    return torch.matmul(L, e) + pw[:, None] * k_last.float()[:, None, None, :]


class StreamSource:
    """Key/value stream of the sustained decode workload: ``gen_tokens`` tokens
    per problem, produced ``buffer`` at a time.  The AR(1) walk runs across
    chunks; each completed 64-token segment may be re-emitted as a noisy copy
    of an earlier segment of the same problem, so the full key history is kept
    (in the workload's dtype) for the copies."""

    def __init__(self, w: Workload, device="cpu", problems: int | None = None,
                 seed: int | None = None):
        self.w = w
        self.P = w.problems if problems is None else problems
        self.device = device
        self.g = _gen(w.seed if seed is None else seed, device)
        self.t = 0
        self.prev = None  # last walk value [P, d] (fp32)
        self.history = torch.empty(self.P, w.gen_tokens, w.head_dim,
                                   dtype=w.torch_dtype, device=device)

    def next_chunk(self):
        """K, V chunks [P, buffer, d] of the next ``buffer`` tokens."""
        w, P, d, L = self.w, self.P, self.w.head_dim, self.w.buffer
        assert L % SEGMENT == 0 and self.t + L <= w.gen_tokens
        c = math.sqrt(1.0 - RHO * RHO)
        k = torch.randn(P, L, d, generator=self.g, device=self.device)
        if self.prev is None:
            _ar1_walk_(k)
        else:
            k[:, 0].mul_(c).add_(self.prev, alpha=RHO)
            _ar1_walk_(k)
        self.prev = k[:, -1].clone()
        v = torch.randn(P, L, d, generator=self.g, device=self.device)
        self.history[:, self.t:self.t + L] = k.to(self.history.dtype)
        _reemit_segments_(k, self.t // SEGMENT, L // SEGMENT, w.repeat_prob,
                          w.copy_noise, self.g, history=self.history)
        self.t += L
        return k.to(w.torch_dtype), v.to(w.torch_dtype)

    def queries(self, k_last: torch.Tensor) -> torch.Tensor:
        return observation_queries(k_last, self.w.gqa, self.w.n_obs, self.g).to(
            self.w.torch_dtype).contiguous()


def random_scores(P: int, N: int, device="cpu", seed: int = 7,
                  tie_levels: int = 0) -> torch.Tensor:
    """fp32 scores [P, N] for exercising a selection in isolation.  With
    ``tie_levels`` > 0 every value is one of that many levels, so exact ties
    are frequent."""
    g = _gen(seed, device)
    if tie_levels > 0:
        z = torch.randint(0, tie_levels, (P, N), generator=g, device=device).float()
        return z / tie_levels - 0.5
    return torch.randn(P, N, generator=g, device=device) * 0.01


def random_indices(P: int, n_cached: int, budget: int, device="cpu",
                   seed: int = 11) -> torch.Tensor:
    """Strictly ascending int32 index rows [P, budget] drawn uniformly from
    0..n_cached-1 (a random kept set, for exercising the copy alone)."""
    g = _gen(seed, device)
    keys = torch.rand(P, n_cached, generator=g, device=device)
    top = torch.topk(keys, budget, dim=1).indices
    return torch.sort(top, dim=1).values.to(torch.int32).contiguous()


# -------------------------------------------------------------- sentences --
# Stand-in for the sentence structure of a reasoning trace (SkipKV review,
# yoonschallenge.tistory.com/1230, row "Method 1": sentences split at
# newlines and punctuation, represented by mean last-layer hidden states;
# redundant reflections repeat earlier sentences).  Sentence lengths are drawn
# uniformly in [SENT_MIN, SENT_MAX] tokens; each sentence's hidden states are
# a random direction (shared by its tokens) plus per-token noise, and with
# probability SENT_REPEAT a sentence restates an earlier one (the earlier
# direction plus a small perturbation), so its mean representation is close
# to that sentence's.  HIDDEN_LLAMA8B is the model width of the Llama-8B
# configuration.
SENT_MIN, SENT_MAX = 8, 48
SENT_REPEAT = 0.3
SENT_TAU = 0.9
HIDDEN_LLAMA8B = 4096


@dataclasses.dataclass
class SentenceInputs:
    token_seg: torch.Tensor   # [S, T] int32, the sentence of each generated token
    hidden: torch.Tensor      # [S, T, hidden] per-token last-layer hidden states
    count: torch.Tensor       # [S] int32, sentences per sequence
    seg_id: torch.Tensor      # [P, N] int32, the sentence of each cached row
    max_sentences: int
    heads: int                # problem p belongs to sequence (p // heads) % S


def make_sentences(S: int, heads_per_seq: int, layers: int, N: int, hidden_dim: int,
                   device="cpu", seed: int = 11, dtype=torch.bfloat16) -> SentenceInputs:
    """Sentences for S sequences of N cached tokens, for P = layers * S *
    heads_per_seq problems ordered (layer, sequence, head)."""
    g = torch.Generator().manual_seed(seed)
    lengths = []
    for s in range(S):
        ls, total = [], 0
        while total < N:
            n = int(torch.randint(SENT_MIN, SENT_MAX + 1, (1,), generator=g))
            ls.append(min(n, N - total))
            total += ls[-1]
        lengths.append(ls)
    M = max(len(ls) for ls in lengths)
    token_seg = torch.full((S, N), -1, dtype=torch.int32)
    count = torch.tensor([len(ls) for ls in lengths], dtype=torch.int32)
    hidden = torch.empty((S, N, hidden_dim))
    for s, ls in enumerate(lengths):
        dirs = []
        t = 0
        for a, n in enumerate(ls):
            if a > 0 and float(torch.rand((1,), generator=g)) < SENT_REPEAT:
                src = int(torch.randint(0, a, (1,), generator=g))
                d = dirs[src] + 0.1 * torch.randn(hidden_dim, generator=g)
            else:
                d = torch.randn(hidden_dim, generator=g)
            dirs.append(d)
            token_seg[s, t:t + n] = a
            hidden[s, t:t + n] = d + 0.5 * torch.randn((n, hidden_dim), generator=g)
            t += n
    seg_id = token_seg.repeat_interleave(heads_per_seq, dim=0).repeat(layers, 1)
    return SentenceInputs(token_seg.to(device), hidden.to(dtype).to(device), count.to(device),
                          seg_id.contiguous().to(device), M, heads_per_seq)
