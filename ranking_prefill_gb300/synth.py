"""Seeded synthetic inputs for the MIS hot path.

This module draws the raw request shapes (prefix token counts, item counts,
item token counts) and the tensor values that both the CUDA path and the CPU
oracle consume. It holds none of the method's arithmetic: it does not pack
sequences, place delimiters, compute positions or masks. The caller gets the
packed length T from its own layout builder and passes it back in.

Recipe (the same for every consumer):
  * shapes: ``numpy.random.default_rng(seed)``, integer-uniform draws with
    inclusive bounds, in the order prefix lengths, item counts, item lengths,
    then label ids (distinct, uniform over the vocabulary);
  * values: a CPU ``torch.Generator`` seeded with ``seed``; fp32 normal draws in
    the order Q, K, V, hidden, W_lm, each rounded to bf16 (round to nearest
    even). Q, K, V and hidden are N(0, 1); W_lm is N(0, 0.02^2).

The "setwise" workload reads a draw as setwise prompts (query, candidates,
one marker per candidate; "Scaling JEV-like Decision Models with SGLang",
Benchmark: Fused-Choice vs. Setwise Scoring).

The five MIS workloads mirror the shapes of the pages' workloads: a long shared
member/profile prefix followed by many short candidate items ("From
Generation to Scoring", Section 6.1 Setup; "Turbocharging LinkedIn's
recommendation systems with SGLang", Results / Figure 3; "Scaling JEV-like
Decision Models with SGLang", Benchmark: Pointwise Decisions).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional, Tuple

import numpy as np


@dataclass(frozen=True)
class Workload:
    """Shape recipe of one synthetic MIS workload."""

    name: str
    seed: int
    batch: int
    prefix: Tuple[int, int]          # inclusive bounds on prefix tokens (excl. DELIM)
    n_items: Tuple[int, int]         # inclusive bounds on items per request
    item_len: Tuple[int, int]        # inclusive bounds on tokens per item (excl. DELIM)
    hq: int
    hkv: int
    head_dim: int
    d_model: int
    vocab: int
    label_sets: Tuple[int, ...] = (2,)   # K of each requested label set
    note: str = ""
    layout: str = "mis"              # "mis": packed MIS requests; "setwise": the same
                                     # lengths read as query / candidates, one marker each


WORKLOADS = {
    "tiny": Workload(
        "tiny", 1, 1, (128, 128), (8, 8), (16, 16), 4, 2, 64, 256, 1024, (2,),
        "batch 1, prefix 128, 8 items x 16 tokens, 265 packed tokens"),
    "qwen3-0.6b-layer": Workload(
        "qwen3-0.6b-layer", 2, 1, (1024, 1024), (100, 100), (24, 24), 16, 8, 128,
        1024, 151936, (2,),
        "batch 1, prefix 1024, 100 items x 24 tokens, Yes/No labels"),
    "varlen-16": Workload(
        "varlen-16", 3, 16, (512, 4096), (50, 500), (8, 64), 16, 8, 128, 1024,
        151936, (2,),
        "16 requests, prefix U[512,4096], items U[50,500] of U[8,64] tokens"),
    "8b-large": Workload(
        "8b-large", 4, 1, (2000, 2000), (500, 500), (32, 32), 32, 8, 128, 4096,
        151936, (2,),
        "batch 1, prefix 2000, 500 items x 32 tokens, d=4096"),
    "decision-256": Workload(
        "decision-256", 5, 256, (256, 256), (3, 10), (64, 64), 16, 8, 128, 1024,
        151936, (2, 3),
        "256 requests, prefix 256, U[3,10] items of 64 tokens, K=2 and K=3"),
    # "Turbocharging LinkedIn's recommendation systems with SGLang", Results /
    # Figure 3: one ranking request of a 12k-token prefix and 50 items of 150
    # tokens (the shape of the page's MIS against single-item scoring with
    # prefix caching); the page names no model, the qwen3-0.6b heads are used
    "prefix12k-50x150": Workload(
        "prefix12k-50x150", 7, 1, (12000, 12000), (50, 50), (150, 150), 16, 8, 128, 1024,
        151936, (2,), "batch 1, prefix 12000, 50 items x 150 tokens"),
    # decision-256's draw (same seed) as setwise prompts: the prefix lengths are
    # the query lengths and the items the candidates, followed by one marker each
    "setwise-256": Workload(
        "setwise-256", 5, 256, (256, 256), (3, 10), (64, 64), 16, 8, 128, 1024,
        151936, (2, 3),
        "decision-256's requests as setwise prompts: query 256, U[3,10] candidates of "
        "64 tokens, one marker per candidate, plain causal", layout="setwise"),
}

# Index order used by tests and the benchmark (1-based, matching the seeds).
WORKLOAD_ORDER = ["tiny", "qwen3-0.6b-layer", "varlen-16", "8b-large", "decision-256"]


@dataclass
class Shapes:
    """Raw per-request lengths plus the label ids, before any packing."""

    prefix_tokens: np.ndarray    # int32 [B]
    n_items: np.ndarray          # int32 [B]
    item_lens: np.ndarray        # int32 [sum n_items]
    label_sets: List[np.ndarray] = field(default_factory=list)  # int32 [K] each


def draw_shapes(w: Workload, seed: Optional[int] = None) -> Shapes:
    """Draw request shapes and label ids for workload ``w``."""
    rng = np.random.default_rng(w.seed if seed is None else seed)
    p = rng.integers(w.prefix[0], w.prefix[1] + 1, size=w.batch).astype(np.int32)
    n = rng.integers(w.n_items[0], w.n_items[1] + 1, size=w.batch).astype(np.int32)
    lens = rng.integers(w.item_len[0], w.item_len[1] + 1,
                        size=int(n.sum())).astype(np.int32)
    labels = [rng.choice(w.vocab, size=k, replace=False).astype(np.int32)
              for k in w.label_sets]
    return Shapes(p, n, lens, labels)


def custom_shapes(prefix_tokens, n_items, item_lens, labels=()) -> Shapes:
    """Wrap explicit lengths (used by small hand-written test cases)."""
    return Shapes(np.asarray(prefix_tokens, np.int32), np.asarray(n_items, np.int32),
                  np.asarray(item_lens, np.int32),
                  [np.asarray(l, np.int32) for l in labels])


def draw_values(seed: int, T: int, hq: int, hkv: int, head_dim: int,
                d_model: int = 0, vocab: int = 0, w_std: float = 0.02,
                want=("q", "k", "v", "hidden", "w_lm")):
    """Draw bf16 tensors (CPU) in the fixed order Q, K, V, hidden, W_lm.

    A tensor that is not in ``want`` is still drawn (so the stream position of
    the others never changes) unless everything after it is also unwanted.
    Returns a dict of CPU torch bf16 tensors: q [T,hq,D], k/v [T,hkv,D],
    hidden [T,d], w_lm [V,d].
    """
    import torch

    g = torch.Generator().manual_seed(int(seed))
    order = [("q", (T, hq, head_dim), 1.0), ("k", (T, hkv, head_dim), 1.0),
             ("v", (T, hkv, head_dim), 1.0), ("hidden", (T, d_model), 1.0),
             ("w_lm", (vocab, d_model), w_std)]
    last = max((i for i, (n, _, _) in enumerate(order) if n in want), default=-1)
    out = {}
    for i, (name, shape, std) in enumerate(order):
        if i > last:
            break
        if 0 in shape:
            out[name] = torch.empty(shape, dtype=torch.bfloat16)
            continue
        x = torch.randn(shape, generator=g, dtype=torch.float32)
        if std != 1.0:
            x.mul_(std)
        t = x.to(torch.bfloat16)
        del x
        if name in want:
            out[name] = t
    return out


def shard_requests(n_requests: int, rank: int, world: int) -> np.ndarray:
    """Requests handled by ``rank`` when independent requests are split over ranks.

    Contiguous blocks, sizes differing by at most one. Requests are
    independent under the MIS mask (no attention crosses a request), so the
    split needs no exchange between ranks.
    """
    if world <= 0 or not (0 <= rank < world):
        raise ValueError("bad rank/world")
    base, extra = divmod(n_requests, world)
    start = rank * base + min(rank, extra)
    stop = start + base + (1 if rank < extra else 0)
    return np.arange(start, stop, dtype=np.int64)


# ---------------------------------------------------------------------------
# Request-size sweep ("From Generation to Scoring", Section 6.4, RQ3 and
# Figure 6): members with one query each and 200 candidates each; for a given
# N every member's candidates are split, in order, into requests of N items,
# and each request carries the member's whole query. Query lengths follow
# Section 6.1's workload (mean 744, median 543, 95th percentile 2,047 tokens):
# log-normal with median 543 and sigma = sqrt(2 ln(744 / 543)), which puts
# its 95th percentile at about 2,000. Members take the distribution's
# quantiles at (i + 1/2) / members (a stratified draw: 16 members already
# give mean 721 and median 544); candidates are nearly constant, U[24, 32]
# tokens (mean 28), drawn from the seed.
# ---------------------------------------------------------------------------

SWEEP_CANDIDATES = 200
SWEEP_N = (1, 2, 5, 10, 20, 50, 100, 200)


@dataclass
class SweepPool:
    query_tokens: np.ndarray     # int32 [members]
    cand_lens: np.ndarray        # int32 [members, SWEEP_CANDIDATES]
    labels: np.ndarray           # int32 [2]


def sweep_pool(members: int, vocab: int = 151936, seed: int = 6) -> SweepPool:
    from statistics import NormalDist
    rng = np.random.default_rng(seed)
    sigma = float(np.sqrt(2.0 * np.log(744.0 / 543.0)))
    z = np.array([NormalDist().inv_cdf((i + 0.5) / members) for i in range(members)])
    q = np.clip(np.rint(543.0 * np.exp(sigma * z)), 1, 16384)
    c = rng.integers(24, 32 + 1, size=(members, SWEEP_CANDIDATES))
    labels = rng.choice(vocab, size=2, replace=False)
    return SweepPool(q.astype(np.int32), c.astype(np.int32), labels.astype(np.int32))


def sweep_shapes(pool: SweepPool, n: int) -> Shapes:
    """The pool as requests of ``n`` items each (``n`` divides 200)."""
    if SWEEP_CANDIDATES % n:
        raise ValueError("N must divide the candidate count")
    per = SWEEP_CANDIDATES // n
    prefix = np.repeat(pool.query_tokens, per).astype(np.int32)
    n_items = np.full(len(prefix), n, np.int32)
    return Shapes(prefix, n_items, pool.cand_lens.reshape(-1).astype(np.int32), [pool.labels])
