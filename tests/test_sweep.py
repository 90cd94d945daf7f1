"""Request-size sweep inputs ("From Generation to Scoring", Section 6.4).

CPU checks: the split of each member's candidates into requests of N items,
the prefill-token ratio the benchmark reports against eq. (5) as the oracle
computes it, and the packed layouts of the split against the oracle.
"""
import numpy as np
import pytest

import oracle as O
from ranking_prefill_gb300 import lib, synth


@pytest.mark.parametrize("n", synth.SWEEP_N)
def test_split_keeps_every_candidate_once_in_order(n):
    pool = synth.sweep_pool(3)
    s = synth.sweep_shapes(pool, n)
    per = synth.SWEEP_CANDIDATES // n
    assert len(s.prefix_tokens) == 3 * per and (s.n_items == n).all()
    assert np.array_equal(s.prefix_tokens, np.repeat(pool.query_tokens, per))
    assert np.array_equal(s.item_lens, pool.cand_lens.reshape(-1))


def test_token_ratio_is_eq5():
    # one member, all 200 candidates in one request against 200 single-item
    # requests: the benchmark's raw-token ratio is eq. (5)'s R(200)
    pool = synth.sweep_pool(1)
    s1, s200 = synth.sweep_shapes(pool, 1), synth.sweep_shapes(pool, 200)
    raw = lambda s: int(s.prefix_tokens.sum()) + int(s.item_lens.sum())
    r = raw(s1) / raw(s200)
    assert abs(r - O.cost_ratio(int(pool.query_tokens[0]), pool.cand_lens[0])) < 1e-12


def test_query_length_distribution_matches_the_pages_figures():
    # Section 6.1: mean 744, median 543, 95th percentile 2,047 tokens
    q = synth.sweep_pool(200000).query_tokens
    assert abs(np.median(q) - 543) / 543 < 0.02
    assert abs(q.mean() - 744) / 744 < 0.02
    assert abs(np.percentile(q, 95) - 2047) / 2047 < 0.05
    assert abs(synth.sweep_pool(50000).cand_lens.mean() - 28) < 0.1


@pytest.mark.parametrize("n", [1, 20, 200])
def test_sweep_layouts_bit_exact(n):
    s = synth.sweep_shapes(synth.sweep_pool(2), n)
    got = lib.mis_build_layout(s.prefix_tokens, s.n_items, s.item_lens)
    ref = O.build_layout(s.prefix_tokens, s.n_items, s.item_lens)
    for f in ("cu_seqlens", "prefix_len", "item_ptr", "item_offsets", "delim_positions",
              "position_ids"):
        assert np.array_equal(getattr(got, f), getattr(ref, f)), f
