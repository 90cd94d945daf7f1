"""Pins for the fp64 oracle: checks against what the pages and the mathematics
fix, never against the oracle's own formula retyped.

* layout: Figure 2's reconstructed mask and position ids (golden fixture),
  the 265-token total of the tiny workload, the pages' position-id rules;
* mask: literal set enumeration on every tiny layout, and a closed-form count
  of visible pairs;
* attention: single-item-scoring equivalence, permutation invariance, the
  N <= 1 reduction to PyTorch's causal SDPA, and closed forms (zero queries
  give the mean of the visible values, constant values pass through, the
  first row returns its own value);
* scoring: PyTorch's log_softmax, W_lm = 0 gives -ln V, probabilities sum to
  one, eq. (2) for two labels;
* tiles: classification against the brute-force mask;
* eq. (5): the pages' printed workload numbers.
"""
import itertools
import math
import os

import numpy as np
import pytest
import torch

import oracle as O
from ranking_prefill_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    sections, cur = {}, None
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line.isalpha() or line.replace("_", "").isalpha():
                cur = line
                sections[cur] = []
            else:
                sections[cur].append(line)
    return sections


def _f64(t):
    return t.to(torch.float64).numpy()


def _rand(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g, dtype=torch.float32).to(torch.bfloat16)


# ---------------------------------------------------------------- layout ----

def test_figure2_mask_and_positions():
    g = _read_golden("fig2_mask.txt")
    want = np.array([[c == "1" for c in row] for row in g["mask"]])
    lay = O.build_layout([3], [3], [1, 1, 1])
    assert lay.T == 10
    assert (O.mask_bruteforce(lay) == want).all()
    assert (O.mask_rows(lay, 0, np.arange(10)) == want).all()
    assert lay.position_ids.tolist() == [int(x) for x in g["position_ids"][0].split()]
    assert lay.delim_positions.tolist() == [int(x) for x in g["readout_rows"][0].split()]


def test_tiny_workload_total_is_265():
    w = synth.WORKLOADS["tiny"]
    s = synth.draw_shapes(w)
    lay = O.build_layout(s.prefix_tokens, s.n_items, s.item_lens)
    assert lay.T == 265 and lay.M == 8
    assert lay.prefix_len.tolist() == [129]


def test_position_ids_follow_the_pages_rules():
    # every item starts at position |Q| and the largest id is |Q| + longest item set - 1
    s = synth.custom_shapes([5, 0, 7], [3, 2, 0], [2, 0, 4, 1, 3])
    lay = O.build_layout(s.prefix_tokens, s.n_items, s.item_lens)
    for b in range(lay.B):
        s0, S = lay.cu_seqlens[b], lay.prefix_len[b]
        assert lay.position_ids[s0:s0 + S].tolist() == list(range(S))
        segs = range(lay.item_ptr[b], lay.item_ptr[b + 1])
        for i in segs:
            a, e = lay.item_offsets[i], lay.item_ends[i]
            assert lay.position_ids[a:e].tolist() == list(range(S, S + e - a))
            assert lay.delim_positions[i] == e - 1
        if len(segs):
            longest = max(lay.item_ends[i] - lay.item_offsets[i] for i in segs)
            e0 = lay.cu_seqlens[b + 1]
            assert lay.position_ids[s0:e0].max() == S + longest - 1


def _tiny_layouts():
    for B in (1, 2):
        for ps in itertools.product(range(0, 3), repeat=B):
            for ns in itertools.product(range(0, 3), repeat=B):
                n = sum(ns)
                for lens in itertools.product(range(0, 3), repeat=n):
                    yield O.build_layout(ps, ns, lens)


def test_mask_matches_set_enumeration_on_all_tiny_layouts():
    count = 0
    for lay in _tiny_layouts():
        dense = O.mask_bruteforce(lay)
        for b in range(lay.B):
            s0, e0 = lay.cu_seqlens[b], lay.cu_seqlens[b + 1]
            got = O.mask_rows(lay, b, np.arange(s0, e0))
            assert (got == dense[s0:e0, s0:e0]).all()
            # nothing crosses a request
            assert not dense[s0:e0, :s0].any() and not dense[s0:e0, e0:].any()
        count += 1
    assert count > 500


def test_mask_matches_set_enumeration_on_sampled_small_layouts():
    # beyond the exhaustive sweep: 400 seeded layouts with up to 3 requests,
    # shared sets of up to 8 rows (prefix <= 7 plus its DELIM), up to 4 items
    # of up to 4 tokens; the interval form, the set enumeration and the
    # closed-form pair count agree on every one
    rng = np.random.default_rng(2024)
    for _ in range(400):
        B = int(rng.integers(1, 4))
        ps = rng.integers(0, 8, B).tolist()
        ns = rng.integers(0, 5, B).tolist()
        lens = rng.integers(0, 5, sum(ns)).tolist()
        lay = O.build_layout(ps, ns, lens)
        dense = O.mask_bruteforce(lay)
        for b in range(lay.B):
            s0, e0 = lay.cu_seqlens[b], lay.cu_seqlens[b + 1]
            assert (O.mask_rows(lay, b, np.arange(s0, e0)) == dense[s0:e0, s0:e0]).all()
        assert int(dense.sum()) == O.pair_count(lay) == _pairs_closed_form(ps, ns, lens)


def _pairs_closed_form(prefix_tokens, n_items, item_lens):
    # S(S+1)/2 for the causal query block, then per item set of n = L+1
    # tokens: n*S (whole query) + n(n+1)/2 (causal inside the item).
    tot, it = 0, 0
    for p, n in zip(prefix_tokens, n_items):
        S = p + 1
        tot += S * (S + 1) // 2
        for _ in range(n):
            m = item_lens[it] + 1
            tot += m * S + m * (m + 1) // 2
            it += 1
    return tot


@pytest.mark.parametrize("name,expect", [("tiny", 27153), ("qwen3-0.6b-layer", 3120825),
                                         ("8b-large", 35300001)])
def test_pair_count_closed_form(name, expect):
    s = synth.draw_shapes(synth.WORKLOADS[name])
    assert _pairs_closed_form(s.prefix_tokens, s.n_items, s.item_lens) == expect
    if name != "8b-large":          # the oracle count itself (8b-large: 18.5K^2 entries)
        lay = O.build_layout(s.prefix_tokens, s.n_items, s.item_lens)
        assert O.pair_count(lay) == expect


def test_pair_count_random_layouts():
    rng = np.random.default_rng(7)
    for _ in range(20):
        B = int(rng.integers(1, 4))
        p = rng.integers(0, 40, B)
        n = rng.integers(0, 6, B)
        lens = rng.integers(0, 20, int(n.sum()))
        lay = O.build_layout(p, n, lens)
        assert O.pair_count(lay) == _pairs_closed_form(p, n, lens)


# ------------------------------------------------------------- attention ----

def _qkv(T, hq, hkv, D, seed):
    v = synth.draw_values(seed, T, hq, hkv, D, want=("q", "k", "v"))
    return _f64(v["q"]), _f64(v["k"]), _f64(v["v"])


def _interval_visible(lay, j):
    """Visible keys of row j written from the interval description of eq. (4)."""
    b = lay.request_of[j]
    s0, S = int(lay.cu_seqlens[b]), int(lay.prefix_len[b])
    if j < s0 + S:
        return np.arange(s0, j + 1)
    i = lay.item_of[j]
    return np.concatenate([np.arange(s0, s0 + S), np.arange(lay.item_offsets[i], j + 1)])


def test_single_item_scoring_equivalence():
    # MIS rows of item i == the item rows of causal attention on [q; c_i] alone
    s = synth.custom_shapes([20, 9], [4, 3], [5, 0, 11, 3, 7, 2, 6])
    lay = O.build_layout(s.prefix_tokens, s.n_items, s.item_lens)
    q, k, v = _qkv(lay.T, 4, 2, 16, 11)
    o, lse = O.attention(q, k, v, lay)
    for i in range(lay.M):
        b = lay.request_of[lay.item_offsets[i]]
        s0, S = lay.cu_seqlens[b], lay.prefix_len[b]
        idx = np.concatenate([np.arange(s0, s0 + S), np.arange(lay.item_offsets[i], lay.item_ends[i])])
        sis = O.causal_layout([len(idx)])
        o2, lse2 = O.attention(q[idx], k[idx], v[idx], sis)
        n = lay.item_ends[i] - lay.item_offsets[i]
        np.testing.assert_allclose(o[lay.item_offsets[i]:lay.item_ends[i]], o2[-n:], rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[lay.item_offsets[i]:lay.item_ends[i]], lse2[-n:], rtol=0, atol=1e-12)
        np.testing.assert_allclose(o[s0:s0 + S], o2[:S], rtol=0, atol=1e-12)


def test_item_permutation_permutes_outputs():
    lens = [4, 9, 1, 6, 3]
    s = synth.custom_shapes([13], [5], lens)
    lay = O.build_layout(s.prefix_tokens, s.n_items, s.item_lens)
    q, k, v = _qkv(lay.T, 2, 1, 8, 3)
    o, _ = O.attention(q, k, v, lay)
    perm = [3, 0, 4, 2, 1]
    lay2 = O.build_layout([13], [5], [lens[p] for p in perm])
    gather = np.concatenate([np.arange(14)] + [np.arange(lay.item_offsets[p], lay.item_ends[p]) for p in perm])
    o2, _ = O.attention(q[gather], k[gather], v[gather], lay2)
    np.testing.assert_allclose(o2, o[gather], rtol=0, atol=1e-12)


@pytest.mark.parametrize("n_items", [0, 1])
def test_single_item_and_no_item_reduce_to_causal_sdpa(n_items):
    lens = [7][:n_items]
    s = synth.custom_shapes([30, 5], [n_items, n_items], lens * 2)
    lay = O.build_layout(s.prefix_tokens, s.n_items, s.item_lens)
    hq, hkv, D = 6, 3, 16
    q, k, v = _qkv(lay.T, hq, hkv, D, 5)
    o, lse = O.attention(q, k, v, lay)
    for b in range(lay.B):
        s0, e0 = lay.cu_seqlens[b], lay.cu_seqlens[b + 1]
        tq = torch.from_numpy(q[s0:e0]).permute(1, 0, 2)
        tk = torch.from_numpy(k[s0:e0]).permute(1, 0, 2).repeat_interleave(hq // hkv, 0)
        tv = torch.from_numpy(v[s0:e0]).permute(1, 0, 2).repeat_interleave(hq // hkv, 0)
        ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=True)
        np.testing.assert_allclose(o[s0:e0], ref.permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)
        # LSE from PyTorch's own logsumexp of the causal scores
        sc = (tq @ tk.transpose(1, 2)) / math.sqrt(D)
        sc = sc.masked_fill(torch.ones(e0 - s0, e0 - s0, dtype=torch.bool).triu(1), float("-inf"))
        np.testing.assert_allclose(lse[s0:e0], torch.logsumexp(sc, -1).T.numpy(), rtol=0, atol=1e-12)


def test_closed_forms():
    s = synth.custom_shapes([17, 4], [3, 2], [6, 0, 9, 2, 5])
    lay = O.build_layout(s.prefix_tokens, s.n_items, s.item_lens)
    _, k, v = _qkv(lay.T, 4, 2, 8, 9)
    # zero queries: uniform weights, output = mean of visible values, lse = ln |A(j)|
    q0 = np.zeros((lay.T, 4, 8))
    o, lse = O.attention(q0, k, v, lay)
    for j in range(lay.T):
        A = _interval_visible(lay, j)
        for h in range(4):
            np.testing.assert_allclose(o[j, h], v[A, h // 2].mean(axis=0), rtol=0, atol=1e-13)
            assert abs(lse[j, h] - math.log(len(A))) < 1e-13
    # constant values pass through unchanged
    q, _, _ = _qkv(lay.T, 4, 2, 8, 10)
    vc = np.full_like(v, 0.375)
    o, _ = O.attention(q, k, vc, lay)
    np.testing.assert_allclose(o, 0.375, rtol=0, atol=1e-14)
    # the first row of each request sees only itself
    o, lse = O.attention(q, k, v, lay)
    for b in range(lay.B):
        s0 = lay.cu_seqlens[b]
        for h in range(4):
            assert (o[s0, h] == v[s0, h // 2]).all()
            assert abs(lse[s0, h] - q[s0, h] @ k[s0, h // 2] / math.sqrt(8)) < 1e-13


def test_scale_override():
    lay = O.build_layout([6], [2], [3, 2])
    q, k, v = _qkv(lay.T, 2, 2, 4, 1)
    o1, _ = O.attention(q * 2.0, k, v, lay, scale=0.25)
    o2, _ = O.attention(q, k, v, lay, scale=0.5)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-14)


def test_row_sampling_matches_full():
    s = synth.custom_shapes([40], [6], [10, 3, 20, 5, 1, 8])
    lay = O.build_layout(s.prefix_tokens, s.n_items, s.item_lens)
    q, k, v = _qkv(lay.T, 4, 2, 8, 4)
    o, lse = O.attention(q, k, v, lay)
    rows = [0, 5, 41, 77, lay.T - 1]
    o2, lse2 = O.attention(q, k, v, lay, rows=rows)
    assert (o2 == o[rows]).all() and (lse2 == lse[rows]).all()


# --------------------------------------------------------------- scoring ----

def test_label_scores_match_torch_log_softmax():
    T, d, V = 50, 32, 300
    h = _f64(_rand((T, d), 1))
    W = _f64(_rand((V, d), 2)) * 0.3
    rows = [3, 17, 49, 0]
    labels = [7, 299, 0, 7]       # caller order kept, duplicates allowed
    lp, ren, lse = O.label_scores(h, W, rows, labels)
    ref = torch.log_softmax(torch.from_numpy(h[rows]) @ torch.from_numpy(W).T, dim=-1)
    np.testing.assert_allclose(lp, ref[:, labels].numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, torch.logsumexp(torch.from_numpy(h[rows]) @ torch.from_numpy(W).T, -1).numpy(),
                               rtol=0, atol=1e-12)
    refr = torch.softmax(torch.from_numpy(h[rows]) @ torch.from_numpy(W[labels]).T, dim=-1)
    np.testing.assert_allclose(ren, refr.numpy(), rtol=0, atol=1e-12)


def test_label_scores_closed_forms():
    T, d, V = 10, 16, 257
    h = _f64(_rand((T, d), 3))
    lp, ren, _ = O.label_scores(h, np.zeros((V, d)), [1, 2], [5, 6])
    np.testing.assert_allclose(lp, -math.log(V), rtol=0, atol=1e-14)
    np.testing.assert_allclose(ren, 0.5, rtol=0, atol=1e-15)
    W = _f64(_rand((V, d), 4))
    lp, _, _ = O.label_scores(h, W, [0, 9], list(range(V)))
    np.testing.assert_allclose(np.exp(lp).sum(axis=1), 1.0, rtol=0, atol=1e-12)
    # eq. (2): two-label renormalisation is the logistic of the logit gap
    lp, ren, _ = O.label_scores(h, W, [4], [11, 200])
    gap = h[4] @ W[11] - h[4] @ W[200]
    assert abs(ren[0, 0] - 1.0 / (1.0 + math.exp(-gap))) < 1e-14
    assert abs(ren[0, 0] + ren[0, 1] - 1.0) < 1e-15


def test_label_scores_item_subset():
    h = _f64(_rand((20, 8), 5))
    W = _f64(_rand((40, 8), 6))
    rows = [1, 5, 9, 12]
    full = O.label_scores(h, W, rows, [3, 4])
    sub = O.label_scores(h, W, rows, [3, 4], items=[2, 0])
    assert (sub[0] == full[0][[2, 0]]).all()


# ------------------------------------------------------------------ tiles ----

def _tiles_from_dense(lay, BM, BN):
    dense = O.mask_bruteforce(lay)
    out = []
    for b in range(lay.B):
        s0, e0 = lay.cu_seqlens[b], lay.cu_seqlens[b + 1]
        for t, r0 in enumerate(range(s0, e0, BM)):
            for u, c0 in enumerate(range(s0, e0, BN)):
                blk = dense[r0:min(r0 + BM, e0), c0:min(c0 + BN, e0)]
                if blk.any():
                    out.append((b, t, u, O.FULL if blk.all() else O.PARTIAL))
    return np.asarray(out, np.int32).reshape(-1, 4)


@pytest.mark.parametrize("BM,BN", [(4, 4), (4, 8), (8, 4), (3, 5)])
def test_tile_map_vs_dense(BM, BN):
    rng = np.random.default_rng(BM * 10 + BN)
    for _ in range(25):
        B = int(rng.integers(1, 3))
        p = rng.integers(0, 12, B)
        n = rng.integers(0, 5, B)
        lens = rng.integers(0, 7, int(n.sum()))
        lay = O.build_layout(p, n, lens)
        assert (O.tile_map(lay, BM, BN) == _tiles_from_dense(lay, BM, BN)).all()


# ------------------------------------------------------------- cost model ----

def test_cost_ratio_against_printed_workload_numbers():
    g = {}
    with open(os.path.join(GOLDEN, "cost_model.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                key, val, tol = line.split()
                g[key] = (float(val), float(tol))
    Lq, Li, N = int(g["query_mean_tokens"][0]), int(g["item_mean_tokens"][0]), int(g["n_items"][0])
    def close(key, x):
        val, tol = g[key]
        assert abs(x - val) <= tol * val + 1e-9, (key, x, val)
    close("mis_request_tokens", Lq + N * Li)
    close("independent_tokens", N * (Lq + Li))
    close("r_200", O.cost_ratio(Lq, [Li] * N))
    close("tokens_per_label_independent", Lq + Li)
    close("tokens_per_label_mis", (Lq + N * Li) / N)
    # the two printed forms of eq. (5) agree: N(1 + rho) / (N + rho), rho = Lq / mean(L)
    rng = np.random.default_rng(0)
    for _ in range(10):
        lens = rng.integers(1, 60, int(rng.integers(1, 300)))
        rho = 700 / lens.mean()
        n = len(lens)
        assert abs(O.cost_ratio(700, lens) - n * (1 + rho) / (n + rho)) < 1e-9
    assert O.cost_ratio(500, [30]) == 1.0      # one item: nothing to share


# ------------------------------------------------------------------ setwise ----

def _setwise_golden():
    g = {}
    with open(os.path.join(GOLDEN, "setwise_example.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                key, *vals = line.split()
                g[key] = vals
    return g


def test_setwise_layout_follows_the_pages_example():
    # three options A, B, C, then one marker per option; one score row per
    # marker, in option order, every marker after the whole option list
    g = _setwise_golden()
    n = int(g["candidates"][0])
    assert int(g["markers"][0]) == n and len(g["row_order"]) == n
    q, lens = 40, [7, 12, 9]
    sl = O.setwise_layout([q], [n], lens)
    assert sl.M == n
    cand_end = sl.cand_offsets[-1] + lens[-1]
    assert int(g["marker_rows_after_last_candidate"][0]) == 1
    assert (sl.marker_positions >= cand_end).all()                 # after the whole list
    assert list(sl.marker_positions) == sorted(sl.marker_positions)  # A, B, C in order
    assert sl.causal.T == q + sum(lens) + n
    # candidate i starts where the text before it ends
    starts = q + np.concatenate([[0], np.cumsum(lens)[:-1]])
    assert list(sl.cand_offsets) == list(starts)
    # every marker sees every candidate token (plain causal: no isolation)
    for m in sl.marker_positions:
        vis = O.mask_rows(sl.causal, 0, np.array([m]))[0]
        assert vis[: cand_end].all()


def test_setwise_attention_is_plain_causal_sdpa():
    sl = O.setwise_layout([11, 0, 5], [3, 2, 0], [4, 0, 6, 3, 2])
    hq, hkv, D = 4, 2, 16
    q, k, v = _qkv(sl.causal.T, hq, hkv, D, 31)
    o, _ = O.attention(q, k, v, sl.causal)
    cu = sl.causal.cu_seqlens
    for b in range(sl.causal.B):
        s0, e0 = cu[b], cu[b + 1]
        tq = torch.from_numpy(q[s0:e0]).permute(1, 0, 2)
        tk = torch.from_numpy(k[s0:e0]).permute(1, 0, 2).repeat_interleave(hq // hkv, 0)
        tv = torch.from_numpy(v[s0:e0]).permute(1, 0, 2).repeat_interleave(hq // hkv, 0)
        ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=True)
        np.testing.assert_allclose(o[s0:e0], ref.permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)


def test_setwise_markers_read_every_candidate_unlike_mis():
    # Changing candidate 1's values moves every marker's output in setwise,
    # while under MIS only item 1's own rows move (eq. 4 isolates items).
    q_t, lens = 9, [5, 6, 4]
    sl = O.setwise_layout([q_t], [3], lens)
    hq, hkv, D = 2, 1, 8
    q, k, v = _qkv(sl.causal.T, hq, hkv, D, 32)
    o1, _ = O.attention(q, k, v, sl.causal)
    v2 = v.copy()
    a = sl.cand_offsets[1]
    v2[a:a + lens[1]] += 1.0
    o2, _ = O.attention(q, k, v2, sl.causal)
    moved = np.abs(o2 - o1).max(axis=(1, 2)) > 1e-9
    assert moved[sl.marker_positions].all()
    assert not moved[:a].any()                       # causal: rows before candidate 1 unchanged
    lay = O.build_layout([q_t], [3], lens)
    qm, km, vm = _qkv(lay.T, hq, hkv, D, 33)
    m1, _ = O.attention(qm, km, vm, lay)
    vm2 = vm.copy()
    vm2[lay.item_offsets[1]:lay.item_ends[1]] += 1.0
    m2, _ = O.attention(qm, km, vm2, lay)
    moved = np.abs(m2 - m1).max(axis=(1, 2)) > 1e-9
    assert moved[lay.delim_positions[1]] and not moved[lay.delim_positions[[0, 2]]].any()


def test_setwise_layout_rejects_bad_requests():
    with pytest.raises(ValueError):
        O.setwise_layout([0], [0], [])                  # empty request
    with pytest.raises(ValueError):
        O.setwise_layout([3], [2], [1])                 # inconsistent counts


# --------------------------------------------------------------------- rope ----

def test_rope_closed_forms():
    x = np.zeros((3, 1, 2))
    x[:, 0, 0] = 1.0
    r = O.rope(x, [0, 1, 5], base=123.0)          # D = 2: one pair, frequency base^0 = 1
    np.testing.assert_allclose(r[:, 0, 0], np.cos([0.0, 1.0, 5.0]), atol=1e-15)
    np.testing.assert_allclose(r[:, 0, 1], np.sin([0.0, 1.0, 5.0]), atol=1e-15)
    y = np.random.default_rng(3).standard_normal((4, 2, 16))
    np.testing.assert_array_equal(O.rope(y, [0, 0, 0, 0]), y)          # position 0: identity


def test_rope_is_a_rotation_by_position():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((6, 3, 32))
    a, b = rng.integers(0, 5000, 6), rng.integers(0, 5000, 6)
    # composing turns adds positions; each (i, i + D/2) pair keeps its length
    np.testing.assert_allclose(O.rope(O.rope(x, a), b), O.rope(x, a + b), atol=1e-9)
    r = O.rope(x, a)
    np.testing.assert_allclose(r[..., :16] ** 2 + r[..., 16:] ** 2,
                               x[..., :16] ** 2 + x[..., 16:] ** 2, atol=1e-12)
    # the same turn written with complex numbers: (x1 + i x2) * exp(i p f)
    f = 1.0e6 ** (-2.0 * np.arange(16) / 32)
    z = (x[..., :16] + 1j * x[..., 16:]) * np.exp(1j * a[:, None, None] * f)
    np.testing.assert_allclose(r, np.concatenate([z.real, z.imag], -1), atol=1e-9)


def test_rope_scores_depend_on_relative_position_only():
    rng = np.random.default_rng(5)
    q, k = rng.standard_normal((1, 1, 64)), rng.standard_normal((1, 1, 64))
    for p, pk, shift in [(10, 3, 700), (900, 900, 12345), (5, 40, 2)]:
        s1 = (O.rope(q, [p]) * O.rope(k, [pk])).sum()
        s2 = (O.rope(q, [p + shift]) * O.rope(k, [pk + shift])).sum()
        s3 = (O.rope(q, [p - pk]) * k).sum()
        assert abs(s1 - s2) < 1e-9 and abs(s1 - s3) < 1e-9


def test_mis_equals_sis_only_with_reused_positions():
    # Section 4.1: the mask alone is not enough; with the reused position ids
    # every item's rows equal those of its own [q; item] prompt
    s = synth.custom_shapes([20], [3], [5, 7, 4])
    lay = O.build_layout(s.prefix_tokens, s.n_items, s.item_lens)
    hq, hkv, D = 2, 1, 16
    q, k, v = _qkv(lay.T, hq, hkv, D, 41)
    o_reuse, _ = O.attention(O.rope(q, lay.position_ids), O.rope(k, lay.position_ids), v, lay)
    packed = np.arange(lay.T)
    o_packed, _ = O.attention(O.rope(q, packed), O.rope(k, packed), v, lay)
    S = int(lay.prefix_len[0])
    for i in range(lay.M):
        rows = np.concatenate([np.arange(S), np.arange(lay.item_offsets[i], lay.item_ends[i])])
        one = O.causal_layout([len(rows)])
        pos = np.arange(len(rows))
        o1, _ = O.attention(O.rope(q[rows], pos), O.rope(k[rows], pos), v[rows], one)
        np.testing.assert_allclose(o_reuse[rows[S:]], o1[S:], rtol=0, atol=1e-12)
        if i > 0:   # a later item at packed positions sees the query from farther away
            assert np.abs(o_packed[rows[S:]] - o1[S:]).max() > 1e-6


# --------------------------------------------------------- cached prefix ----

def _cached_case(seed):
    rng = np.random.default_rng(seed)
    B = 3
    P = rng.integers(1, 60, B)                   # prefix tokens (without DELIM)
    n = rng.integers(1, 5, B)
    lens = rng.integers(0, 9, int(n.sum()))
    S = P + 1
    # prefixes stored back to back in the cache, in reverse order, with a gap
    cstart = np.zeros(B, np.int64)
    t = 3
    for b in reversed(range(B)):
        cstart[b] = t
        t += S[b] + 2
    return P, n, lens, S, cstart, t


def test_cached_prefix_attention_equals_packed_mis():
    # the same prefixes and items packed as MIS requests: identical item rows
    P, n, lens, S, cstart, cache_T = _cached_case(61)
    hq, hkv, D = 4, 2, 16
    packed = O.build_layout(P, n, lens)
    q, k, v = _qkv(packed.T, hq, hkv, D, 62)
    cl = O.cached_layout(cstart, S, n, lens)
    kc = np.zeros((cache_T, hkv, D)); vc = np.zeros((cache_T, hkv, D))
    item_rows = []
    for b in range(packed.B):
        s0 = packed.cu_seqlens[b]
        kc[cstart[b]:cstart[b] + S[b]] = k[s0:s0 + S[b]]
        vc[cstart[b]:cstart[b] + S[b]] = v[s0:s0 + S[b]]
        item_rows.append(np.arange(s0 + S[b], packed.cu_seqlens[b + 1]))
    item_rows = np.concatenate(item_rows)
    assert len(item_rows) == cl.T
    ref, ref_lse = O.attention(q, k, v, packed, rows=item_rows)
    got, got_lse = O.attention_cached(q[item_rows], k[item_rows], v[item_rows], kc, vc, cl)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(got_lse, ref_lse, rtol=0, atol=1e-12)
    assert np.array_equal(cl.position_ids, packed.position_ids[item_rows])
    assert np.array_equal(item_rows[cl.delim_positions], packed.delim_positions)


def test_single_item_requests_over_one_cached_prefix_equal_mis():
    # "single-item scoring with prefix caching": every item its own request
    # over the same cached prefix gives the MIS item rows again
    S, lens = 30, [4, 0, 7]
    hq, hkv, D = 2, 1, 8
    cl = O.cached_layout([0], [S], [3], lens)
    one = O.cached_layout([0, 0, 0], [S, S, S], [1, 1, 1], lens)
    q, k, v = _qkv(cl.T, hq, hkv, D, 63)
    kc, vc, _ = _qkv(S, hq, hkv, D, 64)
    kc, vc = kc[:, :hkv], vc[:, :hkv]
    a, _ = O.attention_cached(q, k, v, kc, vc, cl)
    b, _ = O.attention_cached(q, k, v, kc, vc, one)
    np.testing.assert_array_equal(a, b)


def test_cached_layout_rejects_bad_requests():
    with pytest.raises(ValueError):
        O.cached_layout([0], [0], [1], [3])        # no cached prefix
    with pytest.raises(ValueError):
        O.cached_layout([0], [4], [0], [])         # no item


# ------------------------------------------------- cached-prefix tile map ----

def _cached_mask_bruteforce(cl, b):
    """Visibility of request b's keys from its new rows, by set enumeration.

    Keys are numbered on the request's own axis: its S_b cached prefix keys
    first (cache rows cache_start .. cache_start + S_b - 1), then its new rows
    in order. Eq. (4) of "From Generation to Scoring", Section 4.1: a key is
    visible from row j iff it precedes j and lies in the shared set Q (here:
    the cached prefix, which precedes every new row) or in j's own item set.
    """
    s0, e0 = int(cl.cu_seqlens[b]), int(cl.cu_seqlens[b + 1])
    S = int(cl.cache_len[b])
    Q = {("cache", int(cl.cache_start[b]) + x) for x in range(S)}
    items = [set(range(int(cl.item_offsets[i]), int(cl.item_ends[i])))
             for i in range(int(cl.item_ptr[b]), int(cl.item_ptr[b + 1]))]
    keys = sorted(Q) + [("new", r) for r in range(s0, e0)]
    vis = np.zeros((e0 - s0, len(keys)), dtype=bool)
    for jj, j in enumerate(range(s0, e0)):
        for kk, key in enumerate(keys):
            if key in Q:
                vis[jj, kk] = True                     # the prefix precedes every new row
            else:
                k = key[1]
                vis[jj, kk] = k <= j and any(j in I and k in I for I in items)
    return vis, S


def _cached_tiles_from_dense(cl, BM, BN):
    out = []
    for b in range(cl.B):
        vis, S = _cached_mask_bruteforce(cl, b)
        L = vis.shape[0]
        # key tiles: the cached prefix from its first key, then the new rows from the first one
        kt = [(u * BN, min((u + 1) * BN, S)) for u in range((S + BN - 1) // BN)]
        kt += [(S + u * BN, S + min((u + 1) * BN, L)) for u in range((L + BN - 1) // BN)]
        for t in range((L + BM - 1) // BM):
            rows = vis[t * BM:min((t + 1) * BM, L)]
            for u, (c0, c1) in enumerate(kt):
                blk = rows[:, c0:c1]
                if blk.any():
                    out.append((b, t, u, O.FULL if blk.all() else O.PARTIAL))
    return np.asarray(out, np.int32).reshape(-1, 4)


def test_tile_map_cached_vs_set_enumeration_exhaustive():
    # every one-request layout with S in 1..5, 1..3 items of 0..3 tokens, on
    # tile shapes that split the prefix, the items and the tiles' own edges
    import itertools
    n_cases = 0
    for S in range(1, 6):
        for n in range(1, 4):
            for lens in itertools.product(range(4), repeat=n):
                cl = O.cached_layout([2], [S], [n], list(lens))
                for BM, BN in [(1, 1), (2, 3), (3, 2), (4, 4)]:
                    got = O.tile_map_cached(cl, BM, BN)
                    ref = _cached_tiles_from_dense(cl, BM, BN)
                    assert got.shape == ref.shape and np.array_equal(got, ref), (S, lens, BM, BN)
                    n_cases += 1
    assert n_cases == 5 * (4 + 16 + 64) * 4


@pytest.mark.parametrize("BM,BN", [(4, 4), (4, 8), (8, 4), (3, 5), (16, 16)])
def test_tile_map_cached_vs_set_enumeration_random(BM, BN):
    rng = np.random.default_rng(700 + BM * 10 + BN)
    for _ in range(20):
        B = int(rng.integers(1, 4))
        S = rng.integers(1, 40, B)
        n = rng.integers(1, 5, B)
        lens = rng.integers(0, 12, int(n.sum()))
        cstart = np.zeros(B, np.int64)
        t = int(rng.integers(0, 9))
        for b in rng.permutation(B):             # prefixes anywhere in the cache, in any order
            cstart[b] = t
            t += int(S[b]) + int(rng.integers(0, 9))
        cl = O.cached_layout(cstart, S, n, lens)
        got = O.tile_map_cached(cl, BM, BN)
        ref = _cached_tiles_from_dense(cl, BM, BN)
        assert got.shape == ref.shape and np.array_equal(got, ref)


def test_tile_map_cached_counts_on_a_hand_case():
    # S = 5 cached keys, items of 2 and 1 tokens (+ DELIM): new rows 0-2 are
    # item 0, rows 3-4 item 1. With BM = BN = 2 the key tiles are
    # cache [0,2) [2,4) [4,5) and new rows [0,2) [2,4) [4,5).
    cl = O.cached_layout([0], [5], [2], [2, 1])
    got = O.tile_map_cached(cl, 2, 2)
    want = [
        # q-tile 0 (rows 0, 1: item 0): every cached tile, then new tile 0 (causal corner)
        (0, 0, 0, O.FULL), (0, 0, 1, O.FULL), (0, 0, 2, O.FULL), (0, 0, 3, O.PARTIAL),
        # q-tile 1 (row 2: item 0; row 3: item 1)
        (0, 1, 0, O.FULL), (0, 1, 1, O.FULL), (0, 1, 2, O.FULL), (0, 1, 3, O.PARTIAL),
        (0, 1, 4, O.PARTIAL),
        # q-tile 2 (row 4: item 1): its own item's keys 3 and 4
        (0, 2, 0, O.FULL), (0, 2, 1, O.FULL), (0, 2, 2, O.FULL), (0, 2, 4, O.PARTIAL),
        (0, 2, 5, O.FULL),
    ]
    assert [tuple(int(x) for x in r) for r in got] == want
