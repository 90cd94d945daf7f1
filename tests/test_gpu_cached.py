"""GPU parity of attention over a cached prefix (the in-batch prefix cache of
"Scaling LLM-Based Ranking Systems with Prefill-Only Optimization", the
knock-knock second request of "Turbocharging LinkedIn's recommendation
systems with SGLang") against the fp64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle as O
from ranking_prefill_gb300 import lib, synth
from gpu_helpers import ATTN_TOL, LSE_TOL, f64, forced_schedule

pytestmark = pytest.mark.gpu


def _run_cached(cl, cache_T, q, k, v, kc, vc, hq, hkv, D, lse=True):
    dev = torch.device("cuda")
    plan = lib.CachedPlan(cl.cu_seqlens, cl.item_ptr, cl.item_offsets, cl.cache_start,
                          cl.cache_len, cache_T, hq, hkv, D)
    ws = torch.zeros(plan.workspace_size(), dtype=torch.uint8, device=dev)
    plan.create(ws)
    o = torch.full((cl.T, hq, D), 7.0, dtype=torch.bfloat16, device=dev)
    l = torch.full((hq, cl.T), 7.0, dtype=torch.float32, device=dev) if lse else None
    lib.mis_attention_fwd_cached(plan, q, k, v, kc, vc, o, l)
    o2 = torch.empty_like(o)
    l2 = torch.empty_like(l) if lse else None
    lib.mis_attention_fwd_cached(plan, q, k, v, kc, vc, o2, l2)
    torch.cuda.synchronize()
    assert lib.mis_get_device_status(ws) == lib.MIS_OK
    assert torch.equal(o, o2) and (not lse or torch.equal(l, l2))   # the same bits again
    return o, l, plan.stats()


@pytest.mark.parametrize("seed", range(4))
@pytest.mark.parametrize("mode", [lib.SCHEDULE_PAIR, lib.SCHEDULE_SPLIT], ids=["pair", "split"])
def test_random_cached_batches(seed, mode):
    rng = np.random.default_rng(800 + seed)
    B = int(rng.integers(1, 4))
    S = rng.integers(1, 400, B)
    S[0] = [128, 129, 255, 1][seed]
    n = rng.integers(1, 9, B)
    lens = rng.integers(0, 150, int(n.sum()))
    cstart, t = np.zeros(B, np.int64), int(rng.integers(0, 40))
    for b in rng.permutation(B):
        cstart[b] = t
        t += int(S[b]) + int(rng.integers(0, 70))
    cache_T = t
    hq, hkv, D = [(4, 2, 128), (8, 2, 64), (6, 6, 128), (16, 8, 128)][seed]
    cl = O.cached_layout(cstart, S, n, lens)
    vals = synth.draw_values(900 + seed, cl.T + cache_T, hq, hkv, D, want=("q", "k", "v"))
    dev = torch.device("cuda")
    q = vals["q"][:cl.T].to(dev)
    k, v = vals["k"][:cl.T].to(dev), vals["v"][:cl.T].to(dev)
    kc, vc = vals["k"][cl.T:].to(dev), vals["v"][cl.T:].to(dev)
    with forced_schedule(mode):
        o, l, st = _run_cached(cl, cache_T, q, k, v, kc, vc, hq, hkv, D)
    ro, rl = O.attention_cached(f64(vals["q"][:cl.T]), f64(vals["k"][:cl.T]), f64(vals["v"][:cl.T]),
                                f64(vals["k"][cl.T:]), f64(vals["v"][cl.T:]), cl)
    assert np.abs(f64(o) - ro).max() <= ATTN_TOL
    assert np.abs(f64(l).T - rl).max() <= LSE_TOL


def test_single_item_requests_share_one_cached_prefix():
    # single-item scoring with prefix caching: 12 requests of one item each,
    # all over the same cached rows
    S, lens = 700, list(range(5, 125, 10))
    cl = O.cached_layout([0] * 12, [S] * 12, [1] * 12, lens)
    hq, hkv, D = 8, 4, 128
    vals = synth.draw_values(950, cl.T + S, hq, hkv, D, want=("q", "k", "v"))
    dev = torch.device("cuda")
    o, l, st = _run_cached(cl, S, vals["q"][:cl.T].to(dev), vals["k"][:cl.T].to(dev),
                           vals["v"][:cl.T].to(dev), vals["k"][cl.T:].to(dev), vals["v"][cl.T:].to(dev),
                           hq, hkv, D)
    ro, _ = O.attention_cached(f64(vals["q"][:cl.T]), f64(vals["k"][:cl.T]), f64(vals["v"][:cl.T]),
                               f64(vals["k"][cl.T:]), f64(vals["v"][cl.T:]), cl)
    assert np.abs(f64(o) - ro).max() <= ATTN_TOL


def test_knock_knock_split_of_the_qwen3_workload_matches_packed_mis():
    # the same rows as the packed MIS run: the prefix rows become the cache,
    # the item rows the second request; their outputs must agree
    w = synth.WORKLOADS["qwen3-0.6b-layer"]
    s = synth.draw_shapes(w)
    lay = lib.mis_build_layout(s.prefix_tokens, s.n_items, s.item_lens)
    vals = synth.draw_values(w.seed, lay.T, w.hq, w.hkv, w.head_dim, want=("q", "k", "v"))
    dev = torch.device("cuda")
    q, k, v = (vals[x].to(dev) for x in ("q", "k", "v"))
    o_mis = torch.empty_like(q)
    plan = lib.Plan(lay.cu_seqlens, lay.prefix_len, lay.item_ptr, lay.item_offsets, w.hq, w.hkv,
                    w.head_dim)
    ws = torch.zeros(plan.workspace_size(), dtype=torch.uint8, device=dev)
    plan.create(ws)
    lib.mis_attention_fwd_plan(plan, q, k, v, o_mis, None)
    S = int(lay.prefix_len[0])
    cl = O.cached_layout([0], [S], s.n_items, s.item_lens)
    o, _, st = _run_cached(cl, S, q[S:], k[S:], v[S:], k[:S], v[:S], w.hq, w.hkv, w.head_dim, lse=False)
    assert (o.float() - o_mis[S:].float()).abs().max().item() <= 1e-2
    rows = np.random.default_rng(3).choice(cl.T, 128, replace=False)
    ro, _ = O.attention_cached(f64(vals["q"][S:]), f64(vals["k"][S:]), f64(vals["v"][S:]),
                               f64(vals["k"][:S]), f64(vals["v"][:S]), cl, rows=rows)
    assert np.abs(f64(o[torch.as_tensor(rows, device=dev)]) - ro).max() <= ATTN_TOL
