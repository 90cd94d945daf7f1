"""GPU parity of setwise (multi-marker) scoring against the fp64 oracle.

Setwise prompts ("Scaling JEV-like Decision Models with SGLang", "Benchmark:
Fused-Choice vs. Setwise Scoring") are plain causal sequences scored at one
marker per candidate: the attention call with a causal plan, then the scoring
call at the marker rows, both through the C ABI. Small batches are checked
element by element; the 256-request workload on seeded rows, all marker
rows among them, and on a seeded subset of markers for scoring.
"""
import numpy as np
import pytest
import torch

import oracle as O
from ranking_prefill_gb300 import lib, synth
from gpu_helpers import ATTN_TOL, LSE_TOL, SCORE_TOL, f64

pytestmark = pytest.mark.gpu


def _run(qt, n, lens, hq, hkv, D, d, V, labels, seed, rows=None, items=None):
    sl = lib.mis_build_setwise_layout(qt, n, lens, with_positions=False)
    ref = O.setwise_layout(qt, n, lens)
    assert np.array_equal(sl.marker_positions, ref.marker_positions)
    vals = synth.draw_values(seed, sl.T, hq, hkv, D, d, V)
    dev = torch.device("cuda")
    q, k, v = (vals[x].to(dev) for x in ("q", "k", "v"))
    o = torch.full_like(q, 7.0)
    lse = torch.full((hq, sl.T), 7.0, dtype=torch.float32, device=dev)
    plan = lib.Plan(sl.cu_seqlens, sl.prefix_len, None, None, hq, hkv, D)
    ws = torch.zeros(plan.workspace_size(), dtype=torch.uint8, device=dev)
    plan.create(ws)
    lib.mis_attention_fwd_plan(plan, q, k, v, o, lse)
    out = torch.full((sl.M, len(labels)), 7.0, dtype=torch.float32, device=dev)
    ren = torch.full_like(out, 7.0)
    sws = torch.zeros(lib.mis_label_scores_workspace_size(sl.M, d, V, len(labels)),
                      dtype=torch.uint8, device=dev)
    lib.mis_label_scores(vals["hidden"].to(dev), vals["w_lm"].to(dev),
                         torch.as_tensor(sl.marker_positions, device=dev), labels, out, ren, sws)
    torch.cuda.synchronize()
    assert lib.mis_get_device_status(ws) == lib.MIS_OK
    assert lib.mis_get_device_status(sws) == lib.MIS_OK
    ro, rl = O.attention(f64(vals["q"]), f64(vals["k"]), f64(vals["v"]), ref.causal, rows=rows)
    sel = slice(None) if rows is None else torch.as_tensor(np.asarray(rows), device=dev)
    assert np.abs(f64(o[sel]) - ro).max() <= ATTN_TOL
    gl = f64(lse)[:, np.asarray(rows) if rows is not None else slice(None)].T
    assert np.abs(gl - rl).max() <= LSE_TOL
    lp, rn, _ = O.label_scores(f64(vals["hidden"]), f64(vals["w_lm"]), ref.marker_positions,
                               labels, items=items)
    isel = slice(None) if items is None else np.asarray(items)
    assert np.abs(f64(out)[isel] - lp).max() <= SCORE_TOL
    assert np.abs(f64(ren)[isel] - rn).max() <= SCORE_TOL


@pytest.mark.parametrize("seed", range(3))
def test_small_setwise_batches(seed):
    rng = np.random.default_rng(300 + seed)
    B = int(rng.integers(1, 5))
    qt = rng.integers(1, 300, B)
    n = rng.integers(0, 12, B)
    lens = rng.integers(0, 70, int(n.sum()))
    hq, hkv, D = [(4, 2, 64), (8, 2, 128), (6, 6, 128)][seed]
    _run(qt.tolist(), n.tolist(), lens.tolist(), hq, hkv, D, 256, 3000, [5, 2999, 17][: 1 + seed],
         700 + seed)


def test_pages_example_shape():
    # three options, one marker each, Yes/No label rows per marker
    _run([120], [3], [14, 11, 16], 4, 2, 128, 512, 5000, [11, 22], 710)


def test_setwise_256_sampled():
    w = synth.WORKLOADS["setwise-256"]
    s = synth.draw_shapes(w)
    ref = O.setwise_layout(s.prefix_tokens, s.n_items, s.item_lens)
    rng = np.random.default_rng(w.seed)
    rows = set(rng.choice(ref.causal.T, size=256, replace=False).tolist())
    rows |= set(ref.marker_positions[:: max(1, ref.M // 64)].tolist())
    rows |= {0, ref.causal.T - 1}
    items = np.sort(rng.choice(ref.M, size=48, replace=False))
    _run(s.prefix_tokens, s.n_items, s.item_lens, w.hq, w.hkv, w.head_dim, w.d_model, w.vocab,
         [int(x) for x in s.label_sets[0]], w.seed, rows=sorted(rows), items=items)
