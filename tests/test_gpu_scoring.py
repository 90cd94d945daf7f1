"""GPU parity of mis_label_scores against the fp64 oracle (through the C ABI).

Full element-by-element checks on small and medium cases (ragged vocabulary
tails, item counts around the 128-item tile, d = 64..8192, V = 1..151936,
K = 1..16, repeated and edge label ids), the full qwen3-0.6b-layer workload, and
seeded item samples of the large ones. Tolerance: max-abs 1e-2 on log-probs
and on the label-renormalised scores.
"""
import numpy as np
import pytest
import torch

import oracle as O
from ranking_prefill_gb300 import lib, synth
from gpu_helpers import SCORE_TOL, f64, run_scores

pytestmark = pytest.mark.gpu


def _check(hidden, w, delim, labels, items=None, T=None):
    out, ren, ws = run_scores(hidden.cuda(), w.cuda(), torch.as_tensor(delim, dtype=torch.int32).cuda(),
                              labels, T=T)
    assert lib.mis_get_device_status(ws) == lib.MIS_OK
    lp, rn, _ = O.label_scores(f64(hidden), f64(w), np.asarray(delim), labels, items=items)
    sel = slice(None) if items is None else np.asarray(items)
    g_lp, g_rn = f64(out)[sel], f64(ren)[sel]
    assert np.isfinite(g_lp).all() and np.isfinite(g_rn).all()
    e1, e2 = np.abs(g_lp - lp).max(), np.abs(g_rn - rn).max()
    assert e1 <= SCORE_TOL, f"logprob err {e1}"
    assert e2 <= SCORE_TOL, f"renorm err {e2}"
    return e1


def test_tiny_workload():
    w = synth.WORKLOADS["tiny"]
    s = synth.draw_shapes(w)
    lay = O.build_layout(s.prefix_tokens, s.n_items, s.item_lens)
    v = synth.draw_values(w.seed, lay.T, w.hq, w.hkv, w.head_dim, w.d_model, w.vocab)
    _check(v["hidden"], v["w_lm"], lay.delim_positions, s.label_sets[0].tolist())


@pytest.mark.parametrize("M,d,V,labels", [
    (1, 64, 1000, [0]),
    (100, 256, 4097, [4096, 0, 17]),
    (128, 512, 2048, [5, 5, 2047, 1000]),
    (129, 128, 777, list(range(16))),
    (300, 1024, 5000, [1234, 4321]),
    # one item tile and more vocabulary tiles than SMs: tiles go out from a
    # counter (ragged last tile, labels in the first and last tiles)
    (1, 64, 60000, [59999, 0]),
    (128, 128, 50001, [50000, 3, 25000]),
    (77, 512, 80000, [1, 79999]),
    # the largest model width (d = 8192: 128 k-blocks per tile) and a
    # one-token vocabulary (every log-prob is exactly 0)
    (3, 8192, 700, [0, 699, 350]),
    (5, 64, 1, [0, 0]),
])
def test_random_cases(M, d, V, labels):
    g = torch.Generator().manual_seed(M * 7 + d)
    T = M + 37
    hidden = torch.randn(T, d, generator=g).to(torch.bfloat16)
    w = (torch.randn(V, d, generator=g) * 0.05).to(torch.bfloat16)
    delim = np.random.default_rng(M).choice(T, size=M, replace=M > T).astype(np.int32)
    _check(hidden, w, delim, labels)


def test_strided_hidden_rows():
    g = torch.Generator().manual_seed(3)
    T, d, V = 90, 256, 3000
    buf = torch.randn(T, d + 64, generator=g).to(torch.bfloat16)
    hidden = buf[:, :d]                       # row stride d + 64
    w = (torch.randn(V, d, generator=g) * 0.05).to(torch.bfloat16)
    delim = np.arange(5, 85, 3, dtype=np.int32)
    out, ren, ws = run_scores(buf.cuda()[:, :d], w.cuda(), torch.as_tensor(delim).cuda(), [1, 2])
    lp, rn, _ = O.label_scores(f64(hidden), f64(w), delim, [1, 2])
    assert np.abs(f64(out) - lp).max() <= SCORE_TOL


def test_index_out_of_range_reports_status():
    g = torch.Generator().manual_seed(4)
    hidden = torch.randn(50, 128, generator=g).to(torch.bfloat16).cuda()
    w = (torch.randn(600, 128, generator=g) * 0.05).to(torch.bfloat16).cuda()
    delim = torch.tensor([3, 50, 7], dtype=torch.int32).cuda()       # 50 is outside [0, 50)
    out, ren, ws = run_scores(hidden, w, delim, [1, 2])
    assert lib.mis_get_device_status(ws) == lib.MIS_ERR_DEVICE_INDEX
    # the valid rows are still scored
    lp, _, _ = O.label_scores(f64(hidden), f64(w), [3, 0, 7], [1, 2])
    assert np.abs(f64(out)[[0, 2]] - lp[[0, 2]]).max() <= SCORE_TOL


def test_next_call_clears_the_status():
    # the status words belong to the last call on the workspace: an index
    # error is reported once, and a clean call afterwards reads MIS_OK
    g = torch.Generator().manual_seed(5)
    hidden = torch.randn(40, 128, generator=g).to(torch.bfloat16).cuda()
    w = (torch.randn(700, 128, generator=g) * 0.05).to(torch.bfloat16).cuda()
    out = torch.empty(3, 2, dtype=torch.float32, device="cuda")
    ws = torch.zeros(lib.mis_label_scores_workspace_size(3, 128, 700, 2), dtype=torch.uint8,
                     device="cuda")
    for rows, want in [([1, 40, 2], lib.MIS_ERR_DEVICE_INDEX), ([1, 39, 2], lib.MIS_OK),
                       ([-1, 5, 6], lib.MIS_ERR_DEVICE_INDEX), ([0, 5, 6], lib.MIS_OK)]:
        lib.mis_label_scores(hidden, w, torch.tensor(rows, dtype=torch.int32).cuda(), [3, 4], out,
                             None, ws)
        assert lib.mis_get_device_status(ws) == want
    lp, _, _ = O.label_scores(f64(hidden), f64(w), [0, 5, 6], [3, 4])
    assert np.abs(f64(out) - lp).max() <= SCORE_TOL


def test_zero_items():
    out, ren, ws = run_scores(torch.zeros(4, 64, dtype=torch.bfloat16).cuda(),
                              torch.zeros(10, 64, dtype=torch.bfloat16).cuda(),
                              torch.zeros(0, dtype=torch.int32).cuda(), [1])
    assert lib.mis_get_device_status(ws) == lib.MIS_OK


def test_qwen3_layer_full():
    w = synth.WORKLOADS["qwen3-0.6b-layer"]
    s = synth.draw_shapes(w)
    lay = O.build_layout(s.prefix_tokens, s.n_items, s.item_lens)
    v = synth.draw_values(w.seed, lay.T, w.hq, w.hkv, w.head_dim, w.d_model, w.vocab,
                          want=("hidden", "w_lm"))
    _check(v["hidden"], v["w_lm"], lay.delim_positions, s.label_sets[0].tolist())


@pytest.mark.parametrize("name", ["8b-large", "decision-256", "varlen-16", "prefix12k-50x150"])
def test_large_workloads_sampled_items(name):
    w = synth.WORKLOADS[name]
    s = synth.draw_shapes(w)
    lay = O.build_layout(s.prefix_tokens, s.n_items, s.item_lens)
    v = synth.draw_values(w.seed, lay.T, w.hq, w.hkv, w.head_dim, w.d_model, w.vocab,
                          want=("hidden", "w_lm"))
    rng = np.random.default_rng(w.seed)
    items = sorted(set(rng.choice(lay.M, size=min(96, lay.M), replace=False).tolist()) | {0, lay.M - 1})
    for labels in s.label_sets:
        _check(v["hidden"], v["w_lm"], lay.delim_positions, labels.tolist(), items=items)


def test_one_workspace_for_calls_of_different_shapes_and_after_a_timeout():
    # A workspace sized for the largest call serves calls of other shapes, and
    # a call whose waits ran out leaves nothing behind that later calls on the
    # same workspace would read: they report MIS_OK and stay exact.
    g = torch.Generator().manual_seed(11)
    T = 700
    hidden = torch.randn(T, 256, generator=g).to(torch.bfloat16)
    w_big = (torch.randn(20000, 256, generator=g) * 0.05).to(torch.bfloat16)
    cases = [(np.random.default_rng(1).choice(T, 300, replace=False), w_big[:5000], [7, 4999, 7]),
             (np.random.default_rng(2).choice(T, 40, replace=False), w_big, [19999]),
             (np.random.default_rng(3).choice(T, 260, replace=False), w_big[:9001], list(range(16)))]
    need = max(lib.mis_label_scores_workspace_size(len(r), 256, int(wl.shape[0]), len(lb))
               for r, wl, lb in cases)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    dev_h = hidden.cuda()

    def call(rows, wl, labels):
        out = torch.full((len(rows), len(labels)), 7.0, dtype=torch.float32, device="cuda")
        ren = torch.full_like(out, 7.0)
        lib.mis_label_scores(dev_h, wl.cuda(), torch.as_tensor(rows, dtype=torch.int32).cuda(),
                             labels, out, ren, ws)
        torch.cuda.synchronize()
        return out, ren

    def check(rows, wl, labels):
        out, ren = call(rows, wl, labels)
        assert lib.mis_get_device_status(ws) == lib.MIS_OK
        lp, rn, _ = O.label_scores(f64(hidden), f64(wl), rows, labels)
        assert np.abs(f64(out) - lp).max() <= SCORE_TOL
        assert np.abs(f64(ren) - rn).max() <= SCORE_TOL

    for c in cases:
        check(*c)
    old = lib.mis_set_wait_limit_ns(2_000_000)
    lib.mis_inject_stall(2)
    try:
        call(*cases[0])
        assert lib.mis_get_device_status(ws) == lib.MIS_ERR_DEVICE_TIMEOUT
    finally:
        lib.mis_inject_stall(0)
        lib.mis_set_wait_limit_ns(old)
    for c in reversed(cases):
        check(*c)


def test_counter_fed_tiles_across_back_to_back_calls():
    # One item tile and more vocabulary tiles than SMs: blocks take tiles from a
    # counter in the workspace status words, which the call's first kernel
    # zeroes. Three calls enqueued back to back on one workspace (no sync in
    # between), then a call whose waits ran out, then a clean call again: each
    # clean call scores every vocabulary tile exactly once.
    g = torch.Generator().manual_seed(21)
    T, d, V = 400, 256, 60001
    hidden = torch.randn(T, d, generator=g).to(torch.bfloat16)
    w = (torch.randn(V, d, generator=g) * 0.05).to(torch.bfloat16)
    dh, dw = hidden.cuda(), w.cuda()
    cases = [(np.random.default_rng(s).choice(T, m, replace=False).astype(np.int32), lb)
             for s, m, lb in [(1, 100, [0, 60000]), (2, 128, [777, 30000, 59999]), (3, 1, [5])]]
    ws = torch.zeros(max(lib.mis_label_scores_workspace_size(len(r), d, V, len(lb)) for r, lb in cases),
                     dtype=torch.uint8, device="cuda")
    outs = []
    for rows, lb in cases:
        out = torch.empty(len(rows), len(lb), dtype=torch.float32, device="cuda")
        lib.mis_label_scores(dh, dw, torch.as_tensor(rows).cuda(), lb, out, None, ws)
        outs.append(out)
    torch.cuda.synchronize()
    assert lib.mis_get_device_status(ws) == lib.MIS_OK
    for (rows, lb), out in zip(cases, outs):
        lp, _, _ = O.label_scores(f64(hidden), f64(w), rows, lb)
        assert np.abs(f64(out) - lp).max() <= SCORE_TOL
    old = lib.mis_set_wait_limit_ns(2_000_000)
    lib.mis_inject_stall(2)
    try:
        rows, lb = cases[0]
        out = torch.empty(len(rows), len(lb), dtype=torch.float32, device="cuda")
        lib.mis_label_scores(dh, dw, torch.as_tensor(rows).cuda(), lb, out, None, ws)
        torch.cuda.synchronize()
        assert lib.mis_get_device_status(ws) == lib.MIS_ERR_DEVICE_TIMEOUT
    finally:
        lib.mis_inject_stall(0)
        lib.mis_set_wait_limit_ns(old)
    rows, lb = cases[1]
    out = torch.empty(len(rows), len(lb), dtype=torch.float32, device="cuda")
    lib.mis_label_scores(dh, dw, torch.as_tensor(rows).cuda(), lb, out, None, ws)
    torch.cuda.synchronize()
    assert lib.mis_get_device_status(ws) == lib.MIS_OK
    lp, _, _ = O.label_scores(f64(hidden), f64(w), rows, lb)
    assert np.abs(f64(out) - lp).max() <= SCORE_TOL


def test_scores_repeat_bit_for_bit():
    # Every path's partial (max, sum) pairs are merged in a fixed order: with
    # the vocabulary tiles from a counter (one item tile, more tiles than SMs)
    # each tile keeps its own partial, whichever block ran it; the fixed runs
    # of tiles (one SM or SM pairs) are fixed by construction. So the same call
    # gives the same bits every time.
    g = torch.Generator().manual_seed(33)
    T = 700
    for M, d, V, labels in [(100, 1024, 151936, [3, 151935]), (60, 256, 30000, [7, 8, 29999]),
                            (300, 512, 20000, [0, 19999])]:
        hidden = torch.randn(T, d, generator=g).to(torch.bfloat16).cuda()
        w = (torch.randn(V, d, generator=g) * 0.02).to(torch.bfloat16).cuda()
        rows = torch.as_tensor(np.random.default_rng(M).choice(T, M, replace=False).astype(np.int32)).cuda()
        runs = [run_scores(hidden, w, rows, labels) for _ in range(3)]
        for out, ren, ws in runs:
            assert lib.mis_get_device_status(ws) == lib.MIS_OK
        for out, ren, _ in runs[1:]:
            assert torch.equal(out, runs[0][0]) and torch.equal(ren, runs[0][1]), (M, d, V)
