"""MIS scores equal single-item scores on the GPU ("From Generation to
Scoring", Section 4.1: the mask and reused positions give each item's final
token the same context as in [q; c_i], so eq. (2) yields the independent
score up to floating-point differences).

One member with 200 candidates is run as one N = 200 request and as 200
single-item requests through the same calls. Each item's readout row must
agree between the two runs, for the attention output (all heads) and for the
label scores computed from that output (the attention output used as the
hidden state). The MIS run is also checked against the fp64 oracle on its
readout rows.
"""
import numpy as np
import pytest
import torch

import oracle as O
from ranking_prefill_gb300 import lib, synth
from gpu_helpers import ATTN_TOL, SCORE_TOL, f64

pytestmark = pytest.mark.gpu


def _run(shapes, qkv_rows, vals, hq, hkv, D, w_lm, labels):
    dev = torch.device("cuda")
    lay = lib.mis_build_layout(shapes.prefix_tokens, shapes.n_items, shapes.item_lens)
    idx = torch.as_tensor(qkv_rows, dtype=torch.long)
    q, k, v = (vals[x][idx].to(dev) for x in ("q", "k", "v"))
    o = torch.empty_like(q)
    plan = lib.Plan(lay.cu_seqlens, lay.prefix_len, lay.item_ptr, lay.item_offsets, hq, hkv, D)
    ws = torch.zeros(plan.workspace_size(), dtype=torch.uint8, device=dev)
    plan.create(ws)
    lib.mis_attention_fwd_plan(plan, q, k, v, o, None)
    hidden = o.view(lay.T, hq * D)                     # the attention output as hidden state
    out = torch.empty(lay.M, len(labels), dtype=torch.float32, device=dev)
    sws = torch.zeros(lib.mis_label_scores_workspace_size(lay.M, hq * D, w_lm.shape[0], len(labels)),
                      dtype=torch.uint8, device=dev)
    lib.mis_label_scores(hidden, w_lm, torch.as_tensor(lay.delim_positions, device=dev), labels,
                         out, None, sws)
    torch.cuda.synchronize()
    assert lib.mis_get_device_status(ws) == lib.MIS_OK
    assert lib.mis_get_device_status(sws) == lib.MIS_OK
    return lay, o, out


def test_mis_equals_single_item_scoring_end_to_end():
    pool = synth.sweep_pool(1, vocab=4096, seed=11)
    pool.query_tokens[0] = 600
    hq, hkv, D = 8, 4, 128
    mis = synth.sweep_shapes(pool, 200)
    sis = synth.sweep_shapes(pool, 1)
    lay_m = O.build_layout(mis.prefix_tokens, mis.n_items, mis.item_lens)
    vals = synth.draw_values(12, lay_m.T, hq, hkv, D, want=("q", "k", "v"))
    # SIS rows are gathered from the MIS rows: each request is [Q; item i]
    S = int(lay_m.prefix_len[0])
    rows_sis = np.concatenate([np.concatenate([np.arange(S), np.arange(lay_m.item_offsets[i],
                                                                        lay_m.item_ends[i])])
                               for i in range(lay_m.M)])
    g = torch.Generator().manual_seed(13)
    w_lm = (torch.randn(4096, hq * D, generator=g) * 0.02).to(torch.bfloat16).cuda()
    labels = [int(x) for x in pool.labels]
    lm, om, sm = _run(mis, np.arange(lay_m.T), vals, hq, hkv, D, w_lm, labels)
    ls, os_, ss = _run(sis, rows_sis, vals, hq, hkv, D, w_lm, labels)
    rm = torch.as_tensor(lm.delim_positions, device="cuda", dtype=torch.long)
    rs = torch.as_tensor(ls.delim_positions, device="cuda", dtype=torch.long)
    d_o = (om[rm].float() - os_[rs].float()).abs().max().item()
    d_s = (sm - ss).abs().max().item()
    assert d_o <= 1e-2, d_o                      # two bf16 results of the same exact quantity
    assert d_s <= SCORE_TOL, d_s
    # and the MIS readout rows against the oracle
    ro, _ = O.attention(f64(vals["q"]), f64(vals["k"]), f64(vals["v"]), lay_m,
                        rows=lay_m.delim_positions)
    assert np.abs(f64(om[rm]) - ro).max() <= ATTN_TOL
