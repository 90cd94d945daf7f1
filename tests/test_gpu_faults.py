"""Failure detection without a GPU fault.

Every wait inside the kernels is bounded. mis_inject_stall() makes the
tensor-core thread of each block wait on a barrier that nothing arrives on,
with a 2 ms bound: the kernels must then drain their own copies and
tensor-core work, free tensor memory, return, and report
MIS_ERR_DEVICE_TIMEOUT through the workspace status; afterwards the same
process must still compute correct results.
"""
import numpy as np
import pytest
import torch

import oracle as O
from ranking_prefill_gb300 import lib, synth
from gpu_helpers import check_attention, f64, run_scores

pytestmark = pytest.mark.gpu


def _tiny():
    w = synth.WORKLOADS["tiny"]
    s = synth.draw_shapes(w)
    lay = lib.mis_build_layout(s.prefix_tokens, s.n_items, s.item_lens)
    v = synth.draw_values(w.seed, lay.T, w.hq, w.hkv, w.head_dim, w.d_model, w.vocab)
    return w, s, lay, v


def test_wait_timeout_is_reported_and_context_survives():
    w, s, lay, v = _tiny()
    dev = torch.device("cuda")
    q, k, vv = v["q"].to(dev), v["k"].to(dev), v["v"].to(dev)
    o = torch.zeros_like(q)
    plan = lib.Plan(lay.cu_seqlens, lay.prefix_len, lay.item_ptr, lay.item_offsets,
                    w.hq, w.hkv, w.head_dim)
    ws = torch.zeros(plan.workspace_size(), dtype=torch.uint8, device=dev)
    plan.create(ws)
    delim = torch.as_tensor(lay.delim_positions, device=dev)
    labels = s.label_sets[0].tolist()
    old = lib.mis_set_wait_limit_ns(2_000_000)
    lib.mis_inject_stall(3)
    try:
        lib.mis_attention_fwd_plan(plan, q, k, vv, o, None)
        torch.cuda.synchronize()
        assert lib.mis_get_device_status(ws) == lib.MIS_ERR_DEVICE_TIMEOUT
        out, ren, sws = run_scores(v["hidden"].to(dev), v["w_lm"].to(dev), delim, labels)
        assert lib.mis_get_device_status(sws) == lib.MIS_ERR_DEVICE_TIMEOUT
    finally:
        lib.mis_inject_stall(0)
        lib.mis_set_wait_limit_ns(old)
    # the context is intact: the same calls now succeed and match the oracle
    check_attention(s, w.hq, w.hkv, w.head_dim, w.seed)
    out, ren, sws = run_scores(v["hidden"].to(dev), v["w_lm"].to(dev), delim, labels)
    assert lib.mis_get_device_status(sws) == lib.MIS_OK
    lp, _, _ = O.label_scores(f64(v["hidden"]), f64(v["w_lm"]), lay.delim_positions, labels)
    assert np.abs(f64(out) - lp).max() <= 1e-2
