"""Allocation-free label scoring, through the C ABI.

mis_label_scores_noalloc serves callers that cannot call cudaMalloc (for
example a plugin inside an engine that has reserved all device memory and
offers no allocator). It keeps its scratch in a static device array shared
by every call, so this test checks two calls in a row, with different sizes
and inputs, against the workspace-based mis_label_scores on the same inputs,
within the scoring tolerance. The file name sorts last so that a run that
stops at the first failure has run every other test before it.
"""
import numpy as np
import pytest
import torch

from ranking_prefill_gb300 import lib

pytestmark = pytest.mark.gpu

SCORE_TOL = 1e-2     # the scoring tolerance of the parity tests (max-abs on log-probs)


def _case(seed, M, T, d, V):
    g = torch.Generator().manual_seed(seed)
    hidden = torch.randn(T, d, generator=g).to(torch.bfloat16).cuda()
    w = (torch.randn(V, d, generator=g) * 0.05).to(torch.bfloat16).cuda()
    rows = torch.as_tensor(np.random.default_rng(seed).choice(T, size=M, replace=False),
                           dtype=torch.int32).cuda()
    return hidden, w, rows


def _with_workspace(hidden, w, rows, labels):
    M, K = rows.numel(), len(labels)
    out = torch.empty(M, K, dtype=torch.float32, device="cuda")
    ren = torch.empty(M, K, dtype=torch.float32, device="cuda")
    ws = torch.zeros(lib.mis_label_scores_workspace_size(M, w.shape[1], w.shape[0], K),
                     dtype=torch.uint8, device="cuda")
    lib.mis_label_scores(hidden, w, rows, labels, out, ren, ws)
    torch.cuda.synchronize()
    assert lib.mis_get_device_status(ws) == lib.MIS_OK
    return out, ren


def _no_alloc(hidden, w, rows, labels):
    M, K = rows.numel(), len(labels)
    out = torch.full((M, K), float("nan"), dtype=torch.float32, device="cuda")
    ren = torch.full((M, K), float("nan"), dtype=torch.float32, device="cuda")
    status = torch.full((2,), 0xFFFF, dtype=torch.int32, device="cuda")
    lib.mis_label_scores_noalloc(hidden, w, rows, labels, out, ren, status)
    torch.cuda.synchronize()
    assert int(status[0].item()) == 0
    return out, ren


def test_no_alloc_matches_workspace_entry_point_twice():
    cases = [(_case(1, 300, 700, 1024, 151936), [9, 151935, 17]),
             (_case(2, 100, 250, 512, 20000), [1, 2])]
    for (hidden, w, rows), labels in cases:
        ref_out, ref_ren = _with_workspace(hidden, w, rows, labels)
        got_out, got_ren = _no_alloc(hidden, w, rows, labels)
        assert bool(torch.isfinite(got_out).all()) and bool(torch.isfinite(got_ren).all())
        assert (got_out - ref_out).abs().max().item() <= SCORE_TOL
        assert (got_ren - ref_ren).abs().max().item() <= SCORE_TOL


def test_no_alloc_refuses_sizes_beyond_its_scratch():
    hidden, w, rows = _case(3, 4, 16, 4096, 1000)
    big_rows = torch.zeros(4096, dtype=torch.int32, device="cuda")   # 4096 x 4096 rows > limit
    out = torch.empty(4096, 2, dtype=torch.float32, device="cuda")
    need = lib.mis_label_scores_workspace_size(4096, 4096, 1000, 2)
    assert need > 8650752
    with pytest.raises(lib.MisError) as e:
        lib.mis_label_scores_noalloc(hidden, w, big_rows, [1, 2], out, None, None)
    assert e.value.status == lib.MIS_ERR_UNSUPPORTED
