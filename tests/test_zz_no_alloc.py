"""Allocation-free label scoring, through the C ABI.

mis_label_scores_noalloc serves callers that cannot call cudaMalloc (for
example a plugin inside an engine that has reserved all device memory and
offers no allocator). It keeps its scratch in a static device array shared
by every call, so these tests make calls back to back, with different sizes
and inputs, and compare each with the workspace-based mis_label_scores on
the same inputs. Both run the same kernels, so the results agree bit for
bit, up to the order of one fp32 sum where vocabulary tiles are handed out
at run time; one case is also held against the fp64 oracle within the
scoring tolerance. The cases cover both ways the LM-head kernel hands out
vocabulary tiles: a fixed split when there are several 128-item tiles, and a
counter kept in the shared scratch when one item tile faces more vocabulary
tiles than there are SMs. The file name sorts last so that a run that stops
at the first failure has run every other test before it.
"""
import numpy as np
import pytest
import torch

import oracle as O
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


REGROUP_TOL = 1e-5   # fp32 logsumexp summed in another grouping of vocabulary tiles


def _check_pair(hidden, w, rows, labels, counter_fed=False):
    ref_out, ref_ren = _with_workspace(hidden, w, rows, labels)
    got_out, got_ren = _no_alloc(hidden, w, rows, labels)
    assert bool(torch.isfinite(got_out).all()) and bool(torch.isfinite(got_ren).all())
    # the same kernels on the same inputs. Label logits come from the one tile
    # holding each label, so the label-renormalised scores are identical.
    # With a fixed split of the vocabulary the log-probs are too; with tiles
    # taken from a counter, which block folds which tile into its running
    # logsumexp changes from call to call, and only the fp32 rounding of
    # that sum may differ.
    assert torch.equal(got_ren, ref_ren)
    if counter_fed:
        assert (got_out - ref_out).abs().max().item() <= REGROUP_TOL
    else:
        assert torch.equal(got_out, ref_out)
    return got_out, got_ren


def test_no_alloc_matches_workspace_entry_point_twice():
    # several item tiles: vocabulary tiles split between blocks in fixed runs
    cases = [(_case(1, 300, 700, 1024, 151936), [9, 151935, 17]),
             (_case(2, 100, 250, 512, 20000), [1, 2])]
    for (hidden, w, rows), labels in cases:
        _check_pair(hidden, w, rows, labels)


def test_no_alloc_counter_fed_vocabulary_tiles_twice_and_against_the_oracle():
    # one item tile (M <= 128) and 594 vocabulary tiles of 256: blocks take
    # tiles from a counter that lives in the shared scratch, so the second
    # call must start from a cleared counter
    labels = [151935, 0, 4242]
    first = _case(4, 100, 400, 1024, 151936)
    second = _case(5, 37, 90, 1024, 151936)
    got, ren = _check_pair(*first, labels, counter_fed=True)
    _check_pair(*second, labels, counter_fed=True)
    hidden, w, rows = first
    f64 = lambda t: t.detach().to("cpu", torch.float64).numpy()
    ref_lp, ref_ren, _ = O.label_scores(f64(hidden), f64(w), rows.cpu().numpy(), labels)
    assert np.abs(f64(got) - ref_lp).max() <= SCORE_TOL
    assert np.abs(f64(ren) - ref_ren).max() <= SCORE_TOL


def test_no_alloc_refuses_sizes_beyond_its_scratch():
    hidden, w, rows = _case(3, 4, 16, 4096, 1000)
    big_rows = torch.zeros(4096, dtype=torch.int32, device="cuda")   # 4096 x 4096 rows > limit
    out = torch.empty(4096, 2, dtype=torch.float32, device="cuda")
    need = lib.mis_label_scores_workspace_size(4096, 4096, 1000, 2)
    assert need > 8650752
    with pytest.raises(lib.MisError) as e:
        lib.mis_label_scores_noalloc(hidden, w, big_rows, [1, 2], out, None, None)
    assert e.value.status == lib.MIS_ERR_UNSUPPORTED
