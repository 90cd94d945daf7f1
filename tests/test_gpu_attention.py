"""GPU parity of mis_attention_fwd against the fp64 oracle (through the C ABI).

Element-by-element on small and medium layouts (several tiles, ragged tails,
empty items, D = 64 and 128, GQA groups 1 to 5 and a lone head, strided
rows, varlen batches), on
the full qwen3-0.6b-layer workload, and on seeded row samples of the large
workloads (every readout row plus seeded random rows; rows are independent,
so each sampled row is still an exact element-by-element check). Seeded
random batches also check that a plan's output repeats bit for bit (a race
check) and that the two schedules agree. Tolerances: max-abs 2e-2 on O, 2e-3 on LSE.
"""
import numpy as np
import pytest
import torch

import oracle as O
from ranking_prefill_gb300 import lib, synth
from gpu_helpers import ATTN_TOL, check_attention, f64, forced_schedule, oracle_layout, run_attention

pytestmark = pytest.mark.gpu


@pytest.fixture(params=[lib.SCHEDULE_PAIR, lib.SCHEDULE_SPLIT], ids=["pair", "split"])
def schedule(request):
    """Run the test under both attention schedules (odd GQA groups are always split)."""
    with forced_schedule(request.param):
        yield request.param


def _expect_schedule(st, mode, hq, hkv):
    want = mode if (hq // hkv) % 2 == 0 else lib.SCHEDULE_SPLIT
    assert st["schedule"] == want
    assert st["n_units"] == st["n_qtiles"] * (hq // 2 if want == lib.SCHEDULE_PAIR else hq)


def _sample_rows(lay, n, seed):
    rng = np.random.default_rng(seed)
    rows = set(rng.choice(lay.T, size=min(n, lay.T), replace=False).tolist())
    rows |= set(lay.delim_positions.tolist())          # every readout row: the rows scoring reads
    rows |= {0, lay.T - 1}
    for b in range(lay.B):
        s0 = int(lay.cu_seqlens[b])
        rows |= {s0, s0 + int(lay.prefix_len[b]) - 1, int(lay.cu_seqlens[b + 1]) - 1}
    return sorted(rows)


def test_tiny_workload_full(schedule):
    w = synth.WORKLOADS["tiny"]
    err, st = check_attention(synth.draw_shapes(w), w.hq, w.hkv, w.head_dim, w.seed)
    assert st["n_full"] + st["n_partial"] == 6
    _expect_schedule(st, schedule, w.hq, w.hkv)


@pytest.mark.parametrize("seed", range(6))
def test_random_small_layouts(seed, schedule):
    rng = np.random.default_rng(100 + seed)
    B = int(rng.integers(1, 5))
    p = rng.integers(0, 400, B)
    n = rng.integers(0, 20, B)
    lens = rng.integers(0, 70, int(n.sum()))
    # requests without items must be plain prefixes; keep them valid
    hq, hkv = [(4, 2), (8, 2), (2, 2), (8, 8), (16, 4), (4, 1)][seed]
    D = 64 if seed % 2 else 128
    err, st = check_attention(synth.custom_shapes(p, n, lens), hq, hkv, D, 1000 + seed)
    _expect_schedule(st, schedule, hq, hkv)


@pytest.mark.parametrize("D", [64, 128])
def test_plain_causal_ragged(D, schedule):
    lens = [1, 127, 128, 129, 300, 513]
    s = synth.custom_shapes([L - 1 for L in lens], [0] * len(lens), [])
    check_attention(s, 4, 2, D, 7, causal=True)


@pytest.mark.parametrize("hq,hkv,D", [(6, 2, 128), (3, 1, 64), (1, 1, 128), (10, 2, 64)])
def test_odd_gqa_groups_and_single_head(hq, hkv, D, schedule):
    # odd groups (3, 5) and a lone head cannot pair two heads on one kv head:
    # the split schedule runs them whatever the request
    s = synth.custom_shapes([90, 260], [3, 5], [12, 0, 140, 7, 64, 1, 33, 129])
    err, st = check_attention(s, hq, hkv, D, 40 + hq)
    _expect_schedule(st, schedule, hq, hkv)


def test_single_item_and_empty_items(schedule):
    s = synth.custom_shapes([200, 0, 5], [1, 3, 4], [150, 0, 0, 0, 1, 0, 300, 2])
    check_attention(s, 4, 2, 128, 8)


def test_many_one_tile_units(schedule):
    # 600 requests of at most 113 rows: every unit has a single key tile, so
    # in the split schedule stream 1 has no tile at all and hands its row
    # statistics to the epilogue unit after unit, about 32 units per block
    rng = np.random.default_rng(77)
    B = 600
    p = rng.integers(0, 100, B)
    n = rng.integers(0, 3, B)
    lens = rng.integers(0, 10, int(n.sum()))
    err, st = check_attention(synth.custom_shapes(p, n, lens), 16, 8, 128, 77)
    assert st["n_qtiles"] == B
    assert st["n_full"] + st["n_partial"] == B          # one key tile per query tile
    _expect_schedule(st, schedule, 16, 8)


def test_strided_rows_and_no_lse():
    s = synth.custom_shapes([250, 60], [7, 3], [20, 1, 33, 64, 0, 5, 90, 17, 8, 41])
    check_attention(s, 4, 2, 128, 9, stride_pad=8, with_lse=False)


def test_strided_output_untouched_outside_rows():
    s = synth.custom_shapes([130], [4], [10, 20, 30, 40])
    lay, vals, o, lse, st, obuf = run_attention(s, 4, 2, 64, 10, stride_pad=16)
    pad = obuf[:, 4 * 64:]
    assert bool((pad == 7.0).all())


def test_one_shot_form():
    s = synth.custom_shapes([300], [12], list(range(0, 120, 10)))
    check_attention(s, 8, 4, 128, 11, plan_form=False)


def test_item_permutation_invariance_on_gpu():
    lens = [30, 5, 64, 17, 90, 2, 41, 8]
    perm = [5, 2, 7, 0, 3, 6, 1, 4]
    P = 500
    s1 = synth.custom_shapes([P], [8], lens)
    s2 = synth.custom_shapes([P], [8], [lens[i] for i in perm])
    lay1, v1, o1, _, _, _ = run_attention(s1, 4, 2, 128, 12)
    lay2 = lib.mis_build_layout([P], [8], [lens[i] for i in perm])
    idx = np.concatenate([np.arange(P + 1)] + [np.arange(lay1.item_offsets[i], lay1.item_offsets[i] + lens[i] + 1)
                                               for i in perm])
    dev = torch.device("cuda")
    q = v1["q"][idx].to(dev); k = v1["k"][idx].to(dev); v = v1["v"][idx].to(dev)
    o2 = torch.empty_like(q)
    plan = lib.Plan(lay2.cu_seqlens, lay2.prefix_len, lay2.item_ptr, lay2.item_offsets, 4, 2, 128)
    ws = torch.zeros(plan.workspace_size(), dtype=torch.uint8, device=dev)
    plan.create(ws)
    lib.mis_attention_fwd_plan(plan, q, k, v, o2, None)
    torch.cuda.synchronize()
    diff = (o2.float() - o1[torch.as_tensor(idx, device=dev)].float()).abs().max().item()
    assert diff <= ATTN_TOL


def test_qwen3_layer_full(schedule):
    w = synth.WORKLOADS["qwen3-0.6b-layer"]
    err, st = check_attention(synth.draw_shapes(w), w.hq, w.hkv, w.head_dim, w.seed)
    assert st["visible_pairs"] == 3120825
    _expect_schedule(st, schedule, w.hq, w.hkv)


def test_schedules_agree_on_a_long_unit_mix():
    # the two schedules reduce the same terms in different orders: their
    # outputs differ by rounding only (much less than the oracle tolerance)
    s = synth.custom_shapes([700, 40, 1500], [9, 1, 30], [3 + 3 * i for i in range(40)])
    outs = []
    for mode in (lib.SCHEDULE_PAIR, lib.SCHEDULE_SPLIT):
        with forced_schedule(mode):
            lay, v, o, lse, st, _ = run_attention(s, 8, 2, 128, 21)
            outs.append((o.float(), lse.clone()))
    assert (outs[0][0] - outs[1][0]).abs().max().item() <= 8e-3
    assert (outs[0][1] - outs[1][1]).abs().max().item() <= 1e-4


def test_random_batches_repeat_bit_for_bit_and_schedules_agree():
    # Seeded random batches (up to 12 requests, prefixes up to 1,500 tokens,
    # up to 150 items of up to 80 tokens, several head layouts). Each plan runs
    # twice and must give bit-identical O and LSE: every unit is computed by
    # one block in a fixed order, so any difference would be a race between
    # the kernel's warp roles. The two schedules must agree within rounding,
    # and every fourth batch is held against the oracle on sampled rows.
    rng = np.random.default_rng(4242)
    dev = torch.device("cuda")
    layouts = [(16, 8, 128), (8, 2, 64), (6, 2, 128), (32, 8, 128), (4, 4, 64), (10, 2, 128)]
    for case in range(16):
        B = int(rng.integers(1, 13))
        p = rng.integers(0, 1500, B)
        n = rng.integers(0, 150, B) * (rng.random(B) < 0.85)
        lens = rng.integers(0, 80, int(n.sum()))
        hq, hkv, D = layouts[case % len(layouts)]
        s = synth.custom_shapes(p, n, lens)
        lay = lib.mis_build_layout(s.prefix_tokens, s.n_items, s.item_lens)
        T = lay.T
        vals = synth.draw_values(500 + case, T, hq, hkv, D, want=("q", "k", "v"))
        q, k, v = (vals[x].to(dev) for x in ("q", "k", "v"))
        outs = []
        for mode in (lib.SCHEDULE_PAIR, lib.SCHEDULE_SPLIT):
            with forced_schedule(mode):
                plan = lib.Plan(lay.cu_seqlens, lay.prefix_len, lay.item_ptr, lay.item_offsets, hq, hkv, D)
            ws = torch.zeros(plan.workspace_size(), dtype=torch.uint8, device=dev)
            plan.create(ws)
            runs = []
            for fill in (7.0, 9.0):
                o = torch.full((T, hq, D), fill, dtype=torch.bfloat16, device=dev)
                lse = torch.full((hq, T), fill, dtype=torch.float32, device=dev)
                lib.mis_attention_fwd_plan(plan, q, k, v, o, lse)
                runs.append((o, lse))
            torch.cuda.synchronize()
            assert lib.mis_get_device_status(ws) == lib.MIS_OK
            assert torch.equal(runs[0][0], runs[1][0]) and torch.equal(runs[0][1], runs[1][1]), case
            outs.append(runs[0])
            plan.destroy()
        assert (outs[0][0].float() - outs[1][0].float()).abs().max().item() <= ATTN_TOL, case
        assert (outs[0][1] - outs[1][1]).abs().max().item() <= 2e-3, case
        if case % 4 == 0:
            olay = oracle_layout(s)
            rows = sorted(set(rng.choice(T, size=min(48, T), replace=False).tolist()) |
                          set(olay.delim_positions[:16].tolist()))
            ro, rl = O.attention(f64(vals["q"]), f64(vals["k"]), f64(vals["v"]), olay, rows=rows)
            for o, lse in outs:
                got = f64(o[torch.as_tensor(rows, device=dev)])
                assert np.abs(got - ro).max() <= ATTN_TOL, case
                assert np.abs(f64(lse)[:, rows].T - rl).max() <= 2e-3, case


@pytest.mark.parametrize("name", ["8b-large", "decision-256", "varlen-16", "prefix12k-50x150"])
def test_large_workloads_sampled_rows(name, schedule):
    w = synth.WORKLOADS[name]
    s = synth.draw_shapes(w)
    lay = oracle_layout(s)
    rows = _sample_rows(lay, 384, w.seed)
    check_attention(s, w.hq, w.hkv, w.head_dim, w.seed, rows=rows, cache_key=("sampled", name))


def test_planner_plans_match_oracle_across_buffer_reuse():
    # three batches through one planner: the third reuses the first staging buffer
    planner = lib.Planner()
    dev = torch.device("cuda")
    cases = [synth.custom_shapes([300], [5], [10, 0, 64, 129, 7]),
             synth.custom_shapes([17, 900], [2, 3], [5, 6, 40, 1, 250]),
             synth.custom_shapes([128], [8], [16] * 8)]
    outs = []
    for n, s in enumerate(cases):
        lay = lib.mis_build_layout(s.prefix_tokens, s.n_items, s.item_lens)
        v = synth.draw_values(50 + n, lay.T, 4, 2, 128, want=("q", "k", "v"))
        q, k, vv = v["q"].to(dev), v["k"].to(dev), v["v"].to(dev)
        o = torch.empty_like(q)
        probe = lib.Plan(lay.cu_seqlens, lay.prefix_len, lay.item_ptr, lay.item_offsets, 4, 2, 128)
        wsz = probe.workspace_size()
        ws = torch.full((wsz + 4 * lay.M + 64,), 0xAB, dtype=torch.uint8, device=dev)
        plan = planner.plan(lay.cu_seqlens, lay.prefix_len, lay.item_ptr, lay.item_offsets, 4, 2, 128,
                            ws, extra=lay.delim_positions)
        lib.mis_attention_fwd_plan(plan, q, k, vv, o, None)
        lib.mis_attention_fwd_plan(plan, q, k, vv, o, None)     # a second launch of the same plan
        outs.append((s, v, o, ws, plan, wsz, lay))
    torch.cuda.synchronize()
    for s, v, o, ws, plan, wsz, lay in outs:
        assert lib.mis_get_device_status(ws) == lib.MIS_OK
        # the side payload landed right after the plan
        side = ws[wsz:wsz + 4 * lay.M].view(torch.int32).cpu().numpy()
        assert np.array_equal(side, lay.delim_positions)
        ro, _ = O.attention(f64(v["q"]), f64(v["k"]), f64(v["v"]), oracle_layout(s))
        assert np.abs(f64(o) - ro).max() <= ATTN_TOL
    planner.destroy()


def test_pointer_and_stride_refusals_launch_nothing():
    # Each refusal below comes from the host checks of mis_attention_fwd_plan,
    # before any launch: the output keeps its fill and the status stays clean.
    s = synth.custom_shapes([130], [3], [10, 20, 30])
    lay = lib.mis_build_layout(s.prefix_tokens, s.n_items, s.item_lens)
    dev = torch.device("cuda")
    T, hq, hkv, D = lay.T, 4, 2, 64
    q = torch.zeros(T, hq, D, dtype=torch.bfloat16, device=dev)
    k = torch.zeros(T, hkv, D, dtype=torch.bfloat16, device=dev)
    o = torch.full((T, hq, D), 7.0, dtype=torch.bfloat16, device=dev)
    lse = torch.full((hq, T), 7.0, dtype=torch.float32, device=dev)
    plan = lib.Plan(lay.cu_seqlens, lay.prefix_len, lay.item_ptr, lay.item_offsets, hq, hkv, D)
    ws = torch.zeros(plan.workspace_size(), dtype=torch.uint8, device=dev)
    plan.create(ws)
    L = lib.load()
    qp, kp, op, lp = q.data_ptr(), k.data_ptr(), o.data_ptr(), lse.data_ptr()
    def call(qa=qp, oa=op, la=None, qs=hq * D, ks=hkv * D, os_=hq * D):
        return L.mis_attention_fwd_plan(plan._h, qa, kp, kp, oa, la, qs, ks, ks, os_, None)
    assert call(qa=qp + 2) == lib.MIS_ERR_INVALID_ARG          # Q not 16-byte aligned
    assert call(oa=op + 8) == lib.MIS_ERR_INVALID_ARG          # O not 16-byte aligned
    assert call(la=lp + 2) == lib.MIS_ERR_INVALID_ARG          # LSE not 4-byte aligned
    assert call(qs=hq * D - 8) == lib.MIS_ERR_SHAPE            # Q rows overlap
    assert call(ks=hkv * D + 4) == lib.MIS_ERR_SHAPE           # not a multiple of 8 elements
    torch.cuda.synchronize()
    assert bool((o == 7.0).all()) and bool((lse == 7.0).all())
    assert lib.mis_get_device_status(ws) == lib.MIS_OK
    plan.destroy()

