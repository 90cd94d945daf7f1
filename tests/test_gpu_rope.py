"""GPU parity of mis_rope_qk against the fp64 oracle, and of rotary
attention at the reused position ids ("From Generation to Scoring", Section
4.1: with the mask and the reused position ids every item's rows equal those
of its own single-item prompt)."""
import numpy as np
import pytest
import torch

import oracle as O
from ranking_prefill_gb300 import lib, synth
from gpu_helpers import ATTN_TOL, SCORE_TOL, f64

pytestmark = pytest.mark.gpu

ROPE_TOL = 8e-3    # max |gpu - oracle| / max(|oracle|, 1): bf16 rounding (2^-9) + fp32 angle rounding


def _rope_err(got, ref):
    return float((np.abs(f64(got) - ref) / np.maximum(np.abs(ref), 1.0)).max())


@pytest.mark.parametrize("hq,hkv,D,base,maxpos,pad", [(16, 8, 128, 1e6, 5000, 0),
                                                       (4, 4, 64, 1e4, 20000, 8),
                                                       (32, 8, 128, 5e5, 300, 16)])
def test_rope_matches_oracle(hq, hkv, D, base, maxpos, pad):
    T = 1500
    rng = np.random.default_rng(D + hq)
    pos = rng.integers(0, maxpos, T).astype(np.int32)
    v = synth.draw_values(int(hq + D), T, hq, hkv, D, want=("q", "k"))
    dev = torch.device("cuda")

    def place(t, h):
        buf = torch.zeros(T, h * D + pad, dtype=torch.bfloat16, device=dev)
        view = buf.as_strided((T, h, D), (h * D + pad, D, 1))
        view.copy_(t.to(dev))
        return view
    q, k = place(v["q"], hq), place(v["k"], hkv)
    qo, ko = place(torch.zeros_like(v["q"]), hq), place(torch.zeros_like(v["k"]), hkv)
    pd = torch.as_tensor(pos, device=dev)
    lib.mis_rope_qk(q, k, qo, ko, pd, base)
    torch.cuda.synchronize()
    assert _rope_err(qo, O.rope(f64(v["q"]), pos, base)) <= ROPE_TOL
    assert _rope_err(ko, O.rope(f64(v["k"]), pos, base)) <= ROPE_TOL
    assert bool((q.float() == v["q"].to(dev).float()).all())          # inputs untouched
    # in place gives the same bits as out of place
    lib.mis_rope_qk(q, k, q, k, pd, base)
    torch.cuda.synchronize()
    assert bool((q.float() == qo.float()).all()) and bool((k.float() == ko.float()).all())


def test_rotary_mis_attention_matches_oracle():
    s = synth.custom_shapes([300, 40], [6, 3], [12, 0, 40, 7, 130, 2, 25, 1, 60])
    lay = lib.mis_build_layout(s.prefix_tokens, s.n_items, s.item_lens)
    hq, hkv, D = 8, 2, 128
    v = synth.draw_values(51, lay.T, hq, hkv, D, want=("q", "k", "v"))
    dev = torch.device("cuda")
    q, k, vv = (v[x].to(dev) for x in ("q", "k", "v"))
    qr, kr = torch.empty_like(q), torch.empty_like(k)
    lib.mis_rope_qk(q, k, qr, kr, torch.as_tensor(lay.position_ids, device=dev))
    o = torch.empty_like(q)
    plan = lib.Plan(lay.cu_seqlens, lay.prefix_len, lay.item_ptr, lay.item_offsets, hq, hkv, D)
    ws = torch.zeros(plan.workspace_size(), dtype=torch.uint8, device=dev)
    plan.create(ws)
    lib.mis_attention_fwd_plan(plan, qr, kr, vv, o, None)
    torch.cuda.synchronize()
    assert lib.mis_get_device_status(ws) == lib.MIS_OK
    olay = O.build_layout(s.prefix_tokens, s.n_items, s.item_lens)
    ro, _ = O.attention(O.rope(f64(v["q"]), olay.position_ids), O.rope(f64(v["k"]), olay.position_ids),
                        f64(v["v"]), olay)
    assert np.abs(f64(o) - ro).max() <= ATTN_TOL


def test_rotary_mis_equals_single_item_prompts_on_gpu():
    # one query, 40 items: MIS with reused positions against 40 separate
    # [q; item] prompts at their own positions, through rope -> attention ->
    # scoring (the attention output as hidden state)
    pool = synth.sweep_pool(1, vocab=3000, seed=21)
    pool.query_tokens[0] = 700
    pool.cand_lens = pool.cand_lens[:, :40].copy()
    P, lens = int(pool.query_tokens[0]), pool.cand_lens[0]
    hq, hkv, D = 8, 4, 128
    dev = torch.device("cuda")
    mis = lib.mis_build_layout([P], [40], lens)
    olay = O.build_layout([P], [40], lens)
    v = synth.draw_values(52, mis.T, hq, hkv, D, want=("q", "k", "v"))
    S = P + 1
    rows = np.concatenate([np.concatenate([np.arange(S), np.arange(olay.item_offsets[i], olay.item_ends[i])])
                           for i in range(40)])
    sis = lib.mis_build_layout([P] * 40, [1] * 40, lens)
    g = torch.Generator().manual_seed(53)
    w_lm = (torch.randn(3000, hq * D, generator=g) * 0.02).to(torch.bfloat16).to(dev)
    labels = [int(x) for x in pool.labels]

    def run(lay, idx):
        t = torch.as_tensor(idx, dtype=torch.long)
        q, k, vv = (v[x][t].to(dev) for x in ("q", "k", "v"))
        lib.mis_rope_qk(q, k, q, k, torch.as_tensor(lay.position_ids, device=dev))
        o = torch.empty_like(q)
        plan = lib.Plan(lay.cu_seqlens, lay.prefix_len, lay.item_ptr, lay.item_offsets, hq, hkv, D)
        ws = torch.zeros(plan.workspace_size(), dtype=torch.uint8, device=dev)
        plan.create(ws)
        lib.mis_attention_fwd_plan(plan, q, k, vv, o, None)
        out = torch.empty(lay.M, 2, dtype=torch.float32, device=dev)
        sws = torch.zeros(lib.mis_label_scores_workspace_size(lay.M, hq * D, 3000, 2),
                          dtype=torch.uint8, device=dev)
        rd = torch.as_tensor(lay.delim_positions, device=dev)
        lib.mis_label_scores(o.view(lay.T, hq * D), w_lm, rd, labels, out, None, sws)
        torch.cuda.synchronize()
        assert lib.mis_get_device_status(ws) == lib.MIS_OK
        return o[rd.long()].float(), out
    om, sm = run(mis, np.arange(mis.T))
    os_, ss = run(sis, rows)
    assert (om - os_).abs().max().item() <= 1e-2
    assert (sm - ss).abs().max().item() <= SCORE_TOL


# ------------------------------------------------ Q rotated on load (fused) ----

@pytest.fixture(params=[lib.SCHEDULE_PAIR, lib.SCHEDULE_SPLIT], ids=["pair", "split"])
def schedule(request):
    from gpu_helpers import forced_schedule
    with forced_schedule(request.param):
        yield request.param


def _fused_case(shapes, hq, hkv, D, seed, base=1.0e6, stride_pad=0):
    """Q unrotated through mis_attention_fwd_plan_rope, K rotated by the K-only
    mis_rope_qk at the layout's position ids; returns (oracle layout, O, LSE,
    oracle O, oracle LSE, status, plan stats)."""
    lay = lib.mis_build_layout(shapes.prefix_tokens, shapes.n_items, shapes.item_lens)
    v = synth.draw_values(seed, lay.T, hq, hkv, D, want=("q", "k", "v"))
    dev = torch.device("cuda")
    T = lay.T

    def place(t, h):
        buf = torch.zeros(T, h * D + stride_pad, dtype=torch.bfloat16, device=dev)
        view = buf.as_strided((T, h, D), (h * D + stride_pad, D, 1))
        view.copy_(t.to(dev))
        return view
    q, k, vv = place(v["q"], hq), place(v["k"], hkv), place(v["v"], hkv)
    q_before = q.clone()
    pos = torch.as_tensor(lay.position_ids, device=dev)
    kr = place(torch.zeros_like(v["k"]), hkv)
    lib.mis_rope_qk(None, k, None, kr, pos, base, Hq=hq)
    o = torch.full((T, hq, D), 7.0, dtype=torch.bfloat16, device=dev)
    lse = torch.full((hq, T), 7.0, dtype=torch.float32, device=dev)
    plan = lib.Plan(lay.cu_seqlens, lay.prefix_len, lay.item_ptr, lay.item_offsets, hq, hkv, D)
    ws = torch.zeros(plan.workspace_size(), dtype=torch.uint8, device=dev)
    plan.create(ws)
    lib.mis_attention_fwd_plan_rope(plan, q, kr, vv, o, lse, base)
    o2, lse2 = torch.empty_like(o), torch.empty_like(lse)
    lib.mis_attention_fwd_plan_rope(plan, q, kr, vv, o2, lse2, base)
    torch.cuda.synchronize()
    status = lib.mis_get_device_status(ws)
    assert torch.equal(q, q_before)                     # Q is rotated in shared memory only
    assert torch.equal(o, o2) and torch.equal(lse, lse2)   # the same bits on a second launch
    olay = O.build_layout(shapes.prefix_tokens, shapes.n_items, shapes.item_lens)
    # the rotated Q and K are held in bf16 on the GPU (Q in shared memory, K
    # in HBM): the oracle attends over the fp64 rotation rounded to bf16
    # (nearest even) once, the storage precision the kernel decides in
    bf = lambda x: torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    qr = O.rope(f64(v["q"]), olay.position_ids, base)
    kr64 = O.rope(f64(v["k"]), olay.position_ids, base)
    ro, rl = O.attention(bf(qr), bf(kr64), f64(v["v"]), olay)
    # and over the exact rotation, for the output tolerance of the method
    ro_exact, _ = O.attention(qr, kr64, f64(v["v"]), olay)
    assert np.abs(f64(o) - ro_exact).max() <= ATTN_TOL
    return olay, o, lse, ro, rl, status, plan.stats()


@pytest.mark.parametrize("hq,hkv,D,seed,base", [(8, 2, 128, 61, 1e6), (4, 2, 64, 62, 1e4),
                                                (6, 2, 128, 63, 5e5), (16, 8, 128, 64, 1e6)])
def test_q_rotated_on_load_matches_oracle(hq, hkv, D, seed, base, schedule):
    # several tiles, ragged tails, empty items, long items straddling tiles
    s = synth.custom_shapes([300, 40, 700], [6, 3, 9],
                            [12, 0, 40, 7, 130, 2, 25, 1, 60, 3, 3, 200, 64, 0, 9, 77, 5, 31])
    olay, o, lse, ro, rl, status, st = _fused_case(s, hq, hkv, D, seed, base)
    assert status == lib.MIS_OK
    assert np.abs(f64(o) - ro).max() <= ATTN_TOL
    assert np.abs(f64(lse).T - rl).max() <= 2e-3
    want = schedule if (hq // hkv) % 2 == 0 else lib.SCHEDULE_SPLIT
    assert st["schedule"] == want


def test_q_rotated_on_load_strided_and_qwen3_layer(schedule):
    w = synth.WORKLOADS["qwen3-0.6b-layer"]
    olay, o, lse, ro, rl, status, _ = _fused_case(synth.draw_shapes(w), w.hq, w.hkv, w.head_dim,
                                                  w.seed, stride_pad=8)
    assert status == lib.MIS_OK
    assert np.abs(f64(o) - ro).max() <= ATTN_TOL
    assert np.abs(f64(lse).T - rl).max() <= 2e-3


def test_q_rotated_on_load_long_positions(schedule):
    # a 12k-token shared set: angles up to 12,000 rad, reduced on the device
    s = synth.custom_shapes([12000], [5], [150, 3, 0, 64, 100])
    olay, o, lse, ro, rl, status, _ = _fused_case(s, 4, 2, 128, 67)
    assert status == lib.MIS_OK
    assert np.abs(f64(o) - ro).max() <= ATTN_TOL
    assert np.abs(f64(lse).T - rl).max() <= 2e-3


def test_q_rotated_on_load_equals_rotating_first():
    # the fused form and the two-pass form (mis_rope_qk on Q and K, then the
    # plain attention call) agree to bf16 rounding of the rotated Q
    s = synth.custom_shapes([500, 90], [20, 4], list(range(3, 63, 3)) + [1, 2, 100, 0])
    hq, hkv, D = 16, 8, 128
    lay = lib.mis_build_layout(s.prefix_tokens, s.n_items, s.item_lens)
    v = synth.draw_values(65, lay.T, hq, hkv, D, want=("q", "k", "v"))
    dev = torch.device("cuda")
    q, k, vv = (v[x].to(dev) for x in ("q", "k", "v"))
    pos = torch.as_tensor(lay.position_ids, device=dev)
    qr, kr = torch.empty_like(q), torch.empty_like(k)
    lib.mis_rope_qk(q, k, qr, kr, pos)
    kr2 = torch.empty_like(k)
    lib.mis_rope_qk(None, k, None, kr2, pos, Hq=hq)
    assert torch.equal(kr, kr2)                      # the K-only pass gives the same K bits
    plan = lib.Plan(lay.cu_seqlens, lay.prefix_len, lay.item_ptr, lay.item_offsets, hq, hkv, D)
    ws = torch.zeros(plan.workspace_size(), dtype=torch.uint8, device=dev)
    plan.create(ws)
    o1, o2 = torch.empty_like(q), torch.empty_like(q)
    lib.mis_attention_fwd_plan(plan, qr, kr, vv, o1, None)
    lib.mis_attention_fwd_plan_rope(plan, q, kr, vv, o2, None)
    torch.cuda.synchronize()
    assert lib.mis_get_device_status(ws) == lib.MIS_OK
    assert (o1.float() - o2.float()).abs().max().item() <= 1e-2


def test_fused_rope_refuses_requests_beyond_its_position_range():
    s = synth.custom_shapes([(1 << 17)], [0], [])
    lay = lib.mis_build_layout(s.prefix_tokens, s.n_items, s.item_lens, with_positions=False)
    dev = torch.device("cuda")
    plan = lib.Plan(lay.cu_seqlens, lay.prefix_len, lay.item_ptr, lay.item_offsets, 2, 2, 64)
    ws = torch.zeros(plan.workspace_size(), dtype=torch.uint8, device=dev)
    plan.create(ws)
    q = torch.zeros(lay.T, 2, 64, dtype=torch.bfloat16, device=dev)
    o = torch.full_like(q, 7.0)
    with pytest.raises(lib.MisError) as e:
        lib.mis_attention_fwd_plan_rope(plan, q, q, q, o, None)
    assert e.value.status == lib.MIS_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert bool((o == 7.0).all())                    # nothing was launched


@pytest.mark.parametrize("cached", [False, True], ids=["packed", "cached"])
def test_k_rotated_at_the_plans_positions(cached):
    # mis_rope_k_plan derives the reused position ids from the plan: bit for
    # bit the K of mis_rope_qk at the layout's position ids
    s = synth.custom_shapes([300, 0, 700], [6, 2, 9],
                            [12, 0, 40, 7, 130, 2, 25, 1, 60, 3, 3, 200, 64, 0, 9, 77, 5])
    hkv, D = 4, 128
    dev = torch.device("cuda")
    if cached:
        lay = O.cached_layout([0, 400, 100], [301, 1, 10], s.n_items, s.item_lens)
        pos = lay.position_ids
        plan = lib.CachedPlan(lay.cu_seqlens, lay.item_ptr, lay.item_offsets, [0, 400, 100],
                              [301, 1, 10], 500, 8, hkv, D)
    else:
        lay = lib.mis_build_layout(s.prefix_tokens, s.n_items, s.item_lens)
        pos = lay.position_ids
        plan = lib.Plan(lay.cu_seqlens, lay.prefix_len, lay.item_ptr, lay.item_offsets, 8, hkv, D)
    T = int(lay.cu_seqlens[-1])
    v = synth.draw_values(68, T, 8, hkv, D, want=("k",))
    k = v["k"].to(dev)
    ws = torch.zeros(plan.workspace_size(), dtype=torch.uint8, device=dev)
    plan.create(ws)
    k1, k2 = torch.empty_like(k), torch.empty_like(k)
    lib.mis_rope_qk(None, k, None, k1, torch.as_tensor(pos, device=dev), Hq=8)
    lib.mis_rope_k_plan(plan, k, k2)
    torch.cuda.synchronize()
    assert torch.equal(k1, k2)
    assert _rope_err(k2, O.rope(f64(v["k"]), pos)) <= ROPE_TOL
