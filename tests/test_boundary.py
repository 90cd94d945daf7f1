"""Host-side checks of the C-ABI library (no GPU needed).

* the shared library loads and exports every function include/mis.h declares;
* mis_build_layout equals the oracle's packing bit for bit;
* the planner's tile map and visible-pair count equal the oracle's
  element-by-element classification bit for bit;
* malformed descriptors and arguments return the documented status codes
  before any device work is enqueued.
"""
import ctypes as C
import os
import re

import numpy as np
import pytest

import oracle as O
from ranking_prefill_gb300 import lib, synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(lib.LIB_PATH):
        from ranking_prefill_gb300 import build
        build.build()
    return lib.load()


def test_exports_every_declared_symbol(L):
    hdr = open(os.path.join(ROOT, "include", "mis.h")).read()
    declared = set(re.findall(r"^\s*(?:[\w\s\*]+?)\b(mis_\w+)\s*\(", hdr, flags=re.M))
    assert declared == set(lib.EXPORTS), declared ^ set(lib.EXPORTS)
    for name in declared:
        assert hasattr(L, name)
    assert L.mis_abi_version() == 2
    for st in range(8):
        assert lib.mis_status_string(st) != "unknown status"


def _shapes_cases():
    # every MIS workload the benchmark and the parity tests run (the five
    # configurations plus the page's 12k-prefix shape), then random batches
    for name in ("tiny", "qwen3-0.6b-layer", "varlen-16", "8b-large", "decision-256",
                 "prefix12k-50x150"):
        yield synth.draw_shapes(synth.WORKLOADS[name])
    rng = np.random.default_rng(123)
    for _ in range(30):
        B = int(rng.integers(1, 5))
        p = rng.integers(0, 300, B)
        n = rng.integers(0, 12, B)
        lens = rng.integers(0, 70, int(n.sum()))
        yield synth.custom_shapes(p, n, lens)


def test_layout_bit_exact(L):
    for s in _shapes_cases():
        got = lib.mis_build_layout(s.prefix_tokens, s.n_items, s.item_lens)
        ref = O.build_layout(s.prefix_tokens, s.n_items, s.item_lens)
        for f in ("cu_seqlens", "prefix_len", "item_ptr", "item_offsets", "delim_positions",
                  "position_ids"):
            assert np.array_equal(getattr(got, f), getattr(ref, f)), f


def _plan(lay, hq=4, hkv=2, D=64):
    return lib.Plan(lay.cu_seqlens, lay.prefix_len, lay.item_ptr, lay.item_offsets, hq, hkv, D)


def test_tile_map_and_pairs_bit_exact(L):
    cases = list(_shapes_cases())
    for s in cases:
        lay = O.build_layout(s.prefix_tokens, s.n_items, s.item_lens)
        p = lib.Plan.host_only(lay.cu_seqlens, lay.prefix_len, lay.item_ptr, lay.item_offsets, 4, 2, 64)
        got = p.tile_map()
        ref = O.tile_map(lay, 128, 128)
        assert got.shape == ref.shape and np.array_equal(got, ref)
        st = p.stats()
        assert st["n_full"] == int((ref[:, 3] == O.FULL).sum())
        assert st["n_partial"] == int((ref[:, 3] == O.PARTIAL).sum())
        if lay.T <= 6000:
            assert st["visible_pairs"] == O.pair_count(lay)


def test_schedule_override_and_units(L):
    s = synth.draw_shapes(synth.WORKLOADS["qwen3-0.6b-layer"])
    lay = lib.mis_build_layout(s.prefix_tokens, s.n_items, s.item_lens, with_positions=False)
    args = (lay.cu_seqlens, lay.prefix_len, lay.item_ptr, lay.item_offsets)
    prev = lib.mis_set_schedule(lib.SCHEDULE_AUTO)
    ref_map = lib.Plan.host_only(*args, 16, 8, 128).tile_map()
    try:
        for mode, hq, hkv, want, per_tile in [(lib.SCHEDULE_PAIR, 16, 8, lib.SCHEDULE_PAIR, 8),
                                              (lib.SCHEDULE_SPLIT, 16, 8, lib.SCHEDULE_SPLIT, 16),
                                              (lib.SCHEDULE_PAIR, 12, 4, lib.SCHEDULE_SPLIT, 12),
                                              (lib.SCHEDULE_AUTO, 6, 6, lib.SCHEDULE_SPLIT, 6)]:
            lib.mis_set_schedule(mode)
            st = lib.Plan.host_only(*args, hq, hkv, 128).stats()
            assert st["schedule"] == want                 # odd GQA groups always split
            assert st["n_units"] == st["n_qtiles"] * per_tile
            # the schedule changes the execution order only, never the tile map
            assert np.array_equal(lib.Plan.host_only(*args, hq, hkv, 128).tile_map(), ref_map)
        lib.mis_set_schedule(lib.SCHEDULE_AUTO)
        st = lib.Plan.host_only(*args, 16, 8, 128).stats()
        assert st["schedule"] in (lib.SCHEDULE_PAIR, lib.SCHEDULE_SPLIT)
        with pytest.raises(lib.MisError):
            lib.mis_set_schedule(7)
        assert lib.mis_set_schedule(lib.SCHEDULE_AUTO) == lib.SCHEDULE_AUTO   # 7 changed nothing
    finally:
        lib.mis_set_schedule(prev)


def test_causal_plan_is_plain_causal(L):
    lens = [1, 127, 128, 129, 300]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    p = lib.Plan.host_only(cu, lens, None, None, 4, 2, 128)
    ref = O.tile_map(O.causal_layout(lens), 128, 128)
    assert np.array_equal(p.tile_map(), ref)
    st = p.stats()
    assert st["n_tiles"] == st["n_causal_tiles"]
    assert st["visible_pairs"] == sum(L_ * (L_ + 1) // 2 for L_ in lens)


def test_workspace_size_and_validation(L):
    s = synth.draw_shapes(synth.WORKLOADS["tiny"])
    lay = lib.mis_build_layout(s.prefix_tokens, s.n_items, s.item_lens)
    p = _plan(lay)
    assert p.workspace_size() > 0
    # descriptor errors
    def status(**kw):
        args = dict(cu=lay.cu_seqlens, pl=lay.prefix_len, ip=lay.item_ptr, io=lay.item_offsets,
                    hq=4, hkv=2, D=64)
        args.update(kw)
        pl = lib.Plan(args["cu"], args["pl"], args["ip"], args["io"], args["hq"], args["hkv"], args["D"])
        h = C.c_void_p()
        return L.mis_plan_create(C.byref(pl.desc), None, 0, None, C.byref(h))
    assert status() == lib.MIS_OK                      # host-only plan
    assert status(hq=3) == lib.MIS_ERR_SHAPE
    assert status(D=96) == lib.MIS_ERR_UNSUPPORTED
    assert status(pl=[0]) == lib.MIS_ERR_SHAPE
    assert status(pl=[300]) == lib.MIS_ERR_SHAPE
    bad = lay.item_offsets.copy(); bad[3] += 1
    assert status(io=bad) == lib.MIS_OK                    # still a valid partition
    bad = lay.item_offsets.copy(); bad[0] += 1
    assert status(io=bad) == lib.MIS_ERR_SHAPE            # first item must follow Q
    bad = lay.item_offsets.copy(); bad[4] = bad[3]
    assert status(io=bad) == lib.MIS_ERR_SHAPE            # empty item set
    assert status(ip=None, io=None) == lib.MIS_ERR_SHAPE  # rows after Q belong to nothing
    assert status(ip=None, io=None, pl=[lay.T]) == lib.MIS_OK   # plain causal is valid
    pl = _plan(lay)
    pl.desc.T = lay.T + 1                                  # cu_seqlens[B] != T
    h = C.c_void_p()
    assert L.mis_plan_create(C.byref(pl.desc), None, 0, None, C.byref(h)) == lib.MIS_ERR_SHAPE
    cu = lay.cu_seqlens.copy(); cu[0] = 1
    assert status(cu=cu) == lib.MIS_ERR_SHAPE
    # misaligned workspace
    h = C.c_void_p()
    assert L.mis_plan_create(C.byref(p.desc), C.c_void_p(0x1001), 1 << 30, None, C.byref(h)) == \
        lib.MIS_ERR_WORKSPACE


def test_label_scores_argument_errors(L):
    labels = np.array([1, 2], np.int32)
    def call(M=4, d=128, V=1000, K=2, lab=labels, ws=None, wsb=0, hidden=0x1000, stride=None,
             delim=0x3000):
        return L.mis_label_scores(C.c_void_p(hidden), d if stride is None else stride, 100,
                                  C.c_void_p(0x2000), d, V, C.c_void_p(delim), M,
                                  lab.ctypes.data_as(C.POINTER(C.c_int32)),
                                  K, C.c_void_p(0x4000), None, ws, wsb, None)
    assert call() == lib.MIS_ERR_WORKSPACE
    assert call(d=96) == lib.MIS_ERR_UNSUPPORTED
    assert call(d=8256) == lib.MIS_ERR_UNSUPPORTED              # above the widest model
    assert call(K=0) == lib.MIS_ERR_INVALID_ARG
    assert call(hidden=0x1008) == lib.MIS_ERR_INVALID_ARG      # not 16-byte aligned (TMA)
    assert call(delim=0x3002) == lib.MIS_ERR_INVALID_ARG
    assert call(stride=64) == lib.MIS_ERR_SHAPE                # row stride below d
    assert call(stride=132) == lib.MIS_ERR_SHAPE               # not a multiple of 8 elements
    assert call(K=17, lab=np.arange(17, dtype=np.int32)) == lib.MIS_ERR_UNSUPPORTED
    assert call(lab=np.array([1, 1000], np.int32)) == lib.MIS_ERR_INVALID_ARG
    assert call(lab=np.array([-1, 3], np.int32)) == lib.MIS_ERR_INVALID_ARG
    assert call(M=-1) == lib.MIS_ERR_INVALID_ARG
    assert call(ws=C.c_void_p(0x10010), wsb=1 << 40) == lib.MIS_ERR_WORKSPACE   # misaligned
    need = lib.mis_label_scores_workspace_size(4, 128, 1000, 2)
    assert need > 0
    assert call(ws=C.c_void_p(0x100000), wsb=need - 1) == lib.MIS_ERR_WORKSPACE
    assert lib.mis_label_scores_workspace_size(4, 128, 0, 2) == 0


def test_layout_argument_errors(L):
    with pytest.raises(lib.MisError) as e:
        lib.mis_build_layout([-1], [0], [])
    assert e.value.status == lib.MIS_ERR_INVALID_ARG
    with pytest.raises(lib.MisError):
        lib.mis_build_layout([4], [2], [3, -2])
    with pytest.raises(lib.MisError) as e:
        lib.mis_build_layout([2 ** 31 - 2], [0], [])
    assert e.value.status == lib.MIS_ERR_SHAPE


def test_setwise_layout_bit_exact(L):
    rng = np.random.default_rng(77)
    cases = [([40], [3], [7, 12, 9]), ([0, 5], [2, 0], [3, 4]), ([1], [0], [])]
    sw = synth.draw_shapes(synth.WORKLOADS["setwise-256"])      # the benchmark's setwise batch
    cases.append((sw.prefix_tokens.tolist(), sw.n_items.tolist(), sw.item_lens.tolist()))
    for _ in range(20):
        B = int(rng.integers(1, 6))
        qt = rng.integers(0, 300, B)
        n = rng.integers(0, 12, B)
        qt[(qt == 0) & (n == 0)] = 1
        cases.append((qt.tolist(), n.tolist(), rng.integers(0, 80, int(n.sum())).tolist()))
    for qt, n, lens in cases:
        got = lib.mis_build_setwise_layout(qt, n, lens)
        ref = O.setwise_layout(qt, n, lens)
        assert np.array_equal(got.cu_seqlens, ref.causal.cu_seqlens)
        assert np.array_equal(got.prefix_len, ref.causal.prefix_len)   # plain causal
        assert np.array_equal(got.marker_positions, ref.marker_positions)
        assert np.array_equal(got.position_ids, ref.causal.position_ids)
        # the attention plan of a setwise batch is the causal plan
        p = lib.Plan.host_only(got.cu_seqlens, got.prefix_len, None, None, 4, 2, 64)
        assert np.array_equal(p.tile_map(), O.tile_map(ref.causal, 128, 128))
    with pytest.raises(lib.MisError) as e:
        lib.mis_build_setwise_layout([0, 3], [0, 1], [2])           # empty request
    assert e.value.status == lib.MIS_ERR_SHAPE
    with pytest.raises(lib.MisError) as e:
        lib.mis_build_setwise_layout([3], [1], [-2])
    assert e.value.status == lib.MIS_ERR_INVALID_ARG


def test_rope_argument_checks(L):
    # all rejected (or, for T = 0, accepted) before anything is enqueued
    fake = C.c_void_p(1 << 20)          # 16-byte aligned, never dereferenced
    ok_args = dict(qs=16 * 128, ks=8 * 128, T=4, Hq=16, Hkv=8, D=128, base=1e6)

    def call(q=fake, k=fake, qo=fake, ko=fake, pos=fake, **kw):
        a = dict(ok_args, **kw)
        return L.mis_rope_qk(q, k, qo, ko, a["qs"], a["ks"], a["qs"], a["ks"], a["T"], a["Hq"],
                             a["Hkv"], a["D"], pos, a["base"], None)
    assert call(T=0) == lib.MIS_OK
    assert call(D=96) == lib.MIS_ERR_UNSUPPORTED
    assert call(base=1.0) == lib.MIS_ERR_INVALID_ARG
    assert call(base=float("inf")) == lib.MIS_ERR_INVALID_ARG
    assert call(pos=None) == lib.MIS_ERR_INVALID_ARG
    assert call(q=C.c_void_p((1 << 20) + 8)) == lib.MIS_ERR_INVALID_ARG      # misaligned
    assert call(qs=16 * 128 - 8) == lib.MIS_ERR_SHAPE                         # row too short
    assert call(ks=8 * 128 + 4) == lib.MIS_ERR_SHAPE                          # stride not 8-multiple
    assert call(Hq=0) == lib.MIS_ERR_INVALID_ARG
    # K only: q and q_out both null; one of them alone is refused
    assert call(q=None, qo=None, T=0) == lib.MIS_OK
    assert call(q=None) == lib.MIS_ERR_INVALID_ARG
    assert call(qo=None) == lib.MIS_ERR_INVALID_ARG
    assert call(q=None, qo=None, ks=8 * 128 - 8) == lib.MIS_ERR_SHAPE


def test_fused_rope_attention_argument_checks(L):
    fake = C.c_void_p(1 << 20)
    s = synth.custom_shapes([130], [3], [10, 20, 30])
    lay = lib.mis_build_layout(s.prefix_tokens, s.n_items, s.item_lens)
    args = (lay.cu_seqlens, lay.prefix_len, lay.item_ptr, lay.item_offsets, 4, 2, 64)
    host = lib.Plan.host_only(*args)
    strides = (4 * 64, 2 * 64, 2 * 64, 4 * 64)
    call = lambda h, base=1e6: L.mis_attention_fwd_plan_rope(h, fake, fake, fake, fake, None,
                                                             *strides, base, None)
    assert call(None) == lib.MIS_ERR_INVALID_ARG
    assert call(host._h) == lib.MIS_ERR_WORKSPACE                 # no device workspace
    cl = O.cached_layout([0], [10], [2], [3, 4])
    cached = lib.CachedPlan.host_only(cl.cu_seqlens, cl.item_ptr, cl.item_offsets, [0], [10], 10,
                                      4, 2, 64)
    assert call(cached._h) == lib.MIS_ERR_INVALID_ARG             # cached plans: not this call
    kcall = lambda h, k=fake, ko=fake, ks=2 * 64, base=1e6: L.mis_rope_k_plan(h, k, ko, ks, ks, base,
                                                                            None)
    assert kcall(None) == lib.MIS_ERR_INVALID_ARG
    assert kcall(host._h) == lib.MIS_ERR_WORKSPACE


def _cached_random(rng):
    B = int(rng.integers(1, 4))
    S = rng.integers(1, 400, B)
    n = rng.integers(1, 9, B)
    lens = rng.integers(0, 150, int(n.sum()))
    cstart, t = np.zeros(B, np.int64), int(rng.integers(0, 50))
    for b in rng.permutation(B):
        cstart[b] = t
        t += int(S[b]) + int(rng.integers(0, 70))
    return cstart, S, n, lens, t


def test_cached_plan_tile_map_and_pairs_bit_exact(L):
    rng = np.random.default_rng(91)
    for case in range(25):
        cstart, S, n, lens, cache_T = _cached_random(rng)
        if case == 0:
            S = np.array([128, 129, 127][: len(S)] + [1] * (len(S) - 3))[: len(S)]
        cl = O.cached_layout(cstart, S, n, lens)
        p = lib.CachedPlan.host_only(cl.cu_seqlens, cl.item_ptr, cl.item_offsets, cstart, S,
                                     cache_T, 4, 2, 128)
        assert np.array_equal(p.tile_map(), O.tile_map_cached(cl, 128, 128))
        pairs = sum(int(S[cl.request_of[j]]) + j - int(cl.item_offsets[cl.item_of[j]]) + 1
                    for j in range(cl.T))
        assert p.stats()["visible_pairs"] == pairs
    # errors
    cl = O.cached_layout([0], [10], [2], [3, 4])
    mk = lambda **kw: lib.CachedPlan.host_only(kw.get("cu", cl.cu_seqlens), kw.get("ip", cl.item_ptr),
                                               kw.get("io", cl.item_offsets), kw.get("cs", [0]),
                                               kw.get("cl", [10]), kw.get("T", 10), 4, 2, 64)
    mk()
    for kw, want in [(dict(T=9), lib.MIS_ERR_SHAPE), (dict(cl=[0]), lib.MIS_ERR_SHAPE),
                     (dict(cs=[-1]), lib.MIS_ERR_SHAPE), (dict(ip=[0, 0]), lib.MIS_ERR_SHAPE),
                     (dict(io=[1, 4]), lib.MIS_ERR_SHAPE)]:
        with pytest.raises(lib.MisError) as e:
            mk(**kw)
        assert e.value.status == want, kw


@pytest.mark.parametrize("name", ["tiny", "qwen3-0.6b-layer", "decision-256", "varlen-16"])
@pytest.mark.parametrize("mode", [lib.SCHEDULE_AUTO, lib.SCHEDULE_PAIR, lib.SCHEDULE_SPLIT],
                         ids=["auto", "pair", "split"])
def test_unit_walk_hands_out_every_unit_once_pass_by_pass(name, mode):
    # The attention kernel's blocks take walk position kk * G + c in pass kk.
    # Whatever the order (the snake over the list, or its wave-by-wave
    # longest-first assignment), every unit is handed out exactly once, and
    # pass kk hands out exactly the list's units kk * G .. kk * G + G - 1, so
    # blocks running together work on neighbouring units of the list.
    w = synth.WORKLOADS[name]
    s = synth.draw_shapes(w)
    lay = lib.mis_build_layout(s.prefix_tokens, s.n_items, s.item_lens, with_positions=False)
    prev = lib.mis_set_schedule(mode)
    try:
        p = lib.Plan.host_only(lay.cu_seqlens, lay.prefix_len, lay.item_ptr, lay.item_offsets,
                               w.hq, w.hkv, w.head_dim)
        walk, G = p.unit_walk()
        n = p.stats()["n_units"]
    finally:
        lib.mis_set_schedule(prev)
    assert G == min(n, G) and G >= 1
    got = walk[walk >= 0]
    assert np.array_equal(np.sort(got), np.arange(n))
    for kk in range((len(walk) + G - 1) // G):
        part = walk[kk * G:(kk + 1) * G]
        assert set(part[part >= 0].tolist()) == set(range(kk * G, min((kk + 1) * G, n)))


@pytest.mark.parametrize("name", list(synth.WORKLOADS))
def test_both_bench_arms_size_every_workload_alike(L, name):
    # bench.py's own arm sizes a workload through the library, its reference
    # arm (the oracle) through the oracle's layout: both see the same T and M
    import sys
    sys.path.insert(0, ROOT)
    import bench
    w = synth.WORKLOADS[name]
    s = synth.draw_shapes(w)
    size = lib.mis_setwise_layout_size if w.layout == "setwise" else lib.mis_layout_size
    assert tuple(size(s.prefix_tokens, s.n_items, s.item_lens)) == bench.oracle_sizes(w, s)


def test_attention_calls_refuse_the_wrong_plan_kind_before_any_launch(L):
    # A plan form runs only the plan kind it was made for, and a host-only
    # plan (no workspace) runs nothing; every refusal comes from the host.
    lay = lib.mis_build_layout([40], [2], [5, 6], with_positions=False)
    plain = lib.Plan.host_only(lay.cu_seqlens, lay.prefix_len, lay.item_ptr, lay.item_offsets,
                               4, 2, 64)
    cl = O.cached_layout([0], [10], [2], [3, 4])
    cached = lib.CachedPlan.host_only(cl.cu_seqlens, cl.item_ptr, cl.item_offsets, [0], [10],
                                      10, 4, 2, 64)
    a = C.c_void_p(0x10000)
    def fwd(plan):
        return L.mis_attention_fwd_plan(plan, a, a, a, a, None, 256, 128, 128, 256, None)
    def fwd_cached(plan):
        return L.mis_attention_fwd_cached(plan, a, a, a, a, a, a, None, 256, 128, 128, 128, 128,
                                          256, None)
    assert fwd(None) == lib.MIS_ERR_INVALID_ARG
    assert fwd(cached._h) == lib.MIS_ERR_INVALID_ARG          # needs the cache buffers
    assert fwd(plain._h) == lib.MIS_ERR_WORKSPACE             # host-only plan
    assert fwd_cached(None) == lib.MIS_ERR_INVALID_ARG
    assert fwd_cached(plain._h) == lib.MIS_ERR_INVALID_ARG    # not a cached-prefix plan
    assert fwd_cached(cached._h) == lib.MIS_ERR_WORKSPACE
    plain.destroy()
    cached.destroy()


def _exec_coverage_ok(lay, p):
    """Every visible key of every row is in exactly one executed key tile of its
    query tile, and a tile without the mask flag has only visible entries."""
    et = p.exec_tiles()
    by_qt = {}
    for b, q0, c0, fl in et.tolist():
        by_qt.setdefault((b, q0), []).append((c0, fl))
    assert len(by_qt) == p.stats()["n_qtiles"]
    for (b, q0), tiles in by_qt.items():
        s0, e0 = int(lay.cu_seqlens[b]), int(lay.cu_seqlens[b + 1])
        S = int(lay.prefix_len[b])
        rows = np.arange(q0, min(q0 + 128, e0))
        vis = O.mask_rows(lay, b, rows)                   # [R, L] over keys s0 .. e0 - 1
        seen = np.zeros_like(vis, dtype=np.int32)
        for c0, fl in tiles:
            keys = c0 + np.arange(128)
            inside = (keys >= s0) & (keys < e0)
            cols = keys[inside] - s0
            seen[:, cols] += 1
            if not fl & 1:                                 # unmasked: all entries visible
                assert inside.all() and vis[:, cols].all()
        assert (seen[vis] == 1).all()                      # every visible key exactly once


def test_executed_tiles_cover_every_visible_key_once(L):
    # the executed key-tile lists, checked row by row against the oracle's
    # eq.-(4) mask: shared sets ending at, just past and well past a tile
    # edge, at D = 64 and 128, plus the benchmark's small workloads and a
    # sampled part of decision-256
    rng = np.random.default_rng(2024)
    cases = []
    for D in (64, 128):
        for P in (127, 128, 129, 130, 131, 255, 256, 257, 383):
            n = int(rng.integers(3, 12))
            cases.append((synth.custom_shapes([P, P + 128], [n, 2], rng.integers(0, 90, n + 2)), D))
    for name in ("qwen3-0.6b-layer", "tiny"):
        w = synth.WORKLOADS[name]
        cases.append((synth.draw_shapes(w), w.head_dim))
    d = synth.draw_shapes(synth.WORKLOADS["decision-256"])
    k = int(d.n_items[:12].sum())
    cases.append((synth.custom_shapes(d.prefix_tokens[:12], d.n_items[:12], d.item_lens[:k]), 128))
    for s, D in cases:
        lay = O.build_layout(s.prefix_tokens, s.n_items, s.item_lens)
        p = lib.Plan.host_only(lay.cu_seqlens, lay.prefix_len, lay.item_ptr, lay.item_offsets, 4, 2, D)
        _exec_coverage_ok(lay, p)
        st = p.stats()
        assert len(p.exec_tiles()) == st["n_tiles"]


def test_reference_arm_prints_the_contract_line_on_the_cpu():
    # `bench.py --impl reference` (the oracle on the host cores) prints one
    # JSON line with the main arm's metric, unit, direction and config object,
    # a cpu_baseline and an e2e entry without host-device copies
    import json
    import subprocess
    import sys
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny", "--steps", "2", "--warmup", "3", "--cpu-budget-s", "2"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [x for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    sys.path.insert(0, ROOT)
    import bench
    w = synth.WORKLOADS["tiny"]
    s = synth.draw_shapes(w)
    T, M = bench.oracle_sizes(w, s)
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "items/s"
    assert d["higher_is_better"] is True and d["steps"] == 2 and d["warmup"] == 3
    assert d["config"] == bench.workload_config(w, s, T, M, len(s.label_sets[0]), 1)
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "items/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_layout_tile_map_and_walk_on_generated_batches(L):
    # Property-based: batches hypothesis generates (1 to 6 requests, prefixes
    # of 0 to 700 tokens, 0 to 30 items of 0 to 300 tokens), layout and tile
    # map bit-exact against the oracle, pair count against the closed form,
    # and the unit walk handing out every unit once under either schedule
    hyp = pytest.importorskip("hypothesis")
    st = pytest.importorskip("hypothesis.strategies")

    req = st.tuples(st.integers(0, 700), st.lists(st.integers(0, 300), max_size=30))

    @hyp.settings(max_examples=60, deadline=None, derandomize=True)
    @hyp.given(st.lists(req, min_size=1, max_size=6), st.sampled_from([(4, 2, 64), (16, 8, 128), (6, 2, 128)]))
    def check(reqs, heads):
        P = [r[0] for r in reqs]
        N = [len(r[1]) for r in reqs]
        lens = [x for r in reqs for x in r[1]]
        got = lib.mis_build_layout(P, N, lens)
        ref = O.build_layout(P, N, lens)
        for f in ("cu_seqlens", "prefix_len", "item_ptr", "item_offsets", "delim_positions",
                  "position_ids"):
            assert np.array_equal(getattr(got, f), getattr(ref, f)), f
        hq, hkv, D = heads
        p = lib.Plan.host_only(ref.cu_seqlens, ref.prefix_len, ref.item_ptr, ref.item_offsets, hq, hkv, D)
        assert np.array_equal(p.tile_map(), O.tile_map(ref, 128, 128))
        assert p.stats()["visible_pairs"] == O.pair_count(ref)
        walk, G = p.unit_walk()
        assert np.array_equal(np.sort(walk[walk >= 0]), np.arange(p.stats()["n_units"]))

    check()
