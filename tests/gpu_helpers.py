"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI
and the oracle on the same seeded inputs."""
import numpy as np
import torch

import oracle as O
from ranking_prefill_gb300 import lib, synth

ATTN_TOL = 2e-2      # max-abs on O (bf16 output, fp32 accumulation)
LSE_TOL = 2e-3       # max-abs on the natural-log normaliser (fp32 exp2/log2 path)
SCORE_TOL = 1e-2     # max-abs on label log-probs


class forced_schedule:
    """Plans created inside the block use the given attention schedule."""

    def __init__(self, mode: int):
        self.mode = mode

    def __enter__(self):
        self.prev = lib.mis_set_schedule(self.mode)
        return self

    def __exit__(self, *exc):
        lib.mis_set_schedule(self.prev)


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def run_attention(shapes, hq, hkv, D, seed, with_lse=True, causal=False, stride_pad=0,
                  plan_form=True):
    """Returns (layout, vals, O gpu [T,hq,D] bf16, lse gpu [hq,T] or None, plan stats)."""
    lay = lib.mis_build_layout(shapes.prefix_tokens, shapes.n_items, shapes.item_lens)
    T = lay.T
    vals = synth.draw_values(seed, T, hq, hkv, D, want=("q", "k", "v"))
    dev = torch.device("cuda")
    def place(t, heads):
        if stride_pad == 0:
            return t.to(dev).contiguous()
        buf = torch.zeros(T, heads * D + stride_pad, dtype=torch.bfloat16, device=dev)
        view = buf.as_strided((T, heads, D), (heads * D + stride_pad, D, 1))
        view.copy_(t.to(dev))
        return view
    q, k, v = place(vals["q"], hq), place(vals["k"], hkv), place(vals["v"], hkv)
    if stride_pad:
        obuf = torch.full((T, hq * D + stride_pad), 7.0, dtype=torch.bfloat16, device=dev)
        o = obuf.as_strided((T, hq, D), (hq * D + stride_pad, D, 1))
    else:
        obuf = None
        o = torch.full((T, hq, D), 7.0, dtype=torch.bfloat16, device=dev)
    lse = torch.full((hq, T), 7.0, dtype=torch.float32, device=dev) if with_lse else None
    if causal:
        pl_ = [int(lay.cu_seqlens[b + 1] - lay.cu_seqlens[b]) for b in range(lay.B)]
        plan = lib.Plan(lay.cu_seqlens, pl_, None, None, hq, hkv, D)
    else:
        plan = lib.Plan(lay.cu_seqlens, lay.prefix_len, lay.item_ptr, lay.item_offsets, hq, hkv, D)
    ws = torch.zeros(plan.workspace_size(), dtype=torch.uint8, device=dev)
    if plan_form:
        plan.create(ws)
        lib.mis_attention_fwd_plan(plan, q, k, v, o, lse)
    else:
        lib.mis_attention_fwd(q, k, v, o, lse, plan.cu, plan.pl, plan.ip, plan.io, ws)
        plan.create(ws)   # for stats below (same workspace, after the run)
    torch.cuda.synchronize()
    st = lib.mis_get_device_status(ws)
    assert st == lib.MIS_OK, lib.mis_status_string(st)
    stats = plan.stats()
    return lay, vals, o, lse, stats, obuf


def oracle_layout(shapes):
    return O.build_layout(shapes.prefix_tokens, shapes.n_items, shapes.item_lens)


_ORACLE_CACHE = {}


def check_attention(shapes, hq, hkv, D, seed, rows=None, causal=False, cache_key=None, **kw):
    """GPU attention vs the oracle on the same seeded inputs. With `cache_key`,
    the oracle's result is kept for the next call with the same key (the same
    workload under another schedule)."""
    lay, vals, o, lse, stats, _ = run_attention(shapes, hq, hkv, D, seed, causal=causal, **kw)
    olay = oracle_layout(shapes)
    if causal:
        olay = O.causal_layout(np.diff(olay.cu_seqlens))
    if cache_key is not None and cache_key in _ORACLE_CACHE:
        ro, rl = _ORACLE_CACHE[cache_key]
    else:
        ro, rl = O.attention(f64(vals["q"]), f64(vals["k"]), f64(vals["v"]), olay, rows=rows)
        if cache_key is not None:
            _ORACLE_CACHE[cache_key] = (ro, rl)
    got = f64(o) if rows is None else f64(o[torch.as_tensor(np.asarray(rows), device=o.device)])
    err = np.abs(got - ro).max() if got.size else 0.0
    assert np.isfinite(got).all()
    assert err <= ATTN_TOL, f"max |O - oracle| = {err}"
    if lse is not None:
        gl = f64(lse)[:, np.asarray(rows) if rows is not None else slice(None)].T
        lerr = np.abs(gl - rl).max() if gl.size else 0.0
        assert lerr <= LSE_TOL, f"max |lse - oracle| = {lerr}"
    return err, stats


def run_scores(hidden, w_lm, delim, labels, with_renorm=True, T=None):
    dev = torch.device("cuda")
    M, K = int(delim.numel()), len(labels)
    out = torch.full((max(M, 1), K), 7.0, dtype=torch.float32, device=dev)[:M]
    ren = torch.full((max(M, 1), K), 7.0, dtype=torch.float32, device=dev)[:M] if with_renorm else None
    ws = torch.zeros(lib.mis_label_scores_workspace_size(M, w_lm.shape[1], w_lm.shape[0], K),
                     dtype=torch.uint8, device=dev)
    lib.mis_label_scores(hidden, w_lm, delim, labels, out, ren, ws, T=T)
    torch.cuda.synchronize()
    return out, ren, ws
