"""ctypes binding of the MIS C ABI (include/mis.h).

Argument marshalling only: every step of the hot path runs in the CUDA
library. Functions keep the C names. Torch tensors are accepted where the C
call takes a device pointer (torch is only used for device memory and
streams). Errors raise ``MisError`` carrying the status code.

The shared library is ``libmis_gb300.so`` next to this file, built by
``ranking_prefill_gb300/build.py`` (or ``__graft_entry__.build()``). If it is
missing, loading raises: there is no fallback path.
"""
from __future__ import annotations

import ctypes as C
import os
from dataclasses import dataclass
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmis_gb300.so")

STATUS = {0: "MIS_OK", 1: "MIS_ERR_INVALID_ARG", 2: "MIS_ERR_SHAPE", 3: "MIS_ERR_UNSUPPORTED",
          4: "MIS_ERR_WORKSPACE", 5: "MIS_ERR_CUDA", 6: "MIS_ERR_DEVICE_TIMEOUT",
          7: "MIS_ERR_DEVICE_INDEX"}
for _v, _n in STATUS.items():
    globals()[_n] = _v

# every symbol include/mis.h declares
EXPORTS = ["mis_status_string", "mis_abi_version", "mis_layout_size", "mis_build_layout",
           "mis_plan_workspace_size", "mis_plan_create", "mis_plan_get_stats",
           "mis_plan_tile_map", "mis_plan_unit_walk", "mis_plan_destroy", "mis_attention_fwd_plan",
           "mis_attention_fwd", "mis_label_scores_workspace_size", "mis_label_scores",
           "mis_get_device_status", "mis_set_wait_limit_ns", "mis_label_scores_noalloc",
           "mis_inject_stall", "mis_planner_create", "mis_planner_plan", "mis_planner_destroy",
           "mis_set_schedule", "mis_setwise_layout_size", "mis_build_setwise_layout",
           "mis_rope_qk", "mis_cached_plan_workspace_size", "mis_cached_plan_create",
           "mis_attention_fwd_cached", "mis_attention_fwd_plan_rope", "mis_rope_k_plan",
           "mis_plan_exec_tiles"]


class MisError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)} ({status})")


class mis_attn_desc(C.Structure):
    _fields_ = [("B", C.c_int32), ("T", C.c_int32), ("Hq", C.c_int32), ("Hkv", C.c_int32),
                ("D", C.c_int32), ("scale", C.c_float),
                # const int32_t* fields, passed as plain addresses
                ("cu_seqlens", C.c_void_p), ("prefix_len", C.c_void_p),
                ("item_ptr", C.c_void_p), ("item_offsets", C.c_void_p)]


class mis_cached_desc(C.Structure):
    _fields_ = [("B", C.c_int32), ("T", C.c_int32), ("Hq", C.c_int32), ("Hkv", C.c_int32),
                ("D", C.c_int32), ("scale", C.c_float),
                ("cu_seqlens", C.c_void_p), ("item_ptr", C.c_void_p), ("item_offsets", C.c_void_p),
                ("cache_start", C.c_void_p), ("cache_len", C.c_void_p), ("cache_T", C.c_int32)]


class mis_plan_stats(C.Structure):
    _fields_ = [(n, C.c_int64) for n in ("n_qtiles", "n_tiles", "n_full", "n_partial",
                                           "n_causal_tiles", "visible_pairs", "workspace_bytes",
                                           "schedule", "n_units")]

    def as_dict(self):
        return {n: int(getattr(self, n)) for n, _ in self._fields_}


_lib = None


def load(path: str = LIB_PATH):
    """Load (once) and return the ctypes library handle; raises if not built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"MIS CUDA library not built: {path} is missing "
                           "(run ranking_prefill_gb300/build.py)")
    L = C.CDLL(path)
    i32p = C.c_void_p        # int32 arrays go across as plain addresses (cheap to marshal)
    vp, sz, i64 = C.c_void_p, C.c_size_t, C.c_int64
    sig = {
        "mis_status_string": (C.c_char_p, [C.c_int]),
        "mis_abi_version": (C.c_int, []),
        "mis_layout_size": (C.c_int, [C.c_int32, i32p, i32p, i32p, C.POINTER(i64), C.POINTER(i64)]),
        "mis_build_layout": (C.c_int, [C.c_int32, i32p, i32p, i32p, i32p, i32p, i32p, i32p, i32p,
                                       i32p, i64]),
        "mis_plan_workspace_size": (sz, [C.POINTER(mis_attn_desc)]),
        "mis_plan_create": (C.c_int, [C.POINTER(mis_attn_desc), vp, sz, vp, C.POINTER(vp)]),
        "mis_plan_get_stats": (C.c_int, [vp, C.POINTER(mis_plan_stats)]),
        "mis_plan_tile_map": (C.c_int, [vp, i32p, sz, C.POINTER(sz)]),
        "mis_plan_unit_walk": (C.c_int, [vp, i32p, sz, C.POINTER(sz), C.POINTER(C.c_int32)]),
        "mis_plan_exec_tiles": (C.c_int, [vp, i32p, sz, C.POINTER(sz)]),
        "mis_plan_destroy": (C.c_int, [vp]),
        "mis_attention_fwd_plan": (C.c_int, [vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, vp]),
        "mis_attention_fwd": (C.c_int, [vp, vp, vp, vp, vp, i64, i64, i64, i64,
                                        C.POINTER(mis_attn_desc), vp, sz, vp]),
        "mis_label_scores_workspace_size": (sz, [C.c_int32] * 4),
        "mis_label_scores": (C.c_int, [vp, i64, C.c_int32, vp, C.c_int32, C.c_int32, vp, C.c_int32,
                                       i32p, C.c_int32, vp, vp, vp, sz, vp]),
        "mis_get_device_status": (C.c_int, [vp, vp]),
        "mis_set_wait_limit_ns": (C.c_uint64, [C.c_uint64]),
        "mis_inject_stall": (C.c_uint32, [C.c_uint32]),
        "mis_set_schedule": (C.c_int32, [C.c_int32]),
        "mis_cached_plan_workspace_size": (sz, [C.POINTER(mis_cached_desc)]),
        "mis_cached_plan_create": (C.c_int, [C.POINTER(mis_cached_desc), vp, sz, vp, C.POINTER(vp)]),
        "mis_attention_fwd_cached": (C.c_int, [vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i64,
                                               i64, i64, vp]),
        "mis_rope_qk": (C.c_int, [vp, vp, vp, vp, i64, i64, i64, i64, C.c_int32, C.c_int32,
                                  C.c_int32, C.c_int32, vp, C.c_double, vp]),
        "mis_attention_fwd_plan_rope": (C.c_int, [vp, vp, vp, vp, vp, vp, i64, i64, i64, i64,
                                                  C.c_double, vp]),
        "mis_rope_k_plan": (C.c_int, [vp, vp, vp, i64, i64, C.c_double, vp]),
        "mis_setwise_layout_size": (C.c_int, [C.c_int32, i32p, i32p, i32p, C.POINTER(i64),
                                              C.POINTER(i64)]),
        "mis_build_setwise_layout": (C.c_int, [C.c_int32, i32p, i32p, i32p, i32p, i32p, i32p,
                                               i32p, i64]),
        "mis_planner_create": (C.c_int, [C.POINTER(vp)]),
        "mis_planner_plan": (C.c_int, [vp, C.POINTER(mis_attn_desc), vp, sz, vp, sz, vp,
                                       C.POINTER(vp)]),
        "mis_planner_destroy": (C.c_int, [vp]),
        "mis_label_scores_noalloc": (C.c_int, [vp, i64, C.c_int32, vp, C.c_int32, C.c_int32, vp,
                                               C.c_int32, i32p, C.c_int32, vp, vp, vp, vp]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype, f.argtypes = res, args
    _lib = L
    return L


def lib_status_unknown() -> int:
    return MIS_ERR_INVALID_ARG  # noqa: F821  (defined from STATUS above)


def _check(st: int, where: str):
    if st != 0:
        raise MisError(st, where)


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _ptr_i32(a: np.ndarray) -> int:
    """Address of a contiguous int32 array (the array must outlive the call)."""
    return a.ctypes.data


def _dptr(t) -> Optional[int]:
    """Device (or host) address of a tensor, or None."""
    if t is None:
        return None
    return int(t.data_ptr())


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream) if torch.cuda.is_available() else None
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


# --------------------------------------------------------------------- layout

@dataclass
class Layout:
    cu_seqlens: np.ndarray
    prefix_len: np.ndarray
    item_ptr: np.ndarray
    item_offsets: np.ndarray
    delim_positions: np.ndarray
    position_ids: np.ndarray

    @property
    def T(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def B(self) -> int:
        return len(self.prefix_len)

    @property
    def M(self) -> int:
        return len(self.item_offsets)


def mis_layout_size(prefix_tokens, n_items, item_lens):
    L = load()
    p, n, l = _i32(prefix_tokens), _i32(n_items), _i32(item_lens)
    T, M = C.c_int64(), C.c_int64()
    _check(L.mis_layout_size(len(p), _ptr_i32(p), _ptr_i32(n), _ptr_i32(l) if l.size else None,
                             C.byref(T), C.byref(M)), "mis_layout_size")
    return T.value, M.value


def mis_build_layout(prefix_tokens, n_items, item_lens, with_positions: bool = True) -> Layout:
    L = load()
    p, n, l = _i32(prefix_tokens), _i32(n_items), _i32(item_lens)
    T, M = mis_layout_size(p, n, l)
    B = len(p)
    cu, pl, ip = np.zeros(B + 1, np.int32), np.zeros(B, np.int32), np.zeros(B + 1, np.int32)
    io, dp = np.zeros(max(M, 1), np.int32), np.zeros(max(M, 1), np.int32)
    pos = np.zeros(T if with_positions else 1, np.int32)
    _check(L.mis_build_layout(B, _ptr_i32(p), _ptr_i32(n), _ptr_i32(l) if l.size else None,
                              _ptr_i32(cu), _ptr_i32(pl), _ptr_i32(ip), _ptr_i32(io), _ptr_i32(dp),
                              _ptr_i32(pos) if with_positions else None, T if with_positions else 0),
           "mis_build_layout")
    return Layout(cu, pl, ip, io[:M], dp[:M], pos if with_positions else np.zeros(0, np.int32))


@dataclass
class SetwiseLayout:
    """Setwise prompts: plain causal sequences scored at their marker rows."""
    cu_seqlens: np.ndarray
    prefix_len: np.ndarray        # = request lengths (plain causal)
    marker_positions: np.ndarray  # readout rows, request by request, candidate order
    position_ids: np.ndarray

    @property
    def T(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def B(self) -> int:
        return len(self.prefix_len)

    @property
    def M(self) -> int:
        return len(self.marker_positions)


def mis_setwise_layout_size(query_tokens, n_cands, cand_lens):
    L = load()
    q, n, c = _i32(query_tokens), _i32(n_cands), _i32(cand_lens)
    T, M = C.c_int64(), C.c_int64()
    _check(L.mis_setwise_layout_size(len(q), _ptr_i32(q), _ptr_i32(n), _ptr_i32(c) if c.size else None,
                                     C.byref(T), C.byref(M)), "mis_setwise_layout_size")
    return T.value, M.value


def mis_build_setwise_layout(query_tokens, n_cands, cand_lens,
                             with_positions: bool = True) -> SetwiseLayout:
    L = load()
    q, n, c = _i32(query_tokens), _i32(n_cands), _i32(cand_lens)
    T, M = mis_setwise_layout_size(q, n, c)
    B = len(q)
    cu, pl = np.zeros(B + 1, np.int32), np.zeros(B, np.int32)
    mk = np.zeros(max(M, 1), np.int32)
    pos = np.zeros(T if with_positions else 1, np.int32)
    _check(L.mis_build_setwise_layout(B, _ptr_i32(q), _ptr_i32(n), _ptr_i32(c) if c.size else None,
                                      _ptr_i32(cu), _ptr_i32(pl), _ptr_i32(mk),
                                      _ptr_i32(pos) if with_positions else None,
                                      T if with_positions else 0), "mis_build_setwise_layout")
    return SetwiseLayout(cu, pl, mk[:M], pos if with_positions else np.zeros(0, np.int32))


# ---------------------------------------------------------------------- plan

class Plan:
    """Host handle of a mis_plan_create() plan; keeps its arrays alive."""

    def __init__(self, cu_seqlens, prefix_len, item_ptr, item_offsets, Hq, Hkv, D,
                 scale: float = 0.0, workspace=None, stream=None):
        self._L = load()
        self._h = None
        self.cu, self.pl = _i32(cu_seqlens), _i32(prefix_len)
        self.ip = _i32(item_ptr) if item_ptr is not None else None
        self.io = _i32(item_offsets) if item_offsets is not None else None
        self.desc = mis_attn_desc(
            len(self.pl), int(self.cu[-1]), Hq, Hkv, D, scale, _ptr_i32(self.cu), _ptr_i32(self.pl),
            _ptr_i32(self.ip) if self.ip is not None else None,
            _ptr_i32(self.io) if self.io is not None and self.io.size else None)
        self.T, self.Hq, self.Hkv, self.D = int(self.cu[-1]), Hq, Hkv, D
        self.workspace = workspace
        if workspace is not None:
            self.create(workspace, stream)

    def workspace_size(self) -> int:
        n = self._L.mis_plan_workspace_size(C.byref(self.desc))
        if n == 0:
            # ask mis_plan_create for the reason
            h = C.c_void_p()
            st = self._L.mis_plan_create(C.byref(self.desc), None, 0, None, C.byref(h))
            if st == 0:
                self._L.mis_plan_destroy(h)
            _check(st or lib_status_unknown(), "mis_plan_workspace_size")
        return int(n)

    def create(self, workspace, stream=None):
        """Plan into `workspace` (device uint8 tensor); None makes a host-only plan."""
        self.destroy()
        self.workspace = workspace
        h = C.c_void_p()
        if workspace is None:
            _check(self._L.mis_plan_create(C.byref(self.desc), None, 0, None, C.byref(h)),
                   "mis_plan_create")
        else:
            nbytes = workspace.numel() * workspace.element_size()
            _check(self._L.mis_plan_create(C.byref(self.desc), _dptr(workspace), nbytes,
                                           _stream(stream), C.byref(h)), "mis_plan_create")
        self._h = h
        return self

    @classmethod
    def host_only(cls, cu_seqlens, prefix_len, item_ptr, item_offsets, Hq, Hkv, D, scale=0.0):
        p = cls(cu_seqlens, prefix_len, item_ptr, item_offsets, Hq, Hkv, D, scale)
        return p.create(None)

    def stats(self) -> dict:
        s = mis_plan_stats()
        _check(self._L.mis_plan_get_stats(self._h, C.byref(s)), "mis_plan_get_stats")
        return s.as_dict()

    def unit_walk(self):
        """(walk, G): the unit at each walk position of the attention kernel's
        blocks (-1: none) and the block count G."""
        n = C.c_size_t()
        g = C.c_int32()
        _check(self._L.mis_plan_unit_walk(self._h, None, 0, C.byref(n), C.byref(g)),
               "mis_plan_unit_walk")
        out = np.zeros(max(n.value, 1), np.int32)
        _check(self._L.mis_plan_unit_walk(self._h, _ptr_i32(out), n.value, C.byref(n), C.byref(g)),
               "mis_plan_unit_walk")
        return out[:n.value], int(g.value)

    def tile_map(self) -> np.ndarray:
        n = C.c_size_t()
        _check(self._L.mis_plan_tile_map(self._h, None, 0, C.byref(n)), "mis_plan_tile_map")
        out = np.zeros((max(n.value, 1), 4), np.int32)
        _check(self._L.mis_plan_tile_map(self._h, _ptr_i32(out), n.value, C.byref(n)),
               "mis_plan_tile_map")
        return out[:n.value]

    def exec_tiles(self) -> np.ndarray:
        """(request, first query row, first key row, flags) of every key tile
        the kernel runs; flags bit 0 = masked."""
        n = C.c_size_t()
        _check(self._L.mis_plan_exec_tiles(self._h, None, 0, C.byref(n)), "mis_plan_exec_tiles")
        out = np.zeros((max(n.value, 1), 4), np.int32)
        _check(self._L.mis_plan_exec_tiles(self._h, _ptr_i32(out), n.value, C.byref(n)),
               "mis_plan_exec_tiles")
        return out[:n.value]

    def destroy(self):
        if self._h is not None:
            self._L.mis_plan_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


class CachedPlan(Plan):
    """Plan of item requests over a cached prefix (mis_cached_plan_create)."""

    def __init__(self, cu_seqlens, item_ptr, item_offsets, cache_start, cache_len, cache_T,
                 Hq, Hkv, D, scale: float = 0.0, workspace=None, stream=None):
        self._L = load()
        self._h = None
        self.cu, self.ip, self.io = _i32(cu_seqlens), _i32(item_ptr), _i32(item_offsets)
        self.cs, self.cl = _i32(cache_start), _i32(cache_len)
        self.cdesc = mis_cached_desc(len(self.cl), int(self.cu[-1]), Hq, Hkv, D, scale,
                                     _ptr_i32(self.cu), _ptr_i32(self.ip), _ptr_i32(self.io),
                                     _ptr_i32(self.cs), _ptr_i32(self.cl), int(cache_T))
        self.T, self.Hq, self.Hkv, self.D = int(self.cu[-1]), Hq, Hkv, D
        self.workspace = workspace
        if workspace is not None:
            self.create(workspace, stream)

    def workspace_size(self) -> int:
        n = self._L.mis_cached_plan_workspace_size(C.byref(self.cdesc))
        if n == 0:
            h = C.c_void_p()
            st = self._L.mis_cached_plan_create(C.byref(self.cdesc), None, 0, None, C.byref(h))
            if st == 0:
                self._L.mis_plan_destroy(h)
            _check(st or lib_status_unknown(), "mis_cached_plan_workspace_size")
        return int(n)

    def create(self, workspace, stream=None):
        self.destroy()
        self.workspace = workspace
        h = C.c_void_p()
        if workspace is None:
            _check(self._L.mis_cached_plan_create(C.byref(self.cdesc), None, 0, None, C.byref(h)),
                   "mis_cached_plan_create")
        else:
            nbytes = workspace.numel() * workspace.element_size()
            _check(self._L.mis_cached_plan_create(C.byref(self.cdesc), _dptr(workspace), nbytes,
                                                  _stream(stream), C.byref(h)), "mis_cached_plan_create")
        self._h = h
        return self

    @classmethod
    def host_only(cls, *args, **kw):
        p = cls(*args, **kw)
        return p.create(None)


def mis_attention_fwd_cached(plan: "CachedPlan", q, k, v, k_cache, v_cache, o, lse=None,
                             stream=None):
    L = load()
    _check(L.mis_attention_fwd_cached(plan._h, _dptr(q), _dptr(k), _dptr(v), _dptr(k_cache),
                                      _dptr(v_cache), _dptr(o), _dptr(lse), q.stride(0), k.stride(0),
                                      v.stride(0), k_cache.stride(0), v_cache.stride(0), o.stride(0),
                                      _stream(stream)), "mis_attention_fwd_cached")


class Planner:
    """mis_planner_*: plans uploaded through pinned staging, no stream sync."""

    def __init__(self):
        self._L = load()
        h = C.c_void_p()
        _check(self._L.mis_planner_create(C.byref(h)), "mis_planner_create")
        self._h = h

    def plan(self, cu_seqlens, prefix_len, item_ptr, item_offsets, Hq, Hkv, D, workspace,
             scale: float = 0.0, stream=None, extra: Optional[np.ndarray] = None) -> Plan:
        """`extra` (a contiguous host array, e.g. the readout rows) rides in the
        same upload and lands at workspace byte offset plan.workspace_size()."""
        p = Plan(cu_seqlens, prefix_len, item_ptr, item_offsets, Hq, Hkv, D, scale)
        h = C.c_void_p()
        nbytes = workspace.numel() * workspace.element_size()
        ex = None if extra is None else np.ascontiguousarray(extra)
        _check(self._L.mis_planner_plan(self._h, C.byref(p.desc), _dptr(workspace), nbytes,
                                        None if ex is None else ex.ctypes.data,
                                        0 if ex is None else ex.nbytes,
                                        _stream(stream), C.byref(h)), "mis_planner_plan")
        p._h, p.workspace = h, workspace
        return p

    def destroy(self):
        if self._h is not None:
            self._L.mis_planner_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


def plan_workspace_bytes(cu_seqlens, prefix_len, item_ptr, item_offsets, Hq, Hkv, D) -> int:
    return Plan(cu_seqlens, prefix_len, item_ptr, item_offsets, Hq, Hkv, D).workspace_size()


def mis_attention_fwd_plan(plan: Plan, q, k, v, o, lse=None, stream=None):
    L = load()
    _check(L.mis_attention_fwd_plan(plan._h, _dptr(q), _dptr(k), _dptr(v), _dptr(o), _dptr(lse),
                                    q.stride(0), k.stride(0), v.stride(0), o.stride(0),
                                    _stream(stream)), "mis_attention_fwd_plan")


def mis_attention_fwd(q, k, v, o, lse, cu_seqlens, prefix_len, item_ptr, item_offsets,
                      workspace, scale: float = 0.0, stream=None):
    """One-shot form: plan + launch; `workspace` a device uint8 tensor."""
    L = load()
    p = Plan(cu_seqlens, prefix_len, item_ptr, item_offsets, q.shape[1], k.shape[1], q.shape[2],
             scale)
    nbytes = workspace.numel() * workspace.element_size()
    _check(L.mis_attention_fwd(_dptr(q), _dptr(k), _dptr(v), _dptr(o), _dptr(lse),
                               q.stride(0), k.stride(0), v.stride(0), o.stride(0),
                               C.byref(p.desc), _dptr(workspace), nbytes, _stream(stream)),
           "mis_attention_fwd")


# ------------------------------------------------------------------- scoring

def mis_rope_qk(q, k, q_out, k_out, position_ids, base: float = 1.0e6, stream=None, Hq=None):
    """Rotary embedding of q [T, Hq, D] and k [T, Hkv, D] (bf16 device tensors
    with unit stride inside a row) at device int32 position ids [T]. q and
    q_out None: K only (then Hq, the model's query heads, is passed as is)."""
    L = load()
    T, Hkv, D = k.shape
    if q is not None:
        Hq = q.shape[1]
    elif Hq is None:
        Hq = Hkv
    qs = q.stride(0) if q is not None else 0
    qos = q_out.stride(0) if q_out is not None else 0
    _check(L.mis_rope_qk(_dptr(q), _dptr(k), _dptr(q_out), _dptr(k_out), qs, k.stride(0),
                         qos, k_out.stride(0), T, Hq, Hkv, D, _dptr(position_ids),
                         float(base), _stream(stream)), "mis_rope_qk")


def mis_rope_k_plan(plan, k, k_out, base: float = 1.0e6, stream=None):
    """Rotary embedding of k [T, Hkv, D] at the plan's reused position ids."""
    L = load()
    _check(L.mis_rope_k_plan(plan._h, _dptr(k), _dptr(k_out), k.stride(0), k_out.stride(0),
                             float(base), _stream(stream)), "mis_rope_k_plan")


def mis_attention_fwd_plan_rope(plan: "Plan", q, k, v, o, lse=None, base: float = 1.0e6,
                                stream=None):
    """mis_attention_fwd_plan with Q rotated on load at the reused position
    ids (derived from the plan); K arrives rotated."""
    L = load()
    _check(L.mis_attention_fwd_plan_rope(plan._h, _dptr(q), _dptr(k), _dptr(v), _dptr(o),
                                         _dptr(lse), q.stride(0), k.stride(0), v.stride(0),
                                         o.stride(0), float(base), _stream(stream)),
           "mis_attention_fwd_plan_rope")


def mis_label_scores_workspace_size(M: int, d: int, V: int, K: int) -> int:
    return int(load().mis_label_scores_workspace_size(M, d, V, K))


def mis_label_scores(hidden, w_lm, delim_positions, label_token_ids: Sequence[int], out_logprobs,
                     out_renorm, workspace, T: Optional[int] = None, stream=None):
    L = load()
    labels = _i32(label_token_ids)
    M = int(delim_positions.numel())
    d, V = int(w_lm.shape[1]), int(w_lm.shape[0])
    nbytes = workspace.numel() * workspace.element_size()
    _check(L.mis_label_scores(_dptr(hidden), hidden.stride(0),
                              int(hidden.shape[0]) if T is None else T, _dptr(w_lm), d, V,
                              _dptr(delim_positions), M, _ptr_i32(labels), len(labels),
                              _dptr(out_logprobs), _dptr(out_renorm), _dptr(workspace), nbytes,
                              _stream(stream)), "mis_label_scores")


def mis_label_scores_noalloc(hidden, w_lm, delim_positions, label_token_ids: Sequence[int],
                             out_logprobs, out_renorm=None, device_status=None,
                             T: Optional[int] = None, stream=None):
    """mis_label_scores without a workspace: for callers that cannot allocate
    device memory. The library's static scratch is shared by every call on a
    device, so calls must not overlap on the GPU."""
    L = load()
    labels = _i32(label_token_ids)
    M = int(delim_positions.numel())
    d, V = int(w_lm.shape[1]), int(w_lm.shape[0])
    _check(L.mis_label_scores_noalloc(_dptr(hidden), hidden.stride(0),
                                      int(hidden.shape[0]) if T is None else T, _dptr(w_lm), d, V,
                                      _dptr(delim_positions), M, _ptr_i32(labels), len(labels),
                                      _dptr(out_logprobs), _dptr(out_renorm), _dptr(device_status),
                                      _stream(stream)), "mis_label_scores_noalloc")


def mis_get_device_status(workspace, stream=None) -> int:
    return int(load().mis_get_device_status(_dptr(workspace), _stream(stream)))


def mis_set_wait_limit_ns(ns: int) -> int:
    return int(load().mis_set_wait_limit_ns(int(ns)))


def mis_inject_stall(mask: int) -> int:
    return int(load().mis_inject_stall(int(mask)))


SCHEDULE_AUTO, SCHEDULE_PAIR, SCHEDULE_SPLIT = 0, 1, 2


def mis_set_schedule(mode: int) -> int:
    """Attention schedule of plans created afterwards (process-wide); returns the previous mode."""
    prev = int(load().mis_set_schedule(int(mode)))
    if prev < 0:
        raise MisError(MIS_ERR_INVALID_ARG, "mis_set_schedule")
    return prev


def mis_status_string(st: int) -> str:
    return load().mis_status_string(int(st)).decode()
