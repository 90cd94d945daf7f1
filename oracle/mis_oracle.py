"""CPU oracle for Multiple-Item Scoring (MIS): plain, slow, fp64.

TEST INFRASTRUCTURE ONLY. Nothing on the product path may import, call or
execute this module: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it. It shares
no code with the CUDA library; both sides read the same seeded inputs and
nothing else.

What it computes, and where each step comes from:

* ``build_layout`` — the packed sequence of "From Generation to Scoring"
  (Section 4.1, eq. 3) in the delimiter layout of "Turbocharging LinkedIn's
  recommendation systems with SGLang" (section "Multi-item-scoring: Our
  innovation with SGLang"): ``<prefix><DELIM><item 1><DELIM>...<item N><DELIM>``,
  and the reused position ids of Section 4.1 ("Position IDs encode token
  positions ...").
* ``mask_rows`` — the additive mask of eq. (4), evaluated by set membership:
  key k is visible from row j iff k <= j and (k is in the query set Q, or j and
  k lie in the same item set I_i).
* ``attention`` — softmax attention under that mask, naive: full score rows,
  -inf on masked entries, max-shifted exponentials, normalised sum.
* ``label_scores`` — the answer-token readout of Section 3.3: the next-token
  logits at each item's readout row over the full vocabulary, log-softmax over
  the vocabulary ("Scaling JEV-like Decision Models with SGLang", section "Why a
  Decision Workload Deserves a Scoring Interface": label extraction keeps the
  full-distribution normalisation), then the requested label columns; and the
  label-renormalised score of eq. (2) (``apply_softmax``, same page, "Send a
  Scoring Request").
* ``tile_map`` — which (q-tile, k-tile) blocks of the mask are empty, full or
  partial, counted element by element from ``mask_rows``.
* ``cost_ratio`` — eq. (5), the prefill-token reduction factor R(N).
* ``rope`` — rotary position embedding of Q and K at given position ids, the
  step that consumes the reused position ids of "From Generation to
  Scoring" Section 4.1; the SGLang changes of "Turbocharging ..." also
  adjust the positional encoding so each item sits at its single-item
  position.
* ``cached_layout`` / ``attention_cached`` — items scored over a prefix whose
  K/V was computed earlier and kept in a cache (the in-batch prefix cache
  of "Scaling LLM-Based Ranking Systems with Prefill-Only Optimization",
  Components table, and the knock-knock second request of "Turbocharging
  LinkedIn's recommendation systems with SGLang"): each item row sees its request's
  cached prefix and its own item causally, as in eq. (4).
* ``setwise_layout`` — the anchor-based setwise prompt of "Scaling JEV-like
  Decision Models with SGLang" (section "Benchmark: Fused-Choice vs. Setwise
  Scoring"): query, every candidate, then one marker per candidate, as one
  plain causal sequence, scored at each marker.

Readings taken where the pages are silent or garbled:
  - the leading DELIM belongs to the shared set Q (so |Q| = S = P + 1); each
    trailing DELIM belongs to its own item's set I_i, and is that item's
    readout row (the row that "reads prefix + item k");
  - position ids: query tokens 0..S-1; token at offset d of an item (its
    trailing DELIM has offset L_i) gets S + d;
  - softmax scale 1/sqrt(D) unless given; q head h reads kv head
    h // (Hq / Hkv);
  - log-probabilities are natural-log, normalised over the whole vocabulary;
  - requests in a batch never attend to each other.
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Iterable, List, Optional, Sequence

import numpy as np

EMPTY, FULL, PARTIAL = 0, 1, 2


@dataclass
class Layout:
    """Packed-sequence description of a batch of MIS requests (all int32)."""

    cu_seqlens: np.ndarray       # [B+1] request boundaries in the packed stream
    prefix_len: np.ndarray       # [B]   S_b = prefix tokens + leading DELIM (= |Q|)
    item_ptr: np.ndarray         # [B+1] CSR into item_offsets
    item_offsets: np.ndarray     # [M]   absolute first token of each item segment
    item_ends: np.ndarray        # [M]   absolute one-past-last token of each segment
    delim_positions: np.ndarray  # [M]   absolute row of each item's trailing DELIM
    position_ids: np.ndarray     # [T]   reused position ids
    request_of: np.ndarray       # [T]   request index of every token
    item_of: np.ndarray          # [T]   global item index, -1 for tokens of Q

    @property
    def T(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def B(self) -> int:
        return len(self.prefix_len)

    @property
    def M(self) -> int:
        return len(self.item_offsets)


def build_layout(prefix_tokens: Sequence[int], n_items: Sequence[int],
                 item_lens: Sequence[int]) -> Layout:
    """Pack requests token by token into ``<prefix><DELIM>(<item><DELIM>)*``.

    ``prefix_tokens[b]`` counts the request's prefix tokens without the DELIM;
    ``item_lens`` lists every item's token count (without its DELIM), request
    after request.
    """
    prefix_tokens = [int(x) for x in prefix_tokens]
    n_items = [int(x) for x in n_items]
    item_lens = [int(x) for x in item_lens]
    if len(prefix_tokens) != len(n_items) or sum(n_items) != len(item_lens):
        raise ValueError("inconsistent request description")
    cu, plen, iptr = [0], [], [0]
    offs, ends, delims, pos, req_of, item_of = [], [], [], [], [], []
    t = 0
    it = 0
    for b, (p, n) in enumerate(zip(prefix_tokens, n_items)):
        if p < 0 or n < 0:
            raise ValueError("negative length")
        s = p + 1                        # prefix tokens and the leading DELIM
        for d in range(s):               # query set Q: positions 0..S-1
            pos.append(d)
            req_of.append(b)
            item_of.append(-1)
            t += 1
        plen.append(s)
        for _ in range(n):
            L = item_lens[it]
            if L < 0:
                raise ValueError("negative item length")
            offs.append(t)
            for d in range(L + 1):       # item tokens then its trailing DELIM
                pos.append(s + d)
                req_of.append(b)
                item_of.append(it)
                t += 1
            ends.append(t)
            delims.append(t - 1)         # the trailing DELIM is the readout row
            it += 1
        cu.append(t)
        iptr.append(it)
    i32 = lambda a: np.asarray(a, dtype=np.int32)
    return Layout(i32(cu), i32(plen), i32(iptr), i32(offs), i32(ends), i32(delims),
                  i32(pos), i32(req_of), i32(item_of))


@dataclass
class SetwiseLayout:
    """A batch of setwise prompts: one plain causal sequence per request."""

    causal: Layout               # the attention layout (no item sets)
    cand_offsets: np.ndarray     # [M] absolute first row of each candidate's tokens
    marker_positions: np.ndarray # [M] absolute marker row of each candidate (readout rows)

    @property
    def M(self) -> int:
        return len(self.marker_positions)


@dataclass
class CachedLayout:
    """Item requests over cached prefix K/V (all int32).

    The new sequence holds only item sets (item tokens + trailing DELIM);
    request b's prefix (its |Q| = S_b rows: prefix tokens and the leading
    DELIM) sits in the cache at rows [cache_start[b], cache_start[b] + S_b).
    """

    cu_seqlens: np.ndarray       # [B+1] rows of the new sequence per request
    item_ptr: np.ndarray         # [B+1]
    item_offsets: np.ndarray     # [M] first new-sequence row of each item set
    item_ends: np.ndarray        # [M]
    delim_positions: np.ndarray  # [M] readout rows (new sequence)
    position_ids: np.ndarray     # [T] reused positions S_b + d
    cache_start: np.ndarray      # [B]
    cache_len: np.ndarray        # [B] S_b
    request_of: np.ndarray       # [T]
    item_of: np.ndarray          # [T]

    @property
    def T(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def B(self) -> int:
        return len(self.cache_len)

    @property
    def M(self) -> int:
        return len(self.item_offsets)


def cached_layout(cache_start: Sequence[int], cache_len: Sequence[int],
                  n_items: Sequence[int], item_lens: Sequence[int]) -> CachedLayout:
    """Pack the item sets of each request, token by token, after a cached prefix."""
    cache_start = [int(x) for x in cache_start]
    cache_len = [int(x) for x in cache_len]
    n_items = [int(x) for x in n_items]
    item_lens = [int(x) for x in item_lens]
    if not (len(cache_start) == len(cache_len) == len(n_items)) or sum(n_items) != len(item_lens):
        raise ValueError("inconsistent request description")
    cu, iptr, offs, ends, delims, pos, req_of, item_of = [0], [0], [], [], [], [], [], []
    t = it = 0
    for b, (S, n) in enumerate(zip(cache_len, n_items)):
        if S < 1 or n < 1 or cache_start[b] < 0:
            raise ValueError("each request needs a cached prefix and at least one item")
        for _ in range(n):
            offs.append(t)
            for d in range(item_lens[it] + 1):     # item tokens then its trailing DELIM
                pos.append(S + d)
                req_of.append(b)
                item_of.append(it)
                t += 1
            ends.append(t)
            delims.append(t - 1)
            it += 1
        cu.append(t)
        iptr.append(it)
    i32 = lambda a: np.asarray(a, dtype=np.int32)
    return CachedLayout(i32(cu), i32(iptr), i32(offs), i32(ends), i32(delims), i32(pos),
                        i32(cache_start), i32(cache_len), i32(req_of), i32(item_of))


def attention_cached(q: np.ndarray, k: np.ndarray, v: np.ndarray, k_cache: np.ndarray,
                     v_cache: np.ndarray, lay: CachedLayout, scale: Optional[float] = None,
                     rows: Optional[Iterable[int]] = None):
    """Softmax attention of new-sequence rows over [cached prefix ; own item].

    Row j of item i of request b sees every cached key of b (the prefix
    precedes all item tokens, so eq. (4)'s k <= j holds) and the keys of item i
    up to j. Naive fp64, the cached keys first, then the item keys in order.
    Returns (O [R, Hq, D], LSE [R, Hq]).
    """
    T, Hq, D = q.shape
    group = Hq // k.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    rows = np.arange(T) if rows is None else np.asarray(list(rows), dtype=np.int64)
    out = np.zeros((len(rows), Hq, D), dtype=np.float64)
    lse = np.zeros((len(rows), Hq), dtype=np.float64)
    for n, j in enumerate(rows):
        b, i = int(lay.request_of[j]), int(lay.item_of[j])
        c0, S = int(lay.cache_start[b]), int(lay.cache_len[b])
        keys = np.concatenate([np.asarray(k_cache[c0:c0 + S], np.float64),
                               np.asarray(k[lay.item_offsets[i]:j + 1], np.float64)])
        vals = np.concatenate([np.asarray(v_cache[c0:c0 + S], np.float64),
                               np.asarray(v[lay.item_offsets[i]:j + 1], np.float64)])
        qj = np.asarray(q[j], np.float64)
        for h in range(Hq):
            sc = scale * (keys[:, h // group, :] @ qj[h])
            m = sc.max()
            p = np.exp(sc - m)
            out[n, h] = (p @ vals[:, h // group, :]) / p.sum()
            lse[n, h] = m + np.log(p.sum())
    return out, lse


def tile_map_cached(lay: CachedLayout, BM: int, BN: int) -> np.ndarray:
    """Non-empty (request, q-tile, k-tile, FULL/PARTIAL) blocks of cached-prefix requests.

    Query tiles cover each request's new rows from its first one. Key tiles
    0 .. ceil(S/BN)-1 cover its cached prefix [cache_start, cache_start + S)
    from its first row, and the next ones its new rows from the first one;
    a tile is clipped at the end of its range. Visibility by enumeration:
    every cached key of the request, and keys of the row's own item up to
    the row.
    """
    out = []
    for b in range(lay.B):
        s0, e0 = int(lay.cu_seqlens[b]), int(lay.cu_seqlens[b + 1])
        S = int(lay.cache_len[b])
        nc = (S + BN - 1) // BN
        rows = np.arange(s0, e0)
        item = lay.item_of[s0:e0]
        for t in range(0, (e0 - s0 + BM - 1) // BM):
            r = rows[t * BM:(t + 1) * BM]
            it = item[t * BM:(t + 1) * BM]
            for u in range(nc):                       # cached keys: visible from every row
                n = min(BN, S - u * BN)
                out.append((b, t, u, FULL if n > 0 else EMPTY))
            for u in range(0, (e0 - s0 + BN - 1) // BN):
                kk = np.arange(s0 + u * BN, min(s0 + (u + 1) * BN, e0))
                vis = (item[kk - s0][None, :] == it[:, None]) & (kk[None, :] <= r[:, None])
                if vis.any():
                    out.append((b, t, nc + u, FULL if vis.all() else PARTIAL))
    out = [x for x in out if x[3] != EMPTY]
    return np.asarray(out, dtype=np.int32).reshape(-1, 4)


def setwise_layout(query_tokens: Sequence[int], n_cands: Sequence[int],
                   cand_lens: Sequence[int]) -> SetwiseLayout:
    """Setwise (anchor-based) prompts, token by token.

    Per request: its query tokens (context, question, instruction), then the
    tokens of every candidate in order, then one marker per candidate. The
    prompt "ends with one marker per candidate", the markers "correspond to A,
    B, and C in order", and "all markers follow the complete candidate list, so
    each readout can attend to every candidate" ("Scaling JEV-like Decision
    Models with SGLang", "Benchmark: Fused-Choice vs. Setwise Scoring"); MIS is
    off, so attention is plain causal over the whole request. Marker i of a
    request is the readout row of its candidate i.
    """
    query_tokens = [int(x) for x in query_tokens]
    n_cands = [int(x) for x in n_cands]
    cand_lens = [int(x) for x in cand_lens]
    if len(query_tokens) != len(n_cands) or sum(n_cands) != len(cand_lens):
        raise ValueError("inconsistent request description")
    lengths, offs, marks = [], [], []
    t, c = 0, 0
    for q, n in zip(query_tokens, n_cands):
        if q < 0 or n < 0:
            raise ValueError("negative length")
        start = t
        t += q                                    # query
        for _ in range(n):                        # candidate texts
            if cand_lens[c] < 0:
                raise ValueError("negative candidate length")
            offs.append(t)
            t += cand_lens[c]
            c += 1
        for _ in range(n):                        # one marker per candidate
            marks.append(t)
            t += 1
        if t == start:
            raise ValueError("empty request")
        lengths.append(t - start)
    i32 = lambda a: np.asarray(a, dtype=np.int32)
    return SetwiseLayout(causal_layout(lengths), i32(offs), i32(marks))


def causal_layout(lengths: Sequence[int]) -> Layout:
    """A batch of plain causal sequences: every token is in Q, no items."""
    lengths = [int(x) for x in lengths]
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    T = int(cu[-1])
    req_of = np.repeat(np.arange(len(lengths)), lengths).astype(np.int32)
    pos = np.concatenate([np.arange(L) for L in lengths] or [np.zeros(0)]).astype(np.int32)
    z = np.zeros(0, np.int32)
    return Layout(cu, np.asarray(lengths, np.int32), np.zeros(len(lengths) + 1, np.int32),
                  z, z, z, pos, req_of, np.full(T, -1, np.int32))


# ---------------------------------------------------------------------------
# rotary position embedding at the (reused) position ids
# ---------------------------------------------------------------------------

def rope(x: np.ndarray, positions: Sequence[int], base: float = 1.0e6) -> np.ndarray:
    """Rotate every head vector of ``x`` [T, H, D] by its row's position.

    Rotate-half form: for i < D/2 the pair (x[i], x[i + D/2]) of a row at
    position p turns by the angle p * base^(-2i/D). The pages fix the position
    ids (Section 4.1: query 0..Lq-1, offset d of every item -> Lq + d) but not
    the encoding; rotary embedding with the Qwen3 family's base 10^6 is the
    reading taken for the Qwen3-shaped workloads (the base is a parameter).
    """
    x = np.asarray(x, dtype=np.float64)
    T, H, D = x.shape
    half = D // 2
    pos = np.asarray(positions, dtype=np.float64).reshape(T, 1, 1)
    inv = base ** (-2.0 * np.arange(half, dtype=np.float64) / D)
    ang = pos * inv.reshape(1, 1, half)
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


# ---------------------------------------------------------------------------
# eq. (4): the MIS mask by set membership
# ---------------------------------------------------------------------------

def mask_rows(lay: Layout, b: int, rows: np.ndarray) -> np.ndarray:
    """Boolean visibility [len(rows), L_b] of request ``b``'s keys from ``rows``.

    rows are absolute token indices inside request b. Entry (r, k) is True iff
    key s0+k is visible from row rows[r] under eq. (4).
    """
    s0, e0 = int(lay.cu_seqlens[b]), int(lay.cu_seqlens[b + 1])
    rows = np.asarray(rows, dtype=np.int64)
    keys = np.arange(s0, e0, dtype=np.int64)
    in_q = lay.item_of[s0:e0] < 0                       # k in Q
    item_k = lay.item_of[s0:e0]
    item_j = lay.item_of[rows]
    causal = keys[None, :] <= rows[:, None]             # k <= j
    same_item = (item_j[:, None] == item_k[None, :]) & (item_k[None, :] >= 0)
    return causal & (in_q[None, :] | same_item)


def mask_bruteforce(lay: Layout) -> np.ndarray:
    """Dense [T, T] visibility by literal enumeration of the sets of eq. (4).

    Pure Python; only for tiny layouts. Requests are independent, so keys of
    another request are never visible.
    """
    T = lay.T
    M = np.zeros((T, T), dtype=bool)
    for b in range(lay.B):
        s0 = int(lay.cu_seqlens[b])
        Q = set(range(s0, s0 + int(lay.prefix_len[b])))
        items = [set(range(int(lay.item_offsets[i]), int(lay.item_ends[i])))
                 for i in range(int(lay.item_ptr[b]), int(lay.item_ptr[b + 1]))]
        req = range(s0, int(lay.cu_seqlens[b + 1]))
        for j in req:
            for k in req:
                if k > j:
                    continue
                if k in Q or any(j in I and k in I for I in items):
                    M[j, k] = True
    return M


def pair_count(lay: Layout) -> int:
    """Number of visible (j, k) pairs, counted from the mask."""
    total = 0
    for b in range(lay.B):
        s0, e0 = int(lay.cu_seqlens[b]), int(lay.cu_seqlens[b + 1])
        for r0 in range(s0, e0, 1024):
            total += int(mask_rows(lay, b, np.arange(r0, min(r0 + 1024, e0))).sum())
    return total


# ---------------------------------------------------------------------------
# attention under the mask
# ---------------------------------------------------------------------------

def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, lay: Layout,
              scale: Optional[float] = None, rows: Optional[Iterable[int]] = None,
              row_block: int = 512):
    """Masked softmax attention in fp64.

    q: [T, Hq, D], k/v: [T, Hkv, D] (any float dtype; promoted to fp64).
    Returns (O [R, Hq, D], LSE [R, Hq]) for the requested absolute rows (all
    rows by default, in increasing order). LSE is the natural-log normaliser
    of the scaled scores: lse_j = m_j + ln sum_k exp(s_jk - m_j).
    """
    T, Hq, D = q.shape
    Hkv = k.shape[1]
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    group = Hq // Hkv
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    rows = np.arange(T) if rows is None else np.asarray(list(rows), dtype=np.int64)
    out = np.zeros((len(rows), Hq, D), dtype=np.float64)
    lse = np.zeros((len(rows), Hq), dtype=np.float64)
    if len(rows) == 0:
        return out, lse
    req = lay.request_of[rows]
    for b in np.unique(req):
        sel = np.nonzero(req == b)[0]
        s0, e0 = int(lay.cu_seqlens[b]), int(lay.cu_seqlens[b + 1])
        kb = np.asarray(k[s0:e0], dtype=np.float64)      # [L, Hkv, D]
        vb = np.asarray(v[s0:e0], dtype=np.float64)
        for c0 in range(0, len(sel), row_block):
            idx = sel[c0:c0 + row_block]
            r = rows[idx]
            vis = mask_rows(lay, int(b), r)               # [R, L]
            qr = np.asarray(q[r], dtype=np.float64)       # [R, Hq, D]
            for h in range(Hq):
                g = h // group
                s = scale * (qr[:, h, :] @ kb[:, g, :].T)  # [R, L]
                s = np.where(vis, s, -np.inf)
                m = s.max(axis=1, keepdims=True)
                p = np.exp(s - m)
                l = p.sum(axis=1, keepdims=True)
                out[idx, h, :] = (p @ vb[:, g, :]) / l
                lse[idx, h] = m[:, 0] + np.log(l[:, 0])
    return out, lse


# ---------------------------------------------------------------------------
# answer-token readout
# ---------------------------------------------------------------------------

def label_scores(hidden: np.ndarray, w_lm: np.ndarray, readout_rows: Sequence[int],
                 labels: Sequence[int], items: Optional[Iterable[int]] = None,
                 item_block: int = 64):
    """Full-vocabulary log-softmax at each readout row, then the label columns.

    hidden: [T, d]; w_lm: [V, d] (row v is the output embedding of token v).
    Returns (logprob [R, K], renorm [R, K], lse [R]) for the selected items
    (all by default). renorm is the softmax over the K label logits of each
    item (eq. 2 for K = 2; ``apply_softmax``).
    """
    readout_rows = np.asarray(readout_rows, dtype=np.int64)
    labels = np.asarray(labels, dtype=np.int64)
    sel = np.arange(len(readout_rows)) if items is None else np.asarray(list(items), np.int64)
    V = w_lm.shape[0]
    if labels.size and (labels.min() < 0 or labels.max() >= V):
        raise ValueError("label id outside the vocabulary")
    W = np.asarray(w_lm, dtype=np.float64)
    logp = np.zeros((len(sel), len(labels)), dtype=np.float64)
    ren = np.zeros_like(logp)
    lse = np.zeros(len(sel), dtype=np.float64)
    for c0 in range(0, len(sel), item_block):
        idx = np.arange(c0, min(c0 + item_block, len(sel)))
        h = np.asarray(hidden[readout_rows[sel[idx]]], dtype=np.float64)   # [R, d]
        z = h @ W.T                                                       # [R, V]
        m = z.max(axis=1, keepdims=True)
        l = m[:, 0] + np.log(np.exp(z - m).sum(axis=1))
        zl = z[:, labels]                                                 # [R, K]
        logp[idx] = zl - l[:, None]
        if labels.size:
            mm = zl.max(axis=1, keepdims=True)
            e = np.exp(zl - mm)
            ren[idx] = e / e.sum(axis=1, keepdims=True)
        lse[idx] = l
    return logp, ren, lse


# ---------------------------------------------------------------------------
# tile classification and the cost model
# ---------------------------------------------------------------------------

def tile_map(lay: Layout, BM: int, BN: int) -> np.ndarray:
    """Non-empty (request, q-tile, k-tile, FULL|PARTIAL) blocks, canonical order.

    Tiles are indexed per request: q-tile t covers rows
    [s0 + t*BM, min(s0 + (t+1)*BM, e0)), k-tile u likewise with BN. A block is
    EMPTY iff no entry is visible, FULL iff every entry is, else PARTIAL.
    Returns int32 [n, 4] sorted by (request, q-tile, k-tile).
    """
    out: List[tuple] = []
    for b in range(lay.B):
        s0, e0 = int(lay.cu_seqlens[b]), int(lay.cu_seqlens[b + 1])
        L = e0 - s0
        for t in range((L + BM - 1) // BM):
            r = np.arange(s0 + t * BM, min(s0 + (t + 1) * BM, e0))
            vis = mask_rows(lay, b, r)
            for u in range((L + BN - 1) // BN):
                blk = vis[:, u * BN: min((u + 1) * BN, L)]
                n = int(blk.sum())
                if n == 0:
                    continue
                out.append((b, t, u, FULL if n == blk.size else PARTIAL))
    return np.asarray(out, dtype=np.int32).reshape(-1, 4)


def cost_ratio(Lq: int, item_lens: Sequence[int]) -> float:
    """eq. (5): prefill tokens of N independent requests over one MIS request.

    R(N) = (N * Lq + sum_i L_i) / (Lq + sum_i L_i).
    """
    n = len(item_lens)
    s = float(sum(item_lens))
    return (n * Lq + s) / (Lq + s)


def useful_attention_flops(lay: Layout, hq: int, head_dim: int) -> int:
    """4 * Hq * D per visible pair (one multiply-add each for QK^T and PV)."""
    return 4 * hq * head_dim * pair_count(lay)
