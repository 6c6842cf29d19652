"""CPU oracle for tile-sparse masked softmax attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` import this package.  The product
library never imports, loads or calls it, and it shares no code with the
CUDA path: the mask semantics, tile classification, tile lists, softmax and
gradients here are written out independently from the pages.

Two independent implementations live here:

* ``oracle.c`` (built into ``liboracle.so``): fp64 loops over the visible set
  of every row, evaluating the mask element by element.  Used at every size.
* the numpy twin (``np_*`` functions): an explicit dense [Q, KV] boolean mask
  built by broadcasting, then dense fp64 softmax attention and its analytic
  backward in matrix form.  Used only at tiny sizes, to cross-check the C
  loops.

Every function is pinned by ``tests/test_oracle_pins.py`` to values the pages
print (tile counts of one 65,536-token sequence), closed forms, library
routines on textbook special cases, finite differences and invariants.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

# Node numbering of oracle.c (independent of the product library's numbering).
_OP = {"true": 0, "causal": 1, "same_doc": 2, "window": 3, "sink": 4, "prefix": 5, "and": 6, "or": 7}
_SCORE = {"none": 0, "softcap": 1, "alibi": 2, "relbias": 3}


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (plain -O2 C with OpenMP)."""
    src = os.path.join(_HERE, "oracle.c")
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(src):
        subprocess.run(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", src,
                        "-o", _LIB_PATH, "-lm"], check=True)
    return _LIB_PATH


class _Program(ctypes.Structure):
    _fields_ = [("n", ctypes.c_int32), ("op", ctypes.c_int32 * 16), ("arg", ctypes.c_int64 * 16),
                ("doc", ctypes.POINTER(ctypes.c_int32)), ("sel", ctypes.POINTER(ctypes.c_int8)),
                ("sel_block", ctypes.c_int64), ("sel_nkv", ctypes.c_int64), ("q_off", ctypes.c_int64)]


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.POINTER
        d = P(ctypes.c_double)
        i64p = P(ctypes.c_int64)
        lib.oracle_mask_dense.argtypes = [P(_Program), ctypes.c_int64, ctypes.c_int64, P(ctypes.c_uint8)]
        lib.oracle_classify_tiles.argtypes = [P(_Program), ctypes.c_int64, ctypes.c_int64, ctypes.c_int32,
                                              P(ctypes.c_int8)]
        bias = [d, ctypes.c_int64, ctypes.c_int64]  # the head's bias table, its first distance, its length
        lib.oracle_forward_head.argtypes = [d, d, d, ctypes.c_int64, ctypes.c_int64, ctypes.c_int32, P(_Program),
                                            ctypes.c_int32, ctypes.c_double, ctypes.c_double, i64p,
                                            ctypes.c_int64, d, d] + bias
        lib.oracle_backward_head.argtypes = [d, d, d, d, ctypes.c_int64, ctypes.c_int64, ctypes.c_int32,
                                             P(_Program), ctypes.c_int32, ctypes.c_double, ctypes.c_double,
                                             i64p, ctypes.c_int64, i64p, ctypes.c_int64, d, d, d, d, d] + bias
        lib.oracle_score_param_grad_head.argtypes = [d, d, d, d, ctypes.c_int64, ctypes.c_int64, ctypes.c_int32,
                                                     P(_Program), ctypes.c_int32, ctypes.c_double,
                                                     ctypes.c_double] + bias
        lib.oracle_score_param_grad_head.restype = ctypes.c_double
        lib.oracle_bias_grad_head.argtypes = [d, d, d, d, ctypes.c_int64, ctypes.c_int64, ctypes.c_int32,
                                              P(_Program), d, ctypes.c_int64, ctypes.c_int64, ctypes.c_double, d]
        for f in (lib.oracle_mask_dense, lib.oracle_classify_tiles, lib.oracle_forward_head,
                  lib.oracle_backward_head, lib.oracle_bias_grad_head):
            f.restype = None
        _lib = lib
    return _lib


class Program:
    """A mask program resolved for one batch row (doc ids and prefix length bound).

    ``selection`` (optional, int8 [nq, nkv], see ``selection_from_lists``)
    restricts it to caller-chosen tiles of ``block`` x ``block``: a pair is
    visible when its tile is selected as full (2), or selected as partial (1)
    and the program holds there.  ``q_offset``: query row i sits at position
    i + q_offset of the sequence (CAUSAL, WINDOW, SAME_DOC and ALiBi see that
    position), e.g. new tokens decoded at the end of a cache.
    """

    def __init__(self, mask, doc_row: Optional[np.ndarray] = None, prefix_len: Optional[int] = None,
                 selection: Optional[np.ndarray] = None, block: int = 128, q_offset: int = 0):
        nodes = mask.nodes if hasattr(mask, "nodes") else tuple(mask)
        if len(nodes) > 16:
            raise ValueError("at most 16 nodes")
        self._doc = None
        if any(n[0] == "same_doc" for n in nodes):
            if doc_row is None:
                raise ValueError("same_doc needs document ids")
            self._doc = np.ascontiguousarray(doc_row, dtype=np.int32)
        s = _Program()
        s.n = len(nodes)
        s.q_off = int(q_offset)
        for t, node in enumerate(nodes):
            s.op[t] = _OP[node[0]]
            if node[0] in ("window", "sink"):
                s.arg[t] = int(node[1])
            elif node[0] == "prefix":
                if prefix_len is None:
                    raise ValueError("prefix needs a prefix length")
                s.arg[t] = int(prefix_len)
        if self._doc is not None:
            s.doc = self._doc.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
        self._sel = None
        if selection is not None:
            self._sel = np.ascontiguousarray(selection, dtype=np.int8)
            if self._sel.ndim != 2 or block < 1:
                raise ValueError("selection must be [nq, nkv] with a positive block")
            s.sel = self._sel.ctypes.data_as(ctypes.POINTER(ctypes.c_int8))
            s.sel_block = int(block)
            s.sel_nkv = self._sel.shape[1]
        self.struct = s


def selection_from_lists(kv_num, kv_idx, full_num=None, full_idx=None, nkv: int = 0,
                         drop_invalid: bool = False) -> np.ndarray:
    """Tile selection [nq, nkv] of caller-supplied lists for one (batch, head).

    Row I lists ``kv_num[I]`` partial tiles in ``kv_idx[I, :kv_num[I]]`` and
    ``full_num[I]`` full tiles in ``full_idx[I, :full_num[I]]``, in any order
    (tutorial "FlexAttention in PyTorch", "Decoding and paged KV caches":
    BlockMask.from_kv_blocks).  Result: 0 not listed, 1 partial, 2 full.
    A count outside [0, min(nkv, row length)], an index outside [0, nkv) or a
    tile listed twice is invalid: ValueError, or with ``drop_invalid`` the
    entry is skipped (a count is clamped; a tile in both lists stays full).
    Returns (selection, n_invalid) when ``drop_invalid`` is set.
    """
    kv_num = np.asarray(kv_num)
    nq = kv_num.shape[0]
    sel = np.zeros((nq, nkv), dtype=np.int8)
    bad = 0
    lists = [(kv_num, np.asarray(kv_idx), 1)]
    if full_num is not None:
        lists.append((np.asarray(full_num), np.asarray(full_idx), 2))
    for num, idx, code in lists:
        for I in range(nq):
            n = int(num[I])
            cap = min(nkv, idx.shape[1])
            if n < 0 or n > cap:
                if not drop_invalid:
                    raise ValueError(f"row {I}: count {n} outside [0, {cap}]")
                bad += 1
                n = max(0, min(n, cap))
            for t in range(n):
                J = int(idx[I, t])
                if J < 0 or J >= nkv:
                    if not drop_invalid:
                        raise ValueError(f"row {I}: tile index {J} outside [0, {nkv})")
                    bad += 1
                    continue
                if sel[I, J] != 0:
                    if not drop_invalid:
                        raise ValueError(f"row {I}: tile {J} listed twice")
                    bad += 1
                sel[I, J] = max(int(sel[I, J]), code)
    return (sel, bad) if drop_invalid else sel


def _dptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _i64ptr(a: Optional[np.ndarray]):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))


def mask_dense(prog: Program, q_len: int, kv_len: int) -> np.ndarray:
    M = np.zeros((q_len, kv_len), dtype=np.uint8)
    _load().oracle_mask_dense(ctypes.byref(prog.struct), q_len, kv_len,
                              M.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)))
    return M.astype(bool)


def classify_tiles(prog: Program, q_len: int, kv_len: int, block: int = 128) -> np.ndarray:
    """Brute-force tile classes [nq, nkv]: 0 EMPTY, 1 PARTIAL, 2 FULL."""
    nq = -(-q_len // block)
    nkv = -(-kv_len // block)
    cls = np.zeros((nq, nkv), dtype=np.int8)
    _load().oracle_classify_tiles(ctypes.byref(prog.struct), q_len, kv_len, block,
                                  cls.ctypes.data_as(ctypes.POINTER(ctypes.c_int8)))
    return cls


def tile_lists(cls: np.ndarray) -> dict:
    """Per-row and per-column tile lists from a class grid.

    kv_* lists hold the PARTIAL tiles of each query-tile row, full_kv_* the
    FULL ones; both ascending, zero padded to nkv.  q_* / full_q_* are the
    same per key-tile column (used by the backward), padded to nq.
    """
    nq, nkv = cls.shape
    out = {}
    for name, code in (("kv", 1), ("full_kv", 2)):
        num = np.zeros(nq, dtype=np.int32)
        idx = np.zeros((nq, nkv), dtype=np.int32)
        for I in range(nq):
            js = np.nonzero(cls[I] == code)[0]
            num[I] = len(js)
            idx[I, :len(js)] = js
        out[f"{name}_num_blocks"] = num
        out[f"{name}_indices"] = idx
    for name, code in (("q", 1), ("full_q", 2)):
        num = np.zeros(nkv, dtype=np.int32)
        idx = np.zeros((nkv, nq), dtype=np.int32)
        for J in range(nkv):
            is_ = np.nonzero(cls[:, J] == code)[0]
            num[J] = len(is_)
            idx[J, :len(is_)] = is_
        out[f"{name}_num_blocks"] = num
        out[f"{name}_indices"] = idx
    return out


def _score_args(score: tuple, h: int):
    """(op, scalar parameter, bias table of head h or None, its first distance d0).
    Score tuples: ("none",), ("softcap", c), ("alibi", slopes[H]),
    ("relbias", table[H, L], d0) -- the learned relative-position bias
    s = x + table[h, clamp(q_pos - kv_idx - d0, 0, L - 1)]."""
    kind = score[0]
    if kind == "none":
        return _SCORE["none"], 0.0, None, 0
    if kind == "softcap":
        return _SCORE["softcap"], float(score[1]), None, 0
    if kind == "alibi":
        return _SCORE["alibi"], float(np.float32(score[1][h])), None, 0
    if kind == "relbias":
        table = np.ascontiguousarray(np.asarray(score[1], dtype=np.float32)[h], dtype=np.float64)
        return _SCORE["relbias"], 0.0, table, int(score[2])
    raise ValueError(score)


def _bias_args(table: Optional[np.ndarray], d0: int):
    if table is None:
        return [None, 0, 0]
    return [_dptr(table), int(d0), int(table.shape[0])]


def forward_head(q: np.ndarray, k: np.ndarray, v: np.ndarray, prog: Program, score: tuple, h: int,
                 scale: float, rows: Optional[Sequence[int]] = None):
    """out [n_rows, D], lse [n_rows] for one head; q, k, v float64 [len, D]."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    k = np.ascontiguousarray(k, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float64)
    D = q.shape[1]
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    n = q.shape[0] if r is None else len(r)
    out = np.zeros((n, D), dtype=np.float64)
    lse = np.zeros(n, dtype=np.float64)
    op, param, table, d0 = _score_args(score, h)
    _load().oracle_forward_head(_dptr(q), _dptr(k), _dptr(v), q.shape[0], k.shape[0], D,
                                ctypes.byref(prog.struct), op, param, float(scale), _i64ptr(r),
                                n, _dptr(out), _dptr(lse), *_bias_args(table, d0))
    return out, lse


def backward_head(q, k, v, do, prog: Program, score: tuple, h: int, scale: float,
                  rows: Optional[Sequence[int]] = None, cols: Optional[Sequence[int]] = None):
    """dq [rows], dk, dv [cols], plus lse and delta for every row, for one head."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    k = np.ascontiguousarray(k, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float64)
    do = np.ascontiguousarray(do, dtype=np.float64)
    D = q.shape[1]
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    c = None if cols is None else np.ascontiguousarray(cols, dtype=np.int64)
    nr = q.shape[0] if r is None else len(r)
    nc = k.shape[0] if c is None else len(c)
    dq = np.zeros((nr, D))
    dk = np.zeros((nc, D))
    dv = np.zeros((nc, D))
    lse = np.zeros(q.shape[0])
    delta = np.zeros(q.shape[0])
    op, param, table, d0 = _score_args(score, h)
    _load().oracle_backward_head(_dptr(q), _dptr(k), _dptr(v), _dptr(do), q.shape[0], k.shape[0], D,
                                 ctypes.byref(prog.struct), op, param, float(scale), _i64ptr(r), nr,
                                 _i64ptr(c), nc, _dptr(dq), _dptr(dk), _dptr(dv), _dptr(lse), _dptr(delta),
                                 *_bias_args(table, d0))
    return dq, dk, dv, lse, delta


def paged_gather(pool: np.ndarray, page_table: np.ndarray, kv_len: int, block: int = 128) -> np.ndarray:
    """Logical keys (or values) of a paged cache (tutorial "FlexAttention in
    PyTorch", "Decoding and paged KV caches": logical tile indices go through a
    page table to physical blocks).  pool [H, n_pages * block, D]; page_table
    [B, nkv]: the page holding logical tile J of batch row b.  Returns
    [B, H, kv_len, D] with row j of batch b taken from row j mod block of page
    page_table[b, j // block].  A page index outside [0, n_pages) is an error."""
    H, rows, D = pool.shape
    n_pages = rows // block
    B, nkv = page_table.shape
    if nkv * block < kv_len:
        raise ValueError("page table shorter than kv_len")
    out = np.zeros((B, H, kv_len, D), dtype=pool.dtype)
    for b in range(B):
        for J in range(-(-kv_len // block)):
            page = int(page_table[b, J])
            if page < 0 or page >= n_pages:
                raise ValueError(f"batch {b} tile {J}: page {page} outside [0, {n_pages})")
            n = min(block, kv_len - J * block)
            out[b, :, J * block:J * block + n] = pool[:, page * block:page * block + n]
    return out


def score_param_grad_head(q, k, v, do, prog: Program, score: tuple, h: int, scale: float) -> float:
    """dL/dparam of L = sum(out * dO) for one head: the soft-cap c, or the ALiBi
    slope of head h (0.0 for a score mod without a parameter)."""
    arrs = [np.ascontiguousarray(a, dtype=np.float64) for a in (q, k, v, do)]
    op, param, table, d0 = _score_args(score, h)
    return float(_load().oracle_score_param_grad_head(*(_dptr(a) for a in arrs), arrs[0].shape[0],
                                                      arrs[1].shape[0], arrs[0].shape[1],
                                                      ctypes.byref(prog.struct), op, param, float(scale),
                                                      *_bias_args(table, d0)))


def bias_grad_head(q, k, v, do, prog: Program, score: tuple, h: int, scale: float) -> np.ndarray:
    """dL/dtable[h, :] of L = sum(out * dO) for one (b, h) under ("relbias",
    table, d0): every visible pair's P (dP - Delta) added to the entry of its
    distance (tutorial Pattern 3: a learned relative-position bias trains)."""
    if score[0] != "relbias":
        raise ValueError(score)
    arrs = [np.ascontiguousarray(a, dtype=np.float64) for a in (q, k, v, do)]
    _, _, table, d0 = _score_args(score, h)
    grad = np.zeros(table.shape[0], dtype=np.float64)
    _load().oracle_bias_grad_head(*(_dptr(a) for a in arrs), arrs[0].shape[0], arrs[1].shape[0],
                                  arrs[0].shape[1], ctypes.byref(prog.struct), _dptr(table), int(d0),
                                  table.shape[0], float(scale), _dptr(grad))
    return grad


def head_score(score_kind: tuple, slopes=None, softcap=None) -> tuple:
    """Score tuple for forward_head/backward_head from workload fields."""
    if score_kind[0] == "alibi":
        return ("alibi", slopes)
    if score_kind[0] == "softcap":
        return ("softcap", softcap if softcap is not None else score_kind[1])
    return ("none",)


# ---------------------------------------------------------------------------
# numpy twin (tiny sizes only): dense explicit mask, dense softmax.
# ---------------------------------------------------------------------------

def np_mask(mask, q_len: int, kv_len: int, doc_row=None, prefix_len=None, q_offset: int = 0) -> np.ndarray:
    """Explicit [q_len, kv_len] boolean mask by broadcasting index grids; query
    row i sits at position i + q_offset."""
    i = np.arange(q_offset, q_offset + q_len, dtype=np.int64)[:, None]
    j = np.arange(kv_len, dtype=np.int64)[None, :]
    stack = []
    for node in (mask.nodes if hasattr(mask, "nodes") else mask):
        kind = node[0]
        if kind == "true":
            stack.append(np.ones((q_len, kv_len), dtype=bool))
        elif kind == "causal":
            stack.append(np.broadcast_to(i >= j, (q_len, kv_len)))
        elif kind == "same_doc":
            d = np.asarray(doc_row, dtype=np.int64)
            stack.append(d[q_offset:q_offset + q_len][:, None] == d[:kv_len][None, :])
        elif kind == "window":
            stack.append(np.broadcast_to((i - j) < node[1], (q_len, kv_len)))
        elif kind == "sink":
            stack.append(np.broadcast_to(j < node[1], (q_len, kv_len)))
        elif kind == "prefix":
            stack.append(np.broadcast_to(j < prefix_len, (q_len, kv_len)))
        elif kind in ("and", "or"):
            b = stack.pop()
            a = stack.pop()
            stack.append((a & b) if kind == "and" else (a | b))
        else:
            raise ValueError(node)
    (M,) = stack
    return np.array(M, dtype=bool)


def np_select(M: np.ndarray, selection: np.ndarray, block: int) -> np.ndarray:
    """Mask M restricted to selected tiles (see Program): the selection grid is
    expanded to one code per pair, then full -> visible, partial -> M, else hidden."""
    q_len, kv_len = M.shape
    E = np.repeat(np.repeat(np.asarray(selection), block, axis=0), block, axis=1)[:q_len, :kv_len]
    return (E == 2) | ((E == 1) & M)


def np_classify(M: np.ndarray, block: int, block_kv: Optional[int] = None) -> np.ndarray:
    """Tile classes of an explicit mask: 0 EMPTY (no visible pair), 2 FULL (every
    in-range pair visible), 1 PARTIAL.  Tiles are block x block, or block rows by
    block_kv columns when given (the rectangular tiles attention kernels walk
    over a finer block mask: tutorial, sharp edge 4)."""
    bk = block if block_kv is None else block_kv
    q_len, kv_len = M.shape
    nq, nkv = -(-q_len // block), -(-kv_len // bk)
    cls = np.zeros((nq, nkv), dtype=np.int8)
    for I in range(nq):
        for J in range(nkv):
            t = M[I * block:(I + 1) * block, J * bk:(J + 1) * bk]
            cls[I, J] = 0 if not t.any() else (2 if t.all() else 1)
    return cls


def _np_bias_entry(d0, L, q_len, kv_len, q_offset=0):
    """[q_len, kv_len] table entry of every pair: clip(q_pos - kv_idx - d0, 0, L - 1)."""
    i = np.arange(q_offset, q_offset + q_len)[:, None]
    j = np.arange(kv_len)[None, :]
    return np.clip(i - j - d0, 0, L - 1)


def _np_scores(q, k, score, slope, scale, q_len, kv_len, q_offset=0):
    """Scores and ds/dx.  score: ("none",), ("softcap", c), ("alibi",) with the
    head's slope in `slope`, or ("relbias", table_h [L], d0)."""
    x = scale * (q @ k.T)
    i = np.arange(q_offset, q_offset + q_len)[:, None]
    j = np.arange(kv_len)[None, :]
    if score[0] == "relbias":
        table = np.asarray(score[1], dtype=np.float64)
        return x + table[_np_bias_entry(int(score[2]), len(table), q_len, kv_len, q_offset)], np.ones_like(x)
    if score[0] == "softcap":
        c = float(score[1])
        t = np.tanh(x / c)
        return c * t, 1.0 - t * t
    if score[0] == "alibi":
        return x - slope * (i - j), np.ones_like(x)
    return x, np.ones_like(x)


def np_forward(q, k, v, M, score=("none",), slope=0.0, scale=None, q_offset=0):
    q_len, D = q.shape
    kv_len = k.shape[0]
    scale = 1.0 / np.sqrt(D) if scale is None else scale
    s, _ = _np_scores(q, k, score, slope, scale, q_len, kv_len, q_offset)
    s = np.where(M, s, -np.inf)
    m = s.max(axis=1, keepdims=True)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    e = np.where(M, np.exp(s - m_safe), 0.0)
    l = e.sum(axis=1, keepdims=True)
    with np.errstate(invalid="ignore", divide="ignore"):
        P = np.where(l > 0, e / np.where(l > 0, l, 1.0), 0.0)
        lse = np.where(l[:, 0] > 0, m_safe[:, 0] + np.log(np.where(l[:, 0] > 0, l[:, 0], 1.0)), -np.inf)
    return P @ v, lse, P


def np_backward(q, k, v, do, M, score=("none",), slope=0.0, scale=None, q_offset=0):
    q_len, D = q.shape
    kv_len = k.shape[0]
    scale = 1.0 / np.sqrt(D) if scale is None else scale
    out, lse, P = np_forward(q, k, v, M, score, slope, scale, q_offset)
    _, dsdx = _np_scores(q, k, score, slope, scale, q_len, kv_len, q_offset)
    dP = do @ v.T
    dS = P * (dP - (P * dP).sum(axis=1, keepdims=True)) * dsdx
    dq = scale * dS @ k
    dk = scale * dS.T @ q
    dv = P.T @ do
    return dq, dk, dv


def np_score_param_grad(q, k, v, do, M, score=("none",), slope=0.0, scale=None) -> float:
    """dL/dparam in matrix form: sum of P * (dP - Delta) * ds/dparam over the mask."""
    q_len, D = q.shape
    kv_len = k.shape[0]
    scale = 1.0 / np.sqrt(D) if scale is None else scale
    _, _, P = np_forward(q, k, v, M, score, slope, scale)
    dP = do @ v.T
    delta = (P * dP).sum(axis=1, keepdims=True)
    x = scale * (q @ k.T)
    if score[0] == "softcap":
        c = float(score[1])
        t = np.tanh(x / c)
        dsdp = t - (x / c) * (1.0 - t * t)
    elif score[0] == "alibi":
        dsdp = -(np.arange(q_len)[:, None] - np.arange(kv_len)[None, :]).astype(np.float64)
    else:
        dsdp = np.zeros_like(x)
    return float(np.where(M, P * (dP - delta) * dsdp, 0.0).sum())


def np_bias_grad(q, k, v, do, M, table_h, d0, scale=None, q_offset=0) -> np.ndarray:
    """dL/dtable_h in matrix form: dS = P (dP - Delta) over the mask, summed into
    the entry of each pair's distance."""
    q_len, D = q.shape
    kv_len = k.shape[0]
    scale = 1.0 / np.sqrt(D) if scale is None else scale
    score = ("relbias", table_h, d0)
    _, _, P = np_forward(q, k, v, M, score, 0.0, scale, q_offset)
    dP = do @ v.T
    dS = np.where(M, P * (dP - (P * dP).sum(axis=1, keepdims=True)), 0.0)
    grad = np.zeros(len(table_h))
    np.add.at(grad, _np_bias_entry(int(d0), len(table_h), q_len, kv_len, q_offset), dS)
    return grad
