"""Seeded synthetic workloads shaped like the pages' attention workloads.

Recipe (one place, used by every test and by the bench):

* seed = 1000 + workload number (1..5), unless a test passes its own seed;
* document lengths come from ``numpy.random.Generator(PCG64(seed))``:
  geometric with mean 100 (support 1, 2, ...) for the tiny workload,
  log-normal with median 600 and sigma 1.0, rounded and clipped to
  [16, 16384] for the packed 64K workloads; lengths are drawn until they
  cover S and the last document is cut to fit;
* document ids follow the speedrun notes ("FlexAttention", the code block
  after the Context paragraph): an end-of-text flag marks the first token of
  every document after the first, and the id of a position is the inclusive
  cumulative sum of the flags, so the first document has id 0;
* q, k, v and dO are drawn in that order from ``torch.Generator`` seeded with
  the same seed, as float32 N(0, 1) of shape [B, H, S, D], then rounded to
  bfloat16 (round to nearest even);
* ALiBi slopes are slope_h = 2^(-8 (h + 1) / H), stored as float32.

A mask program is a postfix list of nodes; the product binding and the oracle
each translate it into their own representation.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional, Sequence, Tuple

import numpy as np
import torch

# Node kinds of a mask program (postfix).  Atoms push one predicate, AND/OR pop
# two and push one.
ATOMS = ("true", "causal", "same_doc", "window", "sink", "prefix")
COMBINERS = ("and", "or")


@dataclasses.dataclass(frozen=True)
class MaskProgram:
    """A postfix mask program.

    ``nodes`` is a tuple of tuples: ("causal",), ("same_doc",), ("window", W),
    ("sink", n), ("prefix",), ("true",), ("and",), ("or",).  Window and sink
    carry their integer parameter; the document ids and the per-batch prefix
    lengths are passed beside the program as arrays.
    """

    nodes: Tuple[tuple, ...]

    def with_window(self, w: int) -> "MaskProgram":
        return MaskProgram(tuple(("window", int(w)) if n[0] == "window" else n for n in self.nodes))

    def uses(self, kind: str) -> bool:
        return any(n[0] == kind for n in self.nodes)

    def validate(self) -> None:
        depth = 0
        for n in self.nodes:
            if n[0] in ATOMS:
                depth += 1
            elif n[0] in COMBINERS:
                if depth < 2:
                    raise ValueError(f"combiner {n[0]} needs two operands")
                depth -= 1
            else:
                raise ValueError(f"unknown mask node {n!r}")
        if depth != 1:
            raise ValueError("mask program must leave exactly one value")


def _p(*nodes) -> MaskProgram:
    prog = MaskProgram(tuple(nodes))
    prog.validate()
    return prog


@dataclasses.dataclass(frozen=True)
class Workload:
    number: int
    name: str
    B: int
    H: int
    S: int
    D: int
    mask: MaskProgram
    docs: Optional[tuple]          # ("geometric", mean) | ("lognormal", median, sigma, lo, hi) | None
    score: tuple                   # ("none",) | ("softcap", c) | ("alibi",)
    windows: Tuple[int, ...] = ()  # window sweep (workload 5)
    doc_seed: Optional[int] = None  # seed of the document-length stream, if not the workload's own

    @property
    def seed(self) -> int:
        return 1000 + self.number


_LOGNORMAL = ("lognormal", 600.0, 1.0, 16, 16384)

WORKLOADS = {
    1: Workload(1, "tiny_doc_causal_S512", 1, 2, 512, 64,
                _p(("causal",), ("same_doc",), ("and",)), ("geometric", 100.0), ("none",)),
    2: Workload(2, "packed64k_doc_causal_w1024_D128", 1, 6, 65536, 128,
                _p(("causal",), ("same_doc",), ("and",), ("window", 1024), ("and",)), _LOGNORMAL, ("none",)),
    3: Workload(3, "window1024_sinks4_32k_D64", 1, 16, 32768, 64,
                _p(("causal",), ("window", 1024), ("sink", 4), ("or",), ("and",)), None, ("none",)),
    4: Workload(4, "causal_softcap30_8k_B4_D64", 4, 16, 8192, 64,
                _p(("causal",)), None, ("softcap", 30.0)),
    5: Workload(5, "packed64k_doc_window_sweep_alibi_D128", 1, 16, 65536, 128,
                _p(("causal",), ("same_doc",), ("and",), ("window", 64), ("and",)), _LOGNORMAL, ("alibi",),
                windows=tuple(range(64, 1793, 64)), doc_seed=1002),
}


def doc_lengths(rng: np.random.Generator, dist: tuple, S: int) -> List[int]:
    """Draw document lengths until they cover S; the last one is cut to fit."""
    lens: List[int] = []
    total = 0
    while total < S:
        if dist[0] == "geometric":
            L = int(rng.geometric(1.0 / float(dist[1])))
        elif dist[0] == "lognormal":
            _, median, sigma, lo, hi = dist
            L = int(np.clip(np.rint(rng.lognormal(np.log(median), sigma)), lo, hi))
        else:
            raise ValueError(dist)
        lens.append(L)
        total += L
    lens[-1] -= total - S
    return lens


def doc_ids_from_lengths(lens: Sequence[int]) -> np.ndarray:
    """Document id of every position: inclusive cumsum of end-of-text flags.

    The flag sits on the first token of each document after the first one,
    so ids start at 0 (the speedrun notes' ``cumsum(tokens == EOT)``).
    """
    S = int(sum(lens))
    eot = np.zeros(S, dtype=np.int32)
    starts = np.cumsum(np.asarray(lens, dtype=np.int64))[:-1]
    eot[starts] = 1
    return np.cumsum(eot, dtype=np.int64).astype(np.int32)


def make_doc_ids(dist: tuple, S: int, seed: int, batch: int = 1) -> np.ndarray:
    """[batch, S] int32 document ids, one independent stream per batch row."""
    rng = np.random.Generator(np.random.PCG64(seed))
    rows = [doc_ids_from_lengths(doc_lengths(rng, dist, S)) for _ in range(batch)]
    return np.stack(rows).astype(np.int32)


def make_qkv(B: int, H: int, S: int, D: int, seed: int, with_dout: bool = True,
             kv_len: Optional[int] = None):
    """q, k, v (and dO) as bfloat16 CPU tensors, drawn in that order."""
    g = torch.Generator().manual_seed(seed)
    kv_len = S if kv_len is None else kv_len
    q = torch.randn(B, H, S, D, generator=g, dtype=torch.float32).to(torch.bfloat16)
    k = torch.randn(B, H, kv_len, D, generator=g, dtype=torch.float32).to(torch.bfloat16)
    v = torch.randn(B, H, kv_len, D, generator=g, dtype=torch.float32).to(torch.bfloat16)
    if not with_dout:
        return q, k, v
    do = torch.randn(B, H, S, D, generator=g, dtype=torch.float32).to(torch.bfloat16)
    return q, k, v, do


def make_alibi_slopes(H: int) -> np.ndarray:
    """ALiBi slopes slope_h = 2^(-8 (h+1) / H) as float32 (workload 5's choice)."""
    return np.array([2.0 ** (-8.0 * (h + 1) / H) for h in range(H)], dtype=np.float32)


def make_workload_inputs(w: Workload, S: Optional[int] = None, B: Optional[int] = None,
                         H: Optional[int] = None, seed: Optional[int] = None, with_dout: bool = True):
    """Everything one workload needs, optionally at a smaller S/B/H with the same recipe.

    Returns a dict with q, k, v, (do), docs (int32 [B, S] or None), slopes
    (float32 [H] or None), softcap (float or None), mask (MaskProgram).
    """
    S = w.S if S is None else S
    B = w.B if B is None else B
    H = w.H if H is None else H
    seed = w.seed if seed is None else seed
    out = {}
    t = make_qkv(B, H, S, w.D, seed, with_dout=with_dout)
    out.update(q=t[0], k=t[1], v=t[2])
    if with_dout:
        out["do"] = t[3]
    out["docs"] = None
    if w.docs is not None:
        dseed = w.doc_seed if (w.doc_seed is not None and seed == w.seed) else seed
        out["docs"] = make_doc_ids(w.docs, S, dseed, batch=1)
    out["slopes"] = make_alibi_slopes(H) if w.score[0] == "alibi" else None
    out["softcap"] = float(w.score[1]) if w.score[0] == "softcap" else None
    out["mask"] = w.mask
    out["B"], out["H"], out["S"], out["D"] = B, H, S, w.D
    return out
