"""Helpers shared by the GPU parity tests: seeded inputs on the device, the
mapping of a symbolic mask program to the library's node list, oracle runs per
head, and the tolerance checks.

Tolerances (written here once, used by every parity test):
  out  max |out - out_ref| <= 2e-2 over every element,
  LSE  max |lse - lse_ref| <= 1e-3 over rows whose LSE is finite, and the two
       sides agree on which rows are -inf (rows that see no key),
  grads max |g - g_ref| / max |g_ref| <= 5e-2 for each of dq, dk, dv.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

OUT_TOL = 2e-2
LSE_TOL = 1e-3
GRAD_TOL = 5e-2


def device_nodes(mask, docs=None, prefix=None, window_tensor=None):
    """Binding node list for a synth MaskProgram (docs [Bm, L] / prefix [Bm] as numpy)."""
    nodes = []
    for node in mask.nodes:
        kind = node[0]
        if kind == "same_doc":
            nodes.append(("same_doc", torch.as_tensor(np.ascontiguousarray(docs), dtype=torch.int32).cuda()))
        elif kind == "window":
            nodes.append(("window", window_tensor if window_tensor is not None else int(node[1])))
        elif kind == "sink":
            nodes.append(("sink", int(node[1])))
        elif kind == "prefix":
            nodes.append(("prefix", torch.as_tensor(np.asarray(prefix), dtype=torch.int32).cuda()))
        else:
            nodes.append((kind,))
    return nodes


def score_arg(score_kind, slopes=None, softcap=None):
    if score_kind[0] == "softcap":
        return ("softcap", [float(softcap if softcap is not None else score_kind[1])])
    if score_kind[0] == "alibi":
        return ("alibi", torch.as_tensor(slopes, dtype=torch.float32))
    return None


def oracle_score(score_kind, slopes=None, softcap=None):
    if score_kind[0] == "softcap":
        return ("softcap", float(softcap if softcap is not None else score_kind[1]))
    if score_kind[0] == "alibi":
        return ("alibi", slopes)
    return ("none",)


def head64(t, b, h):
    return t[b, h].to(torch.float64).numpy()


def oracle_program(mask, docs, prefix, b, Bm):
    bm = 0 if Bm == 1 else b
    return oracle.Program(mask, doc_row=None if docs is None else docs[bm],
                          prefix_len=None if prefix is None else int(prefix[bm]))


def check_forward(out, lse, ref_out, ref_lse, what=""):
    out = np.asarray(out, dtype=np.float64)
    lse = np.asarray(lse, dtype=np.float64)
    assert out.shape == ref_out.shape
    err = np.abs(out - ref_out).max() if out.size else 0.0
    assert err <= OUT_TOL, f"{what}: out max-abs error {err:.3e} > {OUT_TOL}"
    inf_gpu = np.isneginf(lse)
    inf_ref = np.isneginf(ref_lse)
    assert np.array_equal(inf_gpu, inf_ref), f"{what}: -inf LSE rows differ"
    fin = ~inf_ref
    if fin.any():
        lerr = np.abs(lse[fin] - ref_lse[fin]).max()
        assert lerr <= LSE_TOL, f"{what}: LSE max-abs error {lerr:.3e} > {LSE_TOL}"
    return err


def check_grad(g, ref, name):
    g = np.asarray(g, dtype=np.float64)
    scale = np.abs(ref).max()
    err = np.abs(g - ref).max()
    rel = err / scale if scale > 0 else err
    assert rel <= GRAD_TOL, f"{name}: max|g - g_ref| / max|g_ref| = {rel:.3e} > {GRAD_TOL}"
    return rel
