"""Learned relative-position bias (tutorial "FlexAttention in PyTorch", Pattern 3:
a score_mod edits every surviving logit, and a learned relative-position bias
trains through the fused backward):

    s = x + table[h, clamp(q_pos - kv_idx - d0, 0, L - 1)].

The forward (128 x 128 and 128 x 64 key tiles, and the short-query kernel), the
backward and the table gradient are compared with the oracle element by
element, on ragged document + window programs where the table is shorter than
the visible distances and d0 > 0, so that both clamped ends are in use, and
with query rows at an offset for decoding.
"""
import numpy as np
import pytest
import torch

import oracle
from fa_testutil import check_forward, check_grad, device_nodes, head64, oracle_program
from synth import MaskProgram, make_doc_ids, make_qkv

pytestmark = pytest.mark.gpu

fa = pytest.importorskip("block_sparse_masked_fa_gb300")

P = lambda *n: MaskProgram(tuple(n))
DOC_WIN = P(("causal",), ("same_doc",), ("and",), ("window", 500), ("and",))


def _table(H, L, seed):
    """A decaying bias with noise, fp32 [H, L]."""
    rng = np.random.default_rng(seed)
    return (-0.01 * np.arange(L)[None, :] + rng.normal(scale=0.5, size=(H, L))).astype(np.float32)


@pytest.mark.parametrize("block", [128, 64])
@pytest.mark.parametrize("D", [64, 128])
def test_forward_backward_and_table_gradient(D, block):
    """Distances 0..499 are visible; with d0 = 5 and L = 300 the first five and
    everything past 304 share the end entries.  The table gradient is summed
    over the batch, overwritten (the buffer starts as NaN), and leaves dk and dv
    bit-identical to a backward without it."""
    B, H, S, d0, L = 2, 2, 1100, 5, 300
    docs = make_doc_ids(("geometric", 300.0), S, 93, batch=B)
    q, k, v, do = make_qkv(B, H, S, D, 94 + D)
    table = _table(H, L, 95)
    score = ("relbias", torch.as_tensor(table), d0)
    bm = fa.fa_create_block_mask(device_nodes(DOC_WIN, docs), B, 1, S, S, block)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    out, lse = fa.fa_forward(qd, kd, vd, bm, score=score)
    dtab = torch.full((H, L), float("nan"), device="cuda")
    grads = fa.fa_backward(qd, kd, vd, out, lse, dod, bm, score=score, score_param_grad=dtab)
    plain = fa.fa_backward(qd, kd, vd, out, lse, dod, bm, score=score)
    torch.cuda.synchronize()
    assert fa.fa_get_status(bm) == 0
    assert torch.equal(grads[1], plain[1]) and torch.equal(grads[2], plain[2])
    osc = ("relbias", table, d0)
    scale = 1.0 / np.sqrt(D)
    ref_tab = np.zeros((H, L))
    for b in range(B):
        prog = oracle_program(DOC_WIN, docs, None, b, B)
        for h in range(H):
            qq, kk, vv, dd = (head64(t, b, h) for t in (q, k, v, do))
            ref_out, ref_lse = oracle.forward_head(qq, kk, vv, prog, osc, h, scale)
            check_forward(out[b, h].float().cpu().numpy(), lse[b, h].cpu().numpy(), ref_out, ref_lse,
                          f"block {block} D{D} b{b} h{h}")
            ref = oracle.backward_head(qq, kk, vv, dd, prog, osc, h, scale)[:3]
            for name, g, r in zip(("dq", "dk", "dv"), grads, ref):
                check_grad(g[b, h].float().cpu().numpy(), r, f"block {block} D{D} b{b} h{h} {name}")
            ref_tab[h] += oracle.bias_grad_head(qq, kk, vv, dd, prog, osc, h, scale)
    got = dtab.cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all() and np.abs(ref_tab[:, 0]).max() > 0 and np.abs(ref_tab[:, -1]).max() > 0
    check_grad(got, ref_tab, f"block {block} D{D} dtable")


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("q_len", [1, 4, 16])
def test_short_query_forward_at_an_offset(D, q_len):
    """q_len new tokens at the end of a 3,000-key cache (query positions
    kv_len - q_len ..), document + window 1,500 + causal, a 1,000-entry table:
    the short-query kernel and the general forward against the oracle."""
    B, H, kv_len, d0, L = 2, 2, 3000, 2, 1000
    off = kv_len - q_len
    q, k, v = make_qkv(B, H, q_len, D, 96 + D + q_len, with_dout=False, kv_len=kv_len)
    docs = make_doc_ids(("geometric", 900.0), kv_len, 97, batch=B)
    mask = P(("causal",), ("same_doc",), ("and",), ("window", 1500), ("and",))
    table = _table(H, L, 98)
    score = ("relbias", torch.as_tensor(table), d0)
    bm = fa.fa_create_block_mask(device_nodes(mask, docs), B, 1, q_len, kv_len, 128, q_offset=off)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    out_d, lse_d = fa.fa_forward_decode(qd, kd, vd, bm, score=score)
    out_f, lse_f = fa.fa_forward(qd, kd, vd, bm, score=score)
    torch.cuda.synchronize()
    assert fa.fa_get_status(bm) == 0
    osc = ("relbias", table, d0)
    for b in range(B):
        prog = oracle.Program(mask, doc_row=docs[b], q_offset=off)
        for h in range(H):
            ref_out, ref_lse = oracle.forward_head(head64(q, b, h), head64(k, b, h), head64(v, b, h), prog, osc, h,
                                                   1.0 / np.sqrt(D))
            for what, o, l in (("decode", out_d, lse_d), ("forward", out_f, lse_f)):
                check_forward(o[b, h].float().cpu().numpy(), l[b, h].cpu().numpy(), ref_out, ref_lse,
                              f"{what} D{D} b{b} h{h}")


def test_alibi_table_equals_alibi():
    """A table holding -slope_h * distance over every visible distance gives the
    ALiBi results (forward outputs, and dq / dk / dv to bf16 rounding)."""
    B, H, S, D = 1, 4, 900, 128
    q, k, v, do = make_qkv(B, H, S, D, 99)
    mask = P(("causal",), ("window", 400), ("and",))
    slopes = np.array([2.0 ** (-8 * (h + 1) / H) for h in range(H)], dtype=np.float32)
    table = (-slopes[:, None].astype(np.float64) * np.arange(400)[None, :]).astype(np.float32)
    bm = fa.fa_create_block_mask(device_nodes(mask), 1, 1, S, S, 128)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    res = {}
    for name, sc in (("alibi", ("alibi", torch.as_tensor(slopes))), ("table", ("relbias", torch.as_tensor(table), 0))):
        out, lse = fa.fa_forward(qd, kd, vd, bm, score=sc)
        res[name] = (out, lse) + tuple(fa.fa_backward(qd, kd, vd, out, lse, dod, bm, score=sc))
    torch.cuda.synchronize()
    assert fa.fa_get_status(bm) == 0
    a, t = res["alibi"], res["table"]
    assert (a[0].float() - t[0].float()).abs().max() <= 2e-2
    assert (a[1] - t[1]).abs().max() <= 1e-3
    for ga, gt in zip(a[2:], t[2:]):
        assert (ga.float() - gt.float()).abs().max() <= 2e-2 * ga.float().abs().max()
