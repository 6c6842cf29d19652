"""The prepared pair: fa_forward_prepare_backward (a forward that also clears
the backward workspace's fp32 dq accumulator while it runs) and
fa_backward_prepared (the backward that takes that accumulator as zero).

The forward's outputs are the same bits as fa_forward's; the workspace's
accumulator, filled with NaN beforehand, is zero afterwards (every CTA's share,
including the last partial copy); the prepared backward's gradients agree with
fa_backward's (dk and dv bit for bit, dq -- summed by reduce-adds in no fixed
order -- to bf16 rounding) and with the oracle on sampled heads.
"""
import numpy as np
import pytest
import torch

import oracle
from fa_testutil import check_grad, device_nodes, head64, oracle_program, oracle_score, score_arg
from synth import MaskProgram, make_alibi_slopes, make_doc_ids, make_qkv

pytestmark = pytest.mark.gpu

fa = pytest.importorskip("block_sparse_masked_fa_gb300")


def _run_pair(B, H, S, D, seed, mask, docs, score):
    q, k, v, do = (t.cuda() for t in make_qkv(B, H, S, D, seed))
    bm = fa.fa_create_block_mask(device_nodes(mask, docs), B if docs is not None and docs.ndim == 2 else 1, 1, S, S,
                                 128)
    ws_bytes = fa.fa_backward_workspace_bytes(B, H, S, D)
    ws = torch.full((ws_bytes,), 0xFF, dtype=torch.uint8, device="cuda")  # fp32 NaN in every word
    out_p, lse_p = fa.fa_forward_prepare_backward(q, k, v, bm, ws, score=score)
    torch.cuda.synchronize()
    acc = ws[: B * H * S * D * 4].view(torch.int32)
    assert int(torch.count_nonzero(acc)) == 0, "dq accumulator not cleared"
    assert bool((ws[B * H * S * D * 4:] == 0xFF).all()), "bytes past the accumulator written"
    out, lse = fa.fa_forward(q, k, v, bm, score=score)
    assert torch.equal(out, out_p) and torch.equal(lse, lse_p)
    g_ref = fa.fa_backward(q, k, v, out, lse, do, bm, score=score)
    g_pre = fa.fa_backward_prepared(q, k, v, out_p, lse_p, do, bm, ws, score=score)
    torch.cuda.synchronize()
    assert fa.fa_get_status(bm) == 0
    assert torch.equal(g_ref[1], g_pre[1]) and torch.equal(g_ref[2], g_pre[2])
    r, g = g_ref[0].float(), g_pre[0].float()
    assert (r - g).abs().max() <= 1e-2 * r.abs().max()
    return (q, k, v, do), g_pre


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("score_kind", [("none",), ("softcap", 20.0), ("alibi",)])
def test_prepared_pair_matches_forward_and_backward(D, score_kind):
    """Ragged length (7 full query tiles and a 104-row tail), documents, a
    window; B = 2 with a per-batch mask.  Gradients of two heads against the
    oracle, every element."""
    B, H, S = 2, 3, 1000
    docs = make_doc_ids(("geometric", 150.0), S, 31 + D, batch=B)
    mask = MaskProgram((("causal",), ("same_doc",), ("and",), ("window", 400), ("and",)))
    slopes = make_alibi_slopes(H)
    score = score_arg(score_kind, slopes=slopes)
    (q, k, v, do), (dq, dk, dv) = _run_pair(B, H, S, D, 700 + D, mask, docs, score)
    inp = {n: t.cpu() for n, t in zip(("q", "k", "v", "do"), (q, k, v, do))}
    ref_score = oracle_score(score_kind, slopes=slopes)
    for b, h in ((0, 0), (1, H - 1)):
        prog = oracle_program(mask, docs, None, b, B)
        ref = oracle.backward_head(head64(inp["q"], b, h), head64(inp["k"], b, h), head64(inp["v"], b, h),
                                   head64(inp["do"], b, h), prog, ref_score, h, 1.0 / np.sqrt(D))[:3]
        for name, gt, rf in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
            check_grad(gt[b, h].float().cpu().numpy(), rf, f"D{D} {score_kind[0]} b{b} h{h} {name}")


def test_prepared_pair_few_items_large_accumulator():
    """Two query tiles per head and one head: the forward runs two CTAs, each of
    which clears half of the accumulator (whole 4 KB copies and a partial
    last one: 200 rows x 128 x 4 bytes is not a multiple of 4 KB per CTA)."""
    mask = MaskProgram((("causal",),))
    _run_pair(1, 1, 200, 128, 77, mask, None, None)


def test_prepared_pair_twice_in_a_row():
    """A training loop: the pair called twice on one workspace.  The second
    forward clears what the first backward accumulated into."""
    B, H, S, D = 1, 2, 1300, 128
    q, k, v, do = (t.cuda() for t in make_qkv(B, H, S, D, 4242))
    bm = fa.fa_create_block_mask([("causal",)], 1, 1, S, S, 128)
    ws = torch.empty(fa.fa_backward_workspace_bytes(B, H, S, D), dtype=torch.uint8, device="cuda")
    out, lse = fa.fa_forward(q, k, v, bm)
    ref = fa.fa_backward(q, k, v, out, lse, do, bm)
    for _ in range(2):
        o2, l2 = fa.fa_forward_prepare_backward(q, k, v, bm, ws)
        got = fa.fa_backward_prepared(q, k, v, o2, l2, do, bm, ws)
        torch.cuda.synchronize()
        assert fa.fa_get_status(bm) == 0
        assert torch.equal(ref[1], got[1]) and torch.equal(ref[2], got[2])
        r, g = ref[0].float(), got[0].float()
        assert (r - g).abs().max() <= 1e-2 * r.abs().max()


@pytest.mark.parametrize("D", [64, 128])
def test_prepared_pair_block64_forward_tiles(D):
    """A block-64 mask: the forward walks 128 x 64 key tiles (its BK = 64
    kernels, which carry the same clearing stream) and the backward 128 x 128.
    Accumulator cleared, outputs equal to fa_forward's, gradients equal to
    fa_backward's."""
    B, H, S = 1, 3, 1000
    docs = make_doc_ids(("geometric", 60.0), S, 41 + D)
    q, k, v, do = (t.cuda() for t in make_qkv(B, H, S, D, 42 + D))
    bm = fa.fa_create_block_mask(device_nodes(MaskProgram((("causal",), ("same_doc",), ("and",))), docs), 1, 1,
                                 S, S, 64)
    ws = torch.full((fa.fa_backward_workspace_bytes(B, H, S, D),), 0xFF, dtype=torch.uint8, device="cuda")
    out_p, lse_p = fa.fa_forward_prepare_backward(q, k, v, bm, ws)
    torch.cuda.synchronize()
    assert int(torch.count_nonzero(ws[: B * H * S * D * 4])) == 0
    out, lse = fa.fa_forward(q, k, v, bm)
    assert torch.equal(out, out_p) and torch.equal(lse, lse_p)
    g_ref = fa.fa_backward(q, k, v, out, lse, do, bm)
    g_pre = fa.fa_backward_prepared(q, k, v, out, lse, do, bm, ws)
    torch.cuda.synchronize()
    assert fa.fa_get_status(bm) == 0
    assert torch.equal(g_ref[1], g_pre[1]) and torch.equal(g_ref[2], g_pre[2])
    r, g = g_ref[0].float(), g_pre[0].float()
    assert r.abs().max() > 0 and (r - g).abs().max() <= 1e-2 * r.abs().max()


@pytest.mark.parametrize("kind", ["alibi", "relbias"])
def test_prepared_pair_with_score_parameter_gradient(kind):
    """The learned ALiBi slopes' and bias table's gradients through
    fa_backward_prepared (its preprocessing kernel still zeroes the gradient
    buffer, NaN beforehand) match fa_backward's."""
    B, H, S, D = 2, 2, 900, 128
    docs = make_doc_ids(("geometric", 200.0), S, 61, batch=B)
    q, k, v, do = (t.cuda() for t in make_qkv(B, H, S, D, 62))
    mask = MaskProgram((("causal",), ("same_doc",), ("and",), ("window", 400), ("and",)))
    bm = fa.fa_create_block_mask(device_nodes(mask, docs), B, 1, S, S, 128)
    if kind == "alibi":
        score = ("alibi", torch.as_tensor(make_alibi_slopes(H)))
        shape = (H,)
    else:
        rng = np.random.default_rng(63)
        score = ("relbias", torch.as_tensor(rng.normal(scale=0.5, size=(H, 250)).astype(np.float32)), 3)
        shape = (H, 250)
    ws = torch.empty(fa.fa_backward_workspace_bytes(B, H, S, D), dtype=torch.uint8, device="cuda")
    out, lse = fa.fa_forward_prepare_backward(q, k, v, bm, ws, score=score)
    g_pre = torch.full(shape, float("nan"), device="cuda")
    grads = fa.fa_backward_prepared(q, k, v, out, lse, do, bm, ws, score=score, score_param_grad=g_pre)
    g_ref = torch.full(shape, float("nan"), device="cuda")
    ref = fa.fa_backward(q, k, v, out, lse, do, bm, score=score, score_param_grad=g_ref)
    torch.cuda.synchronize()
    assert fa.fa_get_status(bm) == 0
    assert torch.equal(grads[1], ref[1]) and torch.equal(grads[2], ref[2])
    a, b = g_pre.double(), g_ref.double()
    assert torch.isfinite(a).all() and b.abs().max() > 0
    assert (a - b).abs().max() <= 1e-3 * b.abs().max()
