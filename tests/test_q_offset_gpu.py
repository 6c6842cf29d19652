"""Query rows at an offset (tutorial "FlexAttention in PyTorch", "Decoding and
paged KV caches": during generation the queries are the newest positions of a
longer key sequence, so a mask built for training shapes is wrong).

With fa_mask_spec.q_offset = o, query row i is position i + o for CAUSAL,
WINDOW, SAME_DOC and ALiBi.  The block mask lists (bit-exact), the forward, the
backward and the short-query forward are compared with the oracle, which takes
the same offset (and is itself pinned to equal the corresponding rows of the
whole sequence).
"""
import numpy as np
import pytest
import torch

import oracle
from fa_testutil import check_forward, check_grad, device_nodes, head64
from synth import MaskProgram, make_alibi_slopes, make_doc_ids, make_qkv

pytestmark = pytest.mark.gpu

fa = pytest.importorskip("block_sparse_masked_fa_gb300")

P = lambda *n: MaskProgram(tuple(n))
DOC_WIN = P(("causal",), ("same_doc",), ("and",), ("window", 300), ("and",))
WIN_SINK = P(("causal",), ("window", 200), ("sink", 24), ("or",), ("and",))


@pytest.mark.parametrize("mask", ["doc_win", "win_sink"])
@pytest.mark.parametrize("q_len,kv_len,off", [(300, 1000, 700), (257, 1000, 501), (1000, 1000, 0), (64, 1300, 1236)])
def test_block_mask_lists_with_offset(mask, q_len, kv_len, off):
    prog = DOC_WIN if mask == "doc_win" else WIN_SINK
    docs = make_doc_ids(("geometric", 90.0), kv_len, 41)
    bm = fa.fa_create_block_mask(device_nodes(prog, docs), 1, 1, q_len, kv_len, 128, q_offset=off)
    torch.cuda.synchronize()
    assert fa.fa_get_status(bm) == 0
    cls = oracle.classify_tiles(oracle.Program(prog, doc_row=docs[0], q_offset=off), q_len, kv_len)
    np.testing.assert_array_equal(bm.tile_class().cpu().numpy()[0, 0], cls)
    L = oracle.tile_lists(cls)
    got = {k: v.cpu().numpy()[0, 0] for k, v in bm.lists().items()}
    for name, ref in L.items():
        np.testing.assert_array_equal(got[name], ref, err_msg=name)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("off", [700, 699])
def test_forward_backward_with_offset(D, off):
    """Queries are the last 300 (or the 300 before the last one) of 1,000 + 1
    positions: document, window and causal mask, ALiBi; every element."""
    H, q_len, kv_len = 2, 300, 1001
    q, k, v, do = make_qkv(1, H, q_len, D, 770 + D, kv_len=kv_len)
    docs = make_doc_ids(("geometric", 80.0), kv_len, 19)
    slopes = make_alibi_slopes(H)
    score = ("alibi", torch.as_tensor(slopes))
    bm = fa.fa_create_block_mask(device_nodes(DOC_WIN, docs), 1, 1, q_len, kv_len, 128, q_offset=off)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    out, lse = fa.fa_forward(qd, kd, vd, bm, score=score)
    grads = fa.fa_backward(qd, kd, vd, out, lse, dod, bm, score=score)
    torch.cuda.synchronize()
    assert fa.fa_get_status(bm) == 0
    prog = oracle.Program(DOC_WIN, doc_row=docs[0], q_offset=off)
    scale = 1.0 / np.sqrt(D)
    for h in range(H):
        qq, kk, vv, dd = (head64(t, 0, h) for t in (q, k, v, do))
        ref_out, ref_lse = oracle.forward_head(qq, kk, vv, prog, ("alibi", slopes), h, scale)
        check_forward(out[0, h].float().cpu().numpy(), lse[0, h].cpu().numpy(), ref_out, ref_lse, f"off {off} h{h}")
        ref = oracle.backward_head(qq, kk, vv, dd, prog, ("alibi", slopes), h, scale)[:3]
        for name, g, r in zip(("dq", "dk", "dv"), grads, ref):
            check_grad(g[0, h].float().cpu().numpy(), r, f"off {off} h{h} {name}")


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("q_len", [1, 4])
def test_decode_newest_tokens(D, q_len):
    """The decoding case: q_len new tokens at the end of a 3,000-key cache with a
    causal, sliding-window, same-document program -- through the short-query
    forward and through the general forward."""
    B, H, kv_len = 2, 2, 3000
    off = kv_len - q_len
    q, k, v = make_qkv(B, H, q_len, D, 880 + D + q_len, with_dout=False, kv_len=kv_len)
    docs = make_doc_ids(("geometric", 900.0), kv_len, 23, batch=B)
    mask = P(("causal",), ("same_doc",), ("and",), ("window", 1500), ("and",))
    bm = fa.fa_create_block_mask(device_nodes(mask, docs), B, 1, q_len, kv_len, 128, q_offset=off)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    out_d, lse_d = fa.fa_forward_decode(qd, kd, vd, bm)
    out_f, lse_f = fa.fa_forward(qd, kd, vd, bm)
    torch.cuda.synchronize()
    assert fa.fa_get_status(bm) == 0
    for b in range(B):
        prog = oracle.Program(mask, doc_row=docs[b], q_offset=off)
        for h in range(H):
            ref_out, ref_lse = oracle.forward_head(head64(q, b, h), head64(k, b, h), head64(v, b, h), prog, ("none",),
                                                   h, 1.0 / np.sqrt(D))
            for what, o, l in (("decode", out_d, lse_d), ("forward", out_f, lse_f)):
                check_forward(o[b, h].float().cpu().numpy(), l[b, h].cpu().numpy(), ref_out, ref_lse,
                              f"{what} b{b} h{h}")


def test_offset_out_of_range_refused():
    """q_offset must keep every query position below max(q_len, kv_len)."""
    with pytest.raises(fa.FaError, match="INVALID"):
        fa.fa_create_block_mask([("causal",)], 1, 1, 300, 1000, 128, q_offset=701)
    with pytest.raises(fa.FaError, match="INVALID"):
        fa.fa_create_block_mask([("causal",)], 1, 1, 300, 1000, 128, q_offset=-1)


def test_long_prefill_chunk_sampled_rows():
    """A prefill chunk: 2,048 queries at positions 14,336 .. 16,383 of a 16,384-key
    sequence, document + window 1,024 + causal, ALiBi, D 128; sampled rows of
    the forward and the backward against the oracle."""
    H, q_len, kv_len, D = 4, 2048, 16384, 128
    off = kv_len - q_len
    q, k, v, do = make_qkv(1, H, q_len, D, 4321, kv_len=kv_len)
    docs = make_doc_ids(("lognormal", 600.0, 1.0, 16, 16384), kv_len, 1002)
    mask = P(("causal",), ("same_doc",), ("and",), ("window", 1024), ("and",))
    slopes = make_alibi_slopes(H)
    score = ("alibi", torch.as_tensor(slopes))
    bm = fa.fa_create_block_mask(device_nodes(mask, docs), 1, 1, q_len, kv_len, 128, q_offset=off)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    out, lse = fa.fa_forward(qd, kd, vd, bm, score=score)
    grads = fa.fa_backward(qd, kd, vd, out, lse, dod, bm, score=score)
    torch.cuda.synchronize()
    assert fa.fa_get_status(bm) == 0
    prog = oracle.Program(mask, doc_row=docs[0], q_offset=off)
    rng = np.random.default_rng(8)
    rows = np.unique(np.concatenate([rng.integers(0, q_len, 32), [0, 127, 128, q_len - 1]]))
    cols = np.unique(np.concatenate([rng.integers(off - 1100, kv_len, 32), [kv_len - 1, off, off - 1]]))
    scale = 1.0 / np.sqrt(D)
    for h in (0, H - 1):
        qq, kk, vv, dd = (head64(t, 0, h) for t in (q, k, v, do))
        ref_out, ref_lse = oracle.forward_head(qq, kk, vv, prog, ("alibi", slopes), h, scale, rows=rows)
        check_forward(out[0, h].float().cpu().numpy()[rows], lse[0, h].cpu().numpy()[rows], ref_out, ref_lse, f"h{h}")
        rdq, rdk, rdv, _, _ = oracle.backward_head(qq, kk, vv, dd, prog, ("alibi", slopes), h, scale, rows=rows,
                                                   cols=cols)
        for name, g, r in zip(("dq", "dk", "dv"), (grads[0][0, h][rows], grads[1][0, h][cols], grads[2][0, h][cols]),
                              (rdq, rdk, rdv)):
            check_grad(g.float().cpu().numpy(), r, f"h{h} {name}")
