"""Block masks with tiles smaller than 128 (tutorial "FlexAttention in PyTorch",
sharp edge 4: a smaller BLOCK_SIZE captures more of a fine-grained mask's
sparsity) through the attention kernels.

The builder derives, from the block-size tile classes, the forward's 128-row by
64-column tiles and the backward's 128 x 128 tiles; their lists must be
bit-exact against the oracle's classes of the same rectangular tiles of the
explicit mask.  Forward and backward results must match the oracle (which
knows nothing of tiles) within the usual tolerances, at block 16, 32 and 64.
"""
import numpy as np
import pytest
import torch

import oracle
from fa_testutil import check_forward, check_grad, device_nodes, head64, oracle_score, score_arg
from synth import MaskProgram, make_alibi_slopes, make_doc_ids, make_qkv

pytestmark = pytest.mark.gpu

fa = pytest.importorskip("block_sparse_masked_fa_gb300")

P = lambda *n: MaskProgram(tuple(n))
DOC_WINDOW = P(("causal",), ("same_doc",), ("and",), ("window", 300), ("and",))
WINDOW_SINK = P(("causal",), ("window", 200), ("sink", 40), ("or",), ("and",))


def _lists_of(cls):
    return oracle.tile_lists(cls)


@pytest.mark.parametrize("block", [16, 32, 64])
@pytest.mark.parametrize("mask", ["doc_window", "window_sink"])
def test_kernel_tiles_bit_exact(block, mask):
    """The coarser lists of a ragged, non-square block mask against the oracle's
    classes of 128 x 64 (forward rows) and 128 x 128 (backward columns) tiles."""
    q_len, kv_len = 1500, 1700
    docs = make_doc_ids(("geometric", 40.0), kv_len, 31)
    prog = DOC_WINDOW if mask == "doc_window" else WINDOW_SINK
    bm = fa.fa_create_block_mask(device_nodes(prog, docs), 1, 1, q_len, kv_len, block)
    torch.cuda.synchronize()
    assert fa.fa_get_status(bm) == 0
    M = oracle.np_mask(prog, q_len, kv_len, doc_row=docs[0])
    got = {k: v.cpu().numpy()[0, 0] for k, v in bm.kernel_lists().items()}
    fcls = oracle.np_classify(M, 128, 64)
    bcls = oracle.np_classify(M, 128, 128)
    np.testing.assert_array_equal(got["fwd_tile_class"], fcls)
    np.testing.assert_array_equal(got["bwd_tile_class"], bcls)
    FL, BL = _lists_of(fcls), _lists_of(bcls)
    for name in ("kv_num_blocks", "kv_indices", "full_kv_num_blocks", "full_kv_indices"):
        np.testing.assert_array_equal(got["fwd_" + name], FL[name])
    for name in ("q_num_blocks", "q_indices", "full_q_num_blocks", "full_q_indices"):
        np.testing.assert_array_equal(got["bwd_" + name], BL[name])
    # and the block mask proper keeps the block-size tiles
    np.testing.assert_array_equal(bm.tile_class().cpu().numpy()[0, 0], oracle.np_classify(M, block))


def _run(q, k, v, do, nodes, block, score, scale=0.0):
    S, kv_len = q.shape[2], k.shape[2]
    bm = fa.fa_create_block_mask(nodes, 1, 1, S, kv_len, block)
    out, lse = fa.fa_forward(q, k, v, bm, score=score, scale=scale)
    grads = fa.fa_backward(q, k, v, out, lse, do, bm, score=score, scale=scale) if do is not None else None
    torch.cuda.synchronize()
    assert fa.fa_get_status(bm) == 0
    return out, lse, grads


@pytest.mark.parametrize("block", [16, 32, 64])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("score", ["none", "softcap", "alibi"])
def test_forward_backward_parity(block, D, score):
    """Every kernel instantiation of the 128 x 64 forward (two head dims, three
    score mods) and the backward on a ragged document + window mask."""
    H, q_len, kv_len = 2, 1100, 1300
    q, k, v, do = make_qkv(1, H, q_len, D, 900 + block + D, kv_len=kv_len)
    docs = make_doc_ids(("geometric", 40.0), kv_len, 77)
    slopes = make_alibi_slopes(H)
    kind = {"none": ("none",), "softcap": ("softcap", 30.0), "alibi": ("alibi",)}[score]
    sc = score_arg(kind, slopes, 30.0)
    out, lse, grads = _run(*(t.cuda() for t in (q, k, v, do)), device_nodes(DOC_WINDOW, docs), block, sc)
    prog = oracle.Program(DOC_WINDOW, doc_row=docs[0])
    osc = oracle_score(kind, slopes, 30.0)
    scale = 1.0 / np.sqrt(D)
    for h in range(H):
        ref_out, ref_lse = oracle.forward_head(head64(q, 0, h), head64(k, 0, h), head64(v, 0, h), prog, osc, h, scale)
        check_forward(out[0, h].float().cpu().numpy(), lse[0, h].cpu().numpy(), ref_out, ref_lse,
                      f"block {block} D{D} {score} h{h}")
        ref = oracle.backward_head(head64(q, 0, h), head64(k, 0, h), head64(v, 0, h), head64(do, 0, h), prog, osc,
                                   h, scale)[:3]
        for name, g, r in zip(("dq", "dk", "dv"), grads, ref):
            check_grad(g[0, h].float().cpu().numpy(), r, f"block {block} D{D} {score} h{h} {name}")


def test_block64_equals_block128_results():
    """The same inputs and program through block 64 and block 128 masks: both are
    exact computations of the same mask, so they agree within the tolerance."""
    q, k, v, do = (t.cuda() for t in make_qkv(1, 2, 2048, 128, 4321))
    docs = make_doc_ids(("geometric", 40.0), 2048, 5)
    nodes = device_nodes(DOC_WINDOW, docs)
    o64, l64, g64 = _run(q, k, v, do, nodes, 64, None)
    o128, l128, g128 = _run(q, k, v, do, nodes, 128, None)
    check_forward(o64.float().cpu().numpy(), l64.cpu().numpy(), o128.double().cpu().numpy(), l128.double().cpu().numpy(),
                  "block 64 vs 128")
    for a, b in zip(g64, g128):
        check_grad(a.float().cpu().numpy(), b.double().cpu().numpy(), "block 64 vs 128")


def test_fine_documents_full_length_sampled_rows():
    """A fine-grained mask at length: 16,384 tokens of documents of geometric mean
    length 40 (causal & same document), block 64; the forward walks fewer 64-wide
    key tiles than the 128-wide count would give, and sampled rows match the oracle."""
    S, H, D = 16384, 2, 128
    q, k, v = make_qkv(1, H, S, D, 2468, with_dout=False)
    docs = make_doc_ids(("geometric", 40.0), S, 13)
    prog = P(("causal",), ("same_doc",), ("and",))
    nodes = device_nodes(prog, docs)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    bm = fa.fa_create_block_mask(nodes, 1, 1, S, S, 64)
    out, lse = fa.fa_forward(qd, kd, vd, bm)
    torch.cuda.synchronize()
    assert fa.fa_get_status(bm) == 0
    L = bm.kernel_lists()
    fwd_tiles = int((L["fwd_kv_num_blocks"] + L["fwd_full_kv_num_blocks"]).sum())
    bm128 = fa.fa_create_block_mask(nodes, 1, 1, S, S, 128)
    e, p_, f_ = fa.fa_block_mask_summary(bm128)
    assert fwd_tiles < 2 * (p_ + f_)  # 64-wide tiles cover fewer key positions than 128-wide ones
    rng = np.random.default_rng(3)
    rows = np.unique(np.concatenate([rng.integers(0, S, 40), [0, S - 1, 127, 128]]))
    pr = oracle.Program(prog, doc_row=docs[0])
    for h in range(H):
        ref_out, ref_lse = oracle.forward_head(head64(q, 0, h), head64(k, 0, h), head64(v, 0, h), pr, ("none",), h,
                                               1.0 / np.sqrt(D), rows=rows)
        check_forward(out[0, h].float().cpu().numpy()[rows], lse[0, h].cpu().numpy()[rows], ref_out, ref_lse,
                      f"h{h}")


def test_small_blocks_refused_where_not_supported():
    """Caller-chosen tiles below block 128, and the paged / short-query forwards
    below block 128, are refused before any GPU work."""
    q, k, v = (t.cuda() for t in make_qkv(1, 1, 256, 64, 1, with_dout=False))
    num = torch.ones(1, 1, 4, dtype=torch.int32, device="cuda")
    idx = torch.zeros(1, 1, 4, 4, dtype=torch.int32, device="cuda")
    idx[0, 0, :, 0] = torch.arange(4, dtype=torch.int32)
    bm = fa.fa_block_mask_from_kv_blocks(num, idx, 256, 256, block=64)
    with pytest.raises(fa.FaError, match="UNSUPPORTED"):
        fa.fa_forward(q, k, v, bm)
    bm64 = fa.fa_create_block_mask([("causal",)], 1, 1, 1, 256, 64)
    with pytest.raises(fa.FaError, match="UNSUPPORTED"):
        fa.fa_forward_decode(q[:, :, :1], k, v, bm64)
