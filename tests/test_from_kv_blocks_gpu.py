"""Caller-chosen tiles (BlockMask.from_kv_blocks of the tutorial "FlexAttention
in PyTorch", section "Decoding and paged KV caches"; block-selection sparse
patterns of its opening section), CUDA path through the C ABI:

* the block mask rebuilt from the caller's lists is bit-exact against the
  oracle's reading of the same lists (class grid, row and column lists, work
  orders), at several block sizes with ragged lengths and unordered lists;
* invalid lists set the status word's check bit and leave the lists of the
  valid entries;
* forward and backward match the oracle restricted to the selected tiles on
  every element (mask program on partial tiles, or none), including a
  decoding shape and an empty selection;
* a program's EMPTY tiles listed as PARTIAL change nothing (-inf is masked).
"""
import numpy as np
import pytest
import torch

import oracle
from fa_testutil import check_forward, check_grad, device_nodes, head64
from synth import MaskProgram, make_alibi_slopes, make_doc_ids, make_qkv
from test_builder_gpu import LIST_NAMES, compare

pytestmark = pytest.mark.gpu

fa = pytest.importorskip("block_sparse_masked_fa_gb300")

P = lambda *n: MaskProgram(tuple(n))
DEVICE_CHECK = 7


def random_lists(rng, Bm, Hm, nq, nkv, stride, p_part=0.3, p_full=0.3):
    """Unordered lists of a random selection per (bm, hm), junk past the counts."""
    sel = np.zeros((Bm, Hm, nq, nkv), np.int8)
    num = np.zeros((Bm, Hm, nq), np.int32)
    fnum = np.zeros((Bm, Hm, nq), np.int32)
    idx = rng.integers(-5, 3 * nkv, size=(Bm, Hm, nq, stride)).astype(np.int32)
    fidx = rng.integers(-5, 3 * nkv, size=(Bm, Hm, nq, stride)).astype(np.int32)
    for b in range(Bm):
        for h in range(Hm):
            u = rng.random((nq, nkv))
            sel[b, h] = np.where(u < p_part, 1, np.where(u < p_part + p_full, 2, 0))
            for I in range(nq):
                p = rng.permutation(np.nonzero(sel[b, h, I] == 1)[0])
                f = rng.permutation(np.nonzero(sel[b, h, I] == 2)[0])
                num[b, h, I], fnum[b, h, I] = len(p), len(f)
                idx[b, h, I, :len(p)] = p
                fidx[b, h, I, :len(f)] = f
    return sel, num, idx, fnum, fidx


def oracle_lists(sel):
    Bm, Hm = sel.shape[:2]
    per = [[oracle.tile_lists(sel[b, h]) for h in range(Hm)] for b in range(Bm)]
    return {n: np.stack([np.stack([per[b][h][n] for h in range(Hm)]) for b in range(Bm)]) for n in LIST_NAMES}


def cuda32(*arrays):
    return [torch.as_tensor(np.ascontiguousarray(a), dtype=torch.int32).cuda() for a in arrays]


@pytest.mark.parametrize("block,q_len,kv_len", [(128, 1000, 700), (64, 515, 1300), (32, 300, 333)])
def test_lists_bit_exact(block, q_len, kv_len):
    rng = np.random.default_rng(block + q_len)
    Bm, Hm = 2, 3
    nq, nkv = -(-q_len // block), -(-kv_len // block)
    sel, num, idx, fnum, fidx = random_lists(rng, Bm, Hm, nq, nkv, nkv + 3)
    bm = fa.fa_block_mask_from_kv_blocks(*cuda32(num, idx), q_len, kv_len, *cuda32(fnum, fidx), block=block)
    compare(bm, sel, oracle_lists(sel))
    np.testing.assert_array_equal(fa.fa_block_mask_summary(bm),
                                  [(sel == 0).sum(), (sel == 1).sum(), (sel == 2).sum()])


def test_partial_lists_only_and_narrow_rows():
    """No full lists, rows narrower than nkv (a top-k style selection of 3)."""
    rng = np.random.default_rng(5)
    q_len = kv_len = 2048
    nq = nkv = 16
    sel = np.zeros((1, 1, nq, nkv), np.int8)
    idx = np.zeros((1, 1, nq, 3), np.int32)
    for I in range(nq):
        js = rng.choice(nkv, 3, replace=False)
        idx[0, 0, I] = js
        sel[0, 0, I, js] = 1
    num = np.full((1, 1, nq), 3, np.int32)
    bm = fa.fa_block_mask_from_kv_blocks(*cuda32(num, idx), q_len, kv_len)
    compare(bm, sel, oracle_lists(sel))


def test_invalid_lists_flagged_and_dropped():
    nq = nkv = 4
    num = np.array([[[1, 2, 5, -1]]], np.int32)          # rows 2, 3: counts outside [0, 4]
    idx = np.array([[[[9, 0, 0, 0],                       # index past the last tile: dropped
                      [1, 1, 0, 0],                       # tile 1 listed twice
                      [0, 1, 2, 3],                       # count 5 clamped to 4
                      [0, 0, 0, 0]]]], np.int32)
    fnum = np.array([[[1, 0, 0, 1]]], np.int32)
    fidx = np.array([[[[2, 0, 0, 0], [0, 0, 0, 0], [0, 0, 0, 0], [3, 0, 0, 0]]]], np.int32)
    bm = fa.fa_block_mask_from_kv_blocks(*cuda32(num, idx), 512, 512, *cuda32(fnum, fidx))
    assert fa.fa_get_status(bm) == DEVICE_CHECK        # read and cleared
    sel, bad = oracle.selection_from_lists(num[0, 0], idx[0, 0], fnum[0, 0], fidx[0, 0], nkv, drop_invalid=True)
    assert bad == 4
    compare(bm, sel[None, None], oracle_lists(sel[None, None]))
    # a tile in both lists is flagged and stays FULL
    bm = fa.fa_block_mask_from_kv_blocks(*cuda32(np.array([[[1, 0, 0, 0]]], np.int32),
                                                 np.array([[[[2, 0, 0, 0]] + [[0] * 4] * 3]], np.int32)),
                                         512, 512,
                                         *cuda32(np.array([[[1, 0, 0, 0]]], np.int32),
                                                 np.array([[[[2, 0, 0, 0]] + [[0] * 4] * 3]], np.int32)))
    assert fa.fa_get_status(bm) == DEVICE_CHECK
    assert bm.tile_class().cpu().numpy()[0, 0, 0].tolist() == [0, 0, 2, 0]


def test_own_lists_round_trip():
    """A program's own lists, given back with the program, rebuild the same
    block mask and the same forward result, bit for bit."""
    S, D = 1500, 64
    docs = make_doc_ids(("geometric", 150.0), S, 11)
    mask = P(("causal",), ("same_doc",), ("and",), ("window", 400), ("and",))
    nodes = device_nodes(mask, docs)
    bm1 = fa.fa_create_block_mask(nodes, 1, 1, S, S, 128)
    L = bm1.lists()
    bm2 = fa.fa_block_mask_from_kv_blocks(L["kv_num_blocks"], L["kv_indices"], S, S, L["full_kv_num_blocks"],
                                          L["full_kv_indices"], nodes=nodes)
    assert fa.fa_get_status(bm2) == 0
    torch.testing.assert_close(bm2.tile_class(), bm1.tile_class(), rtol=0, atol=0)
    for n in LIST_NAMES:
        torch.testing.assert_close(bm2.lists()[n], L[n], rtol=0, atol=0)
    torch.testing.assert_close(bm2.row_segs(), bm1.row_segs(), rtol=0, atol=0)
    q, k, v = (t.cuda() for t in make_qkv(1, 2, S, D, 12, with_dout=False))
    o1, l1 = fa.fa_forward(q, k, v, bm1)
    o2, l2 = fa.fa_forward(q, k, v, bm2)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def _run_and_check(q_len, kv_len, D, B, H, sel, mask, docs, score, seed, what):
    """Forward + backward of the selection (lists per (b, h)) against the
    oracle on every element of every head."""
    q, k, v, do = make_qkv(B, H, q_len, D, seed, kv_len=kv_len)
    nkv = sel.shape[-1]
    num = (sel == 1).sum(-1).astype(np.int32)
    fnum = (sel == 2).sum(-1).astype(np.int32)
    idx = np.zeros(sel.shape, np.int32)
    fidx = np.zeros(sel.shape, np.int32)
    rng = np.random.default_rng(seed)
    for pos in np.ndindex(*sel.shape[:3]):
        p = rng.permutation(np.nonzero(sel[pos] == 1)[0])
        f = rng.permutation(np.nonzero(sel[pos] == 2)[0])
        idx[pos][:len(p)] = p
        fidx[pos][:len(f)] = f
    nodes = None if mask is None else device_nodes(mask, docs)
    bm = fa.fa_block_mask_from_kv_blocks(*cuda32(num, idx), q_len, kv_len, *cuda32(fnum, fidx), nodes=nodes)
    slopes = make_alibi_slopes(H)
    # the learned bias: distances -200 .. 999 in the table, both ends clamped for these lengths
    table = np.random.default_rng(seed + 1).normal(scale=0.6, size=(H, 1200)).astype(np.float32)
    dev_score = {"none": None, "softcap": ("softcap", [20.0]), "alibi": ("alibi", torch.as_tensor(slopes)),
                 "relbias": ("relbias", torch.as_tensor(table), -200)}[score]
    ref_score = {"none": ("none",), "softcap": ("softcap", 20.0), "alibi": ("alibi", slopes),
                 "relbias": ("relbias", table, -200)}[score]
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    out, lse = fa.fa_forward(qd, kd, vd, bm, score=dev_score)
    dq, dk, dv = fa.fa_backward(qd, kd, vd, out, lse, dod, bm, score=dev_score)
    torch.cuda.synchronize()
    assert fa.fa_get_status(bm) == 0
    Bm, Hm = sel.shape[:2]
    for b in range(B):
        for h in range(H):
            s = sel[0 if Bm == 1 else b, 0 if Hm == 1 else h]
            prog = oracle.Program(mask if mask is not None else P(("true",)),
                                  doc_row=None if docs is None else docs[0 if Bm == 1 else b], selection=s, block=128)
            args = [head64(t, b, h) for t in (q, k, v)]
            ref_out, ref_lse = oracle.forward_head(*args, prog, ref_score, h, 1.0 / np.sqrt(D))
            tag = f"{what} b{b} h{h}"
            check_forward(out[b, h].float().cpu().numpy(), lse[b, h].cpu().numpy(), ref_out, ref_lse, tag)
            ref = oracle.backward_head(*args, head64(do, b, h), prog, ref_score, h, 1.0 / np.sqrt(D))[:3]
            for g, r, name in zip((dq, dk, dv), ref, ("dq", "dk", "dv")):
                got = g[b, h].float().cpu().numpy()
                if np.abs(r).max() == 0:
                    assert np.abs(got).max() == 0, f"{tag} {name}: expected zeros"
                else:
                    check_grad(got, r, f"{tag} {name}")
    return out, lse, (dq, dk, dv)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("score", ["none", "softcap", "alibi", "relbias"])
def test_forward_backward_per_head_lists(D, score):
    """Per-(batch, head) random selections (Bm = B, Hm = H), no program: every
    pair of a listed tile is visible; ragged lengths."""
    B, H, q_len, kv_len = 2, 2, 700, 900
    nq, nkv = -(-q_len // 128), -(-kv_len // 128)
    rng = np.random.default_rng(D + len(score))
    sel = random_lists(rng, B, H, nq, nkv, nkv)[0]
    _run_and_check(q_len, kv_len, D, B, H, sel, None, None, score, 70 + D, f"D{D} {score}")


@pytest.mark.parametrize("D", [64, 128])
def test_forward_backward_program_on_partial_tiles(D):
    """A causal document program on the partial tiles, full tiles whole (even
    above the diagonal), one selection broadcast over the heads."""
    B, H, S = 2, 3, 1000
    n = -(-S // 128)
    docs = make_doc_ids(("geometric", 120.0), S, 21)
    sel = random_lists(np.random.default_rng(22 + D), 1, 1, n, n, n, 0.5, 0.2)[0]
    sel[0, 0, :, 0] = 1                           # every row sees its document start through tile 0 at least
    _run_and_check(S, S, D, B, H, sel, P(("causal",), ("same_doc",), ("and",)), docs, "none", 80 + D,
                   f"D{D} doc program")


def test_decoding_shape_block_selection():
    """One query per sequence over a long key cache, a few selected tiles (a
    decoding step of a block-selection sparse pattern)."""
    B, H, kv_len = 3, 4, 4000
    nkv = -(-kv_len // 128)
    rng = np.random.default_rng(31)
    sel = np.zeros((B, 1, 1, nkv), np.int8)
    for b in range(B):
        sel[b, 0, 0, rng.choice(nkv, 6, replace=False)] = 2
        sel[b, 0, 0, nkv - 1] = 1                  # the cut last tile through the program
    _run_and_check(1, kv_len, 128, B, H, sel, P(("true",)), None, "none", 32, "decode q_len 1")


def test_empty_selection():
    """Nothing listed: out = 0, LSE = -inf, zero gradients."""
    S = 300
    sel = np.zeros((1, 1, 3, 3), np.int8)
    out, lse, grads = _run_and_check(S, S, 64, 1, 2, sel, None, None, "none", 33, "empty")
    assert torch.all(out == 0) and torch.all(torch.isneginf(lse))
    assert all(torch.all(g == 0) for g in grads)


def test_empty_tiles_listed_as_partial_change_nothing():
    """-inf is the same as masked (tutorial "The two hooks"; speedrun notes,
    tile summary): listing a program's EMPTY tiles as PARTIAL, where the
    program hides every pair, leaves out, LSE and the gradients as they were."""
    S, D, H = 1000, 64, 2
    docs = make_doc_ids(("geometric", 200.0), S, 41)
    mask = P(("causal",), ("same_doc",), ("and",), ("window", 300), ("and",))
    nodes = device_nodes(mask, docs)
    q, k, v, do = (t.cuda() for t in make_qkv(1, H, S, D, 42))
    bm1 = fa.fa_create_block_mask(nodes, 1, 1, S, S, 128)
    L = {n: t.cpu().numpy() for n, t in bm1.lists().items()}
    cls = bm1.tile_class().cpu().numpy()[0, 0]
    nq, nkv = cls.shape
    num = L["kv_num_blocks"].copy()
    idx = np.zeros((1, 1, nq, nkv), np.int32)
    added = 0
    for I in range(nq):
        part = list(L["kv_indices"][0, 0, I, :num[0, 0, I]])
        empty = [J for J in range(nkv) if cls[I, J] == 0][:3]       # up to three hidden tiles per row
        added += len(empty)
        lst = part + empty
        idx[0, 0, I, :len(lst)] = lst
        num[0, 0, I] = len(lst)
    assert added > 0
    bm2 = fa.fa_block_mask_from_kv_blocks(torch.as_tensor(num).cuda(), torch.as_tensor(idx).cuda(), S, S,
                                          bm1.lists()["full_kv_num_blocks"], bm1.lists()["full_kv_indices"],
                                          nodes=nodes)
    o1, l1 = fa.fa_forward(q, k, v, bm1)
    o2, l2 = fa.fa_forward(q, k, v, bm2)
    g1 = fa.fa_backward(q, k, v, o1, l1, do, bm1)
    g2 = fa.fa_backward(q, k, v, o2, l2, do, bm2)
    torch.cuda.synchronize()
    assert fa.fa_get_status(bm1) == 0 and fa.fa_get_status(bm2) == 0
    assert int((bm2.tile_class() == 1).sum()) == int((bm1.tile_class() == 1).sum()) + added
    check_forward(o2.float().cpu().numpy(), l2.cpu().numpy(), o1.float().cpu().numpy(),
                  l1.cpu().numpy().astype(np.float64), "empty tiles as partial")
    for a, b, name in zip(g2, g1, ("dq", "dk", "dv")):
        check_grad(a.float().cpu().numpy(), b.float().cpu().numpy().astype(np.float64), name)
