"""Short-query forward (tutorial "FlexAttention in PyTorch", "Decoding and
paged KV caches": a decoding path for short queries), CUDA path through the C
ABI, against the oracle on every element: each (head dim, score mod, q_len
bucket), mask programs and caller-chosen tiles on partial tiles, plain and
paged caches, a single long sequence split over many CTAs, an empty
selection, and NaN in pool rows that must never be read."""
import numpy as np
import pytest
import torch

import oracle
from fa_testutil import check_forward, device_nodes
from synth import MaskProgram, make_alibi_slopes, make_doc_ids, make_qkv

pytestmark = pytest.mark.gpu

fa = pytest.importorskip("block_sparse_masked_fa_gb300")

P = lambda *n: MaskProgram(tuple(n))


def scores(kind, H):
    slopes = make_alibi_slopes(H)
    dev = {"none": None, "softcap": ("softcap", [3.0]), "alibi": ("alibi", torch.as_tensor(slopes))}[kind]
    ref = {"none": ("none",), "softcap": ("softcap", 3.0), "alibi": ("alibi", slopes)}[kind]
    return dev, ref


def check_all(out, lse, q, k, v, progs, ref_score, what):
    """progs(b) -> oracle Program for batch row b; every (b, h), every element."""
    B, H, _, D = q.shape
    for b in range(B):
        prog = progs(b)
        for h in range(H):
            ref_out, ref_lse = oracle.forward_head(q[b, h].double().numpy(), k[b, h].double().numpy(),
                                                   v[b, h].double().numpy(), prog, ref_score, h, 1.0 / np.sqrt(D))
            check_forward(out[b, h].float().cpu().numpy(), lse[b, h].cpu().numpy(), ref_out, ref_lse,
                          f"{what} b{b} h{h}")


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("score", ["none", "softcap", "alibi"])
@pytest.mark.parametrize("q_len", [1, 3, 16])
def test_decode_program(D, score, q_len):
    """A document program with sinks (the query rows sit in the first
    document; its keys span several tiles, ragged kv_len)."""
    B, H, kv_len = 2, 3, 1000
    docs = make_doc_ids(("geometric", 300.0), kv_len, 5 + q_len, batch=B)
    mask = P(("same_doc",), ("sink", 40), ("or",))
    q, k, v = make_qkv(B, H, q_len, D, 6 + D, with_dout=False, kv_len=kv_len)
    dev_score, ref_score = scores(score, H)
    bm = fa.fa_create_block_mask(device_nodes(mask, docs), B, 1, q_len, kv_len, 128)
    out, lse = fa.fa_forward_decode(q.cuda(), k.cuda(), v.cuda(), bm, score=dev_score)
    torch.cuda.synchronize()
    assert fa.fa_get_status(bm) == 0
    check_all(out, lse, q, k, v, lambda b: oracle.Program(mask, doc_row=docs[b]), ref_score,
              f"D{D} {score} q{q_len}")
    # the general forward agrees within the same bar
    out2, lse2 = fa.fa_forward(q.cuda(), k.cuda(), v.cuda(), bm, score=dev_score)
    assert (out2.float() - out.float()).abs().max() <= 2e-2


@pytest.mark.parametrize("D", [64, 128])
def test_decode_selected_tiles(D):
    """Block-selection decoding: caller-chosen FULL and PARTIAL tiles per batch
    row, a sink program on the partial ones."""
    B, H, q_len, kv_len = 3, 2, 2, 3000
    nkv = -(-kv_len // 128)
    rng = np.random.default_rng(D)
    sel = np.zeros((B, 1, 1, nkv), np.int8)
    for b in range(B):
        sel[b, 0, 0, rng.choice(nkv, 9, replace=False)] = rng.integers(1, 3, size=9)
    num = (sel == 1).sum(-1).astype(np.int32)
    fnum = (sel == 2).sum(-1).astype(np.int32)
    idx = np.zeros(sel.shape, np.int32)
    fidx = np.zeros(sel.shape, np.int32)
    for b in range(B):
        p_ = np.nonzero(sel[b, 0, 0] == 1)[0]
        f_ = np.nonzero(sel[b, 0, 0] == 2)[0]
        idx[b, 0, 0, :len(p_)] = p_[::-1]
        fidx[b, 0, 0, :len(f_)] = f_
    mask = P(("sink", 1000),)
    cu = lambda a: torch.as_tensor(a).cuda()
    bm = fa.fa_block_mask_from_kv_blocks(cu(num), cu(idx), q_len, kv_len, cu(fnum), cu(fidx),
                                         nodes=device_nodes(mask))
    q, k, v = make_qkv(B, H, q_len, D, 30 + D, with_dout=False, kv_len=kv_len)
    out, lse = fa.fa_forward_decode(q.cuda(), k.cuda(), v.cuda(), bm)
    torch.cuda.synchronize()
    assert fa.fa_get_status(bm) == 0
    check_all(out, lse, q, k, v, lambda b: oracle.Program(mask, selection=sel[b, 0], block=128), ("none",),
              f"D{D} selected")


def test_decode_paged_equals_plain_and_ignores_rows_past_kv_len():
    """Paged decode = plain decode on the gathered tensors, bit for bit, with
    the pool rows past kv_len in each last page set to NaN (never read)."""
    B, H, q_len, kv_len, D = 3, 4, 4, 1100, 128
    nkv = -(-kv_len // 128)
    n_pages = B * nkv + 3
    g = torch.Generator().manual_seed(40)
    kp = torch.randn(H, n_pages * 128, D, generator=g).to(torch.bfloat16)
    vp = torch.randn(H, n_pages * 128, D, generator=g).to(torch.bfloat16)
    table = np.random.default_rng(41).permutation(n_pages)[:B * nkv].reshape(B, nkv).astype(np.int32)
    tail = kv_len - (nkv - 1) * 128
    for b in range(B):
        last = int(table[b, -1])
        kp[:, last * 128 + tail:(last + 1) * 128] = float("nan")
        vp[:, last * 128 + tail:(last + 1) * 128] = float("nan")
    kg = torch.as_tensor(oracle.paged_gather(kp.float().numpy(), table, kv_len)).to(torch.bfloat16)
    vg = torch.as_tensor(oracle.paged_gather(vp.float().numpy(), table, kv_len)).to(torch.bfloat16)
    q = make_qkv(B, H, q_len, D, 42, with_dout=False)[0]
    mask = P(("true",))
    bm = fa.fa_create_block_mask(device_nodes(mask), 1, 1, q_len, kv_len, 128)
    out_p, lse_p = fa.fa_forward_decode(q.cuda(), kp.cuda(), vp.cuda(), bm, page_table=torch.as_tensor(table).cuda())
    out_c, lse_c = fa.fa_forward_decode(q.cuda(), kg.cuda(), vg.cuda(), bm)
    torch.cuda.synchronize()
    assert fa.fa_get_status(bm) == 0
    assert torch.isfinite(out_p.float()).all()
    assert torch.equal(out_p, out_c) and torch.equal(lse_p, lse_c)
    check_all(out_p, lse_p, q, kg, vg, lambda b: oracle.Program(mask), ("none",), "paged")


def test_decode_one_long_sequence_many_splits():
    """B = H = 1 over 160 key tiles: the work is split many ways (a share of a
    few tiles per CTA) and merged."""
    q_len, kv_len, D = 1, 160 * 128 - 5, 128
    assert fa.fa_forward_decode_workspace_bytes(1, 1, q_len, kv_len, D) >= 32 * q_len * (D + 1) * 4
    docs = make_doc_ids(("geometric", 15000.0), kv_len, 50)
    mask = P(("same_doc",), ("sink", 300), ("or",))
    q, k, v = make_qkv(1, 1, q_len, D, 51, with_dout=False, kv_len=kv_len)
    bm = fa.fa_create_block_mask(device_nodes(mask, docs), 1, 1, q_len, kv_len, 128)
    dev_score, ref_score = scores("alibi", 1)
    out, lse = fa.fa_forward_decode(q.cuda(), k.cuda(), v.cuda(), bm, score=dev_score)
    torch.cuda.synchronize()
    assert fa.fa_get_status(bm) == 0
    check_all(out, lse, q, k, v, lambda b: oracle.Program(mask, doc_row=docs[0]), ref_score, "long")


def test_decode_empty_selection():
    q_len, kv_len = 2, 600
    z = torch.zeros(1, 1, 1, dtype=torch.int32).cuda()
    bm = fa.fa_block_mask_from_kv_blocks(z, torch.zeros(1, 1, 1, 5, dtype=torch.int32).cuda(), q_len, kv_len)
    q, k, v = make_qkv(2, 2, q_len, 64, 60, with_dout=False, kv_len=kv_len)
    out, lse = fa.fa_forward_decode(q.cuda(), k.cuda(), v.cuda(), bm)
    torch.cuda.synchronize()
    assert fa.fa_get_status(bm) == 0
    assert torch.all(out == 0) and torch.all(torch.isneginf(lse))


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("paged", [False, True])
def test_decode_bucketed_cache(D, paged):
    """A block mask built once for a cache bucket of 4,096 keys (tutorial
    "Decoding and paged KV caches": bucket the cache length), reused while the
    cache grows: at each kv_len the result is the oracle's over the first
    kv_len keys with the same program.  The cache tensors have the bucket's
    rows; rows past kv_len hold NaN, and (paged) the table entries of tiles past
    kv_len name pages outside the pool: neither may be read."""
    B, H, q_len, cap = 2, 2, 2, 4096
    nkv = cap // 128
    docs = make_doc_ids(("geometric", 700.0), cap, 17, batch=B)
    mask = P(("same_doc",), ("sink", 16), ("or",), ("window", 100000), ("and",))
    q, k, v = make_qkv(B, H, q_len, D, 90 + D, with_dout=False, kv_len=cap)
    bm = fa.fa_create_block_mask(device_nodes(mask, docs), B, 1, q_len, cap, 128)
    for kv_len in (1, 129, 1000, 2500, 4095, 4096):
        kd, vd = k.clone(), v.clone()
        kd[:, :, kv_len:] = float("nan")
        vd[:, :, kv_len:] = float("nan")
        if paged:
            n_pages = B * nkv
            perm = np.random.default_rng(kv_len).permutation(n_pages)
            table = torch.full((B, nkv), 10 ** 6, dtype=torch.int32)          # out of range past kv_len
            kpool = torch.full((H, n_pages * 128, D), float("nan"), dtype=torch.bfloat16)
            vpool = kpool.clone()
            for b in range(B):
                for J in range(-(-kv_len // 128)):
                    pg = int(perm[b * nkv + J])
                    table[b, J] = pg
                    kpool[:, pg * 128:(pg + 1) * 128] = kd[b, :, J * 128:(J + 1) * 128]
                    vpool[:, pg * 128:(pg + 1) * 128] = vd[b, :, J * 128:(J + 1) * 128]
            out, lse = fa.fa_forward_decode(q.cuda(), kpool.cuda(), vpool.cuda(), bm, page_table=table.cuda(),
                                            kv_len=kv_len)
        else:
            out, lse = fa.fa_forward_decode(q.cuda(), kd.cuda(), vd.cuda(), bm, kv_len=kv_len)
        torch.cuda.synchronize()
        assert fa.fa_get_status(bm) == 0
        check_all(out, lse, q, k[:, :, :kv_len], v[:, :, :kv_len], lambda b: oracle.Program(mask, doc_row=docs[b]),
                  ("none",), f"D{D} paged {paged} kv_len {kv_len}")
