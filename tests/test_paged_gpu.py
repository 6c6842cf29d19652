"""Paged keys / values (tutorial "FlexAttention in PyTorch", "Decoding and
paged KV caches"): the paged forward through the C ABI gives the same bits as
the forward on the gathered logical keys and values, and matches the oracle
on the gathered tensors; page-table errors are reported."""
import numpy as np
import pytest
import torch

import oracle
from fa_testutil import check_forward, device_nodes
from synth import MaskProgram, make_alibi_slopes, make_doc_ids, make_qkv

pytestmark = pytest.mark.gpu

fa = pytest.importorskip("block_sparse_masked_fa_gb300")

P = lambda *n: MaskProgram(tuple(n))
DEVICE_CHECK = 7


def make_pool(H, n_pages, D, seed):
    """Pools of finite bf16 values (rows past kv_len in a last page are read)."""
    g = torch.Generator().manual_seed(seed)
    return tuple(torch.randn(H, n_pages * 128, D, generator=g).to(torch.bfloat16) for _ in range(2))


def gather(pool, table, kv_len):
    """Logical [B, H, kv_len, D] from a pool (test plumbing on the device)."""
    rows = (table.long()[:, :, None] * 128 + torch.arange(128, device=table.device)).reshape(table.shape[0], -1)
    return pool[:, rows[:, :kv_len]].permute(1, 0, 2, 3).contiguous()


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("score", ["none", "alibi", "relbias"])
def test_paged_forward_equals_gathered(D, score):
    B, H, q_len, kv_len = 3, 2, 700, 900
    nkv = -(-kv_len // 128)
    n_pages = B * nkv + 7
    kp, vp = make_pool(H, n_pages, D, 1 + D)
    table = torch.as_tensor(np.random.default_rng(2).permutation(n_pages)[:B * nkv].reshape(B, nkv),
                            dtype=torch.int32)
    q = make_qkv(B, H, q_len, D, 3 + D, with_dout=False)[0]
    docs = make_doc_ids(("geometric", 200.0), max(q_len, kv_len), 4, batch=B)
    mask = P(("causal",), ("same_doc",), ("and",), ("window", 500), ("and",))
    slopes = make_alibi_slopes(H)
    btab = np.random.default_rng(5).normal(scale=0.6, size=(H, 300)).astype(np.float32)  # distances 2 .. 301
    dev_score = {"none": None, "alibi": ("alibi", torch.as_tensor(slopes)),
                 "relbias": ("relbias", torch.as_tensor(btab), 2)}[score]
    qd, kpd, vpd, td = q.cuda(), kp.cuda(), vp.cuda(), table.cuda()
    bm = fa.fa_create_block_mask(device_nodes(mask, docs), B, 1, q_len, kv_len, 128)
    out_p, lse_p = fa.fa_forward_paged(qd, kpd, vpd, td, bm, score=dev_score)
    k_log, v_log = gather(kpd, td, kv_len), gather(vpd, td, kv_len)
    out_c, lse_c = fa.fa_forward(qd, k_log, v_log, bm, score=dev_score)
    torch.cuda.synchronize()
    assert fa.fa_get_status(bm) == 0
    assert torch.equal(out_p, out_c) and torch.equal(lse_p, lse_c)
    # the oracle on its own gather of the same pools
    kg = oracle.paged_gather(kp.double().numpy(), table.numpy(), kv_len)
    vg = oracle.paged_gather(vp.double().numpy(), table.numpy(), kv_len)
    ref_score = {"none": ("none",), "alibi": ("alibi", slopes), "relbias": ("relbias", btab, 2)}[score]
    for b, h in ((0, 0), (2, 1)):
        prog = oracle.Program(mask, doc_row=docs[b])
        ref_out, ref_lse = oracle.forward_head(q[b, h].double().numpy(), kg[b, h], vg[b, h], prog, ref_score, h,
                                               1.0 / np.sqrt(D))
        check_forward(out_p[b, h].float().cpu().numpy(), lse_p[b, h].cpu().numpy(), ref_out, ref_lse,
                      f"paged D{D} {score} b{b} h{h}")


def test_paged_decode_with_shared_prefix_pages():
    """One query per sequence (a decoding step); the batch rows share the pages
    of a common prefix, then continue on pages of their own."""
    B, H, kv_len, D = 4, 4, 1500, 128
    nkv = -(-kv_len // 128)
    shared = 5
    n_pages = shared + B * (nkv - shared)
    kp, vp = make_pool(H, n_pages, D, 11)
    table = np.zeros((B, nkv), np.int32)
    own = iter(np.random.default_rng(12).permutation(np.arange(shared, n_pages)))
    for b in range(B):
        table[b, :shared] = np.arange(shared)
        table[b, shared:] = [next(own) for _ in range(nkv - shared)]
    q = make_qkv(B, H, 1, D, 13, with_dout=False)[0]
    td = torch.as_tensor(table).cuda()
    bm = fa.fa_create_block_mask([("true",)], 1, 1, 1, kv_len, 128)
    out, lse = fa.fa_forward_paged(q.cuda(), kp.cuda(), vp.cuda(), td, bm)
    torch.cuda.synchronize()
    assert fa.fa_get_status(bm) == 0
    kg = oracle.paged_gather(kp.double().numpy(), table, kv_len)
    vg = oracle.paged_gather(vp.double().numpy(), table, kv_len)
    for b in range(B):
        for h in range(H):
            ref_out, ref_lse = oracle.forward_head(q[b, h].double().numpy(), kg[b, h], vg[b, h],
                                                   oracle.Program(P(("true",))), ("none",), h, 1.0 / np.sqrt(D))
            check_forward(out[b, h].float().cpu().numpy(), lse[b, h].cpu().numpy(), ref_out, ref_lse, f"b{b} h{h}")


def test_paged_page_out_of_range_reported():
    B, H, S, D = 1, 1, 512, 64
    kp, vp = make_pool(H, 4, D, 21)
    table = torch.tensor([[0, 1, 9, 3]], dtype=torch.int32).cuda()       # page 9 of 4
    q = make_qkv(B, H, S, D, 22, with_dout=False)[0].cuda()
    bm = fa.fa_create_block_mask([("causal",)], 1, 1, S, S, 128)
    fa.fa_forward_paged(q, kp.cuda(), vp.cuda(), table, bm)
    assert fa.fa_get_status(bm) == DEVICE_CHECK
    table[0, 2] = -1
    fa.fa_forward_paged(q, kp.cuda(), vp.cuda(), table, bm)
    assert fa.fa_get_status(bm) == DEVICE_CHECK
    table[0, 2] = 2
    fa.fa_forward_paged(q, kp.cuda(), vp.cuda(), table, bm)
    assert fa.fa_get_status(bm) == 0
