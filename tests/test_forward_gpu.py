"""Forward parity: out and LSE of the CUDA path (through the C ABI) against
the fp64 oracle on the same seeded inputs.

Reduced sizes compare every element (several tiles plus a ragged tail); the
full workload sizes compare sampled rows in the launch configuration the
bench times; edge cases cover empty rows, single tiles and broadcast masks.
"""
import numpy as np
import pytest
import torch

import oracle
from fa_testutil import (check_forward, device_nodes, head64, oracle_program, oracle_score, score_arg)
from synth import WORKLOADS, MaskProgram, make_alibi_slopes, make_doc_ids, make_qkv, make_workload_inputs

pytestmark = pytest.mark.gpu

fa = pytest.importorskip("block_sparse_masked_fa_gb300")


def run_fa(inp, mask, Bm=1, window_tensor=None, prefix=None, score=None, scale=0.0):
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    B, H, S, D = q.shape
    nodes = device_nodes(mask, inp.get("docs"), prefix, window_tensor)
    bm = fa.fa_create_block_mask(nodes, Bm, 1, S, k.shape[2], 128)
    out, lse = fa.fa_forward(q, k, v, bm, score=score, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_get_status(bm) == 0
    return out.float().cpu().numpy(), lse.cpu().numpy(), bm


def oracle_rows(inp, mask, b, h, rows, score, Bm=1, prefix=None, scale=None):
    D = inp["q"].shape[-1]
    scale = 1.0 / np.sqrt(D) if not scale else scale
    prog = oracle_program(mask, inp.get("docs"), prefix, b, Bm)
    return oracle.forward_head(head64(inp["q"], b, h), head64(inp["k"], b, h), head64(inp["v"], b, h), prog,
                               score, h, scale, rows=rows)


@pytest.mark.parametrize("wnum", [1, 2, 3, 4, 5])
@pytest.mark.parametrize("S", [1000, 1280])
def test_workload_recipe_reduced_size_all_elements(wnum, S):
    """Each workload's mask, score mod and head dim at S = 1000 (ragged) / 1280."""
    w = WORKLOADS[wnum]
    H = min(w.H, 3)
    inp = make_workload_inputs(w, S=S, B=1, H=H, seed=7000 + wnum, with_dout=False)
    mask = w.mask.with_window(256) if w.windows else w.mask
    sc = score_arg(w.score, inp["slopes"], inp["softcap"])
    out, lse, _ = run_fa(inp, mask, score=sc)
    for h in range(H):
        ref_out, ref_lse = oracle_rows(inp, mask, 0, h, None, oracle_score(w.score, inp["slopes"], inp["softcap"]))
        check_forward(out[0, h], lse[0, h], ref_out, ref_lse, f"w{wnum} S{S} h{h}")


def _sample_rows(S, rng, n=48):
    tiles = S // 128
    rows = set(rng.integers(0, S, size=n).tolist())
    for I in rng.integers(0, tiles, size=4):
        rows.update([int(I) * 128, int(I) * 128 + 127])
    rows.update([0, S - 1])
    return np.array(sorted(rows), dtype=np.int64)


@pytest.mark.parametrize("wnum", [1, 2, 3, 4, 5])
def test_workload_full_size_sampled_rows(wnum):
    """Full workload shape as timed by the bench; sampled rows of two heads (every row for workload 1)."""
    w = WORKLOADS[wnum]
    inp = make_workload_inputs(w, with_dout=False)
    W = None
    mask = w.mask
    if w.windows:
        W = torch.tensor([1024], dtype=torch.int32, device="cuda")
        mask = w.mask.with_window(1024)
    sc = score_arg(w.score, inp["slopes"], inp["softcap"])
    out, lse, _ = run_fa(inp, mask, window_tensor=W, score=sc)
    rng = np.random.default_rng(wnum)
    heads = [(0, 0), (w.B - 1, w.H - 1)]
    for b, h in heads:
        rows = None if w.S <= 512 else _sample_rows(w.S, rng)
        ref_out, ref_lse = oracle_rows(inp, mask, b, h, rows, oracle_score(w.score, inp["slopes"], inp["softcap"]))
        got_o = out[b, h] if rows is None else out[b, h][rows]
        got_l = lse[b, h] if rows is None else lse[b, h][rows]
        check_forward(got_o, got_l, ref_out, ref_lse, f"w{wnum} b{b} h{h}")


def _inputs(B, H, S, D, seed, kv_len=None, docs=None):
    q, k, v = make_qkv(B, H, S, D, seed, with_dout=False, kv_len=kv_len)
    return {"q": q, "k": k, "v": v, "docs": docs}


P = lambda *n: MaskProgram(tuple(n))


@pytest.mark.parametrize("D", [64, 128])
def test_fully_masked_rows(D):
    """window 0 masks every pair: out = 0, LSE = -inf everywhere; same_doc & sink
    masks exactly the rows of documents that start after the sinks."""
    S = 640
    inp = _inputs(1, 2, S, D, 11)
    out, lse, bm = run_fa(inp, P(("causal",), ("window", 0), ("and",)))
    assert np.all(out == 0) and np.all(np.isneginf(lse))
    assert fa.fa_block_mask_summary(bm)[0] == 25          # every tile EMPTY
    docs = np.repeat(np.arange(5), 128).astype(np.int32)[None]
    docs[0, :200] = 0                                       # doc 0 longer than the tile
    inp["docs"] = docs
    mask = P(("same_doc",), ("sink", 10), ("and",))
    out, lse, _ = run_fa(inp, mask)
    for h in range(2):
        ref_out, ref_lse = oracle_rows(inp, mask, 0, h, None, ("none",))
        check_forward(out[0, h], lse[0, h], ref_out, ref_lse, f"doc&sink h{h}")
    assert np.all(np.isneginf(lse[:, :, 256:]))


@pytest.mark.parametrize("D", [64, 128])
def test_diagonal_only(D):
    """causal & (i - j < 1): out_i = v_i and LSE_i = scale * q_i . k_i."""
    S = 384
    inp = _inputs(1, 1, S, D, 12)
    out, lse, _ = run_fa(inp, P(("causal",), ("window", 1), ("and",)))
    v = inp["v"][0, 0].float().numpy()
    np.testing.assert_allclose(out[0, 0], v, atol=1e-2)
    ref = (inp["q"][0, 0].double() * inp["k"][0, 0].double()).sum(-1).numpy() / np.sqrt(D)
    np.testing.assert_allclose(lse[0, 0], ref, atol=1e-3)


@pytest.mark.parametrize("S", [1, 77, 128, 129])
def test_tiny_and_single_tile(S):
    inp = _inputs(1, 2, S, 64, 13)
    mask = P(("causal",))
    out, lse, _ = run_fa(inp, mask)
    for h in range(2):
        ref_out, ref_lse = oracle_rows(inp, mask, 0, h, None, ("none",))
        check_forward(out[0, h], lse[0, h], ref_out, ref_lse, f"S{S}")


@pytest.mark.parametrize("q_len,kv_len", [(256, 1000), (1000, 300), (130, 515)])
def test_cross_lengths(q_len, kv_len):
    """q_len != kv_len with absolute-index causal plus sinks."""
    inp = _inputs(1, 2, q_len, 128, 14, kv_len=kv_len)
    mask = P(("causal",), ("sink", 5), ("or",))
    out, lse, _ = run_fa(inp, mask)
    for h in range(2):
        ref_out, ref_lse = oracle_rows(inp, mask, 0, h, None, ("none",))
        check_forward(out[0, h], lse[0, h], ref_out, ref_lse, f"{q_len}x{kv_len}")


def test_batch_broadcast_docs_and_prefix():
    """Bm = B = 2: different documents and prefix lengths per batch row; H = 3 broadcast."""
    S = 896
    docs = make_doc_ids(("geometric", 150.0), S, 15, batch=2)
    inp = _inputs(2, 3, S, 64, 16, docs=docs)
    prefix = np.array([100, 300], dtype=np.int32)
    mask = P(("causal",), ("prefix",), ("or",), ("same_doc",), ("and",))
    sl = make_alibi_slopes(3)
    out, lse, _ = run_fa(inp, mask, Bm=2, prefix=prefix, score=("alibi", torch.as_tensor(sl)))
    for b in range(2):
        for h in range(3):
            ref_out, ref_lse = oracle_rows(inp, mask, b, h, None, ("alibi", sl), Bm=2, prefix=prefix)
            check_forward(out[b, h], lse[b, h], ref_out, ref_lse, f"b{b} h{h}")


def test_v_ones_gives_ones():
    S = 700
    inp = _inputs(1, 2, S, 128, 17)
    inp["v"] = torch.ones_like(inp["v"])
    out, lse, _ = run_fa(inp, P(("causal",), ("window", 300), ("and",)), score=("softcap", [30.0]))
    np.testing.assert_allclose(out, 1.0, atol=4e-3)


def test_full_tiles_as_partial_give_same_result():
    """Tutorial, "The two hooks": the mask on a full tile changes nothing (the
    kernel only skips it for speed).  Moving every FULL tile into the PARTIAL
    list must give the same result within rounding."""
    S = 1024
    inp = _inputs(1, 2, S, 64, 18)
    mask = P(("causal",))
    out1, lse1, bm = run_fa(inp, mask)
    L = bm.lists()
    nkv = bm.struct.nkv
    num, idx, fnum, fidx = (L[n].view(-1, *L[n].shape[3:]) for n in
                            ("kv_num_blocks", "kv_indices", "full_kv_num_blocks", "full_kv_indices"))
    for r in range(num.shape[0]):
        merged = sorted(idx[r, :num[r]].tolist() + fidx[r, :fnum[r]].tolist())
        idx[r, :len(merged)] = torch.tensor(merged, dtype=torch.int32, device="cuda")
        num[r] = len(merged)
        fnum[r] = 0
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    out2, lse2 = fa.fa_forward(q, k, v, bm)
    np.testing.assert_allclose(out2.float().cpu().numpy(), out1, atol=2e-2)
    np.testing.assert_allclose(lse2.cpu().numpy(), lse1, atol=1e-4)
    assert nkv == 8


@pytest.mark.parametrize("D", [64, 128])
def test_unsorted_document_ids(D):
    """Document ids that decrease and repeat (doc 2 appears in two separate runs):
    the kernels compare ids one by one instead of using runs."""
    S = 900
    rng = np.random.default_rng(31)
    docs = np.repeat(rng.integers(0, 4, size=9), 100).astype(np.int32)[None]
    inp = _inputs(1, 2, S, D, 32, docs=docs)
    mask = P(("same_doc",), ("window", 500), ("and",))
    out, lse, _ = run_fa(inp, mask)
    for h in range(2):
        ref_out, ref_lse = oracle_rows(inp, mask, 0, h, None, ("none",))
        check_forward(out[0, h], lse[0, h], ref_out, ref_lse, f"unsorted h{h}")


def test_rows_of_three_intervals():
    """sink | (causal & window) | same_doc: a row sees up to three separate key
    ranges, more than the two-interval row summary holds, so the kernels fall
    back to evaluating the program per word; a second program with at most two
    per row takes the summary path.  Both against the oracle."""
    S = 1100
    docs = np.repeat(np.arange(11), 100).astype(np.int32)[None]
    inp = _inputs(1, 2, S, 64, 35, docs=docs)
    for mask in (P(("sink", 10), ("causal",), ("window", 64), ("and",), ("or",), ("same_doc",), ("or",)),
                 P(("sink", 10), ("causal",), ("window", 64), ("and",), ("or",))):
        out, lse, _ = run_fa(inp, mask)
        for h in range(2):
            ref_out, ref_lse = oracle_rows(inp, mask, 0, h, None, ("none",))
            check_forward(out[0, h], lse[0, h], ref_out, ref_lse, f"{len(mask.nodes)} nodes h{h}")


def test_many_items_per_cta_with_per_batch_masks():
    """More query tiles than resident CTAs, so every CTA walks several items:
    the mask arguments change between items (one prefix length and document
    layout per batch row), and many tiles see no key at all (same_doc & (sink |
    prefix) hides every document that starts after the sink and the prefix)."""
    B, H, S = 4, 4, 4096
    docs = make_doc_ids(("geometric", 300.0), S, 41, batch=B)
    inp = _inputs(B, H, S, 64, 42, docs=docs)
    prefix = np.array([0, 200, 700, 1500], dtype=np.int32)
    mask = P(("same_doc",), ("sink", 64), ("prefix",), ("or",), ("and",))
    out, lse, bm = run_fa(inp, mask, Bm=B, prefix=prefix)
    lists = bm.lists()
    visible = (lists["kv_num_blocks"].long() + lists["full_kv_num_blocks"].long()).cpu().numpy()
    assert (visible == 0).any() and (visible > 0).any()
    assert B * H * (S // 128) > 2 * torch.cuda.get_device_properties(0).multi_processor_count
    rng = np.random.default_rng(43)
    rows = np.unique(np.concatenate([rng.choice(S, 80, replace=False), [0, 63, 64, S - 1]])).astype(np.int64)
    for b in range(B):
        for h in (0, H - 1):
            ref_out, ref_lse = oracle_rows(inp, mask, b, h, rows, ("none",), Bm=B, prefix=prefix)
            check_forward(out[b, h][rows], lse[b, h][rows], ref_out, ref_lse, f"b{b} h{h}")
