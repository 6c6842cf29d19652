"""Backward parity: dq, dk, dv of the CUDA path (through the C ABI) against
the fp64 oracle's gradients of L = sum(out * dO) on the same seeded inputs.

Bar: max |g - g_ref| / max |g_ref| <= 5e-2 for each gradient (written once in
fa_testutil).  The CUDA backward consumes the CUDA forward's out and LSE, as a
training step would.
"""
import numpy as np
import pytest
import torch

import oracle
from fa_testutil import (check_forward, check_grad, device_nodes, head64, oracle_program, oracle_score, score_arg)
from synth import WORKLOADS, MaskProgram, make_alibi_slopes, make_doc_ids, make_qkv, make_workload_inputs

pytestmark = pytest.mark.gpu

fa = pytest.importorskip("block_sparse_masked_fa_gb300")

P = lambda *n: MaskProgram(tuple(n))


def run_fa(inp, mask, Bm=1, prefix=None, score=None, window_tensor=None):
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    S, kv_len = q.shape[2], k.shape[2]
    bm = fa.fa_create_block_mask(device_nodes(mask, inp.get("docs"), prefix, window_tensor), Bm, 1, S, kv_len, 128)
    out, lse = fa.fa_forward(q, k, v, bm, score=score)
    dq, dk, dv = fa.fa_backward(q, k, v, out, lse, do, bm, score=score)
    torch.cuda.synchronize()
    assert fa.fa_get_status(bm) == 0
    return tuple(t.float().cpu().numpy() for t in (dq, dk, dv))


def oracle_grads(inp, mask, b, h, score, Bm=1, prefix=None, rows=None, cols=None):
    D = inp["q"].shape[-1]
    prog = oracle_program(mask, inp.get("docs"), prefix, b, Bm)
    dq, dk, dv, _, _ = oracle.backward_head(head64(inp["q"], b, h), head64(inp["k"], b, h), head64(inp["v"], b, h),
                                            head64(inp["do"], b, h), prog, score, h, 1.0 / np.sqrt(D),
                                            rows=rows, cols=cols)
    return dq, dk, dv


def check_all(got, ref, what):
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        check_grad(g, r, f"{what} {name}")


@pytest.mark.parametrize("wnum", [1, 2, 3, 4, 5])
@pytest.mark.parametrize("S", [1000, 1280])
def test_workload_recipe_reduced_size_all_elements(wnum, S):
    w = WORKLOADS[wnum]
    H = min(w.H, 2)
    inp = make_workload_inputs(w, S=S, B=1, H=H, seed=8000 + wnum)
    mask = w.mask.with_window(256) if w.windows else w.mask
    got = run_fa(inp, mask, score=score_arg(w.score, inp["slopes"], inp["softcap"]))
    for h in range(H):
        ref = oracle_grads(inp, mask, 0, h, oracle_score(w.score, inp["slopes"], inp["softcap"]))
        check_all([g[0, h] for g in got], ref, f"w{wnum} S{S} h{h}")


def _sample(S, rng, n=40):
    rows = set(rng.integers(0, S, size=n).tolist())
    rows.update([0, S - 1, 127, 128])
    return np.array(sorted(rows), dtype=np.int64)


@pytest.mark.parametrize("wnum", [1, 2, 3, 4, 5])
def test_workload_full_size_sampled(wnum):
    """Full workload shape; dq on sampled rows, dk / dv on sampled columns of two heads."""
    w = WORKLOADS[wnum]
    inp = make_workload_inputs(w)
    mask, W = w.mask, None
    if w.windows:
        W = torch.tensor([1024], dtype=torch.int32, device="cuda")
        mask = w.mask.with_window(1024)
    got = run_fa(inp, mask, score=score_arg(w.score, inp["slopes"], inp["softcap"]), window_tensor=W)
    rng = np.random.default_rng(100 + wnum)
    for b, h in [(0, 0), (w.B - 1, w.H - 1)]:
        rows = None if w.S <= 512 else _sample(w.S, rng)
        cols = None if w.S <= 512 else _sample(w.S, rng)
        ref = oracle_grads(inp, mask, b, h, oracle_score(w.score, inp["slopes"], inp["softcap"]), rows=rows, cols=cols)
        dq, dk, dv = (g[b, h] for g in got)
        if rows is not None:
            dq, dk, dv = dq[rows], dk[cols], dv[cols]
        check_all((dq, dk, dv), ref, f"w{wnum} b{b} h{h}")


def _inputs(B, H, S, D, seed, kv_len=None, docs=None):
    q, k, v, do = make_qkv(B, H, S, D, seed, kv_len=kv_len)
    return {"q": q, "k": k, "v": v, "do": do, "docs": docs}


@pytest.mark.parametrize("D", [64, 128])
def test_diagonal_only(D):
    """Only the diagonal visible: P = 1, so dv = dO and dq = dk = 0."""
    inp = _inputs(1, 2, 300, D, 21)
    dq, dk, dv = run_fa(inp, P(("causal",), ("window", 1), ("and",)))
    np.testing.assert_allclose(dv, inp["do"].float().numpy(), atol=1e-2)
    assert np.abs(dq).max() < 1e-2 and np.abs(dk).max() < 1e-2


@pytest.mark.parametrize("D", [64, 128])
def test_fully_masked_rows_and_columns(D):
    """same_doc & sink(10): documents after the first see nothing, so their dq
    rows are zero, and only the 10 sink keys get dk / dv."""
    S = 640
    docs = np.repeat(np.arange(5), 128).astype(np.int32)[None]
    docs[0, :200] = 0
    inp = _inputs(1, 2, S, D, 22, docs=docs)
    mask = P(("same_doc",), ("sink", 10), ("and",))
    dq, dk, dv = run_fa(inp, mask)
    assert np.all(dq[:, :, 200:] == 0)
    assert np.all(dk[:, :, 10:] == 0) and np.all(dv[:, :, 10:] == 0)
    for h in range(2):
        check_all([g[0, h] for g in (dq, dk, dv)], oracle_grads(inp, mask, 0, h, ("none",)), f"h{h}")


def test_everything_masked_gives_zero_gradients():
    inp = _inputs(1, 1, 256, 64, 23)
    dq, dk, dv = run_fa(inp, P(("causal",), ("window", 0), ("and",)))
    assert not dq.any() and not dk.any() and not dv.any()


@pytest.mark.parametrize("S", [1, 77, 129])
def test_tiny_sizes(S):
    inp = _inputs(1, 2, S, 128, 24)
    mask = P(("causal",))
    got = run_fa(inp, mask)
    for h in range(2):
        check_all([g[0, h] for g in got], oracle_grads(inp, mask, 0, h, ("none",)), f"S{S} h{h}")


@pytest.mark.parametrize("q_len,kv_len", [(256, 1000), (1000, 300)])
def test_cross_lengths(q_len, kv_len):
    inp = _inputs(1, 2, q_len, 64, 25, kv_len=kv_len)
    mask = P(("causal",), ("sink", 5), ("or",))
    got = run_fa(inp, mask, score=("softcap", [20.0]))
    for h in range(2):
        check_all([g[0, h] for g in got], oracle_grads(inp, mask, 0, h, ("softcap", 20.0)), f"{q_len}x{kv_len}")


def test_batch_broadcast_docs_prefix_alibi():
    S = 768
    docs = make_doc_ids(("geometric", 150.0), S, 26, batch=2)
    inp = _inputs(2, 2, S, 128, 27, docs=docs)
    prefix = np.array([90, 260], dtype=np.int32)
    mask = P(("causal",), ("prefix",), ("or",), ("same_doc",), ("and",))
    sl = make_alibi_slopes(2)
    got = run_fa(inp, mask, Bm=2, prefix=prefix, score=("alibi", torch.as_tensor(sl)))
    for b in range(2):
        for h in range(2):
            ref = oracle_grads(inp, mask, b, h, ("alibi", sl), Bm=2, prefix=prefix)
            check_all([g[b, h] for g in got], ref, f"b{b} h{h}")


def test_unsorted_document_ids():
    S = 900
    rng = np.random.default_rng(33)
    docs = np.repeat(rng.integers(0, 4, size=9), 100).astype(np.int32)[None]
    inp = _inputs(1, 2, S, 64, 34, docs=docs)
    mask = P(("same_doc",), ("window", 500), ("and",))
    got = run_fa(inp, mask)
    for h in range(2):
        check_all([g[0, h] for g in got], oracle_grads(inp, mask, 0, h, ("none",)), f"unsorted h{h}")


def test_rows_of_three_intervals():
    """Key columns seen by up to three separate query ranges (fallback to the
    per-word program) and by at most two (interval summary), against the oracle."""
    S = 1100
    docs = np.repeat(np.arange(11), 100).astype(np.int32)[None]
    inp = _inputs(1, 2, S, 64, 36, docs=docs)
    for mask in (P(("sink", 10), ("causal",), ("window", 64), ("and",), ("or",), ("same_doc",), ("or",)),
                 P(("sink", 10), ("causal",), ("window", 64), ("and",), ("or",))):
        got = run_fa(inp, mask)
        for h in range(2):
            check_all([g[0, h] for g in got], oracle_grads(inp, mask, 0, h, ("none",)), f"{len(mask.nodes)} nodes h{h}")


def test_many_items_per_cta_with_per_batch_masks():
    """More key tiles than resident CTAs, so every CTA walks several items: the
    mask arguments change between items (one prefix length and document layout
    per batch row), and many key tiles see no query at all."""
    B, H, S = 4, 2, 4096
    docs = make_doc_ids(("geometric", 300.0), S, 51, batch=B)
    inp = _inputs(B, H, S, 128, 52, docs=docs)
    prefix = np.array([0, 200, 700, 1500], dtype=np.int32)
    mask = P(("same_doc",), ("sink", 64), ("prefix",), ("or",), ("and",))
    got = run_fa(inp, mask, Bm=B, prefix=prefix)
    assert B * H * (S // 128) > torch.cuda.get_device_properties(0).multi_processor_count
    rng = np.random.default_rng(53)
    for b in range(B):
        h = b % H
        rows, cols = _sample(S, rng), _sample(S, rng)
        ref = oracle_grads(inp, mask, b, h, ("none",), Bm=B, prefix=prefix, rows=rows, cols=cols)
        dq, dk, dv = (g[b, h] for g in got)
        check_all((dq[rows], dk[cols], dv[cols]), ref, f"b{b} h{h}")
        # keys past the sink and the prefix are seen by no query: zero gradients
        hidden = np.arange(S) >= max(64, int(prefix[b]))
        assert not dk[hidden].any() and not dv[hidden].any()


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("score", ["none", "softcap", "alibi"])
def test_every_kernel_instantiation(D, score):
    """Each (head dim, score mod) kernel pair, forward and backward, on every
    element of a ragged size with partial and full tiles."""
    S, H = 700, 2
    inp = _inputs(1, H, S, D, 60 + D + len(score))
    mask = P(("causal",), ("window", 300), ("and",), ("sink", 8), ("or",), ("causal",), ("and",))
    sl = make_alibi_slopes(H)
    dev_score = {"none": None, "softcap": ("softcap", [25.0]), "alibi": ("alibi", torch.as_tensor(sl))}[score]
    ref_score = {"none": ("none",), "softcap": ("softcap", 25.0), "alibi": ("alibi", sl)}[score]
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    bm = fa.fa_create_block_mask(device_nodes(mask), 1, 1, S, S, 128)
    out, lse = fa.fa_forward(q, k, v, bm, score=dev_score)
    dq, dk, dv = fa.fa_backward(q, k, v, out, lse, do, bm, score=dev_score)
    torch.cuda.synchronize()
    assert fa.fa_get_status(bm) == 0
    for h in range(H):
        prog = oracle_program(mask, None, None, 0, 1)
        args = (head64(inp["q"], 0, h), head64(inp["k"], 0, h), head64(inp["v"], 0, h))
        ref_out, ref_lse = oracle.forward_head(*args, prog, ref_score, h, 1.0 / np.sqrt(D))
        check_forward(out[0, h].float().cpu().numpy(), lse[0, h].cpu().numpy(), ref_out, ref_lse, f"D{D} {score} h{h}")
        ref = oracle_grads(inp, mask, 0, h, ref_score)
        check_all([g[0, h].float().cpu().numpy() for g in (dq, dk, dv)], ref, f"D{D} {score} h{h}")


@pytest.mark.parametrize("D", [64, 128])
def test_alibi_slope_gradient(D):
    """dL/dslope[h] of learned ALiBi slopes (tutorial Pattern 3: a learned
    relative-position bias trains through the fused backward) against the
    oracle summed over the batch, on a ragged document + window + sink program.
    dk and dv are the same bits as without the slope gradient; dq, summed by
    reduce-adds in no fixed order, agrees to bf16 rounding."""
    B, H, S = 2, 4, 1900
    docs = make_doc_ids(("geometric", 400.0), S, 90, batch=B)
    inp = _inputs(B, H, S, D, 91 + D, docs=docs)
    mask = P(("causal",), ("same_doc",), ("and",), ("window", 700), ("and",), ("sink", 5), ("or",), ("causal",),
             ("and",))
    slopes = make_alibi_slopes(H)
    score = ("alibi", torch.as_tensor(slopes))
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    bm = fa.fa_create_block_mask(device_nodes(mask, docs), B, 1, S, S, 128)
    out, lse = fa.fa_forward(q, k, v, bm, score=score)
    g_plain = fa.fa_backward(q, k, v, out, lse, do, bm, score=score)
    dslope = torch.full((H,), float("nan"), device="cuda")       # overwritten, not accumulated
    g_slope = fa.fa_backward(q, k, v, out, lse, do, bm, score=score, score_param_grad=dslope)
    dslope2 = torch.full((H,), 7.0, device="cuda")
    fa.fa_backward_noalloc(q, k, v, out, lse, do, bm, score=score, score_param_grad=dslope2)
    torch.cuda.synchronize()
    assert fa.fa_get_status(bm) == 0
    assert torch.equal(g_plain[1], g_slope[1]) and torch.equal(g_plain[2], g_slope[2])
    dq0, dq1 = g_plain[0].float(), g_slope[0].float()
    assert (dq0 - dq1).abs().max() <= 1e-2 * dq0.abs().max()
    ref = np.zeros(H)
    for b in range(B):
        prog = oracle_program(mask, docs, None, b, B)
        for h in range(H):
            ref[h] += oracle.score_param_grad_head(head64(inp["q"], b, h), head64(inp["k"], b, h),
                                                   head64(inp["v"], b, h), head64(inp["do"], b, h), prog,
                                                   ("alibi", slopes), h, 1.0 / np.sqrt(D))
    got = dslope.cpu().numpy().astype(np.float64)
    assert np.abs(ref).max() > 0
    check_grad(got, ref, f"dslope D{D}")
    np.testing.assert_allclose(dslope2.cpu().numpy(), got, rtol=1e-5, atol=1e-6 * np.abs(ref).max())


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("cap", [5.0, 30.0])
def test_softcap_small_and_saturating_logits(D, cap):
    """Soft-cap with logits both well inside the cap (tanh nearly linear) and
    near saturation: query rows scaled by 1 and by 10 put both kinds in the same
    tiles.  Forward and gradients against the oracle, every element."""
    S, H = 640, 2
    q, k, v, do = make_qkv(1, H, S, D, 3100 + D, kv_len=S)
    rows = torch.arange(S)
    q = (q.float() * torch.where((rows // 48) % 2 == 0, 1.0, 10.0)[None, None, :, None]).to(torch.bfloat16)
    inp = {"q": q, "k": k, "v": v, "do": do, "docs": None}
    mask = P(("causal",), ("window", 400), ("and",))
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    bm = fa.fa_create_block_mask(device_nodes(mask), 1, 1, S, S, 128)
    out, lse = fa.fa_forward(qd, kd, vd, bm, score=("softcap", [cap]))
    grads = fa.fa_backward(qd, kd, vd, out, lse, dod, bm, score=("softcap", [cap]))
    torch.cuda.synchronize()
    assert fa.fa_get_status(bm) == 0
    prog = oracle.Program(mask)
    for h in range(H):
        ref_out, ref_lse = oracle.forward_head(head64(q, 0, h), head64(k, 0, h), head64(v, 0, h), prog,
                                               ("softcap", cap), h, 1.0 / np.sqrt(D))
        check_forward(out[0, h].float().cpu().numpy(), lse[0, h].cpu().numpy(), ref_out, ref_lse, f"cap {cap} h{h}")
        ref = oracle_grads(inp, mask, 0, h, ("softcap", cap))
        check_all([g[0, h].float().cpu().numpy() for g in grads], ref, f"cap {cap} D{D} h{h}")


def test_query_tiles_no_key_tile_sees_get_zero_dq():
    """Causal & window 100 with 200 keys and 600 queries: query rows from 300
    on see no key, so query tiles 3 and 4 have no visible key tile and no key
    tile's work ever reaches them; their dq (NaN beforehand) must come out
    zero.  The rest against the oracle."""
    B, H, S, KV, D = 1, 2, 600, 200, 64
    q, k, v, do = (t.cuda() for t in make_qkv(B, H, S, D, 517, kv_len=KV))
    mask = P(("causal",), ("window", 100), ("and",))
    bm = fa.fa_create_block_mask(device_nodes(mask), 1, 1, S, KV, 128)
    assert fa.fa_block_mask_summary(bm)[0] > 0  # some tiles EMPTY
    dq = torch.full_like(q, float("nan"))
    out, lse = fa.fa_forward(q, k, v, bm)
    dq, dk, dv = fa.fa_backward(q, k, v, out, lse, do, bm, dq=dq)
    torch.cuda.synchronize()
    assert fa.fa_get_status(bm) == 0
    assert bool((dq[:, :, 384:] == 0).all())
    inp = {n: t.cpu() for n, t in zip(("q", "k", "v", "do"), (q, k, v, do))}
    prog = oracle_program(mask, None, None, 0, 1)
    for h in range(H):
        ref = oracle.backward_head(head64(inp["q"], 0, h), head64(inp["k"], 0, h), head64(inp["v"], 0, h),
                                   head64(inp["do"], 0, h), prog, ("none",), h, 1.0 / np.sqrt(D))[:3]
        for name, gt, rf in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
            check_grad(gt[0, h].float().cpu().numpy(), rf, f"h{h} {name}")
