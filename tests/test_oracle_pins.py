"""Pins of the CPU oracle to things other than itself (CPU only).

Each test fixes some part of the oracle against what the pages print, a closed
form, a library routine on a special case, finite differences, brute force
with an independent implementation, or an invariant of softmax attention.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from synth import MaskProgram, make_alibi_slopes, make_doc_ids

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def P(*nodes):
    return MaskProgram(tuple(nodes))


CAUSAL = P(("causal",))
DOC_CAUSAL = P(("causal",), ("same_doc",), ("and",))


def _golden_tile_counts():
    rows = []
    with open(os.path.join(GOLDEN, "tile_counts_64k.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            name, S, block, tiles = line.split()[:4]
            rows.append((name, int(S), int(block), int(tiles)))
    return rows


def _golden_program(name, S):
    if name == "causal":
        return oracle.Program(CAUSAL)
    if name == "causal_window1024":
        return oracle.Program(P(("causal",), ("window", 1024), ("and",)))
    if name == "causal_chunks1024":
        return oracle.Program(DOC_CAUSAL, doc_row=(np.arange(S) // 1024).astype(np.int32))
    raise KeyError(name)


# ---------------------------------------------------------------- tile classes

@pytest.mark.parametrize("row", _golden_tile_counts(), ids=lambda r: r[0])
def test_page_tile_counts(row):
    """Brute-force classifier reproduces the page's counts for a 64K sequence."""
    name, S, block, tiles = row
    cls = oracle.classify_tiles(_golden_program(name, S), S, S, block)
    assert int((cls > 0).sum()) == tiles


def test_page_ratios_consistent():
    """57x (dense causal vs chunks) and about 2x (window vs chunks), Record #12."""
    g = {r[0]: r[3] for r in _golden_tile_counts()}
    assert round(g["causal"] / g["causal_chunks1024"]) == 57
    assert abs(g["causal_window1024"] / g["causal_chunks1024"] - 2.0) < 0.05


def _window_closed_form(n, W, B=128):
    """Tile d = I - J of causal & (i - j < W) is non-empty iff 0 <= d <= (W + B - 2) // B,
    full iff 1 <= d <= (W - B) // B (derived from i - j spanning [B d - B + 1, B d + B - 1])."""
    dne = min((W + B - 2) // B, n - 1)
    dfull = min((W - B) // B, n - 1) if W >= B else 0
    nonempty = sum(n - d for d in range(0, dne + 1))
    full = sum(n - d for d in range(1, dfull + 1))
    return nonempty, full


@pytest.mark.parametrize("W", [1, 64, 127, 128, 129, 255, 256, 640, 1024, 1792, 5000])
def test_window_classes_closed_form(W):
    S = 8192
    cls = oracle.classify_tiles(oracle.Program(P(("causal",), ("window", W), ("and",))), S, S)
    nonempty, full = _window_closed_form(S // 128, W)
    assert int((cls > 0).sum()) == nonempty
    assert int((cls == 2).sum()) == full


def test_causal_classes_closed_form():
    """Causal: the diagonal tiles are PARTIAL, the strictly lower ones FULL."""
    S = 4096
    n = S // 128
    cls = oracle.classify_tiles(oracle.Program(CAUSAL), S, S)
    expect = np.tril(np.full((n, n), 2, dtype=np.int8), -1) + np.eye(n, dtype=np.int8)
    np.testing.assert_array_equal(cls, expect)


def test_window_sinks_32k_sparsity():
    """Tutorial Pattern 2: 32k context, 1k window + 4 sinks is about 97% block-sparse."""
    S = 32768
    prog = oracle.Program(P(("causal",), ("window", 1024), ("sink", 4), ("or",), ("and",)))
    cls = oracle.classify_tiles(prog, S, S)
    n = S // 128
    nonempty = int((cls > 0).sum())
    # closed form: the window band plus the first tile column below it
    band, _ = _window_closed_form(n, 1024)
    assert nonempty == band + (n - 9)
    assert 0.95 < 1 - nonempty / (n * n) < 0.98


def _random_program(rng, depth=3):
    atoms = [("causal",), ("same_doc",), ("window", int(rng.integers(0, 400))),
             ("sink", int(rng.integers(0, 200))), ("prefix",), ("true",)]
    if depth == 0 or rng.random() < 0.3:
        return [atoms[int(rng.integers(len(atoms)))]]
    a = _random_program(rng, depth - 1)
    b = _random_program(rng, depth - 1)
    return a + b + [("and",) if rng.random() < 0.6 else ("or",)]


@pytest.mark.parametrize("seed", range(12))
def test_mask_and_classes_match_numpy_twin(seed):
    """C element-wise evaluation vs numpy broadcasting on random and/or programs,
    with ragged lengths and small blocks."""
    rng = np.random.default_rng(seed)
    nodes = _random_program(rng)
    if len(nodes) > 16:
        nodes = nodes[:1]
    prog = MaskProgram(tuple(nodes))
    prog.validate()
    q_len, kv_len = int(rng.integers(1, 300)), int(rng.integers(1, 300))
    docs = make_doc_ids(("geometric", 40.0), max(q_len, kv_len), seed)[0]
    prefix = int(rng.integers(0, 150))
    cp = oracle.Program(prog, doc_row=docs, prefix_len=prefix)
    M_c = oracle.mask_dense(cp, q_len, kv_len)
    M_np = oracle.np_mask(prog, q_len, kv_len, doc_row=docs, prefix_len=prefix)
    np.testing.assert_array_equal(M_c, M_np)
    for block in (16, 32, 64, 128):
        np.testing.assert_array_equal(oracle.classify_tiles(cp, q_len, kv_len, block),
                                      oracle.np_classify(M_np, block))


def test_tile_lists_shape_and_order():
    S = 1000  # ragged: 8 tiles, the last one 104 rows
    docs = make_doc_ids(("geometric", 100.0), S, 7)[0]
    cls = oracle.classify_tiles(oracle.Program(DOC_CAUSAL, doc_row=docs), S, S)
    L = oracle.tile_lists(cls)
    n = cls.shape[0]
    for I in range(n):
        p = L["kv_indices"][I, :L["kv_num_blocks"][I]]
        f = L["full_kv_indices"][I, :L["full_kv_num_blocks"][I]]
        assert list(p) == sorted(p) and list(f) == sorted(f)
        assert set(p).isdisjoint(f)
        assert set(p) | set(f) == set(np.nonzero(cls[I])[0])
        assert not L["kv_indices"][I, L["kv_num_blocks"][I]:].any()
    assert L["q_num_blocks"].sum() == L["kv_num_blocks"].sum()
    assert L["full_q_num_blocks"].sum() == L["full_kv_num_blocks"].sum()


def test_rectangular_tiles_causal_closed_form():
    """Causal over 128-row by 64-column tiles: query-tile row I has FULL key tiles
    J < 2I and PARTIAL J = 2I, 2I + 1 (the diagonal 128-block split in two), and
    nothing after; with square tiles the classes are the C classifier's."""
    S = 1024
    M = oracle.np_mask(CAUSAL, S, S)
    cls = oracle.np_classify(M, 128, 64)
    n = S // 128
    assert cls.shape == (n, 2 * n)
    for I in range(n):
        assert (cls[I, :2 * I] == 2).all() and (cls[I, 2 * I:2 * I + 2] == 1).all() and not cls[I, 2 * I + 2:].any()
    for b in (32, 64, 128):
        np.testing.assert_array_equal(oracle.np_classify(M, b, b), oracle.classify_tiles(oracle.Program(CAUSAL), S, S, b))


def test_column_lists_causal_closed_form():
    """Causal key-tile column J: PARTIAL only on the diagonal (row J), FULL on rows J+1 .. n-1
    (the transpose of the row rule: row I sees J < I whole and J = I in part)."""
    S = 2048
    n = S // 128
    L = oracle.tile_lists(oracle.classify_tiles(oracle.Program(CAUSAL), S, S))
    for J in range(n):
        assert L["q_num_blocks"][J] == 1 and L["q_indices"][J, 0] == J
        assert not L["q_indices"][J, 1:].any()
        nf = n - 1 - J
        assert L["full_q_num_blocks"][J] == nf
        assert list(L["full_q_indices"][J, :nf]) == list(range(J + 1, n))
        assert not L["full_q_indices"][J, nf:].any()


@pytest.mark.parametrize("block", [32, 128])
def test_column_lists_are_rows_of_the_transposed_mask(block):
    """On a ragged, non-square mask that is not symmetric (documents, window, sinks), the
    column lists must equal the row lists of the transposed mask, classified from the numpy
    twin's dense [kv, q] matrix.  A row / column swap in the list builder fails this."""
    q_len, kv_len = 1000, 1300
    docs = make_doc_ids(("geometric", 90.0), kv_len, 11)[0]
    prog = P(("causal",), ("same_doc",), ("and",), ("window", 300), ("sink", 70), ("or",), ("and",))
    cp = oracle.Program(prog, doc_row=docs)
    L = oracle.tile_lists(oracle.classify_tiles(cp, q_len, kv_len, block))
    M = oracle.np_mask(prog, q_len, kv_len, doc_row=docs)
    LT = oracle.tile_lists(oracle.np_classify(np.ascontiguousarray(M.T), block))
    assert L["q_num_blocks"].shape == (-(-kv_len // block),)
    assert L["q_indices"].shape == (-(-kv_len // block), -(-q_len // block))
    for mine, theirs in (("q", "kv"), ("full_q", "full_kv")):
        np.testing.assert_array_equal(L[f"{mine}_num_blocks"], LT[f"{theirs}_num_blocks"])
        np.testing.assert_array_equal(L[f"{mine}_indices"], LT[f"{theirs}_indices"])
    assert L["q_num_blocks"].sum() > 0 and L["full_q_num_blocks"].sum() > 0


# ---------------------------------------------------------------- forward

def _qkv(S, D, seed, kv_len=None):
    g = torch.Generator().manual_seed(seed)
    kv_len = S if kv_len is None else kv_len
    f = lambda n: torch.randn(n, D, generator=g).to(torch.bfloat16).double().numpy()
    return f(S), f(kv_len), f(kv_len), f(S)


def test_forward_matches_sdpa_causal():
    """Causal mask without score_mod is textbook causal attention (torch SDPA, fp64)."""
    S, D = 300, 64
    q, k, v, _ = _qkv(S, D, 1)
    out, lse = oracle.forward_head(q, k, v, oracle.Program(CAUSAL), ("none",), 0, 1 / np.sqrt(D))
    tq, tk, tv = (torch.from_numpy(a)[None, None] for a in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=True)[0, 0].numpy()
    np.testing.assert_allclose(out, ref, atol=1e-12, rtol=0)
    s = (q @ k.T) / np.sqrt(D)
    ref_lse = torch.logsumexp(torch.from_numpy(np.where(np.tril(np.ones((S, S), bool)), s, -np.inf)), 1)
    np.testing.assert_allclose(lse, ref_lse.numpy(), atol=1e-12, rtol=0)


def test_forward_matches_sdpa_doc_mask_and_alibi():
    """Document mask + ALiBi as an additive bias is SDPA with a float mask."""
    S, D, H = 257, 64, 4
    q, k, v, _ = _qkv(S, D, 2)
    docs = make_doc_ids(("geometric", 50.0), S, 3)[0]
    slopes = make_alibi_slopes(H)
    h = 2
    prog = oracle.Program(DOC_CAUSAL, doc_row=docs)
    out, lse = oracle.forward_head(q, k, v, prog, ("alibi", slopes), h, 1 / np.sqrt(D))
    i = np.arange(S)[:, None]
    j = np.arange(S)[None, :]
    visible = (i >= j) & (docs[:, None] == docs[None, :])
    bias = np.where(visible, -float(slopes[h]) * (i - j), -np.inf)
    tq, tk, tv = (torch.from_numpy(a)[None, None] for a in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(
        tq, tk, tv, attn_mask=torch.from_numpy(bias)[None, None])[0, 0].numpy()
    np.testing.assert_allclose(out, ref, atol=1e-12, rtol=0)


def test_forward_q_zero_closed_form():
    """q = 0: every visible logit is 0, so out_i is the mean of visible v_j and LSE_i = ln |V_i|."""
    S, D = 333, 64
    _, k, v, _ = _qkv(S, D, 4)
    q = np.zeros((S, D))
    docs = make_doc_ids(("geometric", 60.0), S, 5)[0]
    prog = oracle.Program(P(("causal",), ("same_doc",), ("and",), ("window", 100), ("and",)), doc_row=docs)
    out, lse = oracle.forward_head(q, k, v, prog, ("none",), 0, 0.125)
    for i in range(S):
        js = [j for j in range(max(0, i - 99), i + 1) if docs[j] == docs[i]]
        np.testing.assert_allclose(out[i], v[js].mean(axis=0), atol=1e-12)
        assert abs(lse[i] - np.log(len(js))) < 1e-12


def test_forward_q_zero_alibi_geometric_weights():
    """q = 0 with ALiBi: weights proportional to exp(-slope (i - j)), a geometric series."""
    S, D = 200, 64
    _, k, v, _ = _qkv(S, D, 6)
    q = np.zeros((S, D))
    slope = 0.25
    out, lse = oracle.forward_head(q, k, v, oracle.Program(CAUSAL), ("alibi", [slope]), 0, 0.125)
    for i in (0, 1, 17, 199):
        r = np.exp(-slope)
        w = r ** (i - np.arange(i + 1))           # j = 0..i
        total = (1 - r ** (i + 1)) / (1 - r)       # geometric sum
        np.testing.assert_allclose(out[i], (w[:, None] * v[:i + 1]).sum(0) / total, atol=1e-12)
        assert abs(lse[i] - np.log(total)) < 1e-12


def test_forward_v_ones_rows_sum_to_one():
    S, D = 260, 128
    q, k, _, _ = _qkv(S, D, 7)
    v = np.ones((S, D))
    out, _ = oracle.forward_head(q, k, v, oracle.Program(CAUSAL), ("softcap", 30.0), 0, 0.3)
    np.testing.assert_allclose(out, 1.0, atol=1e-13)


def test_forward_diagonal_window_one():
    """causal & (i - j < 1) leaves only the diagonal: out_i = v_i, LSE_i = s_ii."""
    S, D = 150, 64
    q, k, v, _ = _qkv(S, D, 8)
    prog = oracle.Program(P(("causal",), ("window", 1), ("and",)))
    out, lse = oracle.forward_head(q, k, v, prog, ("none",), 0, 0.125)
    np.testing.assert_allclose(out, v, atol=1e-14)
    np.testing.assert_allclose(lse, 0.125 * (q * k).sum(1), atol=1e-12)


def test_forward_fully_masked_rows():
    """Rows that see nothing: out = 0, LSE = -inf (window 0 masks everything;
    same_doc & sink(n) masks the rows of every document that starts after n)."""
    S, D = 200, 64
    q, k, v, do = _qkv(S, D, 9)
    out, lse = oracle.forward_head(q, k, v, oracle.Program(P(("causal",), ("window", 0), ("and",))),
                                   ("none",), 0, 0.125)
    assert np.all(out == 0) and np.all(np.isneginf(lse))
    docs = np.repeat(np.arange(4), 50).astype(np.int32)
    prog = oracle.Program(P(("same_doc",), ("sink", 10), ("and",)), doc_row=docs)
    out, lse = oracle.forward_head(q, k, v, prog, ("none",), 0, 0.125)
    assert np.all(np.isfinite(lse[:50])) and np.all(np.isneginf(lse[50:]))
    assert np.all(out[50:] == 0)
    dq, dk, dv, _, _ = oracle.backward_head(q, k, v, do, prog, ("none",), 0, 0.125)
    assert np.all(dq[50:] == 0) and np.all(dk[10:] == 0) and np.all(dv[10:] == 0)


def test_softcap_small_logits_close_to_plain():
    """c tanh(s / c) = s - s^3 / (3 c^2) + ...: tiny logits barely change."""
    S, D = 128, 64
    q, k, v, _ = _qkv(S, D, 10)
    scale = 1e-3
    prog = oracle.Program(CAUSAL)
    o1, l1 = oracle.forward_head(q, k, v, prog, ("softcap", 30.0), 0, scale)
    o0, l0 = oracle.forward_head(q, k, v, prog, ("none",), 0, scale)
    smax = np.abs(scale * q @ k.T).max()
    bound = smax ** 3 / (3 * 30.0 ** 2) * 2
    assert np.abs(l1 - l0).max() <= bound
    assert np.abs(o1 - o0).max() <= 4 * bound * np.abs(v).max()


def test_softcap_saturates():
    """Huge logits are capped to [-c, c], so LSE_i <= c + ln |V_i|."""
    S, D = 128, 64
    q, k, v, _ = _qkv(S, D, 11)
    _, lse = oracle.forward_head(q, k, v, oracle.Program(CAUSAL), ("softcap", 30.0), 0, 1e4)
    assert np.all(lse <= 30.0 + np.log(np.arange(1, S + 1)) + 1e-12)


@pytest.mark.parametrize("score", ["none", "softcap", "alibi"])
def test_forward_matches_numpy_twin(score):
    S, D = 203, 64
    q, k, v, _ = _qkv(S, D, 12, kv_len=190)
    docs = make_doc_ids(("geometric", 30.0), S, 13)[0]
    mask = P(("causal",), ("same_doc",), ("and",), ("window", 70), ("sink", 3), ("or",), ("and",))
    sc = {"none": ("none",), "softcap": ("softcap", 5.0), "alibi": ("alibi", [0.125])}[score]
    prog = oracle.Program(mask, doc_row=docs)
    out, lse = oracle.forward_head(q, k, v, prog, sc, 0, 0.2)
    M = oracle.np_mask(mask, S, 190, doc_row=docs)
    ref, ref_lse, _ = oracle.np_forward(q, k, v, M, sc if score != "alibi" else ("alibi",), 0.125, 0.2)
    np.testing.assert_allclose(out, ref, atol=1e-12)
    np.testing.assert_array_equal(np.isneginf(lse), np.isneginf(ref_lse))
    f = np.isfinite(lse)
    np.testing.assert_allclose(lse[f], ref_lse[f], atol=1e-12)


def test_forward_row_subset_matches_full():
    S, D = 300, 64
    q, k, v, _ = _qkv(S, D, 14)
    prog = oracle.Program(CAUSAL)
    out, lse = oracle.forward_head(q, k, v, prog, ("none",), 0, 0.125)
    rows = [0, 5, 299, 128]
    o2, l2 = oracle.forward_head(q, k, v, prog, ("none",), 0, 0.125, rows=rows)
    np.testing.assert_array_equal(o2, out[rows])
    np.testing.assert_array_equal(l2, lse[rows])


# ---------------------------------------------------------------- backward

def test_backward_matches_sdpa_autograd():
    """Causal, no score_mod: gradients of torch SDPA (fp64 autograd)."""
    S, D = 200, 64
    q, k, v, do = _qkv(S, D, 15)
    dq, dk, dv, _, _ = oracle.backward_head(q, k, v, do, oracle.Program(CAUSAL), ("none",), 0, 1 / np.sqrt(D))
    tq, tk, tv = (torch.from_numpy(a)[None, None].requires_grad_() for a in (q, k, v))
    o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=True)
    o.backward(torch.from_numpy(do)[None, None])
    np.testing.assert_allclose(dq, tq.grad[0, 0].numpy(), atol=1e-11)
    np.testing.assert_allclose(dk, tk.grad[0, 0].numpy(), atol=1e-11)
    np.testing.assert_allclose(dv, tv.grad[0, 0].numpy(), atol=1e-11)


@pytest.mark.parametrize("score", ["none", "softcap", "alibi"])
def test_backward_finite_differences(score):
    """Central differences of L = sum(out * dO) through the oracle forward."""
    S, D = 40, 16
    q, k, v, do = _qkv(S, D, 16)
    docs = make_doc_ids(("geometric", 12.0), S, 17)[0]
    mask = P(("causal",), ("same_doc",), ("and",), ("sink", 2), ("or",))
    prog = oracle.Program(mask, doc_row=docs)
    sc = {"none": ("none",), "softcap": ("softcap", 1.5), "alibi": ("alibi", [0.3])}[score]
    scale = 0.7
    dq, dk, dv, _, _ = oracle.backward_head(q, k, v, do, prog, sc, 0, scale)

    def loss(qq, kk, vv):
        o, _ = oracle.forward_head(qq, kk, vv, prog, sc, 0, scale)
        return float((o * do).sum())

    eps = 1e-6
    rng = np.random.default_rng(0)
    for name, g, arr in (("q", dq, q), ("k", dk, k), ("v", dv, v)):
        for _ in range(12):
            r, c = int(rng.integers(S)), int(rng.integers(D))
            args = {"q": q, "k": k, "v": v}
            plus = {n: a.copy() for n, a in args.items()}
            minus = {n: a.copy() for n, a in args.items()}
            plus[name][r, c] += eps
            minus[name][r, c] -= eps
            num = (loss(plus["q"], plus["k"], plus["v"]) - loss(minus["q"], minus["k"], minus["v"])) / (2 * eps)
            assert abs(num - g[r, c]) < 1e-7 * max(1.0, abs(num)), (name, r, c, num, g[r, c])


@pytest.mark.parametrize("score", ["none", "softcap", "alibi"])
def test_backward_matches_numpy_twin(score):
    S, D = 150, 32
    q, k, v, do = _qkv(S, D, 18, kv_len=170)
    docs = make_doc_ids(("geometric", 30.0), 170, 19)[0]
    mask = P(("causal",), ("same_doc",), ("and",), ("window", 50), ("and",))
    sc = {"none": ("none",), "softcap": ("softcap", 4.0), "alibi": ("alibi", [0.0625])}[score]
    prog = oracle.Program(mask, doc_row=docs)
    dq, dk, dv, _, _ = oracle.backward_head(q, k, v, do, prog, sc, 0, 0.3)
    M = oracle.np_mask(mask, S, 170, doc_row=docs)
    ref = oracle.np_backward(q, k, v, do, M, sc if score != "alibi" else ("alibi",), 0.0625, 0.3)
    for a, b in zip((dq, dk, dv), ref):
        np.testing.assert_allclose(a, b, atol=1e-11)


def test_backward_diagonal_only():
    """Only the diagonal visible: P = 1, so dv = dO and dq = dk = 0."""
    S, D = 100, 64
    q, k, v, do = _qkv(S, D, 20)
    prog = oracle.Program(P(("causal",), ("window", 1), ("and",)))
    dq, dk, dv, _, _ = oracle.backward_head(q, k, v, do, prog, ("none",), 0, 0.125)
    np.testing.assert_allclose(dv, do, atol=1e-14)
    assert np.abs(dq).max() < 1e-14 and np.abs(dk).max() < 1e-14


def test_backward_subsets_match_full():
    S, D = 180, 64
    q, k, v, do = _qkv(S, D, 21)
    prog = oracle.Program(CAUSAL)
    dq, dk, dv, _, _ = oracle.backward_head(q, k, v, do, prog, ("softcap", 3.0), 0, 0.2)
    rows, cols = [3, 179, 64], [0, 100, 177]
    dq2, dk2, dv2, _, _ = oracle.backward_head(q, k, v, do, prog, ("softcap", 3.0), 0, 0.2, rows=rows, cols=cols)
    np.testing.assert_array_equal(dq2, dq[rows])
    np.testing.assert_array_equal(dk2, dk[cols])
    np.testing.assert_array_equal(dv2, dv[cols])


# ------------------------------------------------- caller-chosen tiles (from_kv_blocks)

def _random_selection(rng, nq, nkv, p_partial=0.3, p_full=0.3):
    u = rng.random((nq, nkv))
    return np.where(u < p_partial, 1, np.where(u < p_partial + p_full, 2, 0)).astype(np.int8)


@pytest.mark.parametrize("seed", range(6))
def test_selection_of_own_classes_leaves_mask_unchanged(seed):
    """Selecting exactly a program's own PARTIAL and FULL tiles changes nothing:
    FULL tiles are all visible anyway and EMPTY ones hold no visible pair.  A
    swapped class code or a transposed tile index breaks this for the random,
    asymmetric programs here (ragged lengths, several block sizes)."""
    rng = np.random.default_rng(100 + seed)
    nodes = _random_program(rng)
    if len(nodes) > 16:
        nodes = nodes[:1]
    q_len, kv_len = int(rng.integers(40, 260)), int(rng.integers(40, 260))
    docs = make_doc_ids(("geometric", 30.0), max(q_len, kv_len), seed)[0]
    prefix = int(rng.integers(0, 120))
    plain = oracle.Program(P(*nodes), doc_row=docs, prefix_len=prefix)
    M = oracle.mask_dense(plain, q_len, kv_len)
    for block in (16, 32, 64):
        cls = oracle.classify_tiles(plain, q_len, kv_len, block)
        sel = oracle.Program(P(*nodes), doc_row=docs, prefix_len=prefix, selection=cls, block=block)
        np.testing.assert_array_equal(oracle.mask_dense(sel, q_len, kv_len), M)


def test_selection_lists_round_trip_in_any_order():
    """Lists in any order give the grid they were made from; the class grid's
    own ascending lists give it back too."""
    rng = np.random.default_rng(7)
    nq, nkv = 9, 13
    sel = _random_selection(rng, nq, nkv)
    kv_num = np.zeros(nq, np.int32)
    full_num = np.zeros(nq, np.int32)
    kv_idx = np.full((nq, 5 + nkv), -7, np.int32)      # wider rows, junk past the counts
    full_idx = np.full((nq, nkv), 99, np.int32)
    for I in range(nq):
        p = rng.permutation(np.nonzero(sel[I] == 1)[0])
        f = rng.permutation(np.nonzero(sel[I] == 2)[0])
        kv_num[I], full_num[I] = len(p), len(f)
        kv_idx[I, :len(p)] = p
        full_idx[I, :len(f)] = f
    np.testing.assert_array_equal(oracle.selection_from_lists(kv_num, kv_idx, full_num, full_idx, nkv), sel)
    L = oracle.tile_lists(sel)
    np.testing.assert_array_equal(
        oracle.selection_from_lists(L["kv_num_blocks"], L["kv_indices"], L["full_kv_num_blocks"],
                                    L["full_kv_indices"], nkv), sel)
    # partial lists alone
    np.testing.assert_array_equal(oracle.selection_from_lists(kv_num, kv_idx, nkv=nkv), np.where(sel == 1, 1, 0))


def test_selection_from_lists_rejects_invalid_entries():
    nkv = 4
    ok_num, ok_idx = np.array([1]), np.array([[2, 0, 0, 0]])
    for num, idx, fnum, fidx in [
        (np.array([1]), np.array([[4, 0, 0, 0]]), None, None),       # index past the last tile
        (np.array([1]), np.array([[-1, 0, 0, 0]]), None, None),      # negative index
        (np.array([2]), np.array([[1, 1, 0, 0]]), None, None),       # listed twice
        (np.array([5]), np.array([[0, 1, 2, 3, 0]]), None, None),    # count above nkv
        (np.array([-1]), np.array([[0, 0, 0, 0]]), None, None),      # negative count
        (ok_num, ok_idx, np.array([1]), np.array([[2, 0, 0, 0]])),   # partial and full
    ]:
        with pytest.raises(ValueError):
            oracle.selection_from_lists(num, idx, fnum, fidx, nkv)
    sel, bad = oracle.selection_from_lists(ok_num, ok_idx, np.array([2]), np.array([[2, 5, 0, 0]]), nkv,
                                           drop_invalid=True)
    assert bad == 2 and sel.tolist() == [[0, 0, 2, 0]]   # both-listed tile stays full; index 5 dropped


def test_selection_true_program_is_tile_expansion():
    """With an everywhere-true program the mask is the selected tiles, whole
    (built here tile by tile), cut at ragged lengths."""
    rng = np.random.default_rng(3)
    q_len, kv_len, b = 150, 201, 32
    nq, nkv = -(-q_len // b), -(-kv_len // b)
    sel = _random_selection(rng, nq, nkv)
    M = oracle.mask_dense(oracle.Program(P(("true",)), selection=sel, block=b), q_len, kv_len)
    ref = np.zeros((q_len, kv_len), bool)
    for I in range(nq):
        for J in range(nkv):
            if sel[I, J]:
                ref[I * b:(I + 1) * b, J * b:(J + 1) * b] = True
    np.testing.assert_array_equal(M, ref)


def test_selection_partial_tiles_take_the_program_full_tiles_do_not():
    S, b = 96, 32
    n = S // b
    i, j = np.arange(S)[:, None], np.arange(S)[None, :]
    every = lambda c: np.full((n, n), c, np.int8)
    M = lambda c: oracle.mask_dense(oracle.Program(CAUSAL, selection=every(c), block=b), S, S)
    np.testing.assert_array_equal(M(1), i >= j)                 # partial everywhere: causal
    np.testing.assert_array_equal(M(2), np.ones((S, S), bool))  # full everywhere: dense
    np.testing.assert_array_equal(M(0), np.zeros((S, S), bool))  # nothing listed
    q, k, v, _ = _qkv(S, 64, 30)
    out, lse = oracle.forward_head(q, k, v, oracle.Program(CAUSAL, selection=every(0), block=b), ("none",), 0, 0.125)
    assert np.all(out == 0) and np.all(np.isneginf(lse))


def test_selection_block_diagonal_is_independent_blocks():
    """Each query tile sees only its own key tile (full): per-block textbook
    attention (torch SDPA on each block, fp64)."""
    S, D, b = 200, 64, 64
    q, k, v, _ = _qkv(S, D, 31)
    n = -(-S // b)
    sel = np.eye(n, dtype=np.int8) * 2
    out, lse = oracle.forward_head(q, k, v, oracle.Program(P(("true",)), selection=sel, block=b), ("none",), 0,
                                   1 / np.sqrt(D))
    for I in range(n):
        r = slice(I * b, min(S, (I + 1) * b))
        tq, tk, tv = (torch.from_numpy(a[r])[None, None] for a in (q, k, v))
        ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv)[0, 0].numpy()
        np.testing.assert_allclose(out[r], ref, atol=1e-12, rtol=0)
        ref_lse = torch.logsumexp(torch.from_numpy(q[r] @ k[r].T / np.sqrt(D)), 1).numpy()
        np.testing.assert_allclose(lse[r], ref_lse, atol=1e-12, rtol=0)


def test_selection_q_zero_closed_form():
    """q = 0: out_i is the mean of the v_j it sees and LSE_i = ln |V_i|, where
    V_i holds the keys of its full tiles and the causal keys of its partial ones."""
    S, D, b = 160, 32, 32
    _, k, v, _ = _qkv(S, D, 32)
    q = np.zeros((S, D))
    sel = _random_selection(np.random.default_rng(33), S // b, S // b, 0.4, 0.4)
    sel[:, 0] = 1                                   # every row sees key 0 through a partial tile
    out, lse = oracle.forward_head(q, k, v, oracle.Program(CAUSAL, selection=sel, block=b), ("none",), 0, 0.3)
    for i in range(S):
        js = [j for j in range(S) if sel[i // b, j // b] == 2 or (sel[i // b, j // b] == 1 and j <= i)]
        np.testing.assert_allclose(out[i], v[js].mean(axis=0), atol=1e-12)
        assert abs(lse[i] - np.log(len(js))) < 1e-12


@pytest.mark.parametrize("score", ["none", "softcap", "alibi"])
def test_selection_forward_backward_match_numpy_twin(score):
    """C loops over a selection vs the numpy twin's expanded dense mask."""
    S, kv_len, D, b = 130, 170, 32, 32
    q, k, v, do = _qkv(S, D, 34, kv_len=kv_len)
    docs = make_doc_ids(("geometric", 30.0), kv_len, 35)[0]
    mask = P(("causal",), ("same_doc",), ("and",))
    sel = _random_selection(np.random.default_rng(36), -(-S // b), -(-kv_len // b))
    sc = {"none": ("none",), "softcap": ("softcap", 4.0), "alibi": ("alibi", [0.0625])}[score]
    prog = oracle.Program(mask, doc_row=docs, selection=sel, block=b)
    out, lse = oracle.forward_head(q, k, v, prog, sc, 0, 0.3)
    M = oracle.np_select(oracle.np_mask(mask, S, kv_len, doc_row=docs), sel, b)
    tw = sc if score != "alibi" else ("alibi",)
    ref_out, ref_lse, _ = oracle.np_forward(q, k, v, M, tw, 0.0625, 0.3)
    np.testing.assert_allclose(out, ref_out, atol=1e-12)
    np.testing.assert_array_equal(np.isneginf(lse), np.isneginf(ref_lse))
    fin = np.isfinite(ref_lse)
    np.testing.assert_allclose(lse[fin], ref_lse[fin], atol=1e-12)
    dq, dk, dv, _, _ = oracle.backward_head(q, k, v, do, prog, sc, 0, 0.3)
    for a, r in zip((dq, dk, dv), oracle.np_backward(q, k, v, do, M, tw, 0.0625, 0.3)):
        np.testing.assert_allclose(a, r, atol=1e-11)


# ------------------------------------------------- gradient of the score mod's parameter

@pytest.mark.parametrize("score", ["softcap", "alibi"])
def test_score_param_grad_finite_differences(score):
    """dL/dparam (soft-cap c, ALiBi slope) against central differences of
    L = sum(out * dO) through the oracle forward, on a document program."""
    S, D = 60, 16
    q, k, v, do = _qkv(S, D, 40)
    docs = make_doc_ids(("geometric", 15.0), S, 41)[0]
    prog = oracle.Program(P(("causal",), ("same_doc",), ("and",), ("sink", 3), ("or",)), doc_row=docs)
    base = 1.5 if score == "softcap" else 0.3125   # ALiBi slopes are stored fp32: base +- eps exact there
    scale = 0.7

    def sc(val):
        return ("softcap", val) if score == "softcap" else ("alibi", [val])

    def loss(val):
        o, _ = oracle.forward_head(q, k, v, prog, sc(val), 0, scale)
        return float((o * do).sum())

    g = oracle.score_param_grad_head(q, k, v, do, prog, sc(base), 0, scale)
    eps = 2.0 ** -20
    num = (loss(base + eps) - loss(base - eps)) / (2 * eps)
    assert abs(g) > 1e-3                                   # a non-trivial case
    assert abs(num - g) < 1e-7 * max(1.0, abs(num)), (num, g)


@pytest.mark.parametrize("score", ["none", "softcap", "alibi"])
def test_score_param_grad_matches_numpy_twin(score):
    S, kv_len, D = 120, 150, 32
    q, k, v, do = _qkv(S, D, 42, kv_len=kv_len)
    docs = make_doc_ids(("geometric", 30.0), kv_len, 43)[0]
    mask = P(("causal",), ("same_doc",), ("and",), ("window", 60), ("and",))
    sc = {"none": ("none",), "softcap": ("softcap", 4.0), "alibi": ("alibi", [0.0625])}[score]
    g = oracle.score_param_grad_head(q, k, v, do, oracle.Program(mask, doc_row=docs), sc, 0, 0.3)
    M = oracle.np_mask(mask, S, kv_len, doc_row=docs)
    ref = oracle.np_score_param_grad(q, k, v, do, M, sc if score != "alibi" else ("alibi",), 0.0625, 0.3)
    assert abs(g - ref) < 1e-10 * max(1.0, abs(ref))
    if score == "none":
        assert g == 0.0


def test_score_param_grad_vanishes_where_out_cannot_move():
    """V = 1 makes out = 1 whatever the weights, and a diagonal-only mask gives
    P = 1 on one key: in both dL/dslope is exactly zero (dP - Delta = 0 per row)."""
    S, D = 90, 32
    q, k, v, do = _qkv(S, D, 44)
    g = oracle.score_param_grad_head(q, k, np.ones_like(v), do, oracle.Program(CAUSAL), ("alibi", [0.2]), 0, 0.2)
    assert abs(g) < 1e-12
    diag = oracle.Program(P(("causal",), ("window", 1), ("and",)))
    assert oracle.score_param_grad_head(q, k, v, do, diag, ("alibi", [0.2]), 0, 0.2) == 0.0


# ------------------------------------------------- learned relative-position bias

def _alibi_table(slope, d0, L):
    """The bias table that reproduces ALiBi: entry t (distance d0 + t) = -slope (d0 + t)."""
    return np.array([[-slope * (d0 + t) for t in range(L)]], dtype=np.float32)


@pytest.mark.parametrize("d0,L,off", [(0, 64, 0), (-5, 80, 0), (-2, 70, 37)])
def test_relbias_with_alibi_distances_is_alibi(d0, L, off):
    """A table holding -slope * distance over every visible distance is ALiBi
    (tutorial Pattern 3): forward and backward of the two score mods agree, with
    query rows at an offset too.  A sign slip (j - i), a shifted first distance or
    a missing q_offset in the bias fails this."""
    S, kv_len, D = 50, 90, 16
    q, k, v, do = _qkv(S, D, 60, kv_len=kv_len)
    prog = oracle.Program(P(("causal",), ("window", 60), ("and",)), q_offset=off)
    slope, scale = 0.3125, 0.4
    rb, al = ("relbias", _alibi_table(slope, d0, L), d0), ("alibi", [slope])
    o1, l1 = oracle.forward_head(q, k, v, prog, rb, 0, scale)
    o2, l2 = oracle.forward_head(q, k, v, prog, al, 0, scale)
    np.testing.assert_allclose(o1, o2, atol=1e-12)
    np.testing.assert_allclose(l1, l2, atol=1e-12)
    for a, b in zip(oracle.backward_head(q, k, v, do, prog, rb, 0, scale)[:3],
                    oracle.backward_head(q, k, v, do, prog, al, 0, scale)[:3]):
        np.testing.assert_allclose(a, b, atol=1e-12)


def test_relbias_gradient_contracts_to_the_alibi_slope_gradient():
    """With table[t] = -slope (d0 + t), dL/dslope = sum_t dL/dtable[t] * (-(d0 + t)):
    the table gradient and the independently written slope gradient agree."""
    S, D, d0, L = 70, 16, -3, 90
    q, k, v, do = _qkv(S, D, 61)
    docs = make_doc_ids(("geometric", 20.0), S, 62)[0]
    prog = oracle.Program(P(("causal",), ("same_doc",), ("and",), ("sink", 4), ("or",)), doc_row=docs)
    slope, scale = 0.25, 0.5
    g = oracle.bias_grad_head(q, k, v, do, prog, ("relbias", _alibi_table(slope, d0, L), d0), 0, scale)
    gs = oracle.score_param_grad_head(q, k, v, do, prog, ("alibi", [slope]), 0, scale)
    contracted = float((g * -(d0 + np.arange(L))).sum())
    assert abs(gs) > 1e-3
    assert abs(contracted - gs) < 1e-10 * max(1.0, abs(gs)), (contracted, gs)


def test_relbias_constant_table_shifts_lse_only():
    """A constant bias c leaves the softmax (out) unchanged and adds c to LSE; the
    table gradient of any table sums to zero (softmax is shift invariant: the
    row sums of P (dP - Delta) vanish)."""
    S, D, c = 80, 16, 1.75
    q, k, v, do = _qkv(S, D, 63)
    prog = oracle.Program(P(("causal",), ("window", 30), ("and",)))
    o0, l0 = oracle.forward_head(q, k, v, prog, ("none",), 0, 0.3)
    o1, l1 = oracle.forward_head(q, k, v, prog, ("relbias", np.full((1, 12), c, np.float32), 4), 0, 0.3)
    np.testing.assert_allclose(o1, o0, atol=1e-12)
    np.testing.assert_allclose(l1, l0 + c, atol=1e-12)
    table = np.random.default_rng(64).normal(size=(1, 25)).astype(np.float32)
    g = oracle.bias_grad_head(q, k, v, do, prog, ("relbias", table, 2), 0, 0.3)
    assert np.abs(g).max() > 1e-3
    assert abs(g.sum()) < 1e-10


def test_relbias_gradient_finite_differences():
    """dL/dtable against central differences of L = sum(out * dO) through the
    oracle forward, at an interior entry and at both end entries (which collect
    every distance outside the table)."""
    S, D, d0, L = 60, 16, 3, 20
    q, k, v, do = _qkv(S, D, 65)
    prog = oracle.Program(P(("window", 40), ("sink", 5), ("or",)))  # distances below d0 and past the end
    table = np.random.default_rng(66).normal(scale=0.5, size=(1, L)).astype(np.float32)
    scale = 0.45
    g = oracle.bias_grad_head(q, k, v, do, prog, ("relbias", table, d0), 0, scale)
    eps = 2.0 ** -12  # table entries are fp32: +- eps stays exact for these magnitudes
    for t in (0, 7, L - 1):
        def loss(delta):
            tb = table.copy()
            tb[0, t] += delta
            o, _ = oracle.forward_head(q, k, v, prog, ("relbias", tb, d0), 0, scale)
            return float((o * do).sum())
        num = (loss(eps) - loss(-eps)) / (2 * eps)
        assert abs(g[t]) > 1e-4
        assert abs(num - g[t]) < 1e-6 * max(1.0, abs(num)), (t, num, g[t])


@pytest.mark.parametrize("off", [0, 25])
def test_relbias_matches_numpy_twin(off):
    """The C loops against the numpy twin (explicit mask, dense matrices, the
    table gathered with np.clip): out, LSE, dq, dk, dv and the table gradient,
    on a mask with distances on both sides of a short table."""
    S, kv_len, D, d0, L = 40, 90, 16, -4, 30
    q, k, v, do = _qkv(S, D, 67, kv_len=kv_len)
    docs = make_doc_ids(("geometric", 25.0), kv_len, 68)[0]
    mask = P(("same_doc",), ("window", 45), ("and",))  # no causal: negative distances too
    prog = oracle.Program(mask, doc_row=docs, q_offset=off)
    table = np.random.default_rng(69).normal(scale=0.7, size=(1, L)).astype(np.float32)
    sc = ("relbias", table, d0)
    th = table[0].astype(np.float64)
    M = oracle.np_mask(mask, S, kv_len, doc_row=docs, q_offset=off)
    out, lse = oracle.forward_head(q, k, v, prog, sc, 0, 0.35)
    ro, rl, _ = oracle.np_forward(q, k, v, M, ("relbias", th, d0), 0.0, 0.35, q_offset=off)
    np.testing.assert_allclose(out, ro, atol=1e-12)
    np.testing.assert_allclose(lse, rl, atol=1e-12)
    for a, b in zip(oracle.backward_head(q, k, v, do, prog, sc, 0, 0.35)[:3],
                    oracle.np_backward(q, k, v, do, M, ("relbias", th, d0), 0.0, 0.35, q_offset=off)):
        np.testing.assert_allclose(a, b, atol=1e-12)
    g = oracle.bias_grad_head(q, k, v, do, prog, sc, 0, 0.35)
    np.testing.assert_allclose(g, oracle.np_bias_grad(q, k, v, do, M, th, d0, 0.35, q_offset=off), atol=1e-12)
    assert (g != 0).sum() > L // 2


# ------------------------------------------------- paged key / value cache

def test_paged_gather_inverts_the_scatter_into_pages():
    """Write each logical tile of every batch row into the page its table names
    (pages shuffled across the pool and shared by nothing); the gather gives the
    logical tensor back, ragged last tile included."""
    rng = np.random.default_rng(50)
    B, H, kv_len, D, blk = 3, 2, 300, 8, 64
    nkv = -(-kv_len // blk)
    n_pages = B * nkv + 5
    logical = rng.standard_normal((B, H, kv_len, D))
    table = rng.permutation(n_pages)[:B * nkv].reshape(B, nkv).astype(np.int32)
    pool = np.full((H, n_pages * blk, D), 99.0)
    for b in range(B):
        for J in range(nkv):
            n = min(blk, kv_len - J * blk)
            pool[:, table[b, J] * blk:table[b, J] * blk + n] = logical[b, :, J * blk:J * blk + n]
    np.testing.assert_array_equal(oracle.paged_gather(pool, table, kv_len, blk), logical)


def test_paged_gather_identity_table_and_invalid_pages():
    pool = np.arange(2 * 6 * 4 * 3, dtype=np.float64).reshape(2, 24, 3)   # H=2, 6 pages of 4 rows
    ident = np.arange(6, dtype=np.int32)[None]
    np.testing.assert_array_equal(oracle.paged_gather(pool, ident, 22, 4)[0], pool[:, :22])
    for bad in (6, -1):
        t = ident.copy()
        t[0, 2] = bad
        with pytest.raises(ValueError):
            oracle.paged_gather(pool, t, 22, 4)
    with pytest.raises(ValueError):
        oracle.paged_gather(pool, ident[:, :5], 22, 4)                       # table too short


# ---------------------------------------------------------------- query offset

@pytest.mark.parametrize("seed", range(6))
def test_q_offset_mask_matches_numpy_twin(seed):
    """A query offset in the C element-wise evaluation and in the numpy twin's
    broadcasting, on random programs, ragged lengths and small blocks."""
    rng = np.random.default_rng(50 + seed)
    nodes = _random_program(rng)
    if len(nodes) > 16:
        nodes = nodes[:1]
    prog = MaskProgram(tuple(nodes))
    kv_len = int(rng.integers(60, 300))
    q_len = int(rng.integers(1, kv_len))
    off = int(rng.integers(0, kv_len - q_len + 1))
    docs = make_doc_ids(("geometric", 30.0), kv_len, seed)[0]
    prefix = int(rng.integers(0, 150))
    cp = oracle.Program(prog, doc_row=docs, prefix_len=prefix, q_offset=off)
    M = oracle.mask_dense(cp, q_len, kv_len)
    np.testing.assert_array_equal(M, oracle.np_mask(prog, q_len, kv_len, doc_row=docs, prefix_len=prefix,
                                                    q_offset=off))
    for block in (16, 64):
        np.testing.assert_array_equal(oracle.classify_tiles(cp, q_len, kv_len, block), oracle.np_classify(M, block))


@pytest.mark.parametrize("score", ["none", "alibi", "softcap"])
def test_q_offset_rows_are_rows_of_the_whole_sequence(score):
    """Query rows at an offset (decoding new tokens at the end of a cache) give
    exactly the corresponding rows of the same sequence computed whole; their
    gradients are the whole sequence's with dO zero on every other row."""
    kv_len, q_len, off, D = 300, 7, 290, 16
    docs = make_doc_ids(("geometric", 60.0), kv_len, 3)[0]
    mask = P(("causal",), ("same_doc",), ("window", 100), ("sink", 8), ("or",), ("and",), ("and",))
    sc = {"none": ("none",), "alibi": ("alibi", np.array([0.3], np.float32)), "softcap": ("softcap", 5.0)}[score]
    g = torch.Generator().manual_seed(11)
    qf, k, v, dof = (torch.randn(n, D, generator=g, dtype=torch.float64).numpy() for n in (kv_len, kv_len, kv_len, kv_len))
    dof[:off] = 0.0
    dof[off + q_len:] = 0.0
    q, do = qf[off:off + q_len], dof[off:off + q_len]
    whole = oracle.Program(mask, doc_row=docs)
    part = oracle.Program(mask, doc_row=docs, q_offset=off)
    scale = 1.0 / np.sqrt(D)
    out_w, lse_w = oracle.forward_head(qf, k, v, whole, sc, 0, scale)
    out_p, lse_p = oracle.forward_head(q, k, v, part, sc, 0, scale)
    np.testing.assert_allclose(out_p, out_w[off:off + q_len], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse_p, lse_w[off:off + q_len], rtol=1e-12, atol=1e-12)
    dq_w, dk_w, dv_w, _, _ = oracle.backward_head(qf, k, v, dof, whole, sc, 0, scale)
    dq_p, dk_p, dv_p, _, _ = oracle.backward_head(q, k, v, do, part, sc, 0, scale)
    np.testing.assert_allclose(dq_p, dq_w[off:off + q_len], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dk_p, dk_w, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dv_p, dv_w, rtol=1e-10, atol=1e-12)
    # and the numpy twin, in matrix form, agrees
    M = oracle.np_mask(mask, q_len, kv_len, doc_row=docs, q_offset=off)
    slope = float(np.float32(0.3)) if score == "alibi" else 0.0  # the oracle takes slopes as fp32 values
    o2, l2, _ = oracle.np_forward(q, k, v, M, sc if score != "alibi" else ("alibi",), slope, scale, q_offset=off)
    np.testing.assert_allclose(o2, out_p, rtol=1e-10, atol=1e-12)
