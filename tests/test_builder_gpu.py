"""Block-mask builder parity: every list bit-exact against the oracle's
brute-force tile classifier (CUDA path called through the C ABI)."""
import numpy as np
import pytest
import torch

import oracle
from fa_testutil import device_nodes
from synth import WORKLOADS, MaskProgram, make_doc_ids

pytestmark = pytest.mark.gpu

fa = pytest.importorskip("block_sparse_masked_fa_gb300")

LIST_NAMES = ("kv_num_blocks", "kv_indices", "full_kv_num_blocks", "full_kv_indices",
              "q_num_blocks", "q_indices", "full_q_num_blocks", "full_q_indices")


def expected(mask, docs, prefix, Bm, Hm, q_len, kv_len, block):
    per_b = []
    for bm in range(Bm):
        prog = oracle.Program(mask, doc_row=None if docs is None else docs[bm],
                              prefix_len=None if prefix is None else int(prefix[bm]))
        cls = oracle.classify_tiles(prog, q_len, kv_len, block)
        per_b.append((cls, oracle.tile_lists(cls)))
    cls = np.stack([np.stack([c for _ in range(Hm)]) for c, _ in per_b])
    lists = {n: np.stack([np.stack([L[n] for _ in range(Hm)]) for _, L in per_b]) for n in LIST_NAMES}
    return cls, lists


def compare(bm, cls, lists):
    got = {k: v.cpu().numpy() for k, v in bm.lists().items()}
    np.testing.assert_array_equal(bm.tile_class().cpu().numpy(), cls.astype(np.uint8))
    for n in LIST_NAMES:
        np.testing.assert_array_equal(got[n], lists[n], err_msg=n)
    # work orders in chunks of 32 neighbours: chunks by their longest count (longest
    # bucket first, index order inside a bucket), entries inside a chunk longest first
    # (index order among equals); counts exact for rows, quantized to ceil(cmax / 16)
    # for columns (one bucket when cmax <= 16)
    for field, n_key, f_key, quantized in (("row_order", "kv_num_blocks", "full_kv_num_blocks", False),
                                           ("col_order", "q_num_blocks", "full_q_num_blocks", True)):
        work = (got[n_key] + got[f_key]).reshape(-1)
        off = getattr(bm.struct, field) - bm.buffer.data_ptr()
        order = bm.buffer[off:off + 4 * work.size].view(torch.int32).cpu().numpy()
        cmax = int(work.max())
        qz = (cmax + 1 if cmax <= 16 else -(-cmax // 16)) if quantized else 1
        chunk = np.array([work[(r // 32) * 32:(r // 32) * 32 + 32].max() for r in range(work.size)])
        expect = sorted(range(work.size), key=lambda r: (-(chunk[r] // qz), r // 32, -(work[r] // qz), r))
        np.testing.assert_array_equal(order, np.array(expect), err_msg=field)
    assert fa.fa_get_status(bm) == 0


@pytest.mark.parametrize("wnum", [1, 2, 3, 4, 5])
def test_workload_masks_bit_exact(wnum):
    w = WORKLOADS[wnum]
    docs = None
    if w.docs is not None:
        docs = make_doc_ids(w.docs, w.S, w.doc_seed or w.seed)
    mask = w.mask if not w.windows else w.mask.with_window(1024)
    bm = fa.fa_create_block_mask(device_nodes(mask, docs), 1, 1, w.S, w.S, 128)
    cls, lists = expected(mask, docs, None, 1, 1, w.S, w.S, 128)
    compare(bm, cls, lists)
    counts = fa.fa_block_mask_summary(bm)
    assert counts == (int((cls == 0).sum()), int((cls == 1).sum()), int((cls == 2).sum()))


def test_page_counts_64k():
    """The speedrun notes' 64K-token counts, from the CUDA builder."""
    S = 65536
    for nodes, tiles in (([("causal",)], 131328),
                         ([("causal",), ("window", 1024), ("and",)], 4572),
                         ([("causal",), ("same_doc", torch.arange(S, dtype=torch.int32, device="cuda")[None] // 1024),
                           ("and",)], 2304)):
        bm = fa.fa_create_block_mask(nodes, 1, 1, S, S, 128)
        e, p, f = fa.fa_block_mask_summary(bm)
        assert p + f == tiles


def test_window_sweep_from_device_tensor():
    """Workload 5's sweep: W lives in a device int32 that is overwritten between
    builds; the same kernels rebuild the lists for every W."""
    w = WORKLOADS[5]
    docs = make_doc_ids(w.docs, w.S, w.doc_seed)
    W = torch.zeros(1, dtype=torch.int32, device="cuda")
    nodes = device_nodes(w.mask, docs, window_tensor=W)
    for Wv in w.windows:
        W.fill_(Wv)
        bm = fa.fa_create_block_mask(nodes, 1, 1, w.S, w.S, 128)
        cls, lists = expected(w.mask.with_window(Wv), docs, None, 1, 1, w.S, w.S, 128)
        compare(bm, cls, lists)


def _random_program(rng, depth=3):
    atoms = [("causal",), ("same_doc",), ("window", int(rng.integers(0, 700))),
             ("sink", int(rng.integers(0, 300))), ("prefix",), ("true",)]
    if depth == 0 or rng.random() < 0.3:
        return [atoms[int(rng.integers(len(atoms)))]]
    return _random_program(rng, depth - 1) + _random_program(rng, depth - 1) + \
        [("and",) if rng.random() < 0.6 else ("or",)]


@pytest.mark.parametrize("seed", range(16))
def test_random_programs_ragged_broadcast(seed):
    rng = np.random.default_rng(100 + seed)
    nodes = _random_program(rng)
    if len(nodes) > 16:
        nodes = nodes[:1]
    mask = MaskProgram(tuple(nodes))
    mask.validate()
    block = int(rng.choice([16, 32, 64, 128]))
    q_len, kv_len = int(rng.integers(1, 1500)), int(rng.integers(1, 1500))
    Bm, Hm = int(rng.integers(1, 3)), int(rng.integers(1, 3))
    docs = make_doc_ids(("geometric", float(rng.integers(20, 300))), max(q_len, kv_len), seed, batch=Bm)
    prefix = rng.integers(0, 800, size=Bm).astype(np.int32)
    bm = fa.fa_create_block_mask(device_nodes(mask, docs, prefix), Bm, Hm, q_len, kv_len, block)
    cls, lists = expected(mask, docs, prefix, Bm, Hm, q_len, kv_len, block)
    compare(bm, cls, lists)


def _runs_expected(doc, L):
    d = np.asarray(doc[:L], dtype=np.int64)
    change = np.ones(L, dtype=bool)
    change[1:] = d[1:] != d[:-1]
    starts = np.nonzero(change)[0]
    lo = starts[np.searchsorted(starts, np.arange(L), side="right") - 1]
    ends = np.append(starts[1:], L)
    hi = ends[np.searchsorted(starts, np.arange(L), side="right") - 1]
    return lo, hi, int(np.all(d[1:] >= d[:-1]))


@pytest.mark.parametrize("case", ["sorted_multi_chunk", "unsorted_repeats", "ragged_cross", "one_doc"])
def test_doc_runs_table(case):
    """The per-position run table the kernels use on PARTIAL tiles, bit-exact
    (the ranges for rows with sorted ids, the sorted flag for every row)."""
    rng = np.random.default_rng(7)
    if case == "sorted_multi_chunk":
        q_len = kv_len = 40000                       # several 16K-position chunks
        docs = make_doc_ids(("lognormal", 600.0, 1.0, 16, 16384), q_len, 3, batch=2)
    elif case == "unsorted_repeats":
        q_len = kv_len = 3000
        docs = np.stack([np.repeat(rng.integers(0, 5, size=30), 100).astype(np.int32) for _ in range(2)])
    elif case == "ragged_cross":
        q_len, kv_len = 777, 1300
        docs = make_doc_ids(("geometric", 90.0), 1300, 4, batch=2)
    else:
        q_len = kv_len = 5000
        docs = np.zeros((2, 5000), dtype=np.int32)
    L = max(q_len, kv_len)
    mask = MaskProgram((("causal",), ("same_doc",), ("and",)))
    bm = fa.fa_create_block_mask(device_nodes(mask, docs), 2, 1, q_len, kv_len, 128)
    torch.cuda.synchronize()
    off = bm.struct.doc_runs - bm.buffer.data_ptr()
    raw = bm.buffer[off:off + (2 * L * 2 + 2) * 4].view(torch.int32).cpu().numpy()
    runs = raw[:2 * L * 2].reshape(2, L, 2)
    flags = raw[2 * L * 2:]
    for b in range(2):
        lo, hi, srt = _runs_expected(docs[b], L)
        assert flags[b] == srt
        if srt:  # the kernels use the ranges only for rows whose ids never decrease
            np.testing.assert_array_equal(runs[b, :, 0], lo)
            np.testing.assert_array_equal(runs[b, :, 1], hi)


def _true_runs(v):
    """[lo, hi) runs of True in a boolean vector."""
    d = np.diff(np.concatenate([[0], v.astype(np.int8), [0]]))
    return list(zip(np.nonzero(d == 1)[0], np.nonzero(d == -1)[0]))


def _breaks(mask, transposed):
    """Interval ends the program's atoms contribute for one row (see the row_segs kernel)."""
    per = {"causal": 1, "window": 1, "same_doc": 2, "sink": 0 if transposed else 1, "prefix": 0 if transposed else 1}
    return sum(per.get(n[0], 0) for n in mask.nodes)


def check_row_segs(bm, mask, docs, prefix, Bm, q_len, kv_len):
    """Every summarised row equals the oracle's visible set exactly, and every
    row that two intervals describe is summarised (when the ids are sorted and
    the program has at most seven interval ends)."""
    segs = bm.row_segs().cpu().numpy()
    L = max(q_len, kv_len)
    has_doc = any(n[0] == "same_doc" for n in mask.nodes)
    for b in range(Bm):
        prog = oracle.Program(mask, doc_row=None if docs is None else docs[b],
                              prefix_len=None if prefix is None else int(prefix[b]))
        M = oracle.mask_dense(prog, q_len, kv_len)
        sorted_ids = not has_doc or bool(np.all(np.diff(np.asarray(docs[b][:L], dtype=np.int64)) >= 0))
        for which, R in ((0, M), (1, M.T)):
            must = sorted_ids and _breaks(mask, which == 1) <= 7
            for x in range(R.shape[0]):
                lo0, hi0, lo1, hi1 = (int(v) for v in segs[b, which, x])
                if must and len(_true_runs(R[x])) <= 2:
                    assert lo0 >= 0, (b, which, x)
                if lo0 >= 0:
                    got = np.zeros(R.shape[1], dtype=bool)
                    got[lo0:hi0] = True
                    got[lo1:hi1] = True
                    np.testing.assert_array_equal(got, R[x], err_msg=f"b{b} {'col' if which else 'row'} {x}")


@pytest.mark.parametrize("wnum", [1, 2, 3, 4, 5])
def test_row_segs_workload_programs(wnum):
    """The row interval summary of each workload's program, at reduced sizes
    with a ragged tail and q_len != kv_len."""
    w = WORKLOADS[wnum]
    q_len, kv_len = 1111, 1300
    docs = None if w.docs is None else make_doc_ids(w.docs, max(q_len, kv_len), 40 + wnum, batch=2)
    mask = w.mask.with_window(300) if w.windows else w.mask
    bm = fa.fa_create_block_mask(device_nodes(mask, docs), 2 if docs is not None else 1, 1, q_len, kv_len, 128)
    check_row_segs(bm, mask, docs, None, 2 if docs is not None else 1, q_len, kv_len)


@pytest.mark.parametrize("seed", range(8))
def test_row_segs_random_programs(seed):
    rng = np.random.default_rng(300 + seed)
    nodes = _random_program(rng)
    if len(nodes) > 16:
        nodes = nodes[:1]
    mask = MaskProgram(tuple(nodes))
    q_len, kv_len = int(rng.integers(1, 900)), int(rng.integers(1, 900))
    Bm = 2
    docs = make_doc_ids(("geometric", float(rng.integers(20, 300))), max(q_len, kv_len), seed, batch=Bm)
    prefix = rng.integers(0, 800, size=Bm).astype(np.int32)
    bm = fa.fa_create_block_mask(device_nodes(mask, docs, prefix), Bm, 1, q_len, kv_len, 64)
    check_row_segs(bm, mask, docs, prefix, Bm, q_len, kv_len)


def test_row_segs_unsorted_ids_not_summarised():
    """Ids that decrease somewhere: rows of a SAME_DOC program are left to the
    per-word evaluation (lo0 = -1); a program without SAME_DOC is unaffected."""
    rng = np.random.default_rng(9)
    docs = np.repeat(rng.integers(0, 4, size=9), 100).astype(np.int32)[None]
    for mask, summarised in ((MaskProgram((("same_doc",), ("causal",), ("and",))), False),
                             (MaskProgram((("causal",), ("window", 200), ("and",))), True)):
        bm = fa.fa_create_block_mask(device_nodes(mask, docs), 1, 1, 900, 900, 128)
        segs = bm.row_segs().cpu().numpy()
        assert bool(np.all(segs[0, :, :, 0] >= 0)) == summarised
        check_row_segs(bm, mask, docs, None, 1, 900, 900)
