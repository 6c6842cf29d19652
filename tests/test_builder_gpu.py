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
    order = bm.row_order().cpu().numpy()
    assert sorted(order.tolist()) == list(range(order.size))
    work = (got["kv_num_blocks"] + got["full_kv_num_blocks"]).reshape(-1)[order]
    assert np.all(np.diff(work) <= 0)                     # longest rows first
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
