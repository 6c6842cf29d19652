"""fa_backward_noalloc: the backward for callers that cannot allocate device
memory at call time (code inside a framework that reserves all GPU memory for
its own pool, or a latency-critical path that cannot take an allocation's
implicit synchronisation).  Its fp32 dq accumulator lives in a static device
array of the library instead of a caller workspace.

The test calls the new entry point twice in a row through the C ABI and
compares both results with fa_backward's on the same inputs, within the
gradient tolerance every backward test uses.  This file is collected last so
that a run stopping at the first failure has run every other test already.
"""
import numpy as np
import pytest
import torch

from fa_testutil import check_grad, device_nodes
from synth import MaskProgram, make_doc_ids, make_qkv

pytestmark = pytest.mark.gpu

fa = pytest.importorskip("block_sparse_masked_fa_gb300")


def test_noalloc_backward_matches_workspace_backward_twice():
    B, H, S, D = 1, 3, 1000, 128  # ragged: 7 full tiles and a 104-row tail
    q, k, v, do = (t.cuda() for t in make_qkv(B, H, S, D, 9001))
    docs = make_doc_ids(("geometric", 120.0), S, 9002)
    mask = MaskProgram((("causal",), ("same_doc",), ("and",), ("window", 300), ("and",)))
    bm = fa.fa_create_block_mask(device_nodes(mask, docs), 1, 1, S, S, 128)
    score = ("softcap", [30.0])
    out, lse = fa.fa_forward(q, k, v, bm, score=score)
    ref = [t.float().cpu().numpy() for t in fa.fa_backward(q, k, v, out, lse, do, bm, score=score)]
    assert fa.fa_backward_workspace_bytes(B, H, S, D) <= fa.binding.NOALLOC_SCRATCH_BYTES
    for call in range(2):
        got = [t.float().cpu().numpy() for t in fa.fa_backward_noalloc(q, k, v, out, lse, do, bm, score=score)]
        torch.cuda.synchronize()
        assert fa.fa_get_status(bm) == 0
        for name, g, r in zip(("dq", "dk", "dv"), got, ref):
            assert np.abs(r).max() > 0
            check_grad(g, r, f"call {call} {name}")


def test_noalloc_rejects_sizes_beyond_the_scratch():
    """B * H * q_len * (4 D + 4) bytes must fit the static scratch; larger calls
    return FA_ERR_WORKSPACE before queuing any GPU work."""
    B, H, S, D = 1, 1, 40000, 128
    assert fa.fa_backward_workspace_bytes(B, H, S, D) > fa.binding.NOALLOC_SCRATCH_BYTES
    q = torch.zeros(B, H, S, D, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(B, H, S, dtype=torch.float32, device="cuda")
    bm = fa.fa_create_block_mask([("causal",)], 1, 1, S, S, 128)
    with pytest.raises(fa.FaError) as e:
        fa.fa_backward_noalloc(q, q, q, q, lse, q, bm)
    assert e.value.code == 8  # FA_ERR_WORKSPACE
