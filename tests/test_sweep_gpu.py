"""The window-growth sweep at full size: B=1, H=16, S=65536, D=128, causal &
same document & window W, ALiBi (speedrun notes, Record #13: the window grows
from 64 to 1792 in steps of 64 with no recompilation).

One device int32 holds W and is rewritten between block-mask builds, as the
bench's sweep does; nothing else is rebuilt.  At the two ends of the sweep the
forward (out, LSE on sampled rows) and the backward (dq on sampled rows, dk / dv
on sampled columns) of heads 0 and 15 are compared with the fp64 oracle, at the
tolerances of fa_testutil.
"""
import numpy as np
import pytest
import torch

import oracle
from fa_testutil import check_forward, check_grad, device_nodes, head64, oracle_score
from synth import WORKLOADS, make_workload_inputs

pytestmark = pytest.mark.gpu

fa = pytest.importorskip("block_sparse_masked_fa_gb300")

W5 = WORKLOADS[5]


@pytest.fixture(scope="module")
def sweep():
    inp = make_workload_inputs(W5)
    dev = {n: inp[n].cuda() for n in ("q", "k", "v", "do")}
    W = torch.tensor([W5.windows[len(W5.windows) // 2]], dtype=torch.int32, device="cuda")
    nodes = device_nodes(W5.mask, inp["docs"], window_tensor=W)
    spec = fa.make_mask_spec(nodes)
    buf = torch.empty(fa.fa_block_mask_bytes(1, 1, W5.S, W5.S, 128), dtype=torch.uint8, device="cuda")
    score = fa.make_score_spec("alibi", torch.as_tensor(inp["slopes"]))
    # a build at another window first, so each case rewrites W and the buffer
    fa.fa_create_block_mask(spec, 1, 1, W5.S, W5.S, 128, buffer=buf)
    torch.cuda.synchronize()
    return {"inp": inp, "dev": dev, "W": W, "spec": spec, "buf": buf, "score": score}


def _sample(S, rng, n=40):
    idx = set(rng.integers(0, S, size=n).tolist())
    for I in rng.integers(0, S // 128, size=4):
        idx.update([int(I) * 128, int(I) * 128 + 127])
    idx.update([0, S - 1])
    return np.array(sorted(idx), dtype=np.int64)


@pytest.mark.parametrize("Wv", [64, 1792])
def test_sweep_end_full_size(sweep, Wv):
    inp, d = sweep["inp"], sweep["dev"]
    sweep["W"].fill_(Wv)
    bm = fa.fa_create_block_mask(sweep["spec"], 1, 1, W5.S, W5.S, 128, buffer=sweep["buf"])
    out, lse = fa.fa_forward(d["q"], d["k"], d["v"], bm, score=sweep["score"])
    dq, dk, dv = fa.fa_backward(d["q"], d["k"], d["v"], out, lse, d["do"], bm, score=sweep["score"])
    torch.cuda.synchronize()
    assert fa.fa_get_status(bm) == 0
    # the block mask was built for this W: its visible-tile count is the oracle's
    mask = W5.mask.with_window(Wv)
    prog = oracle.Program(mask, doc_row=inp["docs"][0])
    cls = oracle.classify_tiles(prog, W5.S, W5.S)
    L = bm.lists()
    assert int((L["kv_num_blocks"] + L["full_kv_num_blocks"]).sum()) == int((cls > 0).sum())
    score = oracle_score(W5.score, inp["slopes"])
    scale = 1.0 / np.sqrt(W5.D)
    rng = np.random.default_rng(500 + Wv)
    out_c, lse_c = out.float().cpu().numpy(), lse.cpu().numpy()
    grads = [g.float().cpu().numpy() for g in (dq, dk, dv)]
    for h in (0, W5.H - 1):
        rows, cols = _sample(W5.S, rng), _sample(W5.S, rng)
        q, k, v, do = (head64(inp[n], 0, h) for n in ("q", "k", "v", "do"))
        ref_out, ref_lse = oracle.forward_head(q, k, v, prog, score, h, scale, rows=rows)
        check_forward(out_c[0, h][rows], lse_c[0, h][rows], ref_out, ref_lse, f"W{Wv} h{h}")
        rdq, rdk, rdv, _, _ = oracle.backward_head(q, k, v, do, prog, score, h, scale, rows=rows, cols=cols)
        for name, g, r in zip(("dq", "dk", "dv"), (grads[0][0, h][rows], grads[1][0, h][cols],
                                                   grads[2][0, h][cols]), (rdq, rdk, rdv)):
            check_grad(g, r, f"W{Wv} h{h} {name}")
