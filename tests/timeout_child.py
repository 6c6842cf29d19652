"""Child process of test_timeout_gpu.py (run as a script, never collected).

Binds the Python binding to the test library (the same sources built with
FA_TEST_HOOKS: a 50 ms device wait limit and a hook that starves one wait), then
for the forward and the backward in turn: starves the first key-tile load of
the only CTA, checks that the call comes back with FA_ERR_TIMEOUT in the block
mask's status word within a few seconds, clears the hook, and checks that the
next call passes parity with the oracle.  Prints "timeout path ok" at the end.
Nothing here faults or traps: the starved wait gives up, the CTA drains its
copies and MMAs, frees its TMEM and exits.
"""
import ctypes
import os
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.join(ROOT, "tests"))

import block_sparse_masked_fa_gb300.binding as B  # noqa: E402
from block_sparse_masked_fa_gb300 import build as fa_build  # noqa: E402
import oracle  # noqa: E402
from fa_testutil import check_forward, check_grad  # noqa: E402
from synth import MaskProgram, make_qkv  # noqa: E402

FA_ERR_TIMEOUT = 6


def main():
    lib = B._bind(ctypes.CDLL(fa_build.build_test_hooks()))
    lib.fa_test_hook.argtypes = [ctypes.c_int32]
    lib.fa_test_hook.restype = ctypes.c_int
    B._lib = lib
    torch.cuda.set_device(0)
    S, D = 128, 128                          # one query tile and one key tile: one CTA
    q, k, v, do = make_qkv(1, 1, S, D, 4242)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    bm = B.fa_create_block_mask([("causal",)], 1, 1, S, S, 128)
    torch.cuda.synchronize()
    assert B.fa_get_status(bm) == 0
    prog = oracle.Program(MaskProgram((("causal",),)))
    f64 = lambda t: t[0, 0].double().numpy()
    scale = 1.0 / np.sqrt(D)

    # forward: the starved wait gives up and reports, the next forward is exact
    assert lib.fa_test_hook(1) == 0
    t0 = time.time()
    B.fa_forward(qd, kd, vd, bm)
    torch.cuda.synchronize()
    dt = time.time() - t0
    st = B.fa_get_status(bm)
    assert st == FA_ERR_TIMEOUT, f"forward: status {st}, expected FA_ERR_TIMEOUT"
    assert dt < 10.0, f"forward with a starved wait took {dt:.1f} s"
    assert lib.fa_test_hook(0) == 0
    out, lse = B.fa_forward(qd, kd, vd, bm)
    torch.cuda.synchronize()
    assert B.fa_get_status(bm) == 0
    ref_out, ref_lse = oracle.forward_head(f64(q), f64(k), f64(v), prog, ("none",), 0, scale)
    check_forward(out[0, 0].float().cpu().numpy(), lse[0, 0].cpu().numpy(), ref_out, ref_lse, "after timeout")

    # backward: the same, through the backward's producer
    assert lib.fa_test_hook(2) == 0
    t0 = time.time()
    B.fa_backward(qd, kd, vd, out, lse, dod, bm)
    torch.cuda.synchronize()
    dt = time.time() - t0
    st = B.fa_get_status(bm)
    assert st == FA_ERR_TIMEOUT, f"backward: status {st}, expected FA_ERR_TIMEOUT"
    assert dt < 10.0, f"backward with a starved wait took {dt:.1f} s"
    assert lib.fa_test_hook(0) == 0
    grads = B.fa_backward(qd, kd, vd, out, lse, dod, bm)
    torch.cuda.synchronize()
    assert B.fa_get_status(bm) == 0
    ref = oracle.backward_head(f64(q), f64(k), f64(v), f64(do), prog, ("none",), 0, scale)[:3]
    for name, g, r in zip(("dq", "dk", "dv"), grads, ref):
        check_grad(g[0, 0].float().cpu().numpy(), r, name + " after timeout")
    print("timeout path ok")


if __name__ == "__main__":
    main()
