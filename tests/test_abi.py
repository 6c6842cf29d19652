"""C-ABI checks that need no GPU: the library loads, exports every function
declared in include/fa.h, computes buffer sizes, and rejects bad arguments on
the host before queuing any GPU work.

Every call here fails host validation, so no fake pointer ever reaches CUDA.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")

fa = pytest.importorskip("block_sparse_masked_fa_gb300")
from block_sparse_masked_fa_gb300 import binding as B  # noqa: E402

OK, INVALID, UNSUPPORTED, SHAPE, ALIGN, CUDA, TIMEOUT, CHECK, WORKSPACE = range(9)
FAKE = 0x7F0000000000  # 256-byte aligned, never dereferenced: every call below fails validation first


def declared_functions():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:fa_status|const char\s*\*|int32_t)\s+(fa_\w+)\s*\(", src, re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("fa_create_block_mask", "fa_forward", "fa_backward", "fa_block_mask_bytes",
              "fa_backward_workspace_bytes", "fa_get_status", "fa_block_mask_summary", "fa_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(B.LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(declared_functions()) == set(B.EXPORTED)


def test_version_and_status_strings():
    assert fa.fa_version() == 100
    for code in range(9):
        assert fa.fa_status_string(code) and fa.fa_status_string(code) != "unknown status"
    assert fa.fa_status_string(99) == "unknown status"


def _align(x):
    return (x + 255) // 256 * 256


@pytest.mark.parametrize("Bm,Hm,q,kv,block", [(1, 1, 65536, 65536, 128), (2, 3, 1000, 777, 64), (1, 1, 1, 1, 16)])
def test_block_mask_bytes_layout(Bm, Hm, q, kv, block):
    nq, nkv = -(-q // block), -(-kv // block)
    rows, cols, tiles = Bm * Hm * nq, Bm * Hm * nkv, Bm * Hm * nq * nkv
    sizes = [rows * 4, tiles * 4, rows * 4, tiles * 4, cols * 4, tiles * 4, cols * 4, tiles * 4, rows * 4, cols * 4,
             tiles, Bm * 2 * max(nq, nkv) * 4 * 4, Bm * max(q, kv) * 8 + Bm * 4, Bm * 2 * max(q, kv) * 16, 4]
    if block < 128:  # the attention kernels' coarser tiles: 128 x 64 rows (forward), 128 x 128 columns (backward)
        P, fnq, fnkv, bnkv = Bm * Hm, -(-q // 128), -(-kv // 64), -(-kv // 128)
        sizes += [P * fnq * 4, P * fnq * fnkv * 4, P * fnq * 4, P * fnq * fnkv * 4, P * fnq * 4, P * fnq * fnkv,
                  P * bnkv * 4, P * bnkv * fnq * 4, P * bnkv * 4, P * bnkv * fnq * 4, P * bnkv * 4, P * fnq * bnkv]
    assert fa.fa_block_mask_bytes(Bm, Hm, q, kv, block) == sum(_align(s) for s in sizes)


def _bytes_status(*args):
    n = ctypes.c_size_t()
    return B._lib.fa_block_mask_bytes(*args, ctypes.byref(n))


def test_block_mask_bytes_rejects():
    assert _bytes_status(1, 1, 512, 512, 24) == UNSUPPORTED
    assert _bytes_status(1, 1, 512, 512, 256) == UNSUPPORTED
    assert _bytes_status(1, 1, 512, 512, 8) == UNSUPPORTED
    assert _bytes_status(0, 1, 512, 512, 128) == SHAPE
    assert _bytes_status(1, 1, 0, 512, 128) == SHAPE
    assert _bytes_status(1, 1, 1 << 40, 512, 128) == SHAPE
    assert B._lib.fa_block_mask_bytes(1, 1, 512, 512, 128, None) == INVALID


def _spec(nodes, doc_len=0):
    s = B.MaskSpec()
    s.n = len(nodes)
    s.doc_len = doc_len
    for k, (op, param) in enumerate(nodes):
        s.node[k].op = op
        s.node[k].param = param
    return s


def _create(spec, q=512, kv=512, block=128, buf=FAKE, nbytes=1 << 30, bm=True):
    st = B.BlockMaskStruct()
    return B._lib.fa_create_block_mask(ctypes.byref(spec) if spec is not None else None, 1, 1, q, kv, block, buf,
                                       nbytes, ctypes.byref(st) if bm else None, None)


M = B.MASK_OPS


def test_create_block_mask_rejects():
    causal = _spec([(M["causal"], None)])
    assert _create(None) == INVALID
    assert _create(causal, bm=False) == INVALID
    assert _create(causal, buf=FAKE + 16) == ALIGN
    assert _create(causal, nbytes=100) == WORKSPACE
    assert _create(causal, block=48) == UNSUPPORTED
    assert _create(_spec([])) == INVALID
    assert _create(_spec([(99, None)])) == INVALID
    assert _create(_spec([(M["causal"], None), (M["and"], None)])) == INVALID           # AND with one operand
    assert _create(_spec([(M["causal"], None), (M["causal"], None)])) == INVALID        # two values left
    assert _create(_spec([(M["window"], None)])) == INVALID                             # window needs its W
    assert _create(_spec([(M["window"], FAKE + 2)])) == INVALID                         # misaligned parameter
    assert _create(_spec([(M["same_doc"], FAKE)], doc_len=100)) == SHAPE                # doc ids too short
    two_docs = [(M["same_doc"], FAKE), (M["same_doc"], FAKE + 4096), (M["and"], None)]
    assert _create(_spec(two_docs, doc_len=512)) == INVALID                             # one doc array only
    deep = [(M["causal"], None)] * 9 + [(M["and"], None)] * 7
    assert _create(_spec(deep)) == INVALID                                              # stack deeper than 8
    too_many = B.MaskSpec()
    too_many.n = 17
    assert _create(too_many) == INVALID


def _from_lists(num=FAKE, idx=FAKE, fnum=None, fidx=None, stride=4, spec=None, block=128, buf=FAKE,
                nbytes=1 << 30, bm=True):
    st = B.BlockMaskStruct()
    return B._lib.fa_block_mask_from_kv_blocks(num, idx, fnum, fidx, stride,
                                               ctypes.byref(spec) if spec is not None else None, 1, 1, 512, 512,
                                               block, buf, nbytes, ctypes.byref(st) if bm else None, None)


def test_from_kv_blocks_rejects():
    """Host-side errors of the caller-chosen tiles entry, all before any GPU work."""
    assert _from_lists(num=None) == INVALID
    assert _from_lists(idx=None) == INVALID
    assert _from_lists(fnum=FAKE) == INVALID                       # full counts without indices
    assert _from_lists(fidx=FAKE) == INVALID                       # full indices without counts
    assert _from_lists(idx=FAKE + 2) == ALIGN
    assert _from_lists(fnum=FAKE + 1, fidx=FAKE) == ALIGN
    assert _from_lists(stride=0) == SHAPE
    assert _from_lists(spec=_spec([])) == INVALID                   # an empty program is not "no program"
    assert _from_lists(spec=_spec([(M["window"], None)])) == INVALID
    assert _from_lists(block=48) == UNSUPPORTED
    assert _from_lists(bm=False) == INVALID
    assert _from_lists(buf=FAKE + 16) == ALIGN
    assert _from_lists(nbytes=100) == WORKSPACE


def _bm(block=128, q=1024, kv=1024, Bm=1, Hm=1):
    st = B.BlockMaskStruct()
    st.Bm, st.Hm, st.block, st.q_len, st.kv_len = Bm, Hm, block, q, kv
    st.nq, st.nkv = -(-q // block), -(-kv // block)
    st.status = FAKE
    st.row_order = FAKE
    st.spec.n = 1
    st.spec.node[0].op = M["causal"]
    return st


def _fwd(q=FAKE, D=64, B_=1, H=1, S=1024, bm=None, score=None, scale=0.0, lse=FAKE):
    bm = _bm() if bm is None else bm
    sc = B.ScoreSpec() if score is None else score
    return B._lib.fa_forward(q, FAKE, FAKE, B_, H, S, S, D, ctypes.byref(bm), ctypes.byref(sc), scale, FAKE, lse,
                             None)


def test_forward_rejects():
    assert _fwd(q=None) == INVALID
    assert _fwd(q=FAKE + 8) == ALIGN
    assert _fwd(lse=FAKE + 2) == ALIGN
    assert _fwd(D=96) == UNSUPPORTED
    assert _fwd(D=256) == UNSUPPORTED
    assert _fwd(bm=_bm(block=64)) == INVALID          # block 64 without the builder's coarser lists
    coarse = _bm(block=64)
    coarse.fwd_kv_block, coarse.fwd_kv_num_blocks, coarse.fwd_row_order = 64, FAKE, FAKE
    coarse.from_blocks = 1
    assert _fwd(bm=coarse) == UNSUPPORTED             # caller-chosen tiles below block 128
    assert _fwd(S=2048) == SHAPE                      # block mask built for another length
    assert _fwd(B_=2, bm=_bm(Bm=3)) == SHAPE         # Bm must be 1 or B
    assert _fwd(H=4, bm=_bm(Hm=2)) == SHAPE          # Hm must be 1 or H
    assert _fwd(B_=0) == SHAPE
    assert _fwd(scale=-1.0) == INVALID
    assert _fwd(scale=float("nan")) == INVALID
    bad_score = B.ScoreSpec()
    bad_score.op = 7
    assert _fwd(score=bad_score) == INVALID
    cap_without_param = B.ScoreSpec()
    cap_without_param.op = B.SCORE_OPS["softcap"]
    assert _fwd(score=cap_without_param) == INVALID
    broken = _bm()
    broken.spec.n = 0
    assert _fwd(bm=broken) == INVALID


def test_backward_workspace_and_rejects():
    assert fa.fa_backward_workspace_bytes(2, 3, 1000, 128) == (_align(2 * 3 * 1000 * 128 * 4) + _align(2 * 3 * 8 * 256 * 4)
                                                               + _align(4))
    n = ctypes.c_size_t()
    assert B._lib.fa_backward_workspace_bytes(1, 1, 100, 80, ctypes.byref(n)) == UNSUPPORTED
    bm = _bm()
    sc = B.ScoreSpec()
    args = [FAKE] * 6 + [1, 1, 1024, 1024, 64, ctypes.byref(bm), ctypes.byref(sc), 0.0] + [FAKE] * 4
    assert B._lib.fa_backward(*args, 16, None) == WORKSPACE        # workspace too small
    bad = list(args)
    bad[3] = FAKE + 4
    assert B._lib.fa_backward(*bad, 1 << 30, None) == ALIGN
    bad = list(args)
    bad[0] = None
    assert B._lib.fa_backward(*bad, 1 << 30, None) == INVALID
    bad = list(args)
    bad[10] = 32
    assert B._lib.fa_backward(*bad, 1 << 30, None) == UNSUPPORTED


def test_prepared_pair_rejects():
    """Host-side errors of fa_forward_prepare_backward and fa_backward_prepared,
    before any GPU work: the workspace's size and alignment, and the ordinary
    forward / backward checks."""
    bm = _bm()
    sc = B.ScoreSpec()
    need = fa.fa_backward_workspace_bytes(1, 1, 1024, 64)
    fwd = [FAKE] * 3 + [1, 1, 1024, 1024, 64, ctypes.byref(bm), ctypes.byref(sc), 0.0, FAKE, FAKE, FAKE]
    assert B._lib.fa_forward_prepare_backward(*fwd, need - 1, None) == WORKSPACE
    bad = list(fwd)
    bad[13] = FAKE + 8
    assert B._lib.fa_forward_prepare_backward(*bad, need, None) == ALIGN
    bad = list(fwd)
    bad[13] = None
    assert B._lib.fa_forward_prepare_backward(*bad, need, None) == INVALID
    bad = list(fwd)
    bad[7] = 96
    assert B._lib.fa_forward_prepare_backward(*bad, need, None) == UNSUPPORTED
    bad = list(fwd)
    bad[5] = 2048
    assert B._lib.fa_forward_prepare_backward(*bad, need, None) == SHAPE
    bwd = [FAKE] * 6 + [1, 1, 1024, 1024, 64, ctypes.byref(bm), ctypes.byref(sc), 0.0] + [FAKE] * 4
    assert B._lib.fa_backward_prepared(*bwd, need - 1, None) == WORKSPACE
    bad = list(bwd)
    bad[17] = FAKE + 4
    assert B._lib.fa_backward_prepared(*bad, need, None) == ALIGN


def test_forward_paged_rejects():
    """Host-side errors of the paged forward, before any GPU work."""
    bm = _bm()
    sc = B.ScoreSpec()

    def call(table=FAKE, n_pages=16, q=FAKE, scale=0.0):
        return B._lib.fa_forward_paged(q, FAKE, FAKE, table, n_pages, 1, 1, 1024, 1024, 64, ctypes.byref(bm),
                                       ctypes.byref(sc), scale, FAKE, FAKE, None)
    assert call(q=None) == INVALID
    assert call(table=FAKE + 2) == ALIGN
    assert call(n_pages=0) == SHAPE
    assert call(n_pages=1 << 24) == SHAPE                  # pool rows past 2^31
    assert call(scale=-1.0) == INVALID                     # then the checks of fa_forward


def test_forward_decode_rejects():
    """Host-side errors of the short-query forward, before any device query."""
    bm = _bm(q=1)
    sc = B.ScoreSpec()

    def call(q_len=1, table=None, n_pages=0, ws=FAKE, q=FAKE):
        return B._lib.fa_forward_decode(q, FAKE, FAKE, table, n_pages, 1, 1, q_len, 1024, 64, ctypes.byref(bm),
                                        ctypes.byref(sc), 0.0, FAKE, FAKE, ws, 1 << 30, None)
    assert call(q_len=17) == UNSUPPORTED
    assert call(q_len=0) == SHAPE
    assert call(ws=None) == INVALID
    assert call(ws=FAKE + 8) == ALIGN
    assert call(q=None) == INVALID
    assert call(table=FAKE + 2, n_pages=4) == ALIGN
    assert call(table=FAKE, n_pages=0) == SHAPE
    n = ctypes.c_size_t()
    assert B._lib.fa_forward_decode_workspace_bytes(1, 1, 17, 1024, 64, ctypes.byref(n)) == UNSUPPORTED
    assert B._lib.fa_forward_decode_workspace_bytes(1, 1, 1, 1024, 80, ctypes.byref(n)) == UNSUPPORTED
    assert B._lib.fa_forward_decode_workspace_bytes(1, 1, 1, 1024, 64, None) == INVALID
    assert B._lib.fa_forward_decode_workspace_bytes(256, 256, 1, 1024, 64, ctypes.byref(n)) == UNSUPPORTED
    big = _bm(q=1)
    big_args = [FAKE, FAKE, FAKE, None, 0, 256, 256, 1, 1024, 64, ctypes.byref(big), ctypes.byref(sc), 0.0,
                FAKE, FAKE, FAKE, 1 << 30, None]
    assert B._lib.fa_forward_decode(*big_args) == UNSUPPORTED          # B * H = 65,536 grid rows


def test_score_param_grad_rejects():
    """A gradient buffer for the score parameter: ALiBi slopes (and the learned
    bias table) only, 4-byte aligned; the forward ignores it."""
    bm = _bm()
    base = [FAKE] * 6 + [1, 1, 1024, 1024, 64, ctypes.byref(bm)]
    for op, grad, want in ((0, FAKE, UNSUPPORTED), (1, FAKE, UNSUPPORTED), (2, FAKE + 2, ALIGN)):
        sc = B.ScoreSpec()
        sc.op, sc.param, sc.param_grad = op, (FAKE if op else None), grad
        args = base + [ctypes.byref(sc), 0.0] + [FAKE] * 4
        assert B._lib.fa_backward(*args, 1 << 30, None) == want
        assert B._lib.fa_backward_noalloc(*(base + [ctypes.byref(sc), 0.0] + [FAKE] * 3), None) == want
    # op none with a gradient buffer: the backward refuses it at the score check,
    # the forward passes it and stops at the later scale check instead
    sc = B.ScoreSpec()
    sc.param_grad = FAKE
    assert B._lib.fa_backward(*(base + [ctypes.byref(sc), -1.0] + [FAKE] * 4), 1 << 30, None) == UNSUPPORTED
    assert _fwd(score=sc, scale=-1.0) == INVALID


def test_relbias_table_arguments_checked():
    """The learned bias: a table pointer, a length in [1, 2^24] and a first
    distance in [-2^30, 2^30]; its gradient buffer 4-byte aligned."""
    for length, d0, want in ((0, 0, INVALID), ((1 << 24) + 1, 0, INVALID), (10, (1 << 30) + 1, INVALID),
                             (10, -(1 << 30) - 1, INVALID)):
        sc = B.ScoreSpec()
        sc.op, sc.param, sc.bias_len, sc.bias_d0 = 3, FAKE, length, d0
        assert _fwd(score=sc) == want
    sc = B.ScoreSpec()
    sc.op, sc.param, sc.bias_len = 3, None, 10
    assert _fwd(score=sc) == INVALID
    bm = _bm()
    base = [FAKE] * 6 + [1, 1, 1024, 1024, 64, ctypes.byref(bm)]
    sc = B.ScoreSpec()
    sc.op, sc.param, sc.param_grad, sc.bias_len = 3, FAKE, FAKE + 2, 10
    assert B._lib.fa_backward(*(base + [ctypes.byref(sc), 0.0] + [FAKE] * 4), 1 << 30, None) == ALIGN


def test_status_calls_reject_null():
    assert B._lib.fa_get_status(None, 0, None) == INVALID
    counts = (ctypes.c_int64 * 3)()
    assert B._lib.fa_block_mask_summary(None, ctypes.byref(counts), None) == INVALID


@pytest.mark.parametrize("ctype, cname", [(B.BlockMaskStruct, "fa_block_mask"), (B.MaskSpec, "fa_mask_spec"),
                                          (B.ScoreSpec, "fa_score_spec")])
def test_binding_structs_match_the_header(ctype, cname, tmp_path):
    """The ctypes mirrors of the C structs have the header's size and field offsets
    (a C program compiled against fa.h prints them)."""
    import shutil
    import subprocess

    cc = shutil.which("gcc") or shutil.which("cc")
    cuda_inc = next((d for d in ("/usr/local/cuda/include",) if os.path.exists(os.path.join(d, "cuda_runtime_api.h"))),
                    None)
    if cc is None or cuda_inc is None:
        pytest.skip("needs a C compiler and the CUDA headers")
    fields = [f[0] for f in ctype._fields_]
    lines = [f'printf("{f} %zu\\n", offsetof({cname}, {f}));' for f in fields]
    src = tmp_path / "layout.c"
    src.write_text("#include <stdio.h>\n#include <stddef.h>\n#include \"fa.h\"\nint main(void) {\n"
                   f'printf("sizeof %zu\\n", sizeof({cname}));\n' + "\n".join(lines) + "\nreturn 0;\n}\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-std=c11", "-I", os.path.join(ROOT, "include"), "-I", cuda_inc, str(src), "-o", str(exe)],
                   check=True, capture_output=True)
    got = dict(line.split() for line in subprocess.run([str(exe)], check=True, capture_output=True,
                                                         text=True).stdout.splitlines())
    assert int(got["sizeof"]) == ctypes.sizeof(ctype)
    for f in fields:
        assert int(got[f]) == getattr(ctype, f).offset, f
