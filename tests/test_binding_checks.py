"""The Python binding's own argument checks for the entries that take tensors
(caller-chosen tiles, paged and short-query forwards, the slope gradient):
malformed tensors are refused with ValueError before the C ABI is called, so
these run on CPU."""
import pytest
import torch

B = pytest.importorskip("block_sparse_masked_fa_gb300.binding")


class _Mask:
    """Stand-in for a BlockMask: only the fields the checks read."""

    def __init__(self, q_len=1, kv_len=1000):
        self.struct = B.BlockMaskStruct()
        self.struct.q_len, self.struct.kv_len = q_len, kv_len


def test_from_kv_blocks_refuses_malformed_lists():
    num = torch.zeros(1, 1, 8, dtype=torch.int32)
    idx = torch.zeros(1, 1, 8, 8, dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA"):
        B.fa_block_mask_from_kv_blocks(num, idx, 1024, 1024)                   # host tensors
    with pytest.raises(ValueError):
        B.fa_block_mask_from_kv_blocks(num.long(), idx, 1024, 1024)            # wrong dtype


def test_forward_paged_refuses_bad_pools_and_tables():
    q = torch.zeros(2, 4, 16, 64, dtype=torch.bfloat16)
    mask = _Mask(q_len=16, kv_len=1000)                                         # 8 key tiles
    pool = torch.zeros(4, 10 * 128, 64, dtype=torch.bfloat16)
    table = torch.zeros(2, 8, dtype=torch.int32)
    with pytest.raises(ValueError, match="k_pool"):
        B.fa_forward_paged(q, pool[:, :1000], pool[:, :1000], table, mask)      # rows not whole pages
    with pytest.raises(ValueError, match="k_pool"):
        B.fa_forward_paged(q, pool[:2], pool[:2], table, mask)                  # heads differ from q
    with pytest.raises(ValueError, match="page_table"):
        B.fa_forward_paged(q, pool, pool, table, mask)                          # table on the host
    with pytest.raises(ValueError, match="page_table"):
        B.fa_forward_paged(q, pool, pool, table[:, :7], mask)                   # too few tiles


def test_forward_decode_refuses_bad_page_tables():
    q = torch.zeros(2, 4, 1, 64, dtype=torch.bfloat16)
    pool = torch.zeros(4, 10 * 128, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="page_table"):
        B.fa_forward_decode(q, pool, pool, _Mask(), page_table=torch.zeros(2, 8, dtype=torch.int32))
    with pytest.raises(ValueError, match="same shape"):
        B.fa_forward_decode(q, pool, pool[:, :128], _Mask(), page_table=torch.zeros(2, 8, dtype=torch.int32))


def test_forward_decode_refuses_keys_shorter_than_the_mask():
    q = torch.zeros(2, 4, 1, 64, dtype=torch.bfloat16)
    k = torch.zeros(2, 4, 900, 64, dtype=torch.bfloat16)                      # the mask says 1000 keys
    with pytest.raises(ValueError, match="kv_len"):
        B.fa_forward_decode(q, k, k, _Mask(kv_len=1000))
    with pytest.raises(ValueError, match="q_len"):
        B.fa_forward_decode(q, k, k, _Mask(q_len=2, kv_len=900))


def test_slope_gradient_buffer_checked():
    alibi = B.ScoreSpec()
    alibi.op = B.SCORE_OPS["alibi"]
    score = (alibi, [])                                                          # a prebuilt spec
    with pytest.raises(ValueError, match="score_param_grad"):
        B._backward_score(score, torch.zeros(4), 4)                             # host tensor
    with pytest.raises(ValueError, match="score_param_grad"):
        B._backward_score(score, torch.zeros(4, dtype=torch.float64), 4)
    spec, _ = B._backward_score(score, None, 4)
    assert spec.op == B.SCORE_OPS["alibi"] and not spec.param_grad
    assert spec is not alibi                                                     # the caller's spec is not modified


def test_shape_checks_accept_consistent_tensors():
    q = torch.zeros(2, 3, 100, 64)
    k = torch.zeros(2, 3, 250, 64)
    B._check_shapes(q, kv=(("k", k), ("v", k), ("dk", None)), like_q=(("out", q), ("dq", None)),
                    lse=torch.zeros(2, 3, 100))
    B._check_shapes(q)                                                         # nothing else given


@pytest.mark.parametrize("bad", ["k_heads", "k_dim", "v_len", "out", "lse", "q_rank"])
def test_shape_checks_refuse_disagreeing_tensors(bad):
    q = torch.zeros(2, 3, 100, 64)
    k = torch.zeros(2, 3, 250, 64)
    args = {"kv": [("k", k), ("v", k)], "like_q": [("out", q)], "lse": torch.zeros(2, 3, 100)}
    if bad == "k_heads":
        args["kv"][0] = ("k", torch.zeros(2, 1, 250, 64))
    elif bad == "k_dim":
        args["kv"][0] = ("k", torch.zeros(2, 3, 250, 128))
    elif bad == "v_len":
        args["kv"][1] = ("v", torch.zeros(2, 3, 200, 64))
    elif bad == "out":
        args["like_q"][0] = ("out", torch.zeros(2, 3, 99, 64))
    elif bad == "lse":
        args["lse"] = torch.zeros(2, 3, 101)
    else:
        q = q[0]
    with pytest.raises(ValueError):
        B._check_shapes(q, **args)


def test_forward_refuses_keys_with_other_heads_before_the_library():
    q = torch.zeros(1, 4, 128, 64, dtype=torch.bfloat16)
    k = torch.zeros(1, 2, 128, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="k must be"):
        B.fa_forward(q, k, k, _Mask(q_len=128, kv_len=128))


def test_sparsity_map():
    """The ASCII map of a causal 4 x 4 tile grid, and a coarsened 8 x 8 one."""
    import numpy as np

    causal = np.array([[1, 0, 0, 0], [2, 1, 0, 0], [2, 2, 1, 0], [2, 2, 2, 1]])
    lines = B.sparsity_map(causal, 128).split("\n")
    assert lines[:4] == ["+...", "#+..", "##+.", "###+"]
    assert lines[4] == "4 x 4 tiles of 128 (one cell: 1 x 1): 6 empty, 4 partial, 6 full; 37.50% skipped"
    big = np.kron(causal, np.ones((2, 2), dtype=int))        # 8 x 8, two-by-two cells at max_cols 4
    lines = B.sparsity_map(big, 64, max_cols=4).split("\n")
    assert lines[:4] == ["+...", "#+..", "##+.", "###+"] and "one cell: 2 x 2" in lines[4]


def _fwd_args(S=128, D=64):
    q = torch.zeros(1, 4, S, D, dtype=torch.bfloat16)
    return q, q.clone(), q.clone()


@pytest.mark.parametrize("bad", ["k_expand", "q_transpose", "v_float32", "lse_float64", "out_slice"])
def test_forward_refuses_views_and_wrong_dtypes(bad):
    """Views the kernels cannot address as dense [B, H, len, D] arrays (expanded, transposed,
    sliced) and tensors of another dtype are refused before the library is called."""
    q, k, v = _fwd_args()
    out = lse = None
    match = "contiguous"
    if bad == "k_expand":
        k = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16).expand(1, 4, 128, 64)
    elif bad == "q_transpose":
        q = torch.zeros(1, 4, 64, 128, dtype=torch.bfloat16).transpose(2, 3)
    elif bad == "v_float32":
        v, match = v.float(), "v must be torch.bfloat16"
    elif bad == "lse_float64":
        lse, match = torch.zeros(1, 4, 128, dtype=torch.float64), "lse must be torch.float32"
    else:
        out = torch.zeros(1, 4, 128, 128, dtype=torch.bfloat16)[..., :64]
    with pytest.raises(ValueError, match=match):
        B.fa_forward(q, k, v, _Mask(q_len=128, kv_len=128), out=out, lse=lse)


def test_forward_refuses_host_tensors():
    q, k, v = _fwd_args()
    with pytest.raises(ValueError, match="CUDA"):
        B.fa_forward(q, k, v, _Mask(q_len=128, kv_len=128))


@pytest.mark.parametrize("bad", ["dq_expand", "dk_float32", "dout_transpose", "workspace_float32"])
def test_backward_refuses_views_and_wrong_dtypes(bad):
    q, k, v = _fwd_args()
    out, dout = q.clone(), q.clone()
    lse = torch.zeros(1, 4, 128)
    kw = {}
    match = "contiguous"
    if bad == "dq_expand":
        kw["dq"] = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16).expand(1, 4, 128, 64)
    elif bad == "dk_float32":
        kw["dk"], match = torch.zeros(1, 4, 128, 64), "dk must be torch.bfloat16"
    elif bad == "dout_transpose":
        dout = torch.zeros(1, 4, 64, 128, dtype=torch.bfloat16).transpose(2, 3)
    else:
        kw["workspace"], match = torch.zeros(16, dtype=torch.float32), "workspace must be torch.uint8"
    with pytest.raises(ValueError, match=match):
        B.fa_backward(q, k, v, out, lse, dout, _Mask(q_len=128, kv_len=128), **kw)
    if bad != "workspace_float32":
        with pytest.raises(ValueError, match=match):
            B.fa_backward_noalloc(q, k, v, out, lse, dout, _Mask(q_len=128, kv_len=128), **kw)


def test_block_mask_buffer_checked():
    with pytest.raises(ValueError, match="buffer"):
        B._check_buffer(torch.zeros(64, dtype=torch.uint8))                  # host memory
    with pytest.raises(ValueError, match="buffer"):
        B._check_buffer(torch.zeros(64, dtype=torch.int32))


@pytest.mark.parametrize("bad", ["workspace_float32", "workspace_view", "out_float32", "dq_expand"])
def test_prepared_pair_refuses_views_and_wrong_dtypes(bad):
    """fa_forward_prepare_backward and fa_backward_prepared take the caller's
    workspace: it is checked like every other tensor (contiguous uint8 on q's
    device), and so are the outputs."""
    q, k, v = _fwd_args()
    out, dout = q.clone(), q.clone()
    lse = torch.zeros(1, 4, 128)
    ws = torch.zeros(1 << 16, dtype=torch.uint8)
    kw_f, kw_b = {}, {}
    match = "contiguous"
    if bad == "workspace_float32":
        ws, match = torch.zeros(1 << 14, dtype=torch.float32), "workspace must be torch.uint8"
    elif bad == "workspace_view":
        ws = torch.zeros(2, 1 << 16, dtype=torch.uint8)[:, ::2].reshape(-1)[::2]
    elif bad == "out_float32":
        kw_f["out"], match = torch.zeros(1, 4, 128, 64), "out must be torch.bfloat16"
    else:
        kw_b["dq"] = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16).expand(1, 4, 128, 64)
    mask = _Mask(q_len=128, kv_len=128)
    if bad != "dq_expand":
        with pytest.raises(ValueError, match=match):
            B.fa_forward_prepare_backward(q, k, v, mask, ws, **kw_f)
    if bad != "out_float32":
        with pytest.raises(ValueError, match=match):
            B.fa_backward_prepared(q, k, v, out, lse, dout, mask, ws, **kw_b)
