"""ctypes binding of the C ABI in include/fa.h (argument marshalling only).

Names mirror the C entry points: fa_block_mask_bytes, fa_create_block_mask,
fa_block_mask_from_kv_blocks, fa_forward, fa_forward_paged,
fa_forward_decode_workspace_bytes, fa_forward_decode,
fa_backward_workspace_bytes, fa_backward, fa_forward_prepare_backward,
fa_backward_prepared, fa_get_status, fa_block_mask_summary, fa_status_string.  Tensors are torch CUDA tensors; the binding passes their
device pointers and the current CUDA stream.  Every step
of the computation runs in the library's kernels; importing this module fails
loudly when the library has not been built.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfa_gb300.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build the CUDA library first "
        "(python -c 'import __graft_entry__ as g; g.build()')")

_lib = ctypes.CDLL(LIB_PATH)

MAX_NODES = 16
MASK_OPS = {"true": 0, "causal": 1, "same_doc": 2, "window": 3, "sink": 4, "prefix": 5, "and": 6, "or": 7}
SCORE_OPS = {"none": 0, "softcap": 1, "alibi": 2, "relbias": 3}
STATUS = {0: "FA_OK", 1: "FA_ERR_INVALID_ARG", 2: "FA_ERR_UNSUPPORTED", 3: "FA_ERR_SHAPE",
          4: "FA_ERR_ALIGNMENT", 5: "FA_ERR_CUDA", 6: "FA_ERR_TIMEOUT", 7: "FA_ERR_DEVICE_CHECK",
          8: "FA_ERR_WORKSPACE"}


class FaError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {STATUS.get(code, code)} ({_lib.fa_status_string(code).decode()})")
        self.code = code


class MaskNode(ctypes.Structure):
    _fields_ = [("op", ctypes.c_int32), ("param", ctypes.c_void_p)]


class MaskSpec(ctypes.Structure):
    _fields_ = [("n", ctypes.c_int32), ("doc_len", ctypes.c_int64), ("node", MaskNode * MAX_NODES),
                ("q_offset", ctypes.c_int64)]


class ScoreSpec(ctypes.Structure):
    _fields_ = [("op", ctypes.c_int32), ("param", ctypes.c_void_p), ("param_grad", ctypes.c_void_p),
                ("bias_len", ctypes.c_int32), ("bias_d0", ctypes.c_int32)]


class BlockMaskStruct(ctypes.Structure):
    _fields_ = [("Bm", ctypes.c_int32), ("Hm", ctypes.c_int32), ("block", ctypes.c_int32),
                ("nq", ctypes.c_int32), ("nkv", ctypes.c_int32),
                ("q_len", ctypes.c_int64), ("kv_len", ctypes.c_int64)] + \
               [(name, ctypes.c_void_p) for name in (
                   "kv_num_blocks", "kv_indices", "full_kv_num_blocks", "full_kv_indices",
                   "q_num_blocks", "q_indices", "full_q_num_blocks", "full_q_indices",
                   "row_order", "col_order", "tile_class", "tile_summary", "doc_runs", "row_segs", "status")] + \
               [("spec", MaskSpec), ("from_blocks", ctypes.c_int32)] + \
               [(name, ctypes.c_int32) for name in ("fwd_kv_block", "fwd_nq", "fwd_nkv", "bwd_nq", "bwd_nkv")] + \
               [(name, ctypes.c_void_p) for name in (
                   "fwd_kv_num_blocks", "fwd_kv_indices", "fwd_full_kv_num_blocks", "fwd_full_kv_indices",
                   "fwd_row_order", "fwd_tile_class", "bwd_q_num_blocks", "bwd_q_indices", "bwd_full_q_num_blocks",
                   "bwd_full_q_indices", "bwd_col_order", "bwd_tile_class")]


_c = ctypes


def _bind(lib):
    """Declares the C signatures on a loaded library (the package's own, or the test
    library built from the same sources) and returns it."""
    lib.fa_block_mask_bytes.argtypes = [_c.c_int32, _c.c_int32, _c.c_int64, _c.c_int64, _c.c_int32,
                                         _c.POINTER(_c.c_size_t)]
    lib.fa_create_block_mask.argtypes = [_c.POINTER(MaskSpec), _c.c_int32, _c.c_int32, _c.c_int64, _c.c_int64,
                                          _c.c_int32, _c.c_void_p, _c.c_size_t, _c.POINTER(BlockMaskStruct),
                                          _c.c_void_p]
    lib.fa_block_mask_from_kv_blocks.argtypes = [_c.c_void_p] * 4 + [_c.c_int32, _c.POINTER(MaskSpec), _c.c_int32,
                                                                      _c.c_int32, _c.c_int64, _c.c_int64, _c.c_int32,
                                                                      _c.c_void_p, _c.c_size_t,
                                                                      _c.POINTER(BlockMaskStruct), _c.c_void_p]
    lib.fa_forward.argtypes = [_c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_int32, _c.c_int32, _c.c_int64,
                                _c.c_int64, _c.c_int32, _c.POINTER(BlockMaskStruct), _c.POINTER(ScoreSpec),
                                _c.c_float, _c.c_void_p, _c.c_void_p, _c.c_void_p]
    lib.fa_forward_paged.argtypes = [_c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_int32, _c.c_int32,
                                      _c.c_int32, _c.c_int64, _c.c_int64, _c.c_int32, _c.POINTER(BlockMaskStruct),
                                      _c.POINTER(ScoreSpec), _c.c_float, _c.c_void_p, _c.c_void_p, _c.c_void_p]
    lib.fa_forward_decode_workspace_bytes.argtypes = [_c.c_int32, _c.c_int32, _c.c_int64, _c.c_int64, _c.c_int32,
                                                       _c.POINTER(_c.c_size_t)]
    lib.fa_forward_decode.argtypes = [_c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_int32, _c.c_int32,
                                       _c.c_int32, _c.c_int64, _c.c_int64, _c.c_int32, _c.POINTER(BlockMaskStruct),
                                       _c.POINTER(ScoreSpec), _c.c_float, _c.c_void_p, _c.c_void_p, _c.c_void_p,
                                       _c.c_size_t, _c.c_void_p]
    lib.fa_backward_workspace_bytes.argtypes = [_c.c_int32, _c.c_int32, _c.c_int64, _c.c_int32,
                                                 _c.POINTER(_c.c_size_t)]
    lib.fa_backward.argtypes = [_c.c_void_p] * 6 + [_c.c_int32, _c.c_int32, _c.c_int64, _c.c_int64, _c.c_int32,
                                                     _c.POINTER(BlockMaskStruct), _c.POINTER(ScoreSpec), _c.c_float,
                                                     _c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_void_p,
                                                     _c.c_size_t, _c.c_void_p]
    lib.fa_forward_prepare_backward.argtypes = [_c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_int32, _c.c_int32,
                                                 _c.c_int64, _c.c_int64, _c.c_int32, _c.POINTER(BlockMaskStruct),
                                                 _c.POINTER(ScoreSpec), _c.c_float, _c.c_void_p, _c.c_void_p,
                                                 _c.c_void_p, _c.c_size_t, _c.c_void_p]
    lib.fa_backward_prepared.argtypes = lib.fa_backward.argtypes
    lib.fa_backward_noalloc.argtypes = [_c.c_void_p] * 6 + [_c.c_int32, _c.c_int32, _c.c_int64, _c.c_int64,
                                                             _c.c_int32, _c.POINTER(BlockMaskStruct),
                                                             _c.POINTER(ScoreSpec), _c.c_float, _c.c_void_p,
                                                             _c.c_void_p, _c.c_void_p, _c.c_void_p]
    lib.fa_get_status.argtypes = [_c.POINTER(BlockMaskStruct), _c.c_int32, _c.c_void_p]
    lib.fa_block_mask_summary.argtypes = [_c.POINTER(BlockMaskStruct), _c.POINTER(_c.c_int64 * 3), _c.c_void_p]
    lib.fa_status_string.argtypes = [_c.c_int]
    lib.fa_status_string.restype = _c.c_char_p
    for _f in (lib.fa_block_mask_bytes, lib.fa_create_block_mask, lib.fa_block_mask_from_kv_blocks, lib.fa_forward,
               lib.fa_forward_paged, lib.fa_forward_decode_workspace_bytes, lib.fa_forward_decode, lib.fa_backward_workspace_bytes,
               lib.fa_backward, lib.fa_backward_noalloc, lib.fa_forward_prepare_backward, lib.fa_backward_prepared,
               lib.fa_get_status, lib.fa_block_mask_summary):
        _f.restype = _c.c_int
    lib.fa_version.restype = _c.c_int32
    return lib


_lib = _bind(_lib)

EXPORTED = ("fa_block_mask_bytes", "fa_create_block_mask", "fa_block_mask_from_kv_blocks", "fa_forward",
            "fa_forward_paged", "fa_forward_decode_workspace_bytes", "fa_forward_decode", "fa_backward_workspace_bytes",
            "fa_backward", "fa_backward_noalloc", "fa_forward_prepare_backward", "fa_backward_prepared",
            "fa_get_status", "fa_block_mask_summary", "fa_status_string", "fa_version")
NOALLOC_SCRATCH_BYTES = 16 << 20


def _check(code: int, where: str):
    if code != 0:
        raise FaError(code, where)


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _dev_int32(x, device) -> torch.Tensor:
    if isinstance(x, torch.Tensor):
        if x.dtype != torch.int32 or not x.is_cuda:
            raise TypeError("mask parameters must be int32 CUDA tensors")
        return x.contiguous()
    return torch.as_tensor(x, dtype=torch.int32, device=device).reshape(-1)


def make_mask_spec(nodes: Sequence[tuple], device=None, q_offset: int = 0):
    """Device-side mask spec from a postfix node list.

    Nodes: ("causal",), ("true",), ("same_doc", doc_ids [Bm, doc_len] int32),
    ("window", W), ("sink", n), ("prefix", prefix_len [Bm]), ("and",), ("or",).
    Scalars given as Python ints are copied into fresh device int32 tensors;
    pass an int32 CUDA tensor to change a parameter later without a new spec.
    q_offset: position of query row 0 (e.g. kv_len - q_len when decoding the
    newest tokens of a cache; see fa_mask_spec in fa.h).
    Returns (MaskSpec, keepalive list of tensors).
    """
    device = device or torch.device("cuda", torch.cuda.current_device())
    if not 1 <= len(nodes) <= MAX_NODES:
        raise ValueError("a mask program has 1..16 nodes")
    spec = MaskSpec()
    spec.n = len(nodes)
    keep = []
    doc_len = 0
    for k, node in enumerate(nodes):
        kind = node[0]
        spec.node[k].op = MASK_OPS[kind]
        spec.node[k].param = None
        if kind in ("same_doc", "window", "sink", "prefix"):
            t = _dev_int32(node[1], device)
            keep.append(t)
            spec.node[k].param = t.data_ptr()
            if kind == "same_doc":
                doc_len = int(t.shape[-1])
    spec.doc_len = doc_len
    spec.q_offset = int(q_offset)
    return spec, keep


def make_score_spec(kind: str = "none", param=None, device=None, d0: int = 0):
    """("none"), ("softcap", c), ("alibi", slopes[H]), ("relbias", table[H, L], d0) -- the
    learned relative-position bias s = x + table[h, clamp(q_pos - kv_idx - d0, 0, L - 1)];
    param becomes a device fp32 tensor."""
    device = device or torch.device("cuda", torch.cuda.current_device())
    s = ScoreSpec()
    s.op = SCORE_OPS[kind]
    s.param = None
    keep = []
    if kind != "none":
        t = param if isinstance(param, torch.Tensor) else torch.as_tensor(param, dtype=torch.float32)
        if kind == "relbias":
            if t.dim() != 2:
                raise ValueError("the relbias table must be [H, L]")
            s.bias_len, s.bias_d0 = int(t.shape[1]), int(d0)
        t = t.to(device=device, dtype=torch.float32).reshape(-1).contiguous()
        keep.append(t)
        s.param = t.data_ptr()
    return s, keep


class BlockMask:
    """A built block mask: the caller-owned device buffer plus the C descriptor."""

    def __init__(self, struct: BlockMaskStruct, buffer: torch.Tensor, keep: list):
        self.struct = struct
        self.buffer = buffer
        self._keep = keep

    def _view(self, field: str, shape, dtype=torch.int32) -> torch.Tensor:
        off = getattr(self.struct, field) - self.buffer.data_ptr()
        n = 1
        for s in shape:
            n *= s
        nbytes = n * torch.empty(0, dtype=dtype).element_size()
        return self.buffer[off:off + nbytes].view(dtype).view(*shape)

    def lists(self) -> dict:
        s = self.struct
        r, c = (s.Bm, s.Hm, s.nq), (s.Bm, s.Hm, s.nkv)
        return {
            "kv_num_blocks": self._view("kv_num_blocks", r),
            "kv_indices": self._view("kv_indices", r + (s.nkv,)),
            "full_kv_num_blocks": self._view("full_kv_num_blocks", r),
            "full_kv_indices": self._view("full_kv_indices", r + (s.nkv,)),
            "q_num_blocks": self._view("q_num_blocks", c),
            "q_indices": self._view("q_indices", c + (s.nq,)),
            "full_q_num_blocks": self._view("full_q_num_blocks", c),
            "full_q_indices": self._view("full_q_indices", c + (s.nq,)),
        }

    def kernel_lists(self) -> dict:
        """Below block 128: the coarser tiles the attention kernels walk (see
        fa_block_mask in fa.h) -- the forward's query-tile rows of 128 over key
        tiles of fwd_kv_block, the backward's key-tile columns of 128 over query
        tiles of 128, with their class grids.  Empty at block 128."""
        s = self.struct
        if not s.fwd_kv_num_blocks:
            return {}
        fr, br = (s.Bm, s.Hm, s.fwd_nq), (s.Bm, s.Hm, s.bwd_nkv)
        return {
            "fwd_kv_num_blocks": self._view("fwd_kv_num_blocks", fr),
            "fwd_kv_indices": self._view("fwd_kv_indices", fr + (s.fwd_nkv,)),
            "fwd_full_kv_num_blocks": self._view("fwd_full_kv_num_blocks", fr),
            "fwd_full_kv_indices": self._view("fwd_full_kv_indices", fr + (s.fwd_nkv,)),
            "fwd_tile_class": self._view("fwd_tile_class", fr + (s.fwd_nkv,), torch.uint8),
            "bwd_q_num_blocks": self._view("bwd_q_num_blocks", br),
            "bwd_q_indices": self._view("bwd_q_indices", br + (s.bwd_nq,)),
            "bwd_full_q_num_blocks": self._view("bwd_full_q_num_blocks", br),
            "bwd_full_q_indices": self._view("bwd_full_q_indices", br + (s.bwd_nq,)),
            "bwd_tile_class": self._view("bwd_tile_class", (s.Bm, s.Hm, s.bwd_nq, s.bwd_nkv), torch.uint8),
        }

    def tile_class(self) -> torch.Tensor:
        s = self.struct
        return self._view("tile_class", (s.Bm, s.Hm, s.nq, s.nkv), torch.uint8)

    def row_order(self) -> torch.Tensor:
        s = self.struct
        return self._view("row_order", (s.Bm * s.Hm * s.nq,))

    def row_segs(self) -> torch.Tensor:
        """[Bm, 2, max(q_len, kv_len), 4] int32: per query row (0) / key column (1)
        the visible intervals [lo0, hi0) and [lo1, hi1), lo0 = -1 if not summarised."""
        s = self.struct
        return self._view("row_segs", (s.Bm, 2, max(s.q_len, s.kv_len), 4))

    def to_string(self, bm: int = 0, hm: int = 0, max_cols: int = 64) -> str:
        """ASCII map of the tile classes of (bm, hm) and the share of tiles skipped
        (tutorial, sharp edge 6: check the mask visually)."""
        s = self.struct
        return sparsity_map(self.tile_class()[bm, hm].cpu().numpy(), s.block, max_cols)


def sparsity_map(cls, block: int, max_cols: int = 64) -> str:
    """ASCII map of a tile-class grid [nq, nkv] (0 empty, 1 partial, 2 full):
    '.' every tile of a cell skipped, '#' every tile full, '+' otherwise.  A cell
    covers ceil(n / max_cols) tiles a side when the grid is wider than max_cols.
    The last line gives the counts and the share of tiles skipped."""
    import numpy as np

    cls = np.asarray(cls)
    nq, nkv = cls.shape
    f = max(1, -(-max(nq, nkv) // max_cols))
    lines = []
    for r0 in range(0, nq, f):
        row = []
        for c0 in range(0, nkv, f):
            cell = cls[r0:r0 + f, c0:c0 + f]
            row.append("." if not cell.any() else ("#" if (cell == 2).all() else "+"))
        lines.append("".join(row))
    empty, part, full = int((cls == 0).sum()), int((cls == 1).sum()), int((cls == 2).sum())
    total = max(1, cls.size)
    lines.append(f"{nq} x {nkv} tiles of {block} (one cell: {f} x {f}): {empty} empty, {part} partial, "
                 f"{full} full; {100.0 * empty / total:.2f}% skipped")
    return "\n".join(lines)


def fa_block_mask_bytes(Bm: int, Hm: int, q_len: int, kv_len: int, block: int = 128) -> int:
    n = ctypes.c_size_t()
    _check(_lib.fa_block_mask_bytes(Bm, Hm, q_len, kv_len, block, ctypes.byref(n)), "fa_block_mask_bytes")
    return n.value


def _check_buffer(buffer: torch.Tensor):
    """A block-mask buffer is a contiguous uint8 CUDA tensor (its numel is the byte count the library checks)."""
    if buffer.dtype != torch.uint8 or not buffer.is_contiguous() or not buffer.is_cuda:
        raise ValueError("the block-mask buffer must be a contiguous uint8 CUDA tensor")


def fa_create_block_mask(nodes: Sequence[tuple], Bm: int, Hm: int, q_len: int, kv_len: int, block: int = 128,
                         buffer: Optional[torch.Tensor] = None, stream=None, q_offset: int = 0) -> BlockMask:
    """Builds the block mask of a postfix mask program (see make_mask_spec;
    q_offset applies to a node list, a prebuilt spec carries its own)."""
    spec, keep = (nodes if isinstance(nodes, tuple) and isinstance(nodes[0], MaskSpec)
                  else make_mask_spec(nodes, q_offset=q_offset))
    nbytes = fa_block_mask_bytes(Bm, Hm, q_len, kv_len, block)
    if buffer is None:
        buffer = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    _check_buffer(buffer)
    st = BlockMaskStruct()
    _check(_lib.fa_create_block_mask(ctypes.byref(spec), Bm, Hm, q_len, kv_len, block, buffer.data_ptr(),
                                     buffer.numel(), ctypes.byref(st), _stream(stream)), "fa_create_block_mask")
    return BlockMask(st, buffer, keep + [spec])


def fa_block_mask_from_kv_blocks(kv_num_blocks: torch.Tensor, kv_indices: torch.Tensor, q_len: int, kv_len: int,
                                 full_kv_num_blocks: Optional[torch.Tensor] = None,
                                 full_kv_indices: Optional[torch.Tensor] = None, block: int = 128,
                                 nodes: Optional[Sequence[tuple]] = None, buffer: Optional[torch.Tensor] = None,
                                 stream=None) -> BlockMask:
    """Block mask of caller-chosen tiles: int32 CUDA tensors kv_num_blocks
    [Bm, Hm, nq] and kv_indices [Bm, Hm, nq, stride] (PARTIAL tiles, any
    order), optionally the same for FULL tiles.  ``nodes``: the mask program
    applied on PARTIAL tiles (None: all their pairs are visible).  Invalid
    lists are reported by fa_get_status (FA_ERR_DEVICE_CHECK)."""
    tensors = [kv_num_blocks, kv_indices] + ([] if full_kv_num_blocks is None else
                                             [full_kv_num_blocks, full_kv_indices])
    for t in tensors:
        if t is None or t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous():
            raise ValueError("tile lists must be contiguous int32 CUDA tensors")
    if kv_num_blocks.dim() != 3 or kv_indices.dim() != 4 or kv_indices.shape[:3] != kv_num_blocks.shape:
        raise ValueError("kv_num_blocks must be [Bm, Hm, nq] and kv_indices [Bm, Hm, nq, stride]")
    if full_kv_num_blocks is not None and (full_kv_num_blocks.shape != kv_num_blocks.shape or
                                           full_kv_indices.shape != kv_indices.shape):
        raise ValueError("full lists must be shaped like the partial ones")
    Bm, Hm, nq = kv_num_blocks.shape
    if nq != -(-q_len // block):
        raise ValueError(f"lists have {nq} query-tile rows; q_len {q_len} at block {block} has {-(-q_len // block)}")
    keep = list(tensors)
    spec = None
    if nodes is not None:
        spec, k2 = nodes if isinstance(nodes, tuple) and isinstance(nodes[0], MaskSpec) else make_mask_spec(nodes)
        keep += k2 + [spec]
    nbytes = fa_block_mask_bytes(Bm, Hm, q_len, kv_len, block)
    if buffer is None:
        buffer = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    _check_buffer(buffer)
    st = BlockMaskStruct()
    _check(_lib.fa_block_mask_from_kv_blocks(_ptr(kv_num_blocks), _ptr(kv_indices), _ptr(full_kv_num_blocks),
                                             _ptr(full_kv_indices), kv_indices.shape[3],
                                             ctypes.byref(spec) if spec is not None else None, Bm, Hm, q_len,
                                             kv_len, block, buffer.data_ptr(), buffer.numel(), ctypes.byref(st),
                                             _stream(stream)), "fa_block_mask_from_kv_blocks")
    return BlockMask(st, buffer, keep)


def _check_shapes(q, kv=(), like_q=(), lse=None):
    """Refuses tensors whose sizes disagree with q [B, H, q_len, D] (the kernels'
    tensor maps are built from these sizes): keys, values and their gradients
    [B, H, kv_len, D] with one kv_len, out / dO / dq shaped as q, LSE [B, H, q_len].
    None entries are skipped."""
    if q.dim() != 4:
        raise ValueError("q must be [B, H, q_len, D]")
    B, H, q_len, D = q.shape
    kv_len = None
    for name, t in kv:
        if t is None:
            continue
        if t.dim() != 4 or t.shape[0] != B or t.shape[1] != H or t.shape[3] != D:
            raise ValueError(f"{name} must be [{B}, {H}, kv_len, {D}], got {tuple(t.shape)}")
        if kv_len is None:
            kv_len = t.shape[2]
        elif t.shape[2] != kv_len:
            raise ValueError(f"{name} has {t.shape[2]} rows, the other keys / values {kv_len}")
    for name, t in like_q:
        if t is not None and tuple(t.shape) != tuple(q.shape):
            raise ValueError(f"{name} must be shaped like q {tuple(q.shape)}, got {tuple(t.shape)}")
    if lse is not None and tuple(lse.shape) != (B, H, q_len):
        raise ValueError(f"lse must be [{B}, {H}, {q_len}], got {tuple(lse.shape)}")


_BF16, _F32, _I32, _U8 = torch.bfloat16, torch.float32, torch.int32, torch.uint8


def _check_storage(q, tensors):
    """Refuses tensors the kernels cannot address as plain dense arrays: the
    library gets bare device pointers and builds its tensor maps (and the dq
    conversion its indexing) on dense [B, H, len, D] storage, so an expanded,
    transposed or sliced view would make it read and write outside the tensor.
    Each (name, tensor, dtype) must have that dtype, be contiguous and live on
    q's CUDA device; None entries are skipped.  q itself is checked as bf16."""
    given = [(name, t, dtype) for name, t, dtype in (("q", q, _BF16),) + tuple(tensors) if t is not None]
    for name, t, dtype in given:
        if t.dtype != dtype:
            raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    for name, t, _ in given:
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous (an expanded, transposed or sliced view is not), "
                             f"got strides {tuple(t.stride())} for shape {tuple(t.shape)}")
    for name, t, _ in given:
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if t.device != q.device:
            raise ValueError(f"{name} is on {t.device}, q on {q.device}")


def _score(score, H: int):
    """The score spec of a score tuple, with its parameter's size checked against
    the H heads the kernels index it by (a prebuilt (ScoreSpec, keep) pair is
    taken as it is)."""
    if score is None:
        return make_score_spec("none")
    if isinstance(score, tuple) and isinstance(score[0], ScoreSpec):
        return score
    if isinstance(score, str):
        return make_score_spec(score)
    spec, keep = make_score_spec(score[0], score[1] if len(score) > 1 else None, d0=score[2] if len(score) > 2 else 0)
    need = {"softcap": 1, "alibi": H, "relbias": H * spec.bias_len}.get(score[0], 0)
    if keep and keep[0].numel() != need:
        raise ValueError(f"{score[0]} parameter has {keep[0].numel()} values, {need} needed for {H} heads")
    return spec, keep


def fa_forward(q, k, v, block_mask: BlockMask, score=None, scale: float = 0.0, out=None, lse=None, stream=None):
    """out [B,H,q_len,D] bf16 and lse [B,H,q_len] fp32."""
    _check_shapes(q, kv=(("k", k), ("v", v)), like_q=(("out", out),), lse=lse)
    B, H, q_len, D = q.shape
    kv_len = k.shape[2]
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(B, H, q_len, dtype=torch.float32, device=q.device)
    _check_storage(q, (("k", k, _BF16), ("v", v, _BF16), ("out", out, _BF16), ("lse", lse, _F32)))
    sspec, keep = _score(score, H)
    _check(_lib.fa_forward(_ptr(q), _ptr(k), _ptr(v), B, H, q_len, kv_len, D, ctypes.byref(block_mask.struct),
                           ctypes.byref(sspec), float(scale), _ptr(out), _ptr(lse), _stream(stream)), "fa_forward")
    return out, lse


def fa_forward_prepare_backward(q, k, v, block_mask: BlockMask, workspace, score=None, scale: float = 0.0,
                                out=None, lse=None, stream=None):
    """fa_forward that also sets ``workspace``'s dq accumulator to zero while it
    runs (uint8 CUDA tensor of at least fa_backward_workspace_bytes(B, H,
    q_len, D)); pass the same workspace to fa_backward_prepared."""
    _check_shapes(q, kv=(("k", k), ("v", v)), like_q=(("out", out),), lse=lse)
    B, H, q_len, D = q.shape
    kv_len = k.shape[2]
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(B, H, q_len, dtype=torch.float32, device=q.device)
    _check_storage(q, (("k", k, _BF16), ("v", v, _BF16), ("out", out, _BF16), ("lse", lse, _F32),
                       ("workspace", workspace, _U8)))
    sspec, keep = _score(score, H)
    _check(_lib.fa_forward_prepare_backward(_ptr(q), _ptr(k), _ptr(v), B, H, q_len, kv_len, D,
                                            ctypes.byref(block_mask.struct), ctypes.byref(sspec), float(scale),
                                            _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel(),
                                            _stream(stream)), "fa_forward_prepare_backward")
    return out, lse


def _backward_score(score, score_param_grad, H: int):
    """Score spec for the backward: a copy of the caller's, with the device
    pointer of ``score_param_grad`` (fp32, receives dL/dslope [H] for ALiBi or
    dL/dtable [H, L] for the learned relative-position bias)."""
    sspec, keep = _score(score, H)
    spec = ScoreSpec()
    spec.op, spec.param, spec.param_grad = sspec.op, sspec.param, None
    spec.bias_len, spec.bias_d0 = sspec.bias_len, sspec.bias_d0
    if score_param_grad is not None:
        g = score_param_grad
        n = H * sspec.bias_len if sspec.op == SCORE_OPS["relbias"] else H
        if g.dtype != torch.float32 or not g.is_cuda or not g.is_contiguous() or g.numel() != n:
            raise ValueError(f"score_param_grad must be a contiguous fp32 CUDA tensor of {n} elements")
        spec.param_grad = g.data_ptr()
    return spec, keep + [sspec]


def fa_forward_paged(q, k_pool, v_pool, page_table, block_mask: BlockMask, score=None, scale: float = 0.0, out=None,
                     lse=None, stream=None):
    """Forward over paged keys / values: k_pool, v_pool bf16 [H, n_pages * 128, D],
    page_table int32 [B, nkv] (page of each logical key tile).  out, lse as fa_forward."""
    _check_shapes(q, like_q=(("out", out),), lse=lse)
    B, H, q_len, D = q.shape
    kv_len = block_mask.struct.kv_len
    nkv = -(-kv_len // 128)
    if k_pool.dim() != 3 or k_pool.shape != v_pool.shape or k_pool.shape[0] != H or k_pool.shape[2] != D \
            or k_pool.shape[1] % 128 != 0:
        raise ValueError("k_pool / v_pool must be [H, n_pages * 128, D]")
    if page_table.dtype != torch.int32 or not page_table.is_cuda or not page_table.is_contiguous() \
            or tuple(page_table.shape) != (B, nkv):
        raise ValueError(f"page_table must be a contiguous int32 CUDA tensor [B, {nkv}]")
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(B, H, q_len, dtype=torch.float32, device=q.device)
    _check_storage(q, (("k_pool", k_pool, _BF16), ("v_pool", v_pool, _BF16), ("page_table", page_table, _I32),
                       ("out", out, _BF16), ("lse", lse, _F32)))
    sspec, keep = _score(score, H)
    _check(_lib.fa_forward_paged(_ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(page_table), k_pool.shape[1] // 128, B, H,
                                 q_len, kv_len, D, ctypes.byref(block_mask.struct), ctypes.byref(sspec), float(scale),
                                 _ptr(out), _ptr(lse), _stream(stream)), "fa_forward_paged")
    return out, lse


DECODE_MAX_Q = 16


def fa_forward_decode_workspace_bytes(B: int, H: int, q_len: int, kv_len: int, D: int) -> int:
    n = ctypes.c_size_t()
    _check(_lib.fa_forward_decode_workspace_bytes(B, H, q_len, kv_len, D, ctypes.byref(n)),
           "fa_forward_decode_workspace_bytes")
    return n.value


def fa_forward_decode(q, k, v, block_mask: BlockMask, score=None, scale: float = 0.0, page_table=None, out=None,
                      lse=None, workspace=None, stream=None, kv_len: Optional[int] = None):
    """Short-query forward (q_len <= 16) over the keys [0, kv_len): k, v
    [B, H, C, D] with C the block mask's kv_len; or, with an int32 page_table
    [B, nkv], pools [H, n_pages * 128, D].  kv_len defaults to C; a smaller one
    runs a block mask built for a bucketed cache length C on the current cache.
    out, lse as fa_forward."""
    _check_shapes(q, like_q=(("out", out),), lse=lse)
    B, H, q_len, D = q.shape
    cap = block_mask.struct.kv_len
    kv_len = cap if kv_len is None else int(kv_len)
    if not 1 <= kv_len <= cap:
        raise ValueError(f"kv_len {kv_len} must be in [1, {cap}] (the block mask's key length)")
    if q_len != block_mask.struct.q_len:
        raise ValueError(f"q has {q_len} rows; the block mask was built for q_len {block_mask.struct.q_len}")
    n_pages = 0
    if page_table is None and (tuple(k.shape) != (B, H, cap, D) or tuple(v.shape) != (B, H, cap, D)):
        raise ValueError(f"k and v must be [{B}, {H}, {cap}, {D}] (kv_len of the block mask)")
    if page_table is not None and v.shape != k.shape:
        raise ValueError("paged k and v pools must have the same shape")
    if page_table is not None:
        if page_table.dtype != torch.int32 or not page_table.is_cuda or not page_table.is_contiguous() \
                or tuple(page_table.shape) != (B, -(-cap // 128)):
            raise ValueError("page_table must be a contiguous int32 CUDA tensor [B, nkv]")
        if k.dim() != 3 or k.shape[1] % 128 != 0:
            raise ValueError("paged k / v must be [H, n_pages * 128, D]")
        n_pages = k.shape[1] // 128
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(B, H, q_len, dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = torch.empty(fa_forward_decode_workspace_bytes(B, H, q_len, kv_len, D), dtype=torch.uint8,
                                device=q.device)
    _check_storage(q, (("k", k, _BF16), ("v", v, _BF16), ("page_table", page_table, _I32), ("out", out, _BF16),
                       ("lse", lse, _F32), ("workspace", workspace, _U8)))
    sspec, keep = _score(score, H)
    _check(_lib.fa_forward_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(page_table), n_pages, B, H, q_len, kv_len, D,
                                  ctypes.byref(block_mask.struct), ctypes.byref(sspec), float(scale), _ptr(out),
                                  _ptr(lse), _ptr(workspace), workspace.numel(), _stream(stream)),
           "fa_forward_decode")
    return out, lse


def fa_backward_workspace_bytes(B: int, H: int, q_len: int, D: int) -> int:
    n = ctypes.c_size_t()
    _check(_lib.fa_backward_workspace_bytes(B, H, q_len, D, ctypes.byref(n)), "fa_backward_workspace_bytes")
    return n.value


def _backward_tensors(k, v, out, lse, dout, dq, dk, dv):
    return (("k", k, _BF16), ("v", v, _BF16), ("out", out, _BF16), ("lse", lse, _F32), ("dout", dout, _BF16),
            ("dq", dq, _BF16), ("dk", dk, _BF16), ("dv", dv, _BF16))


def fa_backward(q, k, v, out, lse, dout, block_mask: BlockMask, score=None, scale: float = 0.0,
                dq=None, dk=None, dv=None, workspace=None, stream=None, score_param_grad=None):
    """dq, dk, dv (bf16, shaped like q, k, v); with ALiBi, ``score_param_grad``
    (fp32 [H] CUDA tensor) receives dL/dslope of every head, and with the
    learned relative-position bias (fp32 [H, L]) dL/dtable."""
    _check_shapes(q, kv=(("k", k), ("v", v), ("dk", dk), ("dv", dv)),
                  like_q=(("out", out), ("dout", dout), ("dq", dq)), lse=lse)
    B, H, q_len, D = q.shape
    kv_len = k.shape[2]
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if workspace is None:
        workspace = torch.empty(fa_backward_workspace_bytes(B, H, q_len, D), dtype=torch.uint8, device=q.device)
    _check_storage(q, _backward_tensors(k, v, out, lse, dout, dq, dk, dv) + (("workspace", workspace, _U8),))
    sspec, keep = _backward_score(score, score_param_grad, H)
    _check(_lib.fa_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout), B, H, q_len, kv_len, D,
                            ctypes.byref(block_mask.struct), ctypes.byref(sspec), float(scale), _ptr(dq), _ptr(dk),
                            _ptr(dv), _ptr(workspace), workspace.numel(), _stream(stream)), "fa_backward")
    return dq, dk, dv


def fa_backward_prepared(q, k, v, out, lse, dout, block_mask: BlockMask, workspace, score=None, scale: float = 0.0,
                         dq=None, dk=None, dv=None, stream=None, score_param_grad=None):
    """fa_backward on a workspace prepared by fa_forward_prepare_backward (its
    dq accumulator taken as zero)."""
    _check_shapes(q, kv=(("k", k), ("v", v), ("dk", dk), ("dv", dv)),
                  like_q=(("out", out), ("dout", dout), ("dq", dq)), lse=lse)
    B, H, q_len, D = q.shape
    kv_len = k.shape[2]
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _check_storage(q, _backward_tensors(k, v, out, lse, dout, dq, dk, dv) + (("workspace", workspace, _U8),))
    sspec, keep = _backward_score(score, score_param_grad, H)
    _check(_lib.fa_backward_prepared(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout), B, H, q_len,
                                     kv_len, D, ctypes.byref(block_mask.struct), ctypes.byref(sspec), float(scale),
                                     _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace), workspace.numel(),
                                     _stream(stream)), "fa_backward_prepared")
    return dq, dk, dv


def fa_backward_noalloc(q, k, v, out, lse, dout, block_mask: BlockMask, score=None, scale: float = 0.0,
                        dq=None, dk=None, dv=None, stream=None, score_param_grad=None):
    """fa_backward without a workspace: for callers that cannot allocate device
    memory at call time (the library's static scratch holds the fp32 dq
    accumulator; see include/fa.h for the size limit and the sharing rules)."""
    _check_shapes(q, kv=(("k", k), ("v", v), ("dk", dk), ("dv", dv)),
                  like_q=(("out", out), ("dout", dout), ("dq", dq)), lse=lse)
    B, H, q_len, D = q.shape
    kv_len = k.shape[2]
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _check_storage(q, _backward_tensors(k, v, out, lse, dout, dq, dk, dv))
    sspec, keep = _backward_score(score, score_param_grad, H)
    _check(_lib.fa_backward_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout), B, H, q_len, kv_len,
                                    D, ctypes.byref(block_mask.struct), ctypes.byref(sspec), float(scale), _ptr(dq),
                                    _ptr(dk), _ptr(dv), _stream(stream)), "fa_backward_noalloc")
    return dq, dk, dv


def fa_get_status(block_mask: BlockMask, clear: bool = True, stream=None) -> int:
    return _lib.fa_get_status(ctypes.byref(block_mask.struct), 1 if clear else 0, _stream(stream))


def fa_block_mask_summary(block_mask: BlockMask, stream=None):
    counts = (ctypes.c_int64 * 3)()
    _check(_lib.fa_block_mask_summary(ctypes.byref(block_mask.struct), ctypes.byref(counts), _stream(stream)),
           "fa_block_mask_summary")
    return tuple(int(c) for c in counts)


def fa_status_string(code: int) -> str:
    return _lib.fa_status_string(code).decode()


def fa_version() -> int:
    return int(_lib.fa_version())
