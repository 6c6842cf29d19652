"""block_sparse_masked_fa_gb300: tile-sparse masked softmax attention for one GB300 (sm_103a).

The CUDA library (``libfa_gb300.so``, C ABI in ``include/fa.h``) holds the
whole hot path: the block-mask builder, the forward and the backward.  This
package only marshals torch tensors into that ABI; importing it fails when the
library has not been built (there is no CPU fallback).
"""
from .binding import (  # noqa: F401
    EXPORTED,
    BlockMask,
    FaError,
    fa_backward,
    fa_backward_noalloc,
    fa_backward_prepared,
    fa_backward_workspace_bytes,
    fa_block_mask_bytes,
    fa_block_mask_from_kv_blocks,
    fa_block_mask_summary,
    fa_create_block_mask,
    fa_forward,
    fa_forward_decode,
    fa_forward_decode_workspace_bytes,
    fa_forward_paged,
    fa_forward_prepare_backward,
    fa_get_status,
    fa_status_string,
    fa_version,
    make_mask_spec,
    make_score_spec,
)
