"""XAttention block-sparse chunked prefill for GB300 (sm_103a).

The compute lives in libbsxattn.so (hand-written CUDA, C ABI declared in
include/bsxattn.h).  This package holds the ctypes binding (same names as the
C entry points), the in-tree build script and the seeded input generator.
Importing the package does not load the library; the first call does, and it
raises if the library has not been built.
"""
from ._lib import (  # noqa: F401
    BSX_F8E4M3,
    BSX_FORCE_FIRST_LAST,
    BSX_STEP_E4M3_ESTIMATE,
    BSX_STEP_FUSED,
    BSX_STEP_OFFLOAD,
    BsxChunkBuffers,
    BsxError,
    BsxShape,
    bsx_bsa_prefill,
    bsx_bsa_prefill_split,
    bsx_chunk_prefill,
    bsx_chunk_prefill_workspace_bytes,
    bsx_chunk_step,
    bsx_chunk_step_host,
    bsx_cpu_block_mask,
    bsx_debug_drop_ring_item,
    bsx_debug_fused_skip_row,
    bsx_estimate_workspace_bytes,
    bsx_last_error,
    bsx_map_mask_to_cpu_blocks,
    bsx_merge_attn,
    bsx_quantize_e4m3,
    bsx_version,
    bsx_xattn_estimate,
    bsx_xattn_estimate_noalloc,
    load,
    make_chunk_buffers,
    shape_of,
)
