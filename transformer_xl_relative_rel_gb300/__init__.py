"""GB300-native Transformer-XL segment-level relative attention.

The compute lives in ``libtxl.so`` (hand-written sm_103a CUDA behind the C-ABI
declared in ``include/txl.h``); ``abi`` is the thin ctypes binding with the same
entry-point names.  Importing this package does not load the library; the first
call does, and raises ``TxlError`` if it was not built.
"""
from .abi import (TxlError, TXL_F32, TXL_BF16, rel_attn_fwd, rel_attn_fwd_ring,  # noqa: F401
                  rel_attn_fwd_padded, project_heads, project_qkv, project_qkv_cells, rel_table, mem_update, ring_append, check,
                  load_library, library_path, status_string, rel_attn_bwd,
                  rel_attn_bwd_workspace_bytes, rel_attn_fwd_mem, rel_attn_fwd_mem_cells, rel_attn_fwd_plan,
                  rel_attn_fwd_noalloc, selftest_wait)

__all__ = ["TxlError", "TXL_F32", "TXL_BF16", "rel_attn_fwd", "rel_attn_fwd_ring", "mem_update",
           "ring_append", "rel_attn_fwd_padded", "project_heads", "project_qkv", "project_qkv_cells", "rel_table", "check", "load_library",
           "library_path", "status_string", "rel_attn_bwd", "rel_attn_bwd_workspace_bytes",
           "rel_attn_fwd_mem", "rel_attn_fwd_mem_cells", "rel_attn_fwd_plan", "rel_attn_fwd_noalloc", "selftest_wait"]
