"""GB300 (sm_103a) library for attention of new tokens against a read-only
cached KV segment: gist-compressed items gathered by id, or a paged cache read
through a block table.

The compute lives in ``_lib/libgistattn.so`` (C ABI in include/gist_attn.h);
``binding`` marshals torch tensors into it; ``workloads`` draws seeded
synthetic inputs.  The library is loaded on first use and every call fails
loudly if it has not been built.
"""
from .binding import (FLAG_PREROTATED, GistAttnError, STATUS_BAD_BLOCK, STATUS_RANGE, STATUS_TIMEOUT, gist_attn_fwd,
                      gist_attn_fwd_block_mass, gist_attn_fwd_fp8kv, gist_attn_fwd_gist_mask,
                      gist_attn_fwd_ws, workspace_bytes,
                      gist_kv_append, gist_kv_store, gist_out_proj, gist_qkv_rope,
                      gist_attn_gather_debug, kv_bytes_batch, kv_bytes_per_item,
                      kv_bytes_per_position, load_library, status_string)

__all__ = ["FLAG_PREROTATED", "GistAttnError", "STATUS_BAD_BLOCK", "STATUS_RANGE", "STATUS_TIMEOUT", "gist_attn_fwd", "gist_attn_fwd_fp8kv",
           "gist_attn_fwd_block_mass", "gist_attn_fwd_gist_mask", "gist_attn_fwd_ws", "workspace_bytes",
           "gist_kv_append", "gist_kv_store",
           "gist_qkv_rope", "gist_out_proj",
           "gist_attn_gather_debug", "kv_bytes_batch", "kv_bytes_per_item",
           "kv_bytes_per_position", "load_library", "status_string"]
