"""Paged KV-cache attention for GB300 (sm_103a).

``ops`` binds libpagedkv.so (kv_store, paged_decode_attn,
paged_varlen_prefill_attn); ``metadata`` builds the host-side int32 arrays
they consume; ``workloads`` draws seeded synthetic inputs.
"""

from . import metadata, ops, workloads  # noqa: F401
from .ops import (  # noqa: F401
    copy_blocks,
    decode_workspace,
    decode_workspace_bytes,
    device_error,
    kv_store,
    kv_store_fp8,
    paged_decode_attn,
    paged_decode_attn_fp8,
    paged_decode_attn_noalloc,
    paged_varlen_prefill_attn,
    paged_verify_attn,
    prefill_workspace,
    prefill_workspace_bytes,
)

__all__ = [
    "copy_blocks", "kv_store", "kv_store_fp8", "paged_decode_attn", "paged_decode_attn_fp8",
    "paged_decode_attn_noalloc", "paged_varlen_prefill_attn", "paged_verify_attn", "decode_workspace",
    "decode_workspace_bytes", "prefill_workspace", "prefill_workspace_bytes", "device_error", "metadata", "ops",
    "workloads",
]
