"""GB300 (sm_103a) exact attention: FlashAttention-style prefill (forward and backward) and paged-KV decode.

The compute path is the CUDA shared library built from ``csrc/`` (C-ABI declared in
``include/attn_gb300.h``).  ``binding`` marshals torch tensors into that ABI; it has no
fallback: if the library is missing, every call raises.
"""
from .binding import (  # noqa: F401
    AttnError,
    attn_bwd,
    attn_bwd_workspace_size,
    attn_check_device_status,
    attn_last_device_status,
    attn_selftest_bounded_wait,
    attn_fwd,
    attn_fwd_gqa,
    attn_fwd_kvlen,
    attn_status_string,
    kv_quantize_fp8,
    library_path,
    load_library,
    paged_attn_decode,
    paged_attn_decode_fp8,
    paged_attn_decode_gqa,
    paged_attn_decode_noalloc,
    paged_attn_prefill,
    paged_attn_prefill_fp8,
    paged_kv_append,
    paged_kv_append_fp8,
    paged_attn_decode_gqa_workspace_size,
    paged_attn_decode_workspace_size,
    paged_attn_decode_workspace_size_ctx,
)
