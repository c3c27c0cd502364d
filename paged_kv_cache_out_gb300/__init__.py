"""Attention over a paged KV cache for NVIDIA GB300 (sm_103a).

The CUDA library ``libpkv.so`` (C ABI declared in ``include/pkv.h``) holds the
kernels; this package builds it in-tree and binds it with ctypes.
"""
from .binding import (  # noqa: F401
    DEV_BAD_CUSEQ,
    DEV_BAD_PAGE,
    DEV_BAD_SEQLEN,
    DEV_BAD_SHARED,
    DEV_BAD_SLOT,
    DEV_BAD_WORKSPACE,
    DEV_TIMEOUT,
    PkvError,
    decode_workspace,
    decode_workspace_size,
    kv_store,
    load_library,
    paged_decode_attn,
    paged_decode_attn_store,
    paged_prefill_attn,
    paged_prefill_attn_shared,
    prefill_workspace,
)
