"""ctypes binding of libpkv.so: the same three calls, taking torch tensors.

This module only marshals arguments (pointers, sizes, the current CUDA stream)
and turns status codes into exceptions; every step of the computation runs in
the library's CUDA kernels.  There is no fallback: when the library is missing
the calls raise.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from .build import LIB_PATH

_lock = threading.Lock()
_lib = None

OK, EINVAL, EUNSUPPORTED, ECUDA = 0, 1, 2, 3
DEV_BAD_SLOT, DEV_BAD_PAGE, DEV_BAD_SEQLEN, DEV_BAD_CUSEQ, DEV_TIMEOUT = 1, 2, 4, 8, 16
DEV_BAD_WORKSPACE, DEV_BAD_SHARED = 32, 64

_P = ctypes.c_void_p
_I32, _I64, _F32, _SZ = ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t

SIGNATURES = {
    "pkv_status_string": ([_I32], ctypes.c_char_p),
    "pkv_version": ([], _I32),
    "pkv_kv_store": ([_P, _P, _P, _I64, _P, _P, _I64, _I32, _I32, _I32, _P, _P], _I32),
    "pkv_decode_workspace_size": ([_I32, _I32, _I32, _I32], _SZ),
    "pkv_paged_decode_attn": ([_P, _P, _P, _P, _I64, _P, _I32, _I32, _I32, _I32, _I32, _I64,
                               _F32, _P, _SZ, _P, _P, _P], _I32),
    "pkv_paged_decode_attn_store": ([_P, _P, _P, _P, _P, _P, _P, _I64, _P, _I32, _I32, _I32,
                                     _I32, _I32, _I64, _F32, _P, _SZ, _P, _P, _P], _I32),
    "pkv_paged_prefill_attn": ([_P, _P, _P, _P, _P, _I64, _P, _I32, _I64, _I32, _I32, _I32,
                                _I32, _I32, _I64, _F32, _P, _SZ, _P, _P, _P], _I32),
    "pkv_prefill_workspace_size": ([], _SZ),
    "pkv_paged_prefill_attn_shared": ([_P, _P, _P, _P, _P, _I64, _P, _I32, _I64, _I32, _I32, _I32,
                                       _I32, _I32, _I64, _F32, _P, _P, _I32, _I32, _P, _SZ, _P, _P,
                                       _P], _I32),
    "pkv_paged_decode_attn_noalloc": ([_P, _P, _P, _P, _I64, _P, _I32, _I32, _I32, _I32, _I32,
                                       _I64, _F32, _P, _P, _P], _I32),
}


class PkvError(RuntimeError):
    def __init__(self, fn: str, status: int):
        msg = load_library().pkv_status_string(status).decode()
        super().__init__(f"{fn} returned {status} ({msg})")
        self.status = status


def load_library(path: str | None = None):
    """Load libpkv.so (built by ``paged_kv_cache_out_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or LIB_PATH
            if not os.path.exists(p):
                raise RuntimeError(f"the CUDA library {p} is not built: run "
                                   "paged_kv_cache_out_gb300.build.build() first")
            lib = ctypes.CDLL(p)
            for name, (args, res) in SIGNATURES.items():
                f = getattr(lib, name)
                f.argtypes, f.restype = args, res
            _lib = lib
    return _lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(fn, status):
    if status != OK:
        raise PkvError(fn, status)


def _bf16(t, name):
    if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA bfloat16 tensor")


def _i32(t, name):
    if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA int32 tensor")


def kv_store(k_new, v_new, out_loc, k_cache, v_cache, dev_status=None, stream=None):
    """Copy new K/V rows [T, Hkv, d] into pool slots out_loc (pool [P, ps, Hkv, d])."""
    for t, n in ((k_new, "k_new"), (v_new, "v_new"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _bf16(t, n)
    _i32(out_loc, "out_loc")
    P, ps, Hkv, d = k_cache.shape
    T = out_loc.shape[0]
    if k_new.shape != (T, Hkv, d) or v_new.shape != (T, Hkv, d) or v_cache.shape != k_cache.shape:
        raise ValueError("shape mismatch")
    st = load_library().pkv_kv_store(_ptr(k_new), _ptr(v_new), _ptr(out_loc), T, _ptr(k_cache),
                                     _ptr(v_cache), P, ps, Hkv, d, _ptr(dev_status), _stream(stream))
    _check("pkv_kv_store", st)


def decode_workspace_size(batch, num_q_heads, num_kv_heads, head_dim) -> int:
    return int(load_library().pkv_decode_workspace_size(batch, num_q_heads, num_kv_heads, head_dim))


def decode_workspace(batch, num_q_heads, num_kv_heads, head_dim, device=None):
    n = decode_workspace_size(batch, num_q_heads, num_kv_heads, head_dim)
    return torch.empty(max(n, 16), dtype=torch.uint8, device=device or "cuda")


def paged_decode_attn(q, k_cache, v_cache, page_table, seq_lens, softmax_scale, workspace=None,
                      dev_status=None, out=None, stream=None):
    """Decode attention: q [B, Hq, d] over the pool through page_table [B, stride]."""
    _bf16(q, "q"), _bf16(k_cache, "k_cache"), _bf16(v_cache, "v_cache")
    _i32(seq_lens, "seq_lens")
    if page_table.dtype != torch.int32 or page_table.dim() != 2 or page_table.stride(1) != 1:
        raise ValueError("page_table must be a 2-D int32 tensor with unit column stride")
    B, Hq, d = q.shape
    P, ps, Hkv, d2 = k_cache.shape
    if d2 != d or v_cache.shape != k_cache.shape or seq_lens.shape[0] != B:
        raise ValueError("shape mismatch")
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        workspace = decode_workspace(B, Hq, Hkv, d, q.device)
    st = load_library().pkv_paged_decode_attn(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(page_table), page_table.stride(0),
        _ptr(seq_lens), B, Hq, Hkv, d, ps, P, float(softmax_scale), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(dev_status), _ptr(out), _stream(stream))
    _check("pkv_paged_decode_attn", st)
    return out


def paged_decode_attn_store(q, k_new, v_new, out_loc, k_cache, v_cache, page_table, seq_lens,
                            softmax_scale, workspace=None, dev_status=None, out=None, stream=None):
    """kv_store of the decode rows k_new/v_new [B, Hkv, d] at out_loc [B] fused
    into decode attention (same results as kv_store followed by paged_decode_attn)."""
    for t, n in ((q, "q"), (k_new, "k_new"), (v_new, "v_new"), (k_cache, "k_cache"),
                 (v_cache, "v_cache")):
        _bf16(t, n)
    _i32(seq_lens, "seq_lens"), _i32(out_loc, "out_loc")
    if page_table.dtype != torch.int32 or page_table.dim() != 2 or page_table.stride(1) != 1:
        raise ValueError("page_table must be a 2-D int32 tensor with unit column stride")
    B, Hq, d = q.shape
    P, ps, Hkv, d2 = k_cache.shape
    if (d2 != d or v_cache.shape != k_cache.shape or seq_lens.shape[0] != B
            or out_loc.shape[0] != B or k_new.shape != (B, Hkv, d) or v_new.shape != (B, Hkv, d)):
        raise ValueError("shape mismatch")
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        workspace = decode_workspace(B, Hq, Hkv, d, q.device)
    st = load_library().pkv_paged_decode_attn_store(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(out_loc), _ptr(k_cache), _ptr(v_cache),
        _ptr(page_table), page_table.stride(0), _ptr(seq_lens), B, Hq, Hkv, d, ps, P,
        float(softmax_scale), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _ptr(dev_status), _ptr(out), _stream(stream))
    _check("pkv_paged_decode_attn_store", st)
    return out


def prefill_workspace(device=None):
    """A zero-filled prefill workspace (the queue counters must start at zero;
    every call leaves them at zero)."""
    n = int(load_library().pkv_prefill_workspace_size())
    return torch.zeros(max(n, 16), dtype=torch.uint8, device=device or "cuda")


def paged_prefill_attn(q, cu_seqlens_q, k_cache, v_cache, page_table, seq_lens, softmax_scale,
                       max_q_len, workspace=None, dev_status=None, out=None, stream=None):
    """Ragged causal prefill: q [Tq, Hq, d] with offsets cu_seqlens_q [B+1].

    workspace: from prefill_workspace(); calls that may overlap on the GPU
    need separate workspaces.  Without one, a fresh zeroed one is made."""
    _bf16(q, "q"), _bf16(k_cache, "k_cache"), _bf16(v_cache, "v_cache")
    _i32(seq_lens, "seq_lens"), _i32(cu_seqlens_q, "cu_seqlens_q")
    if page_table.dtype != torch.int32 or page_table.dim() != 2 or page_table.stride(1) != 1:
        raise ValueError("page_table must be a 2-D int32 tensor with unit column stride")
    Tq, Hq, d = q.shape
    P, ps, Hkv, d2 = k_cache.shape
    B = seq_lens.shape[0]
    if d2 != d or v_cache.shape != k_cache.shape or cu_seqlens_q.shape[0] != B + 1:
        raise ValueError("shape mismatch")
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        workspace = prefill_workspace(q.device)
    st = load_library().pkv_paged_prefill_attn(
        _ptr(q), _ptr(cu_seqlens_q), _ptr(k_cache), _ptr(v_cache), _ptr(page_table),
        page_table.stride(0), _ptr(seq_lens), B, Tq, int(max_q_len), Hq, Hkv, d, ps, P,
        float(softmax_scale), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _ptr(dev_status), _ptr(out), _stream(stream))
    _check("pkv_paged_prefill_attn", st)
    return out


def paged_prefill_attn_shared(q, cu_seqlens_q, k_cache, v_cache, page_table, seq_lens,
                              softmax_scale, max_q_len, prefix_group_start, prefix_len,
                              max_group_tokens, workspace=None, dev_status=None, out=None,
                              stream=None):
    """Ragged causal prefill for requests that share cached prefixes.

    prefix_group_start [n_groups + 1] int32: group g is requests
    prefix_group_start[g] .. prefix_group_start[g+1]-1 (the groups partition
    the batch in order); prefix_len [n_groups] int32: the keys they share
    (whole pages, listed first in every member's page-table row; 0 for a
    request that shares nothing).  max_group_tokens bounds the new tokens of
    any group.  The result equals paged_prefill_attn on the same arguments.
    workspace: from prefill_workspace()."""
    _bf16(q, "q"), _bf16(k_cache, "k_cache"), _bf16(v_cache, "v_cache")
    _i32(seq_lens, "seq_lens"), _i32(cu_seqlens_q, "cu_seqlens_q")
    _i32(prefix_group_start, "prefix_group_start"), _i32(prefix_len, "prefix_len")
    if page_table.dtype != torch.int32 or page_table.dim() != 2 or page_table.stride(1) != 1:
        raise ValueError("page_table must be a 2-D int32 tensor with unit column stride")
    Tq, Hq, d = q.shape
    P, ps, Hkv, d2 = k_cache.shape
    B = seq_lens.shape[0]
    n_groups = prefix_len.shape[0]
    if (d2 != d or v_cache.shape != k_cache.shape or cu_seqlens_q.shape[0] != B + 1
            or prefix_group_start.shape[0] != n_groups + 1):
        raise ValueError("shape mismatch")
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        workspace = prefill_workspace(q.device)
    st = load_library().pkv_paged_prefill_attn_shared(
        _ptr(q), _ptr(cu_seqlens_q), _ptr(k_cache), _ptr(v_cache), _ptr(page_table),
        page_table.stride(0), _ptr(seq_lens), B, Tq, int(max_q_len), Hq, Hkv, d, ps, P,
        float(softmax_scale), _ptr(prefix_group_start), _ptr(prefix_len), n_groups,
        int(max_group_tokens), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _ptr(dev_status), _ptr(out), _stream(stream))
    _check("pkv_paged_prefill_attn_shared", st)
    return out
