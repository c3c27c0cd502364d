"""Decode attention through the entry point that allocates nothing.

pkv_paged_decode_attn_noalloc serves callers that cannot allocate device
memory for a workspace (a runtime that plans all of its memory ahead, a
plugin that only receives its inputs and outputs): it keeps its scratch in a
fixed array inside the library.  This file is collected last so that a run
stopping at the first failure has run every other test before it.  Two calls
in a row, on different inputs, must each match the regular entry point with a
caller-provided workspace.
"""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_cache_out_gb300 as pkv
from synth import make_inputs
from tests.gpu_util import TOL, Run, as_f64

pytestmark = pytest.mark.gpu


def _call_noalloc(r, out):
    lib = pkv.load_library()
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    x = r.x
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.pkv_paged_decode_attn_noalloc(
        ptr(r.q), ptr(r.k), ptr(r.v), ptr(r.page_table), r.page_table.stride(0), ptr(r.seq_lens),
        x.B, x.Hq, x.Hkv, x.d, x.page_size, x.num_pages, float(x.scale), ptr(r.status), ptr(out),
        stream)


def _inputs(seed):
    lens = np.random.default_rng(seed).integers(1, 6000, size=24)
    lens[0] = 20000  # one long sequence: its keys are split over many blocks
    return make_inputs(seed=seed, Hq=16, Hkv=8, d=128, page_size=16,
                       new_lens=np.ones(len(lens), np.int64), prefix_lens=lens - 1)


def test_noalloc_matches_workspace_entry_point_twice():
    for seed in (70, 71):
        r = Run(_inputs(seed)).store()
        ref = r.decode()                      # regular entry point, torch-allocated workspace
        out = torch.full_like(ref, float("nan"))
        assert _call_noalloc(r, out) == 0
        assert r.dev_status() == 0
        got, want = as_f64(out), as_f64(ref)
        assert np.isfinite(got).all()
        assert float(np.abs(got - want).max()) <= TOL


def test_noalloc_rejects_sizes_beyond_its_scratch():
    lib = pkv.load_library()
    # 16 query heads per KV head at head_dim 128 need more than the fixed scratch
    need = lib.pkv_decode_workspace_size(4096, 128, 8, 128)
    assert need > 4194304
    null = ctypes.c_void_p(0x100)   # never dereferenced: the size check comes first
    st = lib.pkv_paged_decode_attn_noalloc(null, null, null, null, 64, null, 4096, 128, 8, 128, 16,
                                           1024, 0.1, None, null, None)
    assert st == pkv.binding.EUNSUPPORTED
