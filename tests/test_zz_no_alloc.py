"""Decode attention through the entry point that allocates nothing.

pkv_paged_decode_attn_noalloc serves callers that cannot allocate device
memory for a workspace (a runtime that plans all of its memory ahead, a
plugin that only receives its inputs and outputs): it keeps its scratch in a
fixed array inside the library.  This file is collected last so that a run
stopping at the first failure has run every other test before it.  Two calls
in a row, on different inputs, must each give bit for bit what the regular
entry point gives with a caller-provided workspace (the same kernels run on
the same inputs), and match the oracle.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_out_gb300 as pkv
from synth import make_inputs
from tests.gpu_util import TOL, Run, as_f64, max_err

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 4194304  # PKV_NOALLOC_SCRATCH_BYTES in include/pkv.h


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
        x = _inputs(seed)
        r = Run(x).store()
        ref = r.decode()                      # regular entry point, torch-allocated workspace
        out = torch.full_like(ref, float("nan"))
        assert _call_noalloc(r, out) == 0
        assert r.dev_status() == 0
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
        assert max_err(as_f64(out), oracle.run_inputs(x)) <= TOL


def test_every_supported_shape_fits_the_scratch_on_this_gpu():
    lib = pkv.load_library()
    for d in (64, 128):
        for G in (1, 2, 4, 8):
            need = lib.pkv_decode_workspace_size(4096, 8 * G, 8, d)  # the largest batch
            assert 0 < need <= SCRATCH_BYTES, (d, G, need)


def test_unsupported_gqa_ratio_is_rejected_without_a_launch():
    lib = pkv.load_library()
    null = ctypes.c_void_p(0x100)   # never dereferenced: the shape check comes first
    # 16 query heads per KV head is not a built shape
    st = lib.pkv_paged_decode_attn_noalloc(null, null, null, null, 64, null, 4096, 128, 8, 128, 16,
                                           1024, 0.1, None, null, None)
    assert st == pkv.binding.EUNSUPPORTED
