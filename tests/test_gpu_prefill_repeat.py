"""The persistent prefill kernel hands out its work through a queue counter
that every call resets when its last block finishes: many calls in a row, of
different sizes, must all do all of their work (bit-identical results, no
device error)."""
import pytest
import torch

import paged_kv_cache_out_gb300 as pkv
from synth import make_config, make_inputs
from tests.gpu_util import Run

pytestmark = pytest.mark.gpu


def test_many_calls_of_two_sizes_repeat_bit_for_bit():
    big = Run(make_config("ragged_prefill", seed=3)).store()
    small = Run(make_inputs(seed=4, Hq=16, Hkv=8, d=128, page_size=16, new_lens=[70, 5, 200],
                            prefix_lens=[30, 0, 64])).store()
    ref_big, ref_small = big.prefill(), small.prefill()
    assert big.dev_status() == 0 and small.dev_status() == 0
    out_big, out_small = torch.empty_like(ref_big), torch.empty_like(ref_small)
    for i in range(300):
        big.prefill(out=out_big)
        small.prefill(out=out_small)
        if i % 50 == 49:
            assert big.dev_status() == 0 and small.dev_status() == 0
            assert torch.equal(out_big.view(torch.int16), ref_big.view(torch.int16))
            assert torch.equal(out_small.view(torch.int16), ref_small.view(torch.int16))


def test_dirty_workspace_is_reported_and_left_clean():
    """A workspace whose counters are not zero when a call starts (never
    cleared, or shared with a call running at the same time) makes that call
    raise PKV_DEV_BAD_WORKSPACE; the call still returns the counters to zero,
    so the next call on the same workspace is correct."""
    r = Run(make_config("ragged_prefill", seed=5)).store()
    ref = r.prefill()
    assert r.dev_status() == 0
    r.pws.view(torch.int32)[0] = 5          # as if 5 queue entries were already taken
    r.prefill()
    assert r.dev_status() & pkv.DEV_BAD_WORKSPACE
    assert int(r.pws.view(torch.int32)[:3].abs().sum().item()) == 0
    r.status.zero_()
    out = r.prefill()
    assert r.dev_status() == 0
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
