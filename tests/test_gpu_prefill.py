"""Ragged causal prefill on the GPU against the oracle (max abs error <= 2e-2)."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_out_gb300 as pkv
from synth import make_inputs
from tests.gpu_util import TOL, Run, as_f64, max_err

pytestmark = pytest.mark.gpu


def check(x, threads=8):
    r = Run(x).store()
    out = r.prefill()
    assert r.dev_status() == 0
    ref = oracle.run_inputs(x, threads=threads)
    err = max_err(as_f64(out), ref)
    assert err <= TOL, err
    return out, err


def test_basic():
    check(make_inputs(seed=1, Hq=16, Hkv=8, d=128, page_size=16, new_lens=[70, 5, 130],
                      prefix_lens=[33, 0, 200]))


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("ps", [1, 16, 256])
def test_shapes(d, G, ps):
    check(make_inputs(seed=40 + G, Hq=2 * G, Hkv=2, d=d, page_size=ps,
                      new_lens=[1, 17, 128, 129, 300], prefix_lens=[0, 100, 5, 256, 77]))


@pytest.mark.parametrize("ps", [2, 4, 8, 32, 64, 128])
def test_other_page_sizes(ps):
    check(make_inputs(seed=50, Hq=16, Hkv=8, d=128, page_size=ps, new_lens=[200, 33],
                      prefix_lens=[60, 400]))


def test_long_prefix_short_suffix():
    check(make_inputs(seed=51, Hq=16, Hkv=8, d=128, page_size=16, new_lens=[200, 1],
                      prefix_lens=[3000, 5000]))


def test_empty_request_in_the_middle():
    check(make_inputs(seed=52, Hq=16, Hkv=8, d=128, page_size=16, new_lens=[40, 0, 90],
                      prefix_lens=[10, 30, 0]))


def test_decode_shaped_prefill_matches_decode_kernel():
    lens = np.array([77, 300, 1024])
    x = make_inputs(seed=53, Hq=16, Hkv=8, d=128, page_size=16, new_lens=np.ones(3, np.int64),
                    prefix_lens=lens - 1)
    r = Run(x).store()
    a = as_f64(r.prefill())
    b = as_f64(r.decode())
    assert r.dev_status() == 0
    ref = oracle.run_inputs(x)
    assert max_err(a, ref) <= TOL and max_err(b, ref) <= TOL


def test_bad_page_is_flagged():
    x = make_inputs(seed=54, Hq=16, Hkv=8, d=128, page_size=16, new_lens=[50, 60], prefix_lens=[0, 10])
    r = Run(x).store()
    r.page_table[0, 1] = -3
    out = r.prefill()
    assert r.dev_status() & pkv.DEV_BAD_PAGE
    got = as_f64(out)
    assert np.isnan(got[:50]).all()
    assert max_err(got[50:], oracle.run_inputs(x)[50:]) <= TOL


def test_bad_seq_len_is_flagged():
    x = make_inputs(seed=55, Hq=16, Hkv=8, d=128, page_size=16, new_lens=[50, 60], prefix_lens=[0, 10])
    r = Run(x).store()
    r.seq_lens[1] = 20          # fewer keys than new tokens
    out = r.prefill()
    assert r.dev_status() & pkv.DEV_BAD_SEQLEN
    got = as_f64(out)
    assert np.isnan(got[50:]).all()
    assert max_err(got[:50], oracle.run_inputs(x)[:50]) <= TOL


def test_deterministic():
    x = make_inputs(seed=56, Hq=16, Hkv=8, d=128, page_size=16, new_lens=[333, 70], prefix_lens=[100, 0])
    r = Run(x).store()
    a, b = r.prefill(), r.prefill()
    torch.cuda.synchronize()
    assert torch.equal(a, b)
