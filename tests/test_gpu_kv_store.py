"""kv_store on the GPU against the oracle: bit-exact."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_out_gb300 as pkv
from synth import make_config, make_inputs
from tests.gpu_util import Run, to_dev, to_host_bits

pytestmark = pytest.mark.gpu


def _oracle_pool(x, out_loc=None):
    k, v = x.k_cache.copy(), x.v_cache.copy()
    oracle.kv_store(x.k_new, x.v_new, x.out_loc if out_loc is None else out_loc, k, v)
    return k, v


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_tiny_decode_store_bit_exact(seed):
    x = make_config("tiny_decode", seed=seed)
    r = Run(x).store()
    assert r.dev_status() == 0
    k, v = _oracle_pool(x)
    assert np.array_equal(to_host_bits(r.k), k)
    assert np.array_equal(to_host_bits(r.v), v)


@pytest.mark.parametrize("Hkv,d,ps", [(8, 128, 16), (8, 64, 256), (2, 64, 1), (1, 128, 4), (4, 64, 32)])
def test_prefill_store_bit_exact(Hkv, d, ps):
    x = make_inputs(seed=3, Hq=Hkv * 2, Hkv=Hkv, d=d, page_size=ps, new_lens=[300, 1, 77, 0, 513],
                    prefix_lens=[10, 0, 200, 5, 31])
    r = Run(x).store()
    assert r.dev_status() == 0
    k, v = _oracle_pool(x)
    assert np.array_equal(to_host_bits(r.k), k)
    assert np.array_equal(to_host_bits(r.v), v)


def test_negative_slots_are_skipped_and_bad_slots_flagged():
    x = make_inputs(seed=4, Hq=16, Hkv=8, d=128, page_size=16, new_lens=[40, 9], prefix_lens=[3, 0])
    loc = x.out_loc.copy()
    loc[3] = -1
    loc[7] = -5
    bad = loc.copy()
    bad[11] = x.num_pages * x.page_size          # one past the pool
    r = Run(x)
    pkv.kv_store(r.k_new, r.v_new, to_dev(bad), r.k, r.v, dev_status=r.status)
    assert r.dev_status() == pkv.DEV_BAD_SLOT
    skip = bad.copy()
    skip[11] = -1                                 # the bad token is skipped, the rest stored
    k, v = _oracle_pool(x, skip)
    assert np.array_equal(to_host_bits(r.k), k)
    assert np.array_equal(to_host_bits(r.v), v)


def test_large_store_matches_oracle_sampled():
    x = make_config("mixed_step", seed=0)
    r = Run(x).store()
    assert r.dev_status() == 0
    rows = np.random.default_rng(0).choice(x.Tq, 300, replace=False)
    slots = x.out_loc[rows].astype(np.int64)
    got_k = to_host_bits(r.k.view(-1, x.Hkv, x.d)[torch.from_numpy(slots).cuda()])
    got_v = to_host_bits(r.v.view(-1, x.Hkv, x.d)[torch.from_numpy(slots).cuda()])
    assert np.array_equal(got_k, x.k_new[rows]) and np.array_equal(got_v, x.v_new[rows])
    # untouched slots stay as they were (sample of pool slots not written)
    written = np.zeros(x.num_pages * x.page_size, bool)
    written[x.out_loc] = True
    others = np.flatnonzero(~written)[:: max(1, (~written).sum() // 500)]
    got = to_host_bits(r.k.view(-1, x.Hkv, x.d)[torch.from_numpy(others).cuda()])
    assert np.array_equal(got, x.k_cache.reshape(-1, x.Hkv, x.d)[others])
