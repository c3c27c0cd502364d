"""Requests whose page-table rows share their leading pages (a common prefix
kept once in the pool, as prefix caching does: zero-to-sglang chapter 1 on
prefix reuse; miniVLLM block_tables for cross-sequence prefix reuse) attend
to the same physical keys.  Decode and prefill must match the oracle."""
import numpy as np
import pytest
import torch

import oracle
from synth import make_inputs
from tests.gpu_util import TOL, Run, as_f64, max_err

pytestmark = pytest.mark.gpu


def _share_prefix(x, donor, takers, shared_pages):
    """Point the first `shared_pages` entries of the takers' rows at the donor's pages."""
    pt = x.page_table.copy()
    for r in takers:
        pt[r, :shared_pages] = pt[donor, :shared_pages]
    x.page_table = pt
    return x


def test_decode_with_shared_prefix_pages():
    lens = np.array([900, 700, 1500, 64])
    x = make_inputs(seed=80, Hq=16, Hkv=8, d=128, page_size=16, new_lens=np.ones(4, np.int64),
                    prefix_lens=lens - 1)
    x = _share_prefix(x, donor=0, takers=[1, 2], shared_pages=30)   # 480 shared tokens
    r = Run(x).store()
    out = r.decode()
    assert r.dev_status() == 0
    assert max_err(as_f64(out), oracle.run_inputs(x)) <= TOL


def test_prefill_with_shared_prefix_pages():
    x = make_inputs(seed=81, Hq=16, Hkv=8, d=128, page_size=16, new_lens=[100, 60, 200],
                    prefix_lens=[320, 320, 320])
    x = _share_prefix(x, donor=0, takers=[1, 2], shared_pages=20)   # the whole cached prefix
    r = Run(x).store()
    out = r.prefill()
    assert r.dev_status() == 0
    assert max_err(as_f64(out), oracle.run_inputs(x)) <= TOL


# ---- the shared-prefix prefill entry point (pkv_paged_prefill_attn_shared)

from synth import make_config, share_prefix  # noqa: E402
import paged_kv_cache_out_gb300 as pkv  # noqa: E402


def _groups_case(seed, d, G, ps, new_lens, prefix_lens, groups):
    x = make_inputs(seed=seed, Hq=8 * G if G < 8 else 16, Hkv=8 if G < 8 else 2, d=d,
                    page_size=ps, new_lens=new_lens, prefix_lens=prefix_lens)
    return share_prefix(x, groups)


# shared lengths: whole pages, not always whole 128-key tiles; groups of one,
# several and no shared keys; a request in no group (a group of one sharing
# nothing); groups whose packed new tokens span several 128-row query tiles
# and token blocks that span several requests
CASES = [
    # d, G, ps, new_lens, prefix_lens, groups (first, end, shared tokens)
    (128, 2, 16, [100, 60, 200, 33, 70, 90], [320, 400, 320, 160, 208, 50],
     [(0, 3, 320), (3, 5, 144)]),
    (128, 1, 16, [5, 300, 17], [256, 256, 300], [(0, 3, 256)]),
    (128, 4, 16, [64, 64, 1, 129], [80, 96, 80, 81], [(0, 4, 80)]),
    (128, 8, 1, [40, 70], [37, 37], [(0, 2, 37)]),
    (64, 2, 4, [50, 90, 10], [128, 200, 130], [(0, 2, 128), (2, 3, 0)]),
    (64, 4, 256, [100, 300], [512, 700], [(0, 2, 512)]),
    (128, 2, 256, [30, 30, 30], [1024, 1100, 1500], [(0, 3, 768)]),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_shared_prefix_prefill_matches_oracle_and_plain_prefill(case):
    d, G, ps, n, c, groups = CASES[case]
    x = _groups_case(90 + case, d, G, ps, n, c, groups)
    r = Run(x).store()
    plain = r.prefill()
    assert r.dev_status() == 0
    got = r.prefill_shared()
    assert r.dev_status() == 0
    ref = oracle.run_inputs(x)
    assert max_err(as_f64(got), ref) <= TOL
    # the same attention as the plain call, summed in another order
    assert max_err(as_f64(got), as_f64(plain)) <= TOL


def test_no_groups_is_the_plain_prefill_bit_for_bit():
    x = make_inputs(seed=97, Hq=16, Hkv=8, d=128, page_size=16, new_lens=[70, 130],
                    prefix_lens=[50, 300])
    r = Run(x).store()
    plain = r.prefill()
    got = r.prefill_shared(group_start=[0], prefix_len=np.zeros(0, np.int32))
    assert r.dev_status() == 0
    assert (plain.view(torch.int16) == got.view(torch.int16)).all()


def test_many_short_requests_in_one_group():
    """Requests of 1-9 new tokens: one 128-row tile holds many requests, each
    with its own private key tiles; requests with no new tokens in between."""
    rng = np.random.default_rng(7)
    n = rng.integers(0, 10, size=40)
    n[0] = 3
    x = make_inputs(seed=101, Hq=16, Hkv=8, d=128, page_size=16, new_lens=n,
                    prefix_lens=np.full(40, 272))
    x = share_prefix(x, [(0, 40, 256)])
    r = Run(x).store()
    got = r.prefill_shared()
    assert r.dev_status() == 0
    assert max_err(as_f64(got), oracle.run_inputs(x)) <= TOL


def test_shared_prefix_workload_sampled_rows():
    x = make_config("shared_prefix_prefill", seed=1)
    r = Run(x).store()
    got = r.prefill_shared()
    assert r.dev_status() == 0
    rows = np.random.default_rng(3).choice(x.Tq * x.Hq, 600, replace=False)
    ref = oracle.run_inputs(x, rows=rows, threads=16)
    g = as_f64(got).reshape(-1, x.d)[rows]
    assert max_err(g, ref) <= TOL


def test_bad_shared_length_and_mismatched_pages_are_reported():
    # shared length not a whole number of pages
    x = _groups_case(98, 128, 2, 16, [20, 30], [64, 64], [(0, 2, 64)])
    r = Run(x).store()
    r.prefill_shared(prefix_len=[40])
    assert r.dev_status() & pkv.DEV_BAD_SHARED
    # groups that do not partition the batch
    x = _groups_case(98, 128, 2, 16, [20, 30], [64, 64], [(0, 2, 64)])
    r = Run(x).store()
    r.prefill_shared(group_start=[0, 1], prefix_len=[64])
    assert r.dev_status() & pkv.DEV_BAD_SHARED
    # a member whose row lists other pages for the shared keys
    x = _groups_case(99, 128, 2, 16, [20, 30], [64, 64], [(0, 2, 64)])
    x.page_table[1, 0] = x.page_table[1, 5]   # its own (unshared) page instead
    r = Run(x).store()
    r.prefill_shared()
    assert r.dev_status() & pkv.DEV_BAD_SHARED
    # a shared length beyond a member's cached prefix: that request's rows are NaN
    x = _groups_case(100, 128, 2, 16, [20, 30], [64, 96], [(0, 2, 64)])
    r = Run(x).store()
    out = r.prefill_shared(prefix_len=[96])
    assert r.dev_status() & pkv.DEV_BAD_SHARED
    assert torch.isnan(out[:20].float()).all()
