"""Requests whose page-table rows share their leading pages (a common prefix
kept once in the pool, as prefix caching does: zero-to-sglang chapter 1 on
prefix reuse; miniVLLM block_tables for cross-sequence prefix reuse) attend
to the same physical keys.  Decode and prefill must match the oracle."""
import numpy as np
import pytest

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
