"""The five named workloads at full size, on the GPU, against the oracle.

Decode configs are checked on every row; the prefill and mixed configs on a
sample of rows (the oracle computes them one by one) that always includes
each request's first and last new token."""
import os

import numpy as np
import pytest
import torch

import oracle
from synth import make_config
from tests.gpu_util import TOL, Run, as_f64, max_err

pytestmark = pytest.mark.gpu
THREADS = os.cpu_count() or 8


@pytest.mark.parametrize("name", ["tiny_decode", "qwen3_decode", "llama_long_decode"])
def test_decode_config_all_rows(name):
    x = make_config(name, seed=0)
    r = Run(x).store()
    out = r.decode()
    assert r.dev_status() == 0
    ref = oracle.run_inputs(x, threads=THREADS)
    assert max_err(as_f64(out), ref) <= TOL


def _sample_rows(x, n, seed):
    rng = np.random.default_rng(seed)
    toks = set(rng.choice(x.Tq, size=min(n, x.Tq), replace=False).tolist())
    cu = x.cu_seqlens_q
    for r in range(x.B):
        if cu[r + 1] > cu[r]:
            toks.update([int(cu[r]), int(cu[r + 1]) - 1])
    toks = np.array(sorted(toks))
    heads = rng.integers(0, x.Hq, size=len(toks))
    return toks, heads


def test_ragged_prefill_config_sampled():
    x = make_config("ragged_prefill", seed=0)
    r = Run(x).store()
    out = as_f64(r.prefill())
    assert r.dev_status() == 0
    toks, heads = _sample_rows(x, 1500, 0)
    ref = oracle.run_inputs(x, rows=toks * x.Hq + heads, threads=THREADS)
    assert max_err(out[toks, heads], ref) <= TOL


def test_mixed_step_config_sampled():
    x = make_config("mixed_step", seed=0)
    npre = x.meta["n_prefill"]
    r = Run(x).store()
    pre = x.subset(0, npre)
    dec = x.subset(npre, x.B)
    t_pre = int(x.cu_seqlens_q[npre])
    import paged_kv_cache_out_gb300 as pkv
    out_pre = pkv.paged_prefill_attn(r.q[:t_pre], r.cu[: npre + 1], r.k, r.v, r.page_table[:npre],
                                     r.seq_lens[:npre], x.scale, pre.max_q_len, dev_status=r.status)
    out_dec = pkv.paged_decode_attn(r.q[t_pre:], r.k, r.v, r.page_table[npre:], r.seq_lens[npre:],
                                    x.scale, dev_status=r.status)
    assert r.dev_status() == 0
    toks, heads = _sample_rows(x, 1200, 1)
    ref = oracle.run_inputs(x, rows=toks * x.Hq + heads, threads=THREADS)
    got = np.concatenate([as_f64(out_pre), as_f64(out_dec)])[toks, heads]
    assert max_err(got, ref) <= TOL
