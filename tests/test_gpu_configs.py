"""The five named workloads at full size, on the GPU, against the oracle.

Every output row of every config is compared, for seeds 0, 1 and 2 (the tiny
config for seed 0; it is also covered by the smaller tests).  The mixed step
runs its prefill chunks and its decode sequences through the two calls over
one pool, as one layer of the step does."""
import os

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_out_gb300 as pkv
from synth import make_config
from tests.gpu_util import TOL, Run, as_f64, max_err

pytestmark = pytest.mark.gpu
THREADS = os.cpu_count() or 8
SEEDS = (0, 1, 2)


@pytest.mark.parametrize("name,seed", [("tiny_decode", 0)] +
                         [(n, s) for n in ("qwen3_decode", "llama_long_decode") for s in SEEDS])
def test_decode_config_all_rows(name, seed):
    x = make_config(name, seed=seed)
    r = Run(x).store()
    out = r.decode()
    assert r.dev_status() == 0
    ref = oracle.run_inputs(x, threads=THREADS)
    assert max_err(as_f64(out), ref) <= TOL


@pytest.mark.parametrize("seed", SEEDS)
def test_ragged_prefill_config_all_rows(seed):
    x = make_config("ragged_prefill", seed=seed)
    r = Run(x).store()
    out = as_f64(r.prefill())
    assert r.dev_status() == 0
    ref = oracle.run_inputs(x, threads=THREADS)
    assert max_err(out, ref) <= TOL


@pytest.mark.parametrize("seed", SEEDS)
def test_mixed_step_config_all_rows(seed):
    x = make_config("mixed_step", seed=seed)
    npre = x.meta["n_prefill"]
    r = Run(x).store()
    pre = x.subset(0, npre)
    t_pre = int(x.cu_seqlens_q[npre])
    out_pre = pkv.paged_prefill_attn(r.q[:t_pre], r.cu[: npre + 1], r.k, r.v, r.page_table[:npre],
                                     r.seq_lens[:npre], x.scale, pre.max_q_len, workspace=r.pws,
                                     dev_status=r.status)
    out_dec = pkv.paged_decode_attn(r.q[t_pre:], r.k, r.v, r.page_table[npre:], r.seq_lens[npre:],
                                    x.scale, dev_status=r.status)
    assert r.dev_status() == 0
    got = np.concatenate([as_f64(out_pre), as_f64(out_dec)])
    ref = oracle.run_inputs(x, threads=THREADS)
    assert max_err(got, ref) <= TOL
