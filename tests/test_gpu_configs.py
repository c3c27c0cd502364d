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


def test_mixed_step_two_streams_in_a_graph_match_the_serial_step():
    """The bench's concurrent mixed step: the chunks' kv_store + prefill on one
    stream and the decode rows' fused store + decode on another (their pages
    are disjoint), captured in a CUDA graph.  Its output equals the serial
    step's bit for bit and matches the oracle."""
    x = make_config("mixed_step", seed=0)
    npre = x.meta["n_prefill"]
    t_pre = int(x.cu_seqlens_q[npre])
    pre = x.subset(0, npre)
    serial = Run(x).store()
    ref_pre = pkv.paged_prefill_attn(serial.q[:t_pre], serial.cu[:npre + 1], serial.k, serial.v,
                                     serial.page_table[:npre], serial.seq_lens[:npre], x.scale,
                                     pre.max_q_len, workspace=serial.pws, dev_status=serial.status)
    ref_dec = pkv.paged_decode_attn(serial.q[t_pre:], serial.k, serial.v, serial.page_table[npre:],
                                    serial.seq_lens[npre:], x.scale, dev_status=serial.status)
    assert serial.dev_status() == 0
    r = Run(x)  # pool without the new tokens: the graph stores them
    out = torch.empty_like(r.q)
    ws = pkv.decode_workspace(x.B - npre, x.Hq, x.Hkv, x.d)
    main, side = torch.cuda.Stream(), torch.cuda.Stream()
    fork, join = torch.cuda.Event(), torch.cuda.Event()

    def layer():
        fork.record(main)
        side.wait_event(fork)
        pkv.kv_store(r.k_new[:t_pre], r.v_new[:t_pre], r.out_loc[:t_pre], r.k, r.v,
                     dev_status=r.status, stream=main)
        pkv.paged_prefill_attn(r.q[:t_pre], r.cu[:npre + 1], r.k, r.v, r.page_table[:npre],
                               r.seq_lens[:npre], x.scale, pre.max_q_len, workspace=r.pws,
                               dev_status=r.status, out=out[:t_pre], stream=main)
        pkv.paged_decode_attn_store(r.q[t_pre:], r.k_new[t_pre:], r.v_new[t_pre:], r.out_loc[t_pre:],
                                    r.k, r.v, r.page_table[npre:], r.seq_lens[npre:], x.scale,
                                    workspace=ws, dev_status=r.status, out=out[t_pre:], stream=side)
        join.record(side)
        main.wait_event(join)

    main.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    side.wait_stream(main)
    with torch.cuda.graph(g, stream=main):
        layer()
    g.replay()
    torch.cuda.synchronize()
    assert r.dev_status() == 0
    assert torch.equal(out[:t_pre].view(torch.int16), ref_pre.view(torch.int16))
    assert torch.equal(out[t_pre:].view(torch.int16), ref_dec.view(torch.int16))
    ref = oracle.run_inputs(x, threads=THREADS)
    assert max_err(as_f64(out), ref) <= TOL
