"""The three calls can be captured in a CUDA graph and replayed (the engines
replay decode steps from captured graphs: miniVLLM "Engine Architecture",
CUDA graph optimization; mini-sglang "Engine Class", CUDA Graph Optimization).
Replays with new inputs copied into the captured buffers match the oracle."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_out_gb300 as pkv
from synth import make_inputs
from tests.gpu_util import TOL, as_f64, max_err, to_dev

pytestmark = pytest.mark.gpu


def _decode_inputs(seed, lens, pool_pages):
    lens = np.asarray(lens)
    return make_inputs(seed=seed, Hq=16, Hkv=8, d=128, page_size=16,
                       new_lens=np.ones(len(lens), np.int64), prefix_lens=lens - 1,
                       pool_pages=pool_pages, pt_stride=64)


def test_decode_step_graph_replay_with_new_inputs():
    a = _decode_inputs(60, [100, 700, 33, 1000], pool_pages=400)
    b = _decode_inputs(61, [5, 1024, 512, 64], pool_pages=400)
    # captured buffers
    k, v = to_dev(a.k_cache), to_dev(a.v_cache)
    q, kn, vn, loc = to_dev(a.q), to_dev(a.k_new), to_dev(a.v_new), to_dev(a.out_loc)
    pt, sl = to_dev(a.page_table), to_dev(a.seq_lens)
    out = torch.empty_like(q)
    ws = pkv.decode_workspace(a.B, a.Hq, a.Hkv, a.d)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        # warm-up call outside the capture (first call sets kernel attributes)
        pkv.kv_store(kn, vn, loc, k, v, dev_status=status, stream=s)
        pkv.paged_decode_attn(q, k, v, pt, sl, a.scale, workspace=ws, dev_status=status, out=out, stream=s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        pkv.kv_store(kn, vn, loc, k, v, dev_status=status, stream=s)
        pkv.paged_decode_attn(q, k, v, pt, sl, a.scale, workspace=ws, dev_status=status, out=out, stream=s)
    for x in (a, b, a):
        k.copy_(to_dev(x.k_cache)), v.copy_(to_dev(x.v_cache))
        q.copy_(to_dev(x.q)), kn.copy_(to_dev(x.k_new)), vn.copy_(to_dev(x.v_new))
        loc.copy_(to_dev(x.out_loc)), pt.copy_(to_dev(x.page_table)), sl.copy_(to_dev(x.seq_lens))
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert max_err(as_f64(out), oracle.run_inputs(x)) <= TOL


def test_prefill_graph_replay():
    x = make_inputs(seed=62, Hq=16, Hkv=8, d=128, page_size=16, new_lens=[90, 200],
                    prefix_lens=[17, 300])
    k, v = to_dev(x.k_cache), to_dev(x.v_cache)
    q, kn, vn, loc = to_dev(x.q), to_dev(x.k_new), to_dev(x.v_new), to_dev(x.out_loc)
    pt, sl, cu = to_dev(x.page_table), to_dev(x.seq_lens), to_dev(x.cu_seqlens_q)
    out = torch.empty_like(q)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        pkv.paged_prefill_attn(q, cu, k, v, pt, sl, x.scale, x.max_q_len, dev_status=status, out=out, stream=s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        pkv.kv_store(kn, vn, loc, k, v, dev_status=status, stream=s)
        pkv.paged_prefill_attn(q, cu, k, v, pt, sl, x.scale, x.max_q_len, dev_status=status, out=out, stream=s)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert max_err(as_f64(out), oracle.run_inputs(x)) <= TOL


def test_two_captured_prefill_graphs_replayed_alternately():
    """Each captured prefill call owns its workspace, so two graphs replayed in
    turn (or any number of captures) never share queue counters."""
    xs = [make_inputs(seed=63, Hq=16, Hkv=8, d=128, page_size=16, new_lens=[300, 41, 700],
                      prefix_lens=[0, 512, 100]),
          make_inputs(seed=64, Hq=16, Hkv=8, d=128, page_size=16, new_lens=[129, 1000],
                      prefix_lens=[64, 0])]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    runs = []
    for x in xs:
        k, v = to_dev(x.k_cache), to_dev(x.v_cache)
        q, kn, vn, loc = to_dev(x.q), to_dev(x.k_new), to_dev(x.v_new), to_dev(x.out_loc)
        pt, sl, cu = to_dev(x.page_table), to_dev(x.seq_lens), to_dev(x.cu_seqlens_q)
        out = torch.empty_like(q)
        pws = pkv.prefill_workspace()
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        with torch.cuda.stream(s):
            pkv.kv_store(kn, vn, loc, k, v, dev_status=status, stream=s)
            pkv.paged_prefill_attn(q, cu, k, v, pt, sl, x.scale, x.max_q_len, workspace=pws,
                                   dev_status=status, out=out, stream=s)
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            pkv.paged_prefill_attn(q, cu, k, v, pt, sl, x.scale, x.max_q_len, workspace=pws,
                                   dev_status=status, out=out, stream=s)
        # the graph holds raw pointers: keep every buffer it uses alive
        runs.append((x, g, out, status, (k, v, q, kn, vn, loc, pt, sl, cu, pws)))
    refs = [oracle.run_inputs(x) for x in xs]
    for rep in range(6):
        x, g, out, status, _ = runs[rep % 2]
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert max_err(as_f64(out), refs[rep % 2]) <= TOL


@pytest.mark.parametrize("fused", [False, True])
def test_padded_replay_at_a_fixed_maximum_batch(fused):
    """The engines capture decode at a few batch sizes and replay a smaller
    batch padded to the next captured size with dummy rows (mini-sglang
    "Engine Class", CUDA Graph Optimization).  Padding rows have seq_len 0
    and out_loc -1: they produce zero rows and write nothing to the pool."""
    B_max, B_real = 8, 5
    x = _decode_inputs(65, [300, 17, 1024, 5, 999], pool_pages=400)
    Hq, Hkv, d = x.Hq, x.Hkv, x.d
    pad = B_max - B_real

    def padded(a, fill):
        a = np.asarray(a)
        return np.concatenate([a, np.full((pad,) + a.shape[1:], fill, dtype=a.dtype)])

    nan_bits = np.uint16(0x7FC0)
    q = to_dev(padded(x.q, nan_bits))
    kn, vn = to_dev(padded(x.k_new, nan_bits)), to_dev(padded(x.v_new, nan_bits))
    loc = to_dev(padded(x.out_loc, -1))
    pt = to_dev(padded(x.page_table, -1))
    sl = to_dev(padded(x.seq_lens, 0))
    k, v = to_dev(x.k_cache), to_dev(x.v_cache)
    out = torch.full((B_max, Hq, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = pkv.decode_workspace(B_max, Hq, Hkv, d)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")

    def step(stream):
        if fused:
            pkv.paged_decode_attn_store(q, kn, vn, loc, k, v, pt, sl, x.scale, workspace=ws,
                                        dev_status=status, out=out, stream=stream)
        else:
            pkv.kv_store(kn, vn, loc, k, v, dev_status=status, stream=stream)
            pkv.paged_decode_attn(q, k, v, pt, sl, x.scale, workspace=ws, dev_status=status,
                                  out=out, stream=stream)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step(s)          # first call outside the capture
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step(s)
    # fresh pool, then one replay
    k.copy_(to_dev(x.k_cache)), v.copy_(to_dev(x.v_cache))
    out.fill_(float("nan"))
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = as_f64(out)
    assert max_err(got[:B_real], oracle.run_inputs(x)) <= TOL
    assert (got[B_real:] == 0).all()
    # the pool holds the five new rows at their slots and nothing else changed
    want_k = x.k_cache.copy().reshape(-1, Hkv, d)
    want_v = x.v_cache.copy().reshape(-1, Hkv, d)
    want_k[x.out_loc] = x.k_new
    want_v[x.out_loc] = x.v_new
    got_k = k.view(torch.int16).cpu().numpy().view(np.uint16).reshape(-1, Hkv, d)
    got_v = v.view(torch.int16).cpu().numpy().view(np.uint16).reshape(-1, Hkv, d)
    assert np.array_equal(got_k, want_k) and np.array_equal(got_v, want_v)


def test_shared_prefix_prefill_graph_replay():
    """The shared-prefix prefill captured once and replayed twice: the same
    output as the eager call, bit for bit, and the work-queue counters left
    zeroed (the eager call after the replays is still correct)."""
    from synth import share_prefix
    x = make_inputs(seed=64, Hq=16, Hkv=8, d=128, page_size=16, new_lens=[40, 90, 7, 130, 60],
                    prefix_lens=[256, 300, 256, 400, 10])
    x = share_prefix(x, [(0, 4, 256)])
    from tests.gpu_util import Run
    r = Run(x).store()
    eager = r.prefill_shared()
    torch.cuda.synchronize()
    assert int(r.status.item()) == 0
    gs, gl = to_dev(x.meta["prefix_group_start"]), to_dev(x.meta["prefix_len"])
    cu64 = x.cu_seqlens_q.astype(np.int64)
    starts = x.meta["prefix_group_start"]
    max_group = int(max(cu64[starts[g + 1]] - cu64[starts[g]] for g in range(len(starts) - 1)))
    out = torch.empty_like(eager)
    ws = pkv.prefill_workspace()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        pkv.paged_prefill_attn_shared(r.q, r.cu, r.k, r.v, r.page_table, r.seq_lens, x.scale,
                                      x.max_q_len, gs, gl, max_group, workspace=ws,
                                      dev_status=r.status, out=out, stream=s)
    for _ in range(2):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert int(r.status.item()) == 0
        assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
    assert int(ws.view(torch.int32)[:3].abs().sum().item()) == 0
    assert max_err(as_f64(out), oracle.run_inputs(x)) <= TOL
