"""kv_store fused into decode attention on the GPU: the pool must match the
oracle's kv_store bit for bit and the output the oracle's attention over that
pool (max abs error <= 2e-2)."""
import copy

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_out_gb300 as pkv
from synth import make_config, make_inputs
from tests.gpu_util import TOL, Run, as_f64, max_err, to_dev, to_host_bits

pytestmark = pytest.mark.gpu


def decode_case(seed, lens, Hq=16, Hkv=8, d=128, ps=16):
    lens = np.asarray(lens)
    return make_inputs(seed=seed, Hq=Hq, Hkv=Hkv, d=d, page_size=ps,
                       new_lens=np.ones(len(lens), np.int64), prefix_lens=lens - 1)


def fused(r, out_loc=None, k_new=None, v_new=None):
    return pkv.paged_decode_attn_store(
        r.q, r.k_new if k_new is None else k_new, r.v_new if v_new is None else v_new,
        r.out_loc if out_loc is None else out_loc, r.k, r.v, r.page_table, r.seq_lens,
        r.x.scale, dev_status=r.status)


def oracle_pool(x, out_loc=None):
    k, v = x.k_cache.copy(), x.v_cache.copy()
    oracle.kv_store(x.k_new, x.v_new, x.out_loc if out_loc is None else out_loc, k, v)
    return k, v


def check(x, threads=8):
    r = Run(x)
    out = fused(r)
    assert r.dev_status() == 0
    k, v = oracle_pool(x)
    assert np.array_equal(to_host_bits(r.k), k)
    assert np.array_equal(to_host_bits(r.v), v)
    ref = oracle.run_inputs(x, threads=threads)
    err = max_err(as_f64(out), ref)
    assert err <= TOL, err
    return r, out


@pytest.mark.parametrize("seed", [0, 1])
def test_tiny_decode(seed):
    check(make_config("tiny_decode", seed=seed))


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("ps", [1, 16, 256])
def test_shapes(d, G, ps):
    lens = [1, 15, 16, 17, 33, 64, 65, 300, 1000]
    check(decode_case(40 + G, lens, Hq=4 * G, Hkv=4, d=d, ps=ps))


def test_same_bits_as_store_then_decode():
    # the staged row holds the same bits the pool would: identical arithmetic
    x = decode_case(50, [3, 64, 129, 4000, 31], Hq=32, Hkv=8, d=128, ps=16)
    a = Run(x)
    out_f = fused(a)
    b = Run(x).store()
    out_u = b.decode()
    assert a.dev_status() == 0 and b.dev_status() == 0
    assert torch.equal(out_f.view(torch.int16), out_u.view(torch.int16))


def test_last_tile_in_another_block():
    # long sequences are cut over many blocks; the store rides on the last piece
    check(decode_case(51, [20000, 5, 9000, 1], Hq=16, Hkv=8, d=128, ps=16))
    check(decode_case(52, [16384, 30000, 17000], Hq=32, Hkv=8, d=64, ps=256))


def test_negative_slot_reads_the_pool_as_it_is():
    x = decode_case(53, [40, 7, 90, 1], Hq=16, Hkv=8, d=128, ps=16)
    k, v = oracle_pool(x)             # the pool already holds every new row
    x_stored = copy.deepcopy(x)
    x_stored.k_cache[...] = k
    x_stored.v_cache[...] = v
    r = Run(x_stored)
    loc = x.out_loc.copy()
    loc[1] = -1
    loc[3] = -7
    junk = torch.full_like(r.k_new, 3.0)
    kn, vn = r.k_new.clone(), r.v_new.clone()
    kn[1], vn[1], kn[3], vn[3] = junk[1], junk[1], junk[3], junk[3]
    out = fused(r, out_loc=to_dev(loc), k_new=kn, v_new=vn)
    assert r.dev_status() == 0
    # skipped rows: neither stored nor used; the pool's copy is attended to
    assert np.array_equal(to_host_bits(r.k), k)
    assert np.array_equal(to_host_bits(r.v), v)
    ref = oracle.run_inputs(x)
    assert max_err(as_f64(out), ref) <= TOL


def test_zero_length_sequence_still_stores_its_row():
    x = decode_case(54, [40, 7, 90], Hq=16, Hkv=8, d=128, ps=16)
    r = Run(x)
    r.seq_lens[1] = 0
    out = fused(r)
    assert r.dev_status() == 0
    k, v = oracle_pool(x)
    assert np.array_equal(to_host_bits(r.k), k)
    assert np.array_equal(to_host_bits(r.v), v)
    got = as_f64(out)
    assert (got[1] == 0).all()
    ref = oracle.run_inputs(x)
    assert np.abs(got[[0, 2]] - ref[[0, 2]]).max() <= TOL


def _unused_slot(x):
    used = set(np.unique(x.page_table[x.page_table >= 0]).tolist())
    free = [p for p in range(x.num_pages) if p not in used]
    assert free
    return free[0] * x.page_size + 3


def test_slot_beyond_pool_is_flagged_and_skipped():
    x = decode_case(55, [40, 7, 90], Hq=16, Hkv=8, d=128, ps=16)
    r = Run(x)
    loc = x.out_loc.copy()
    loc[2] = x.num_pages * x.page_size
    fused(r, out_loc=to_dev(loc))
    assert r.dev_status() == pkv.DEV_BAD_SLOT
    skip = loc.copy()
    skip[2] = -1
    k, v = oracle_pool(x, skip)
    assert np.array_equal(to_host_bits(r.k), k)
    assert np.array_equal(to_host_bits(r.v), v)


def test_slot_of_another_position_is_flagged_and_stored():
    x = decode_case(56, [40, 7, 90], Hq=16, Hkv=8, d=128, ps=16)
    r = Run(x)
    loc = x.out_loc.copy()
    loc[0] = _unused_slot(x)
    fused(r, out_loc=to_dev(loc))
    assert r.dev_status() == pkv.DEV_BAD_SLOT
    k, v = oracle_pool(x, loc)
    assert np.array_equal(to_host_bits(r.k), k)
    assert np.array_equal(to_host_bits(r.v), v)


def test_decode_workload_sampled():
    # the Qwen3-shaped decode batch (Hq 16, Hkv 8, d 128, lengths 512-4096), sampled rows
    x = make_config("qwen3_decode", seed=7)
    r = Run(x)
    out = fused(r)
    assert r.dev_status() == 0
    rng = np.random.default_rng(7)
    seqs = np.sort(rng.choice(x.B, size=24, replace=False))
    flat = (seqs[:, None] * x.Hq + np.arange(x.Hq)[None, :]).ravel()  # every head of each
    ref = oracle.run_inputs(x, rows=flat, threads=8)
    assert max_err(as_f64(out)[seqs].reshape(-1, x.d), ref) <= TOL
    k, v = oracle_pool(x)
    slots = x.out_loc
    kb, vb = to_host_bits(r.k).reshape(-1, x.Hkv, x.d), to_host_bits(r.v).reshape(-1, x.Hkv, x.d)
    assert np.array_equal(kb[slots], k.reshape(-1, x.Hkv, x.d)[slots])
    assert np.array_equal(vb[slots], v.reshape(-1, x.Hkv, x.d)[slots])


def test_graph_replay_matches_eager():
    x = decode_case(57, [5, 300, 77, 1024], Hq=16, Hkv=8, d=128, ps=16)
    r = Run(x)
    ws = pkv.decode_workspace(x.B, x.Hq, x.Hkv, x.d)
    out = torch.empty_like(r.q)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        pkv.paged_decode_attn_store(r.q, r.k_new, r.v_new, r.out_loc, r.k, r.v, r.page_table,
                                    r.seq_lens, x.scale, workspace=ws, out=out, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    eager = out.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        pkv.paged_decode_attn_store(r.q, r.k_new, r.v_new, r.out_loc, r.k, r.v, r.page_table,
                                    r.seq_lens, x.scale, workspace=ws, out=out)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
