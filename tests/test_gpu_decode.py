"""Paged decode attention on the GPU against the oracle (max abs error <= 2e-2)."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_out_gb300 as pkv
from synth import make_config, make_inputs
from tests.gpu_util import TOL, Run, as_f64, max_err, to_dev

pytestmark = pytest.mark.gpu


def decode_case(seed, lens, Hq=16, Hkv=8, d=128, ps=16, **kw):
    lens = np.asarray(lens)
    return make_inputs(seed=seed, Hq=Hq, Hkv=Hkv, d=d, page_size=ps, new_lens=np.ones(len(lens), np.int64),
                       prefix_lens=lens - 1, **kw)


def check(x, threads=8):
    r = Run(x).store()
    out = r.decode()
    assert r.dev_status() == 0
    ref = oracle.run_inputs(x, threads=threads)
    err = max_err(as_f64(out), ref)
    assert err <= TOL, err
    return out, err


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_tiny_decode(seed):
    check(make_config("tiny_decode", seed=seed))


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("ps", [1, 16, 256])
def test_shapes(d, G, ps):
    lens = [1, 15, 16, 17, 33, 64, 65, 300, 1000]
    check(decode_case(10 + G, lens, Hq=4 * G, Hkv=4, d=d, ps=ps))


@pytest.mark.parametrize("ps", [2, 4, 8, 32, 64, 128])
def test_other_page_sizes(ps):
    check(decode_case(20, [5, 130, 257, 700], Hq=16, Hkv=8, d=128, ps=ps))


def test_long_sequences_split_over_many_blocks():
    # a few long sequences: every block gets a slice of some sequence
    check(decode_case(30, [20000, 5, 9000, 1], Hq=16, Hkv=8, d=128, ps=16))


def test_long_context_llama_shape_split():
    check(decode_case(31, [16384, 30000, 17000], Hq=32, Hkv=8, d=64, ps=256))


def test_many_short_sequences():
    lens = np.random.default_rng(32).integers(1, 300, size=700)
    check(decode_case(32, lens, Hq=16, Hkv=8, d=128, ps=16))


@pytest.mark.parametrize("d,Hq", [(128, 16), (64, 32)])
@pytest.mark.parametrize("ps", [1, 16])
def test_maximum_batch(d, Hq, ps):
    # 4096 sequences: the per-sequence arrays in shared memory leave room for
    # one block per SM, which still splits its registers between consumers
    # and producers; page size 1 has all four producer warps gathering
    lens = np.random.default_rng(33).integers(1, 49, size=4096)
    check(decode_case(33, lens, Hq=Hq, Hkv=8, d=d, ps=ps), threads=16)


def test_single_token_sequence_returns_its_value():
    x = decode_case(33, [1], Hq=8, Hkv=2, d=64, ps=16)
    out, _ = check(x)
    v = x.v_new.astype(np.uint32) << 16
    vf = v.view(np.float32)
    got = as_f64(out)
    for h in range(8):
        assert np.array_equal(got[0, h], vf[0, h // 4].astype(np.float64))


def test_zero_length_rows_are_zero():
    x = decode_case(34, [40, 7, 90], Hq=16, Hkv=8, d=128, ps=16)
    r = Run(x).store()
    r.seq_lens[1] = 0
    out = r.decode()
    assert r.dev_status() == 0
    got = as_f64(out)
    assert (got[1] == 0).all()
    ref = oracle.run_inputs(x)
    assert max_err(got[[0, 2]], ref[[0, 2]]) <= TOL


def test_bad_page_id_is_flagged_and_poisons_only_its_sequence():
    x = decode_case(35, [100, 50, 3000], Hq=16, Hkv=8, d=128, ps=16)
    r = Run(x).store()
    r.page_table[1, 2] = x.num_pages + 7
    out = r.decode()
    st = r.dev_status()
    assert st & pkv.DEV_BAD_PAGE
    got = as_f64(out)
    assert np.isnan(got[1]).all()
    ref = oracle.run_inputs(x)
    assert max_err(got[[0, 2]], ref[[0, 2]]) <= TOL


def test_bad_seq_len_is_flagged():
    x = decode_case(36, [100, 50], Hq=16, Hkv=8, d=128, ps=16)
    r = Run(x).store()
    r.seq_lens[0] = x.page_table.shape[1] * x.page_size + 1
    out = r.decode()
    assert r.dev_status() & pkv.DEV_BAD_SEQLEN
    got = as_f64(out)
    assert np.isnan(got[0]).all()
    assert max_err(got[[1]], oracle.run_inputs(x)[[1]]) <= TOL


def test_deterministic_and_page_placement_invariant():
    a = decode_case(37, [700, 33, 4000], ps=16, contiguous_pages=True)
    b = decode_case(37, [700, 33, 4000], ps=16, contiguous_pages=True)
    # move b's pages to other physical places
    perm = np.random.default_rng(5).permutation(b.num_pages)
    k2, v2 = np.empty_like(b.k_cache), np.empty_like(b.v_cache)
    k2[perm], v2[perm] = b.k_cache, b.v_cache
    b.k_cache, b.v_cache = k2, v2
    b.page_table = np.where(b.page_table >= 0, perm[np.maximum(b.page_table, 0)], -1).astype(np.int32)
    b.out_loc = (perm[b.out_loc // b.page_size] * b.page_size + b.out_loc % b.page_size).astype(np.int32)
    ra, rb = Run(a).store(), Run(b).store()
    o1, o2, o3 = ra.decode(), ra.decode(), rb.decode()
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)
    assert torch.equal(o1, o3)


def test_explicit_workspace_and_stream():
    x = decode_case(38, [500, 20], ps=16)
    r = Run(x).store()
    ws = pkv.decode_workspace(x.B, x.Hq, x.Hkv, x.d)
    s = torch.cuda.Stream()
    torch.cuda.current_stream().synchronize()
    with torch.cuda.stream(s):
        out = r.decode(workspace=ws, stream=s)
    s.synchronize()
    assert max_err(as_f64(out), oracle.run_inputs(x)) <= TOL


def test_workspace_too_small_is_rejected():
    x = decode_case(39, [50], ps=16)
    r = Run(x).store()
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(pkv.PkvError) as e:
        r.decode(workspace=ws)
    assert e.value.status == pkv.binding.EINVAL
