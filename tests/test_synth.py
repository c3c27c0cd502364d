"""The seeded workload generator: shapes, ranges and page bookkeeping."""
import json
import os

import numpy as np
import pytest

from synth import bf16_bits_to_f32, f32_to_bf16_bits, make_config, make_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_bf16_rounding_is_nearest_even_and_exact_on_representables():
    x = np.array([1.0, -2.5, 3.140625, 0.0, 65280.0], np.float32)
    assert np.array_equal(bf16_bits_to_f32(f32_to_bf16_bits(x)), x)
    # 1 + 2^-8 is half way between 1 and 1 + 2^-7: ties go to the even mantissa (1.0)
    assert bf16_bits_to_f32(f32_to_bf16_bits(np.array([1 + 2 ** -8], np.float32)))[0] == 1.0
    assert bf16_bits_to_f32(f32_to_bf16_bits(np.array([1 + 3 * 2 ** -8], np.float32)))[0] == 1 + 2 ** -6
    assert f32_to_bf16_bits(np.array([np.nan], np.float32))[0] == 0x7FC0


def test_same_seed_same_inputs():
    a = make_config("tiny_decode", seed=3)
    b = make_config("tiny_decode", seed=3)
    c = make_config("tiny_decode", seed=4)
    assert np.array_equal(a.k_cache, b.k_cache) and np.array_equal(a.page_table, b.page_table)
    assert not np.array_equal(a.page_table, c.page_table)


def test_tiny_decode_shape():
    x = make_config("tiny_decode", seed=0)
    assert x.seq_lens.tolist() == [37, 100, 255, 513]
    assert x.num_pages == 256 and x.page_size == 16
    assert x.q.shape == (4, 16, 128) and x.k_new.shape == (4, 8, 128)
    assert x.cu_seqlens_q.tolist() == [0, 1, 2, 3, 4]


def test_pages_are_distinct_and_inside_the_pool():
    x = make_inputs(seed=0, Hq=4, Hkv=2, d=8, page_size=16, new_lens=[3, 1, 40],
                    prefix_lens=[100, 0, 7])
    used = x.page_table[x.page_table >= 0]
    assert len(np.unique(used)) == len(used)
    assert used.max() < x.num_pages
    need = (x.seq_lens + 15) // 16
    assert ((x.page_table >= 0).sum(axis=1) == need).all()
    assert x.num_pages == int(np.ceil(1.1 * need.sum()))


def test_out_loc_slots_are_distinct_and_in_the_listed_pages():
    x = make_inputs(seed=1, Hq=4, Hkv=2, d=8, page_size=4, new_lens=[5, 3, 4],
                    prefix_lens=[2, 9, 0])
    assert len(np.unique(x.out_loc)) == len(x.out_loc)
    for r in range(x.B):
        t0, t1 = x.cu_seqlens_q[r], x.cu_seqlens_q[r + 1]
        pages = set(x.page_table[r][x.page_table[r] >= 0].tolist())
        assert set((x.out_loc[t0:t1] // 4).tolist()) <= pages


def test_block_bytes_golden():
    g = json.load(open(os.path.join(GOLDEN, "kv_block_bytes.json")))
    assert g["block_size"] * 2 * g["num_layers"] * g["num_kv_heads"] * g["head_dim"] * g["itemsize"] == g["block_bytes"]
    assert 2 * g["num_kv_heads"] * g["head_dim"] * g["itemsize"] == g["kv_bytes_per_token_per_layer"]


@pytest.mark.parametrize("name", ["qwen3_decode", "llama_long_decode", "ragged_prefill", "mixed_step"])
def test_config_ranges(name, monkeypatch):
    # small stand-ins keep the pools tiny: only the drawn lengths are checked
    import synth.workloads as w
    captured = {}

    def fake(**kw):
        captured.update(kw)
        raise StopIteration

    monkeypatch.setattr(w, "make_inputs", fake)
    with pytest.raises(StopIteration):
        make_config(name, seed=0)
    new = np.asarray(captured["new_lens"])
    pre = np.asarray(captured["prefix_lens"])
    L = new + pre
    if name == "qwen3_decode":
        assert len(L) == 128 and (new == 1).all() and L.min() >= 512 and L.max() <= 4096
        assert captured["page_size"] == 16 and captured["d"] == 128
    elif name == "llama_long_decode":
        assert len(L) == 8 and L.min() >= 16384 and L.max() <= 32768
        assert captured["page_size"] == 256 and captured["d"] == 64 and captured["Hq"] == 32
    elif name == "ragged_prefill":
        assert len(L) == 8 and new.min() >= 128 and new.max() <= 2048
        assert (pre <= new // 2).all()
    else:
        assert new[:4].sum() == 1024 and (new[:4] >= 1).all() and (pre[:4] <= 2048).all()
        assert (new[4:] == 1).all() and len(new) == 260
        assert L[4:].min() >= 1 and L[4:].max() <= 8192


def test_share_prefix_aliases_pages_and_partitions_the_batch():
    from synth import make_inputs
    from synth.workloads import share_prefix
    B, ps = 8, 16
    x = make_inputs(seed=3, Hq=4, Hkv=2, d=64, page_size=ps, new_lens=np.full(B, 5, np.int64),
                    prefix_lens=np.array([40, 48, 33, 64, 50, 32, 47, 36], np.int64))
    before = x.page_table.copy()
    x = share_prefix(x, [(1, 4, 32), (5, 7, 16)])
    starts = x.meta["prefix_group_start"].tolist()
    lens = x.meta["prefix_len"].tolist()
    # groups: {0}, {1,2,3} sharing 32 tokens, {4}, {5,6} sharing 16, {7}
    assert starts == [0, 1, 4, 5, 7, 8] and lens == [0, 32, 0, 16, 0]
    for first, end, shared in ((1, 4, 32), (5, 7, 16)):
        for r in range(first, end):
            assert (x.page_table[r, :shared // ps] == before[first, :shared // ps]).all()
            assert (x.page_table[r, shared // ps:] == before[r, shared // ps:]).all()
    for r in (0, 4, 7):
        assert (x.page_table[r] == before[r]).all()
    # every new token's slot lies in a page its own row still holds past the shared part
    for b in range(B):
        L = int(x.prefix_lens[b] + x.new_lens[b])
        pages = set(x.page_table[b, :(L + ps - 1) // ps].tolist())
        shared_pages = set(x.page_table[b, :lens[next(i for i in range(len(lens)) if starts[i] <= b < starts[i + 1])] // ps].tolist())
        t0 = int(x.cu_seqlens_q[b])
        for slot in x.out_loc[t0:t0 + int(x.new_lens[b])].tolist():
            assert slot // ps in pages and slot // ps not in shared_pages
