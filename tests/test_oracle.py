"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each check fixes a part of the definition that a plausible slip would break:
the library attention routine (torch SDPA in float64) pins the softmax, the
scale, the causal offset of a cached prefix and the GQA head map; permuting
physical pages and changing the page size pin the page-table addressing; the
closed forms pin the normalisation; the log-sum-exp merge pins the returned
LSE; the pages' printed cu_seqlens example pins the ragged offsets.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from synth import bf16_bits_to_f32, cu_seqlens_from_lengths, f32_to_bf16_bits, make_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _small(seed=0, Hq=4, Hkv=2, d=16, ps=4, new=(1, 1, 1), pre=(0, 5, 12), **kw):
    return make_inputs(seed=seed, Hq=Hq, Hkv=Hkv, d=d, page_size=ps,
                       new_lens=np.array(new), prefix_lens=np.array(pre), **kw)


def _stored_pool(x):
    k, v = x.k_cache.copy(), x.v_cache.copy()
    oracle.kv_store(x.k_new, x.v_new, x.out_loc, k, v)
    return k, v


def _contiguous(x, cache, r):
    """Rows 0..seq_len-1 of request r, gathered through its page-table row."""
    L = int(x.seq_lens[r])
    pos = np.arange(L)
    slots = x.page_table[r, pos // x.page_size].astype(np.int64) * x.page_size + pos % x.page_size
    return cache.reshape(-1, x.Hkv, x.d)[slots]


def _sdpa_reference(x, r):
    """torch SDPA (CPU, float64) on request r's contiguous K/V."""
    k_cache, v_cache = _stored_pool(x)
    K = bf16_bits_to_f32(_contiguous(x, k_cache, r)).astype(np.float64)   # [L,Hkv,d]
    V = bf16_bits_to_f32(_contiguous(x, v_cache, r)).astype(np.float64)
    t0, t1 = int(x.cu_seqlens_q[r]), int(x.cu_seqlens_q[r + 1])
    Q = bf16_bits_to_f32(x.q[t0:t1]).astype(np.float64)                   # [n,Hq,d]
    n, L = t1 - t0, int(x.seq_lens[r])
    c = L - n
    G = x.Hq // x.Hkv
    qt = torch.from_numpy(Q).permute(1, 0, 2)[None]                       # [1,Hq,n,d]
    kt = torch.from_numpy(K).permute(1, 0, 2).repeat_interleave(G, dim=0)[None]
    vt = torch.from_numpy(V).permute(1, 0, 2).repeat_interleave(G, dim=0)[None]
    i = torch.arange(n)[:, None]
    j = torch.arange(L)[None, :]
    mask = j <= (c + i)
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=x.scale)
    return o[0].permute(1, 0, 2).numpy()                                  # [n,Hq,d]


# --- kv_store ------------------------------------------------------------

def test_kv_store_equals_numpy_scatter():
    x = _small(seed=1, new=(3, 1, 7), pre=(2, 9, 0))
    k, v = _stored_pool(x)
    k_ref, v_ref = x.k_cache.copy(), x.v_cache.copy()
    k_ref.reshape(-1, x.Hkv, x.d)[x.out_loc] = x.k_new
    v_ref.reshape(-1, x.Hkv, x.d)[x.out_loc] = x.v_new
    assert np.array_equal(k, k_ref) and np.array_equal(v, v_ref)


def test_kv_store_round_trip_through_page_table():
    x = _small(seed=2, new=(4, 1, 6), pre=(3, 17, 0))
    k, v = _stored_pool(x)
    for r in range(x.B):
        t0, t1 = int(x.cu_seqlens_q[r]), int(x.cu_seqlens_q[r + 1])
        n = t1 - t0
        assert np.array_equal(_contiguous(x, k, r)[-n:], x.k_new[t0:t1])
        assert np.array_equal(_contiguous(x, v, r)[-n:], x.v_new[t0:t1])


def test_kv_store_negative_slot_is_skipped_and_others_untouched():
    x = _small(seed=3, new=(2, 2, 2), pre=(1, 1, 1))
    loc = x.out_loc.copy()
    loc[1] = -1
    k, v = x.k_cache.copy(), x.v_cache.copy()
    oracle.kv_store(x.k_new, x.v_new, loc, k, v)
    k_ref = x.k_cache.copy()
    keep = loc >= 0
    k_ref.reshape(-1, x.Hkv, x.d)[loc[keep]] = x.k_new[keep]
    assert np.array_equal(k, k_ref)


def test_kv_store_slot_beyond_pool_is_an_error():
    x = _small(seed=4)
    loc = x.out_loc.copy()
    loc[0] = x.num_pages * x.page_size
    k = x.k_cache.copy()
    with pytest.raises(oracle.OracleError) as e:
        oracle.kv_store(x.k_new, x.v_new, loc, k, x.v_cache.copy())
    assert e.value.code == 5
    assert np.array_equal(k, x.k_cache)


# --- attention against the library routine --------------------------------

@pytest.mark.parametrize("case", [
    dict(Hq=4, Hkv=2, d=16, ps=4, new=(1, 1, 1), pre=(0, 5, 12)),         # decode, GQA 2
    dict(Hq=8, Hkv=2, d=8, ps=2, new=(5, 3, 4), pre=(0, 0, 0)),          # prefill, GQA 4
    dict(Hq=4, Hkv=4, d=32, ps=8, new=(6, 1, 9), pre=(11, 3, 2)),        # prefix + MHA
    dict(Hq=6, Hkv=3, d=16, ps=1, new=(2, 4), pre=(7, 0)),               # token-granular
    dict(Hq=2, Hkv=1, d=64, ps=16, new=(17,), pre=(40,)),                # MQA, ragged pages
])
def test_attention_matches_torch_sdpa(case):
    x = _small(seed=5, Hq=case["Hq"], Hkv=case["Hkv"], d=case["d"], ps=case["ps"],
               new=case["new"], pre=case["pre"])
    out = oracle.run_inputs(x)
    for r in range(x.B):
        t0, t1 = int(x.cu_seqlens_q[r]), int(x.cu_seqlens_q[r + 1])
        ref = _sdpa_reference(x, r)
        np.testing.assert_allclose(out[t0:t1], ref, rtol=0, atol=1e-12)


def test_scale_is_applied_to_scores():
    x = _small(seed=6, new=(3,), pre=(9,), scale=0.37)
    out = oracle.run_inputs(x)
    np.testing.assert_allclose(out, _sdpa_reference(x, 0), rtol=0, atol=1e-12)


# --- closed forms -----------------------------------------------------------

def test_single_key_returns_its_value_exactly():
    x = _small(seed=7, new=(1, 1), pre=(0, 0))
    out = oracle.run_inputs(x)
    G = x.Hq // x.Hkv
    v = bf16_bits_to_f32(x.v_new).astype(np.float64)            # [B,Hkv,d]
    for h in range(x.Hq):
        assert np.array_equal(out[:, h], v[:, h // G])


def test_identical_keys_give_the_mean_value():
    x = _small(seed=8, new=(1,), pre=(10,), ps=4)
    k, v = _stored_pool(x)
    rows = _contiguous(x, k, 0)
    first = rows[0].copy()
    kf = k.reshape(-1, x.Hkv, x.d)
    L = int(x.seq_lens[0])
    pos = np.arange(L)
    slots = x.page_table[0, pos // x.page_size].astype(np.int64) * x.page_size + pos % x.page_size
    kf[slots] = first
    out = oracle.attention(x.q, x.cu_seqlens_q, k, v, x.page_table, x.seq_lens, x.scale)
    mean_v = bf16_bits_to_f32(_contiguous(x, v, 0)).astype(np.float64).mean(axis=0)  # [Hkv,d]
    G = x.Hq // x.Hkv
    for h in range(x.Hq):
        np.testing.assert_allclose(out[0, h], mean_v[h // G], rtol=0, atol=1e-12)


def test_dominant_key_selects_its_value():
    x = _small(seed=9, Hq=2, Hkv=1, d=8, new=(1,), pre=(6,), ps=4)
    k, v = _stored_pool(x)
    q = np.zeros_like(x.q)
    q[0, :, 0] = f32_to_bf16_bits(np.array([64.0], np.float32))[0]
    kf = k.reshape(-1, x.Hkv, x.d)
    L = int(x.seq_lens[0])
    pos = np.arange(L)
    slots = x.page_table[0, pos // x.page_size].astype(np.int64) * x.page_size + pos % x.page_size
    kf[slots] = 0
    kf[slots[3], 0, 0] = f32_to_bf16_bits(np.array([16.0], np.float32))[0]
    out = oracle.attention(q, x.cu_seqlens_q, k, v, x.page_table, x.seq_lens, scale=1.0)
    vd = bf16_bits_to_f32(v.reshape(-1, x.Hkv, x.d)[slots[3], 0]).astype(np.float64)
    # every other key scores 0, the chosen one 1024: exp(1024) overflows a double,
    # so this also pins the subtraction of the row maximum
    np.testing.assert_allclose(out[0, 0], vd, rtol=0, atol=1e-200)


def test_zero_query_gives_the_mean_value():
    x = _small(seed=10, new=(1,), pre=(13,))
    q = np.zeros_like(x.q)
    k, v = _stored_pool(x)
    out = oracle.attention(q, x.cu_seqlens_q, k, v, x.page_table, x.seq_lens, x.scale)
    mean_v = bf16_bits_to_f32(_contiguous(x, v, 0)).astype(np.float64).mean(axis=0)
    G = x.Hq // x.Hkv
    for h in range(x.Hq):
        np.testing.assert_allclose(out[0, h], mean_v[h // G], rtol=0, atol=1e-12)


# --- addressing invariants -------------------------------------------------

def test_physical_page_permutation_does_not_change_the_result():
    a = _small(seed=11, new=(3, 1), pre=(20, 33), ps=4, contiguous_pages=True)
    b = _small(seed=11, new=(3, 1), pre=(20, 33), ps=4, contiguous_pages=True)
    # move every page of b to a new physical place
    perm = np.random.default_rng(99).permutation(b.num_pages)
    k2 = np.empty_like(b.k_cache)
    v2 = np.empty_like(b.v_cache)
    k2[perm] = b.k_cache
    v2[perm] = b.v_cache
    pt2 = np.where(b.page_table >= 0, perm[np.maximum(b.page_table, 0)], -1).astype(np.int32)
    loc_page = b.out_loc // b.page_size
    loc2 = (perm[loc_page] * b.page_size + b.out_loc % b.page_size).astype(np.int32)
    out_a = oracle.run_inputs(a)
    k2s, v2s = k2.copy(), v2.copy()
    oracle.kv_store(b.k_new, b.v_new, loc2, k2s, v2s)
    out_b = oracle.attention(b.q, b.cu_seqlens_q, k2s, v2s, pt2, b.seq_lens, b.scale)
    assert np.array_equal(out_a, out_b)


@pytest.mark.parametrize("ps_other", [1, 16, 256])
def test_page_size_does_not_change_the_result(ps_other):
    base = _small(seed=12, new=(1, 5, 2), pre=(300, 0, 40), ps=4, d=8)
    k, v = _stored_pool(base)
    out_base = oracle.attention(base.q, base.cu_seqlens_q, k, v, base.page_table,
                                base.seq_lens, base.scale)
    # rebuild the same logical rows in a pool of another page size
    ps = ps_other
    pages = (base.seq_lens.astype(np.int64) + ps - 1) // ps
    P = int(pages.sum()) + 3
    order = np.random.default_rng(5).permutation(P)
    pt = np.full((base.B, int(pages.max())), -1, np.int32)
    kk = np.full((P, ps, base.Hkv, base.d), 0x7FC0, np.uint16)
    vv = kk.copy()
    o = 0
    for r in range(base.B):
        pt[r, :pages[r]] = order[o:o + pages[r]]
        o += pages[r]
        L = int(base.seq_lens[r])
        pos = np.arange(L)
        slots = pt[r, pos // ps].astype(np.int64) * ps + pos % ps
        kk.reshape(-1, base.Hkv, base.d)[slots] = _contiguous(base, k, r)
        vv.reshape(-1, base.Hkv, base.d)[slots] = _contiguous(base, v, r)
    out = oracle.attention(base.q, base.cu_seqlens_q, kk, vv, pt, base.seq_lens, base.scale)
    assert np.array_equal(out, out_base)


def test_gqa_equals_repeated_kv_heads():
    x = _small(seed=13, Hq=8, Hkv=2, d=16, new=(3, 1), pre=(5, 9))
    k, v = _stored_pool(x)
    out = oracle.attention(x.q, x.cu_seqlens_q, k, v, x.page_table, x.seq_lens, x.scale)
    G = x.Hq // x.Hkv
    k_rep = np.ascontiguousarray(np.repeat(k, G, axis=2))
    v_rep = np.ascontiguousarray(np.repeat(v, G, axis=2))
    out_rep = oracle.attention(x.q, x.cu_seqlens_q, k_rep, v_rep, x.page_table, x.seq_lens,
                               x.scale)
    assert np.array_equal(out, out_rep)


# --- consistency between phases ------------------------------------------

def test_decode_equals_last_row_of_prefill():
    L = 29
    pre = _small(seed=14, new=(L,), pre=(0,), ps=4)
    k, v = _stored_pool(pre)
    full = oracle.attention(pre.q, pre.cu_seqlens_q, k, v, pre.page_table, pre.seq_lens,
                            pre.scale)
    q_last = np.ascontiguousarray(pre.q[L - 1:L])
    dec = oracle.attention(q_last, np.array([0, 1], np.int32), k, v, pre.page_table,
                           pre.seq_lens, pre.scale)
    assert np.array_equal(dec[0], full[L - 1])


def test_cached_prefix_rows_equal_the_tail_of_a_full_prefill():
    c, n = 23, 9
    full = _small(seed=15, new=(c + n,), pre=(0,), ps=4)
    k, v = _stored_pool(full)
    out_full = oracle.attention(full.q, full.cu_seqlens_q, k, v, full.page_table,
                                full.seq_lens, full.scale)
    q_tail = np.ascontiguousarray(full.q[c:])
    out_tail = oracle.attention(q_tail, np.array([0, n], np.int32), k, v, full.page_table,
                                full.seq_lens, full.scale)
    assert np.array_equal(out_tail, out_full[c:])


def test_log_sum_exp_merge_of_two_key_ranges():
    ps, L, a = 4, 37, 16                     # split at a page boundary
    x = _small(seed=16, new=(1,), pre=(L - 1,), ps=ps, Hq=4, Hkv=2, d=16)
    k, v = _stored_pool(x)
    o, lse = oracle.attention(x.q, x.cu_seqlens_q, k, v, x.page_table, x.seq_lens, x.scale,
                              return_lse=True)
    # keys [0, a): same page table row, a keys
    o1, l1 = oracle.attention(x.q, x.cu_seqlens_q, k, v, x.page_table,
                              np.array([a], np.int32), x.scale, return_lse=True)
    # keys [a, L): the row shifted by a / ps pages
    pt2 = np.ascontiguousarray(x.page_table[:, a // ps:])
    o2, l2 = oracle.attention(x.q, x.cu_seqlens_q, k, v, pt2,
                              np.array([L - a], np.int32), x.scale, return_lse=True)
    M = np.maximum(l1, l2)
    w1, w2 = np.exp(l1 - M), np.exp(l2 - M)
    merged = (w1[..., None] * o1 + w2[..., None] * o2) / (w1 + w2)[..., None]
    np.testing.assert_allclose(merged, o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(M + np.log(w1 + w2), lse, rtol=0, atol=1e-12)


# --- ragged offsets: the pages' printed example ---------------------------

def test_cu_seqlens_golden_example():
    g = json.load(open(os.path.join(GOLDEN, "cu_seqlens_example.json")))
    cu = cu_seqlens_from_lengths(g["new_token_counts"])
    assert cu.tolist() == g["cu_seqlens_q"]
    # the oracle assigns flat token t to request owner_of_token[t]: each row
    # equals the same request computed alone
    x = _small(seed=17, new=tuple(g["new_token_counts"]), pre=(2, 0, 5), d=8)
    assert x.cu_seqlens_q.tolist() == g["cu_seqlens_q"]
    k, v = _stored_pool(x)
    out = oracle.attention(x.q, x.cu_seqlens_q, k, v, x.page_table, x.seq_lens, x.scale)
    for t, r in enumerate(g["owner_of_token"]):
        t0, t1 = int(x.cu_seqlens_q[r]), int(x.cu_seqlens_q[r + 1])
        alone = oracle.attention(np.ascontiguousarray(x.q[t0:t1]),
                                 np.array([0, t1 - t0], np.int32), k, v,
                                 np.ascontiguousarray(x.page_table[r:r + 1]),
                                 np.ascontiguousarray(x.seq_lens[r:r + 1]), x.scale)
        assert np.array_equal(out[t], alone[t - t0])


def test_rows_subset_equals_full_rows():
    x = _small(seed=18, new=(4, 1, 3), pre=(6, 20, 0))
    full = oracle.run_inputs(x)
    rows = np.array([0, 5, 17, x.Tq * x.Hq - 1])
    sub = oracle.run_inputs(x, rows=rows, threads=2)
    assert np.array_equal(sub, full.reshape(-1, x.d)[rows])


# --- errors -------------------------------------------------------------------

def test_bad_page_id_is_an_error():
    x = _small(seed=19)
    k, v = _stored_pool(x)
    pt = x.page_table.copy()
    pt[1, 0] = x.num_pages
    with pytest.raises(oracle.OracleError) as e:
        oracle.attention(x.q, x.cu_seqlens_q, k, v, pt, x.seq_lens, x.scale)
    assert e.value.code == 2


def test_seq_len_beyond_table_row_is_an_error():
    x = _small(seed=20)
    sl = x.seq_lens.copy()
    sl[2] = x.page_table.shape[1] * x.page_size + 1
    with pytest.raises(oracle.OracleError) as e:
        oracle.attention(x.q, x.cu_seqlens_q, x.k_cache, x.v_cache, x.page_table, sl, x.scale)
    assert e.value.code == 3


def test_unused_pool_slots_are_never_read():
    # the generator fills every unused slot with NaN: any stray read would show
    x = _small(seed=21, new=(2, 1), pre=(5, 30), ps=16)
    out = oracle.run_inputs(x)
    assert np.isfinite(out).all()
    assert math.isnan(bf16_bits_to_f32(x.k_cache.reshape(-1)[-1:])[0])
