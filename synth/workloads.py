"""Seeded synthetic workloads shaped like the engines' paged-attention batches.

What is emulated (and where the pages describe it):

* The KV pool is one tensor per K and per V of shape
  ``[num_pages, page_size, num_kv_heads, head_dim]`` (miniVLLM "Engine
  Architecture", section ``allocate_kv_cache``: the pool tensor is
  ``(2, num_layers, num_blocks, block_size, num_kv_heads, head_dim)`` and each
  layer gets its K and V slice).
* Each request owns ``ceil(seq_len / page_size)`` physical pages, listed in its
  row of the page table (mini-sglang "Engine Class", attribute ``page_table``;
  miniVLLM "Engine Architecture", ``prepare_prefill`` / ``prepare_decode``,
  ``block_tables``).  Pages are drawn from a random permutation of the pool, the
  way a block manager hands out free pages after churn.
* The new tokens of a step are listed flat with ``cu_seqlens_q`` (miniVLLM
  ``prepare_prefill``: cumulative query lengths such as ``[0, 5, 8, 12]``),
  and each one has a physical slot in ``out_loc`` / ``slot_mapping``
  (mini-sglang ``forward_batch``; miniVLLM ``prepare_prefill``).  Tokens of the
  cached prefix (``num_cached_tokens``) are already resident in their pages.

Values are fp32 N(0,1) draws from ``numpy.random.default_rng(seed)`` rounded to
bf16 (round to nearest even).  Pool slots that hold no token of any request
are filled with a quiet NaN, so a reader that touches them shows up at once.

This module draws numbers and lays them out; it computes nothing of the
attention method itself.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

BF16_QNAN = np.uint16(0x7FC0)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); return the raw bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    out = np.empty(u.shape, dtype=np.uint16)
    flat_u = u.reshape(-1)
    flat_o = out.reshape(-1)
    step = 1 << 24
    for s in range(0, flat_u.size, step):
        c = flat_u[s:s + step]
        bias = ((c >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
        flat_o[s:s + step] = ((c + bias) >> np.uint32(16)).astype(np.uint16)
        nan = (c & np.uint32(0x7FFFFFFF)) > np.uint32(0x7F800000)
        if nan.any():
            flat_o[s:s + step][nan] = BF16_QNAN
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen raw bf16 bits to fp32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal_bf16(rng: np.random.Generator, shape) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    step = 1 << 24
    for s in range(0, n, step):
        m = min(step, n - s)
        out[s:s + m] = f32_to_bf16_bits(rng.standard_normal(m, dtype=np.float32))
    return out.reshape(shape)


def cu_seqlens_from_lengths(lengths) -> np.ndarray:
    """Cumulative new-token offsets ``[0, n0, n0+n1, ...]`` (int32)."""
    lengths = np.asarray(lengths, dtype=np.int64)
    cu = np.zeros(len(lengths) + 1, dtype=np.int64)
    np.cumsum(lengths, out=cu[1:])
    return cu.astype(np.int32)


@dataclass
class PagedInputs:
    """One step's worth of paged-attention inputs (raw bf16 bits as uint16).

    Shapes (Tq = total new tokens, B = requests, P = pool pages):
      q        [Tq, Hq, d]          queries of the new tokens
      k_new    [Tq, Hkv, d]         keys of the new tokens (not yet in the pool)
      v_new    [Tq, Hkv, d]         values of the new tokens
      out_loc  [Tq] int32           pool slot of each new token
      k_cache  [P, ps, Hkv, d]      pool with the cached prefixes resident
      v_cache  [P, ps, Hkv, d]
      page_table [B, pt_stride] int32, -1 past a request's last page
      seq_lens [B] int32            prefix + new tokens of each request
      cu_seqlens_q [B+1] int32      offsets of each request's new tokens
    """

    Hq: int
    Hkv: int
    d: int
    page_size: int
    q: np.ndarray
    k_new: np.ndarray
    v_new: np.ndarray
    out_loc: np.ndarray
    k_cache: np.ndarray
    v_cache: np.ndarray
    page_table: np.ndarray
    seq_lens: np.ndarray
    cu_seqlens_q: np.ndarray
    scale: float
    meta: dict = field(default_factory=dict)

    @property
    def B(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def Tq(self) -> int:
        return int(self.q.shape[0])

    @property
    def num_pages(self) -> int:
        return int(self.k_cache.shape[0])

    @property
    def new_lens(self) -> np.ndarray:
        return np.diff(self.cu_seqlens_q.astype(np.int64))

    @property
    def prefix_lens(self) -> np.ndarray:
        return self.seq_lens.astype(np.int64) - self.new_lens

    @property
    def max_q_len(self) -> int:
        return int(self.new_lens.max()) if self.B else 0

    def subset(self, lo: int, hi: int) -> "PagedInputs":
        """Requests ``lo..hi-1`` over the same pool (arrays are views)."""
        cu = self.cu_seqlens_q
        t0, t1 = int(cu[lo]), int(cu[hi])
        return PagedInputs(
            Hq=self.Hq, Hkv=self.Hkv, d=self.d, page_size=self.page_size,
            q=self.q[t0:t1], k_new=self.k_new[t0:t1], v_new=self.v_new[t0:t1],
            out_loc=self.out_loc[t0:t1], k_cache=self.k_cache, v_cache=self.v_cache,
            page_table=self.page_table[lo:hi], seq_lens=self.seq_lens[lo:hi],
            cu_seqlens_q=(cu[lo:hi + 1] - cu[lo]).astype(np.int32),
            scale=self.scale, meta=dict(self.meta),
        )


def make_inputs(*, seed: int, Hq: int, Hkv: int, d: int, page_size: int,
                new_lens, prefix_lens, pool_pages: int | None = None,
                pool_factor: float = 1.1, pt_stride: int | None = None,
                rng: np.random.Generator | None = None,
                scale: float | None = None, contiguous_pages: bool = False,
                poison_unused: bool = True) -> PagedInputs:
    """Lay out one batch of requests over a randomly permuted page pool.

    ``new_lens[r]`` tokens of request r arrive this step, after
    ``prefix_lens[r]`` tokens that are already cached.  Pages are assigned
    from ``rng.permutation(pool_pages)`` in request order (or in pool order
    when ``contiguous_pages``).
    """
    if rng is None:
        rng = np.random.default_rng(seed)
    new_lens = np.asarray(new_lens, dtype=np.int64)
    prefix_lens = np.asarray(prefix_lens, dtype=np.int64)
    assert new_lens.shape == prefix_lens.shape
    assert (new_lens >= 0).all() and (prefix_lens >= 0).all()
    B = len(new_lens)
    ps = int(page_size)
    seq_lens = prefix_lens + new_lens
    pages_per_req = (seq_lens + ps - 1) // ps
    total_pages = int(pages_per_req.sum())
    if pool_pages is None:
        pool_pages = max(1, int(math.ceil(pool_factor * total_pages)))
    assert pool_pages >= total_pages, "pool too small for the batch"
    if pt_stride is None:
        pt_stride = max(1, int(pages_per_req.max()) if B else 1)
    assert pt_stride >= (int(pages_per_req.max()) if B else 0)

    order = np.arange(pool_pages) if contiguous_pages else rng.permutation(pool_pages)
    page_table = np.full((B, pt_stride), -1, dtype=np.int32)
    starts = np.zeros(B + 1, dtype=np.int64)
    np.cumsum(pages_per_req, out=starts[1:])
    for r in range(B):
        page_table[r, :pages_per_req[r]] = order[starts[r]:starts[r + 1]]

    Tq = int(new_lens.sum())
    q = _normal_bf16(rng, (Tq, Hq, d))
    k_new = _normal_bf16(rng, (Tq, Hkv, d))
    v_new = _normal_bf16(rng, (Tq, Hkv, d))

    # Physical slot of token position j of request r: the page that the
    # table lists for j's logical page, at offset j mod page_size.
    def slots_of(r: int, lo: int, hi: int) -> np.ndarray:
        pos = np.arange(lo, hi, dtype=np.int64)
        return page_table[r, pos // ps].astype(np.int64) * ps + pos % ps

    out_loc = np.concatenate(
        [slots_of(r, int(prefix_lens[r]), int(seq_lens[r])) for r in range(B)]
        or [np.zeros(0, np.int64)]).astype(np.int32)
    prefix_slots = np.concatenate(
        [slots_of(r, 0, int(prefix_lens[r])) for r in range(B)]
        or [np.zeros(0, np.int64)])

    fill = BF16_QNAN if poison_unused else np.uint16(0)
    k_cache = np.full((pool_pages, ps, Hkv, d), fill, dtype=np.uint16)
    v_cache = np.full((pool_pages, ps, Hkv, d), fill, dtype=np.uint16)
    k_cache.reshape(-1, Hkv, d)[prefix_slots] = _normal_bf16(rng, (len(prefix_slots), Hkv, d))
    v_cache.reshape(-1, Hkv, d)[prefix_slots] = _normal_bf16(rng, (len(prefix_slots), Hkv, d))

    return PagedInputs(
        Hq=Hq, Hkv=Hkv, d=d, page_size=ps, q=q, k_new=k_new, v_new=v_new,
        out_loc=out_loc, k_cache=k_cache, v_cache=v_cache, page_table=page_table,
        seq_lens=seq_lens.astype(np.int32),
        cu_seqlens_q=cu_seqlens_from_lengths(new_lens),
        scale=(1.0 / math.sqrt(d)) if scale is None else float(scale),
        meta={"seed": seed},
    )


# ---------------------------------------------------------------------------
# The five named workloads.  Model shapes: Qwen3-0.6B (16 query heads, 8 KV
# heads, head_dim 128, 28 layers) and Llama-3.2-1B (32 query heads, 8 KV heads,
# head_dim 64), from the miniVLLM "LLMEngine" page (model config keys) and the
# mini-sglang "Engine Class" example; page_size 16 (mini-sglang example) and
# block_size 256 (miniVLLM default).
# ---------------------------------------------------------------------------

def _tiny_decode(seed, **kw):
    lens = np.array([37, 100, 255, 513])
    args = dict(Hq=16, Hkv=8, d=128, page_size=16, new_lens=np.ones(4, np.int64),
                prefix_lens=lens - 1, pool_pages=256)
    args.update(kw)
    x = make_inputs(seed=seed, **args)
    x.meta.update(name="tiny_decode", phase="decode")
    return x


def _qwen3_decode(seed, B=128, **kw):
    rng = np.random.default_rng(seed)
    lens = rng.integers(512, 4096 + 1, size=B)
    args = dict(Hq=16, Hkv=8, d=128, page_size=16, new_lens=np.ones(B, np.int64),
                prefix_lens=lens - 1, pool_factor=1.1, pt_stride=4096 // 16)
    args.update(kw)
    x = make_inputs(seed=seed, rng=rng, **args)
    x.meta.update(name="qwen3_decode", phase="decode")
    return x


def _llama_long_decode(seed, B=8, **kw):
    rng = np.random.default_rng(seed)
    lens = rng.integers(16384, 32768 + 1, size=B)
    args = dict(Hq=32, Hkv=8, d=64, page_size=256, new_lens=np.ones(B, np.int64),
                prefix_lens=lens - 1, pool_factor=1.1, pt_stride=32768 // 256)
    args.update(kw)
    x = make_inputs(seed=seed, rng=rng, **args)
    x.meta.update(name="llama_long_decode", phase="decode")
    return x


def _ragged_prefill(seed, B=8, **kw):
    rng = np.random.default_rng(seed)
    n = rng.integers(128, 2048 + 1, size=B)
    u = rng.uniform(0.0, 0.5, size=B)
    c = np.floor(u * n).astype(np.int64)
    args = dict(Hq=16, Hkv=8, d=128, page_size=16, new_lens=n, prefix_lens=c,
                pool_factor=1.1)
    args.update(kw)
    x = make_inputs(seed=seed, rng=rng, **args)
    x.meta.update(name="ragged_prefill", phase="prefill")
    return x


def _mixed_step(seed, n_chunks=4, chunk_tokens=1024, n_decode=256, **kw):
    """Prefill chunks then decode sequences over one shared pool.

    Requests ``0..n_chunks-1`` are prefill chunks (new lengths from sorted
    uniform cut points of ``chunk_tokens``, prior context uniform in
    0..2048); the remaining ``n_decode`` requests decode one token with
    context lengths log-uniform in 1..8192.
    """
    rng = np.random.default_rng(seed)
    cuts = np.sort(rng.choice(np.arange(1, chunk_tokens), size=n_chunks - 1, replace=False))
    n_pre = np.diff(np.concatenate([[0], cuts, [chunk_tokens]]))
    c_pre = rng.integers(0, 2048 + 1, size=n_chunks)
    L_dec = np.clip(np.rint(np.exp(rng.uniform(0.0, math.log(8192.0), size=n_decode))), 1, 8192)
    L_dec = L_dec.astype(np.int64)
    new = np.concatenate([n_pre, np.ones(n_decode, np.int64)])
    pre = np.concatenate([c_pre, L_dec - 1])
    args = dict(Hq=16, Hkv=8, d=128, page_size=16, new_lens=new, prefix_lens=pre,
                pool_factor=1.1)
    args.update(kw)
    x = make_inputs(seed=seed, rng=rng, **args)
    x.meta.update(name="mixed_step", phase="mixed", n_prefill=n_chunks,
                  n_decode=n_decode, layers=28)
    return x


def share_prefix(x: PagedInputs, groups) -> PagedInputs:
    """Make groups of consecutive requests share their leading cached pages.

    ``groups`` lists ``(first, end, shared_tokens)``: requests first..end-1
    take the first ``shared_tokens // page_size`` page ids of request
    ``first``'s row, the way a prefix cache lets several requests point at
    one cached copy of a common prefix (zero-to-sglang chapter 1, roadmap on
    prefix caching; miniVLLM prepare_prefill, block_tables shared across
    sequences).  ``shared_tokens`` must be a whole number of pages within
    every member's cached prefix, so the new tokens' slots are untouched.
    The pages the members held before stay in the pool, unreferenced.  The
    groups, with every request outside them as a group of one sharing
    nothing, are recorded in ``x.meta`` as ``prefix_group_start`` ([n + 1],
    a partition of the batch) and ``prefix_len`` ([n]) int32 arrays.
    """
    ps = x.page_size
    pt = x.page_table.copy()
    starts, lens = [0], []
    for first, end, shared in sorted(groups):
        assert shared % ps == 0 and first < end and first >= starts[-1]
        assert (x.prefix_lens[first:end] >= shared).all()
        pt[first + 1:end, :shared // ps] = pt[first, :shared // ps]
        for r in range(starts[-1], first):  # requests before the group share nothing
            starts.append(r + 1)
            lens.append(0)
        starts.append(end)
        lens.append(shared)
    for r in range(starts[-1], x.B):
        starts.append(r + 1)
        lens.append(0)
    x.page_table = pt
    x.meta["prefix_group_start"] = np.asarray(starts, dtype=np.int32)
    x.meta["prefix_len"] = np.asarray(lens, dtype=np.int32)
    return x


def _shared_prefix_prefill(seed, B=128, prefix=2048, n_lo=16, n_hi=128, **kw):
    """Many requests after one common cached prefix (a shared system prompt):
    ``prefix`` cached tokens on the same pages for all B requests, then each
    request's own new tokens, uniform in n_lo..n_hi."""
    rng = np.random.default_rng(seed)
    n = rng.integers(n_lo, n_hi + 1, size=B)
    args = dict(Hq=16, Hkv=8, d=128, page_size=16, new_lens=n,
                prefix_lens=np.full(B, prefix, np.int64), pool_factor=1.1)
    args.update(kw)
    x = make_inputs(seed=seed, rng=rng, **args)
    x = share_prefix(x, [(0, B, prefix)])
    x.meta.update(name="shared_prefix_prefill", phase="prefill")
    return x


CONFIGS = {
    "tiny_decode": _tiny_decode,
    "qwen3_decode": _qwen3_decode,
    "llama_long_decode": _llama_long_decode,
    "ragged_prefill": _ragged_prefill,
    "mixed_step": _mixed_step,
    "shared_prefix_prefill": _shared_prefix_prefill,
}


def make_config(name: str, seed: int = 0, **overrides) -> PagedInputs:
    """Build one of the five named workloads for ``seed``."""
    return CONFIGS[name](seed, **overrides)
