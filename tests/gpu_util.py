"""Helpers shared by the GPU parity tests (inputs to the device, one call)."""
import numpy as np
import torch

import paged_kv_cache_out_gb300 as pkv

TOL = 2e-2  # max abs error, bf16 output with fp32 accumulation


def dev():
    return torch.device("cuda:0")


def to_dev(a):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if a.dtype == np.uint16:
        t = t.view(torch.int16).view(torch.bfloat16)
    return t.to(dev())


def to_host_bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


class Run:
    """Device copies of one PagedInputs plus the kernels' outputs."""

    def __init__(self, x):
        self.x = x
        self.k = to_dev(x.k_cache)
        self.v = to_dev(x.v_cache)
        self.q = to_dev(x.q)
        self.k_new = to_dev(x.k_new)
        self.v_new = to_dev(x.v_new)
        self.out_loc = to_dev(x.out_loc)
        self.page_table = to_dev(x.page_table)
        self.seq_lens = to_dev(x.seq_lens)
        self.cu = to_dev(x.cu_seqlens_q)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev())
        self.pws = pkv.prefill_workspace(dev())

    def store(self):
        pkv.kv_store(self.k_new, self.v_new, self.out_loc, self.k, self.v, dev_status=self.status)
        return self

    def decode(self, **kw):
        return pkv.paged_decode_attn(self.q, self.k, self.v, self.page_table, self.seq_lens,
                                     self.x.scale, dev_status=self.status, **kw)

    def prefill(self, **kw):
        kw.setdefault("workspace", self.pws)
        return pkv.paged_prefill_attn(self.q, self.cu, self.k, self.v, self.page_table,
                                      self.seq_lens, self.x.scale, self.x.max_q_len,
                                      dev_status=self.status, **kw)

    def prefill_shared(self, group_start=None, prefix_len=None, **kw):
        """The shared-prefix prefill with the groups recorded in x.meta (or given)."""
        gs = np.asarray(self.x.meta["prefix_group_start"] if group_start is None else group_start,
                        np.int32)
        gl = np.asarray(self.x.meta["prefix_len"] if prefix_len is None else prefix_len, np.int32)
        cu = self.x.cu_seqlens_q.astype(np.int64)
        max_group = max([int(cu[gs[g + 1]] - cu[gs[g]]) for g in range(len(gl))] + [0])
        return pkv.paged_prefill_attn_shared(self.q, self.cu, self.k, self.v, self.page_table,
                                             self.seq_lens, self.x.scale, self.x.max_q_len,
                                             to_dev(gs), to_dev(gl), max_group,
                                             dev_status=self.status, **kw)

    def dev_status(self):
        torch.cuda.synchronize()
        return int(self.status.item())


def as_f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def max_err(got, ref):
    got = np.asarray(got, np.float64)
    assert got.shape == ref.shape
    assert np.isfinite(got).all(), "non-finite output"
    return float(np.abs(got - ref).max())
