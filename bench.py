"""Benchmark of one paged-attention layer step on GB300.

Default workload (N=1): the Qwen3-0.6B-shaped decode layer -- 128 sequences,
16 query / 8 KV heads, head_dim 128, page_size 16, context lengths uniform in
512..4096 over a randomly permuted pool 1.1x the pages in use.  One step is
the whole hot path for that batch: kv_store of the 128 new tokens' K/V rows,
then paged decode attention (main kernel + log-sum-exp merge).

  value     algorithmic HBM bytes of the step / step time (GB/s); inputs
            resident in HBM; the 1.3 GB KV pool is larger than L2, so no flush
  e2e       the same bytes over the time of the same step through the public
            API with host buffers: pinned host -> device copies of the step's
            inputs, the calls, and the device -> host read of the output
  roofline  decode call (main + merge kernel) bytes / its CUDA-event time,
            against the measured HBM copy bandwidth
  prefill   the ragged-prefill workload (8 requests, 128..2048 new tokens,
            0-50 % cached prefix) in TFLOP/s against the measured bf16 peak,
            L2 flushed between repetitions
  long_decode   the Llama-3.2-1B-shaped long-context decode (8 sequences of
                16K-32K keys, page_size 256): decode call GB/s
  mixed_step    the continuous-batching step over 28 layers (kv_store of 1280
                new tokens, 4-chunk prefill, 256-sequence decode per layer, each
                layer its own KV pool), eager and CUDA-graph replayed
  cpu_baseline  the CPU oracle on a bounded sample of the same step

--impl reference times the CPU oracle on the same workload (bounded samples).
--gpus N under torchrun runs N independent replicas (one per GPU, no
collective in the data path) and reports the aggregate.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode attn HBM GB/s (% of peak) + tokens/s; prefill TFLOP/s (% peak)"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ------------------------------------------------------------------ workload accounting
def decode_bytes(x) -> int:
    """Algorithmic bytes of one paged decode call: every key/value row of every
    sequence read once, q read, output written, the page-table entries and
    seq_lens read."""
    L = x.seq_lens.astype(np.int64)
    kv = int(L.sum()) * x.Hkv * x.d * 2 * 2
    qo = 2 * x.B * x.Hq * x.d * 2
    pt = int(((L + x.page_size - 1) // x.page_size).sum()) * 4 + x.B * 4
    return kv + qo + pt


def store_bytes(x) -> int:
    """kv_store: read each new K and V row, write it to its slot, read out_loc."""
    return 2 * 2 * x.Tq * x.Hkv * x.d * 2 + x.Tq * 4


def prefill_flops(x) -> int:
    """Unmasked QK^T and PV multiply-adds: 4 * d * Hq * sum_r (n_r c_r + n_r (n_r + 1) / 2)."""
    n = x.new_lens.astype(np.int64)
    c = x.prefix_lens.astype(np.int64)
    pairs = int((n * c + n * (n + 1) // 2).sum())
    return 4 * x.d * x.Hq * pairs


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            j = json.load(open(p))
            return (float(j["hbm_gbs"]), float(j["bf16_tflops"]),
                    float(j.get("bf16_tflops_sustained", j["bf16_tflops"])), "measured")
        except Exception:  # noqa: BLE001
            pass
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


def source_digest(*names, src_dir=None) -> str:
    """Digest of the named kernel sources with comments and whitespace removed,
    so that a profile's recorded figures stay valid across comment edits and
    are dropped by any change to the code."""
    src_dir = src_dir or os.path.join(ROOT, "paged_kv_cache_out_gb300", "csrc")
    h = hashlib.sha256()
    for n in names:
        text = open(os.path.join(src_dir, n)).read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(summary: str, digest: str):
    """DRAM bytes per launch from a committed ncu summary, if its source digest matches."""
    p = os.path.join(ROOT, "profiles", summary)
    if not os.path.exists(p):
        return None
    vals = {}
    for line in open(p):
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("source_digest") != digest:
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            self.f = os.fdopen(fd, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not self.path:
            return None
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ------------------------------------------------------------------ GPU arm
def to_dev(a, dev):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a))
    if a.dtype == np.uint16:
        t = t.view(torch.int16).view(torch.bfloat16)
    return t.to(dev)


def prime(stream):
    """Queue ~0.5 ms of device work ahead of a timed region, so the host has
    enqueued the first timed launches before the device reaches the start event
    (with few timed steps, the host's launch latency would otherwise be timed)."""
    import torch
    with torch.cuda.stream(stream):
        torch.cuda._sleep(1_000_000)


def batch_override(args):
    return {"B": args.batch} if args.batch else {}


def run_gpu(args, rank, world):
    import torch
    import paged_kv_cache_out_gb300 as pkv
    from synth import make_config

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    pkv.load_library()
    hbm_peak, bf16_peak, bf16_sus, peak_kind = measured_peaks()

    x = make_config(args.workload, seed=args.seed + rank, **batch_override(args))
    assert x.meta["phase"] == "decode", "the GPU arm times a decode workload"
    stream = torch.cuda.Stream(device=dev)
    k, v = to_dev(x.k_cache, dev), to_dev(x.v_cache, dev)
    q, k_new, v_new = to_dev(x.q, dev), to_dev(x.k_new, dev), to_dev(x.v_new, dev)
    out_loc, pt, sl = to_dev(x.out_loc, dev), to_dev(x.page_table, dev), to_dev(x.seq_lens, dev)
    out = torch.empty_like(q)
    ws = pkv.decode_workspace(x.B, x.Hq, x.Hkv, x.d, dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def step():
        pkv.kv_store(k_new, v_new, out_loc, k, v, dev_status=status, stream=stream)
        pkv.paged_decode_attn(q, k, v, pt, sl, x.scale, workspace=ws, dev_status=status, out=out,
                              stream=stream)

    B_dec = decode_bytes(x)
    B_step = B_dec + store_bytes(x)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    stream.synchronize()
    assert int(status.item()) == 0, f"device status {int(status.item())}"

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    # ---- timed region: K steps back to back (events only around the whole
    # region, so kv_store and decode keep their programmatic-dependent-launch
    # overlap)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clocks:
        prime(stream)
        with torch.cuda.stream(stream):
            t0.record(stream)
            for i in range(args.steps):
                step()
            t1.record(stream)
        stream.synchronize()
    barrier()
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / args.steps
    ms_all = reduce_max(ms, world)

    # ---- the decode call alone (main + merge kernel), back to back: the roofline
    d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    prime(stream)
    with torch.cuda.stream(stream):
        d0.record(stream)
        for i in range(args.steps):
            pkv.paged_decode_attn(q, k, v, pt, sl, x.scale, workspace=ws, dev_status=status, out=out,
                                  stream=stream)
        d1.record(stream)
    stream.synchronize()
    dec_ms = d0.elapsed_time(d1) / args.steps

    # ---- end to end through the public API with host buffers: every step
    # copies its inputs in from pinned host memory and its output back, on
    # two copy streams, with device buffers doubled so that step i's copies
    # overlap steps i-1's and i+1's kernels (the pipelining a serving loop does)
    pin = lambda a: to_dev(a, "cpu").pin_memory()  # noqa: E731
    h_in = [pin(x.q), pin(x.k_new), pin(x.v_new), pin(x.out_loc), pin(x.page_table), pin(x.seq_lens)]
    d_in = [[torch.empty_like(t, device=dev) for t in h_in] for _ in range(2)]
    d_out = [torch.empty_like(out) for _ in range(2)]
    h_out = [torch.empty(out.shape, dtype=out.dtype, pin_memory=True) for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in h_in)
    d2h = h_out[0].numel() * h_out[0].element_size()
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]     # buffer b's inputs are on the device
    ev_done = [torch.cuda.Event() for _ in range(2)]   # buffer b's kernels are done
    ev_out = [torch.cuda.Event() for _ in range(2)]    # buffer b's output is on the host

    def copy_in(i):
        b = i % 2
        s_in.wait_event(ev_done[b])  # its buffers' last users (step i - 2) are done
        with torch.cuda.stream(s_in):
            for h, d in zip(h_in, d_in[b]):
                d.copy_(h, non_blocking=True)
        ev_in[b].record(s_in)

    def compute_and_copy_out(i):
        b = i % 2
        stream.wait_event(ev_in[b])
        stream.wait_event(ev_out[b])  # step i - 2's output has left d_out[b]
        di = d_in[b]
        pkv.kv_store(di[1], di[2], di[3], k, v, dev_status=status, stream=stream)
        pkv.paged_decode_attn(di[0], k, v, di[4], di[5], x.scale, workspace=ws, dev_status=status,
                              out=d_out[b], stream=stream)
        ev_done[b].record(stream)
        s_out.wait_event(ev_done[b])
        with torch.cuda.stream(s_out):
            h_out[b].copy_(d_out[b], non_blocking=True)
        ev_out[b].record(s_out)

    def e2e_run(n):
        copy_in(0)
        for i in range(n):
            if i + 1 < n:
                copy_in(i + 1)
            compute_and_copy_out(i)

    e2e_run(args.warmup)
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    prime(s_in)
    e0.record(s_in)
    e2e_run(args.steps)
    stream.wait_stream(s_out)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = reduce_max(e0.elapsed_time(e1) / args.steps, world)
    assert int(status.item()) == 0

    # ---- the same step through the fused entry point (kv_store inside decode)
    def fused_step():
        pkv.paged_decode_attn_store(q, k_new, v_new, out_loc, k, v, pt, sl, x.scale, workspace=ws,
                                    dev_status=status, out=out, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            fused_step()
        stream.synchronize()
        barrier()
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        prime(stream)
        f0.record(stream)
        for _ in range(args.steps):
            fused_step()
        f1.record(stream)
    stream.synchronize()
    fused_ms = reduce_max(f0.elapsed_time(f1) / args.steps, world)
    assert int(status.item()) == 0

    # ---- prefill TFLOP/s on the ragged-prefill workload, the long-context decode
    # and the mixed continuous-batching step (rank 0 reports)
    prefill = long_dec = mixed = page_sizes = shared_prefix = None
    legs = set(args.legs.split(",")) if args.legs != "all" else {"prefill", "long_decode", "mixed",
                                                                   "page_sizes", "shared_prefix"}
    if rank == 0:
        if "prefill" in legs or "page_sizes" in legs:
            prefill = time_prefill(args, dev, stream, bf16_peak, bf16_sus, peak_kind)
        if "long_decode" in legs:
            long_dec = time_long_decode(args, dev, stream, hbm_peak, peak_kind)
        if "mixed" in legs:
            mixed = time_mixed_step(args, dev, stream)
        if "page_sizes" in legs:
            page_sizes = time_page_sizes(args, dev, stream, prefill, hbm_peak, bf16_peak)
        if "shared_prefix" in legs:
            shared_prefix = time_shared_prefix(args, dev, stream, bf16_peak)

    value = world * B_step / (ms_all * 1e-3) / 1e9
    dec_gbs = B_dec / (dec_ms * 1e-3) / 1e9
    digest = source_digest("decode.cu", "common.cuh")
    traffic = profiled_traffic("decode_kernel_qwen3_decode.md", digest)
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_all, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": dict(workload_config(args, x),
                       l2="KV pool 1.3 GB > 129 MB L2: inputs larger than L2, no flush",
                       parallelism=f"replicas x{world}"),
        "pct_of_peak": round(100.0 * value / world / hbm_peak, 2),
        "tokens_per_s": round(world * x.B / (ms_all * 1e-3), 1),
        "roofline": {
            "bound": "hbm",
            "kernel": "paged_decode_attn (decode_kernel + decode_merge_kernel)",
            "achieved": round(dec_gbs, 2),
            "peak": hbm_peak,
            "peak_kind": f"{peak_kind} HBM copy GB/s",
            "unit": "GB/s",
            "frac": round(dec_gbs / hbm_peak, 4),
            "traffic": traffic,
            "algorithmic_bytes": B_dec,
            "ms": round(dec_ms, 5),
        },
        "e2e": {
            "value": round(world * B_step / (e2e_ms * 1e-3) / 1e9, 2),
            "unit": "GB/s",
            "ms_per_step": round(e2e_ms, 5),
            "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h,
            "schedule": "each step's inputs copied in from pinned host memory and its output "
                        "copied out, on two copy streams; device buffers doubled so the copies "
                        "overlap the neighbouring steps' kernels",
        },
        "fused_step": {
            "entry": "pkv_paged_decode_attn_store (kv_store fused into decode, 2 launches)",
            "value": round(world * B_step / (fused_ms * 1e-3) / 1e9, 2),
            "unit": "GB/s",
            "ms_per_step": round(fused_ms, 5),
        },
        "gpu_launches": 3 * args.steps,
        "clocks": clocks.summary(),
    }
    for key, val in (("prefill", prefill), ("long_decode", long_dec), ("mixed_step", mixed),
                     ("page_sizes", page_sizes), ("shared_prefix", shared_prefix)):
        if val is not None:
            line[key] = val
    return line


def prefill_ms(x, dev, stream, reps, warmup, shared=False):
    """Median CUDA-event time of one ragged-prefill call on x, L2 flushed before
    each repetition (shared: the shared-prefix entry point with x's groups)."""
    import torch
    import paged_kv_cache_out_gb300 as pkv
    k, v = to_dev(x.k_cache, dev), to_dev(x.v_cache, dev)
    q, pt, sl, cu = (to_dev(x.q, dev), to_dev(x.page_table, dev), to_dev(x.seq_lens, dev),
                     to_dev(x.cu_seqlens_q, dev))
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    pkv.kv_store(to_dev(x.k_new, dev), to_dev(x.v_new, dev), to_dev(x.out_loc, dev), k, v,
                 dev_status=status, stream=stream)
    out = torch.empty_like(q)
    if shared:
        gs = x.meta["prefix_group_start"]
        gsd, gld = to_dev(gs, dev), to_dev(x.meta["prefix_len"], dev)
        cu64 = x.cu_seqlens_q.astype("int64")
        max_group = int(max(cu64[gs[g + 1]] - cu64[gs[g]] for g in range(len(gs) - 1)))
    pws = pkv.prefill_workspace(dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    times = []
    with torch.cuda.stream(stream):
        for i in range(warmup + reps):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            if shared:
                pkv.paged_prefill_attn_shared(q, cu, k, v, pt, sl, x.scale, x.max_q_len, gsd, gld,
                                              max_group, workspace=pws, dev_status=status, out=out,
                                              stream=stream)
            else:
                pkv.paged_prefill_attn(q, cu, k, v, pt, sl, x.scale, x.max_q_len, workspace=pws,
                                       dev_status=status, out=out, stream=stream)
            b.record(stream)
            b.synchronize()
            if i >= warmup:
                times.append(a.elapsed_time(b))
    assert int(status.item()) == 0
    return statistics.median(times)


def decode_ms(x, dev, stream, reps, warmup):
    """Mean CUDA-event time of one decode call on x, calls back to back (the
    K/V read per call is larger than L2)."""
    import torch
    import paged_kv_cache_out_gb300 as pkv
    k, v = to_dev(x.k_cache, dev), to_dev(x.v_cache, dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    pkv.kv_store(to_dev(x.k_new, dev), to_dev(x.v_new, dev), to_dev(x.out_loc, dev), k, v,
                 dev_status=status, stream=stream)
    q, pt, sl = to_dev(x.q, dev), to_dev(x.page_table, dev), to_dev(x.seq_lens, dev)
    out = torch.empty_like(q)
    ws = pkv.decode_workspace(x.B, x.Hq, x.Hkv, x.d, dev)
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            pkv.paged_decode_attn(q, k, v, pt, sl, x.scale, workspace=ws, dev_status=status, out=out,
                                  stream=stream)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        prime(stream)
        a.record(stream)
        for _ in range(reps):
            pkv.paged_decode_attn(q, k, v, pt, sl, x.scale, workspace=ws, dev_status=status, out=out,
                                  stream=stream)
        b.record(stream)
        stream.synchronize()
    assert int(status.item()) == 0
    return a.elapsed_time(b) / reps


def time_page_sizes(args, dev, stream, prefill16, hbm_peak, bf16_peak):
    """The engines' two other page layouts: miniVLLM's block_size 256 and
    mini-sglang's token-granular table (page_size 1), for ragged prefill and the
    Qwen3 decode layer, next to page_size 16."""
    import torch
    from synth import make_config
    res = {"prefill": {}, "decode": {}}
    for ps in (256, 1):
        x = make_config("ragged_prefill", seed=args.seed, page_size=ps)
        ms = prefill_ms(x, dev, stream, max(5, min(args.steps, 20)), args.warmup)
        tf = prefill_flops(x) / (ms * 1e-3) / 1e12
        res["prefill"][f"page_size_{ps}"] = {"tflops": round(tf, 2), "ms": round(ms, 5),
                                             "frac": round(tf / bf16_peak, 4),
                                             "vs_page_size_16": round(prefill16["ms"] / ms, 4)}
        torch.cuda.empty_cache()
    for ps in (16, 256, 1):
        x = make_config("qwen3_decode", seed=args.seed, page_size=ps, pt_stride=4096 // ps)
        ms = decode_ms(x, dev, stream, max(20, min(args.steps, 200)), args.warmup)
        gbs = decode_bytes(x) / (ms * 1e-3) / 1e9
        res["decode"][f"page_size_{ps}"] = {"gbs": round(gbs, 2), "ms": round(ms, 5),
                                            "frac": round(gbs / hbm_peak, 4)}
        torch.cuda.empty_cache()
    d16 = res["decode"]["page_size_16"]["ms"]
    for ps in (256, 1):
        res["decode"][f"page_size_{ps}"]["vs_page_size_16"] = round(d16 / res["decode"][f"page_size_{ps}"]["ms"], 4)
    res["workloads"] = ("ragged_prefill and qwen3_decode (seed as the run) laid out with the page size named; "
                        "vs_page_size_16 = time at page_size 16 / time at this page size")
    return res


def time_prefill(args, dev, stream, bf16_peak, bf16_sus, peak_kind):
    from synth import make_config

    x = make_config("ragged_prefill", seed=args.seed)
    ms = prefill_ms(x, dev, stream, max(5, args.steps), args.warmup)
    fl = prefill_flops(x)
    tf = fl / (ms * 1e-3) / 1e12
    return {"workload": "ragged_prefill: 8 requests, n~U[128,2048], prefix 0-50 %, Hq=16, "
                        "Hkv=8, d=128, page_size=16",
            "tflops": round(tf, 2), "ms": round(ms, 5), "flops": fl,
            "peak": bf16_peak, "peak_kind": f"{peak_kind} bf16 dense burst",
            "frac": round(tf / bf16_peak, 4), "l2": "flushed (512 MB write) before each rep"}


def time_shared_prefix(args, dev, stream, bf16_peak):
    """Many requests after one common cached prefix: the plain prefill (each
    request reads the shared pages for itself) against the shared-prefix entry
    point (the group's new tokens packed into dense query tiles that read each
    shared K/V tile once), same inputs, same useful FLOPs."""
    from synth import make_config

    x = make_config("shared_prefix_prefill", seed=args.seed)
    reps = max(5, min(args.steps, 20))
    ms_plain = prefill_ms(x, dev, stream, reps, args.warmup)
    ms_shared = prefill_ms(x, dev, stream, reps, args.warmup, shared=True)
    fl = prefill_flops(x)
    return {"workload": f"shared_prefix_prefill: {x.B} requests, {int(x.meta['prefix_len'][0])} shared "
                        f"cached tokens, new tokens U[16,128] ({x.Tq} in all), Hq=16, Hkv=8, d=128, "
                        f"page_size 16",
            "ms_plain": round(ms_plain, 5), "ms_shared": round(ms_shared, 5),
            "speedup": round(ms_plain / ms_shared, 3), "flops": fl,
            "tflops_shared": round(fl / (ms_shared * 1e-3) / 1e12, 2),
            "frac_shared": round(fl / (ms_shared * 1e-3) / 1e12 / bf16_peak, 4),
            "l2": "flushed (512 MB write) before each rep"}


def time_long_decode(args, dev, stream, hbm_peak, peak_kind):
    """Decode call alone on the Llama-3.2-1B-shaped long-context workload."""
    from synth import make_config

    x = make_config("llama_long_decode", seed=args.seed)
    # back to back: the 0.36 GB of K/V rows read per call is three times L2
    ms = decode_ms(x, dev, stream, max(20, min(args.steps, 500)), args.warmup)
    nb = decode_bytes(x)
    gbs = nb / (ms * 1e-3) / 1e9
    return {"workload": f"llama_long_decode: B={x.B}, Hq={x.Hq}, Hkv={x.Hkv}, d={x.d}, "
                        f"page_size={x.page_size}, kv tokens={int(x.seq_lens.sum())}",
            "gbs": round(gbs, 2), "ms": round(ms, 5), "bytes": nb, "peak": hbm_peak,
            "peak_kind": f"{peak_kind} HBM copy GB/s", "frac": round(gbs / hbm_peak, 4),
            "tokens_per_s": round(x.B / (ms * 1e-3), 1),
            "traffic": profiled_traffic("decode_kernel_llama_long_decode.md",
                                        source_digest("decode.cu", "common.cuh")),
            "l2": "back-to-back calls; 0.36 GB read per call > 129 MB L2, no flush"}


def time_mixed_step(args, dev, stream):
    """The continuous-batching step over 28 layers, each layer with its own KV
    pool.  Serial form: kv_store of all new tokens, prefill of the chunks,
    decode of the rest, on one stream.  Concurrent form (the headline): per
    layer the chunks' kv_store + prefill on one stream and the decode rows'
    fused store + decode on a second stream (their pages are disjoint), joined
    before the next layer; both forms are also replayed from CUDA graphs."""
    import torch
    import paged_kv_cache_out_gb300 as pkv
    from synth import make_config

    x = make_config("mixed_step", seed=args.seed)
    layers = x.meta["layers"]
    npre = x.meta["n_prefill"]
    t_pre = int(x.cu_seqlens_q[npre])
    k0, v0 = to_dev(x.k_cache, dev), to_dev(x.v_cache, dev)
    pools = [(k0.clone(), v0.clone()) for _ in range(layers)]
    del k0, v0
    q, kn, vn = to_dev(x.q, dev), to_dev(x.k_new, dev), to_dev(x.v_new, dev)
    loc, pt, sl, cu = (to_dev(x.out_loc, dev), to_dev(x.page_table, dev), to_dev(x.seq_lens, dev),
                       to_dev(x.cu_seqlens_q, dev))
    pre_max_q = int(x.new_lens[:npre].max())
    out = torch.empty_like(q)
    ws = pkv.decode_workspace(x.B - npre, x.Hq, x.Hkv, x.d, dev)
    pws = pkv.prefill_workspace(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    side = torch.cuda.Stream(device=dev)
    fork, join = torch.cuda.Event(), torch.cuda.Event()

    def step_serial():
        for k, v in pools:
            pkv.kv_store(kn, vn, loc, k, v, dev_status=status, stream=stream)
            pkv.paged_prefill_attn(q[:t_pre], cu[:npre + 1], k, v, pt[:npre], sl[:npre], x.scale,
                                   pre_max_q, workspace=pws, dev_status=status, out=out[:t_pre],
                                   stream=stream)
            pkv.paged_decode_attn(q[t_pre:], k, v, pt[npre:], sl[npre:], x.scale, workspace=ws,
                                  dev_status=status, out=out[t_pre:], stream=stream)

    def step_concurrent():
        for k, v in pools:
            fork.record(stream)
            side.wait_event(fork)
            pkv.kv_store(kn[:t_pre], vn[:t_pre], loc[:t_pre], k, v, dev_status=status, stream=stream)
            pkv.paged_prefill_attn(q[:t_pre], cu[:npre + 1], k, v, pt[:npre], sl[:npre], x.scale,
                                   pre_max_q, workspace=pws, dev_status=status, out=out[:t_pre],
                                   stream=stream)
            pkv.paged_decode_attn_store(q[t_pre:], kn[t_pre:], vn[t_pre:], loc[t_pre:], k, v,
                                        pt[npre:], sl[npre:], x.scale, workspace=ws,
                                        dev_status=status, out=out[t_pre:], stream=side)
            join.record(side)
            stream.wait_event(join)

    reps = max(5, min(args.steps, 50))

    def timed(fn):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                fn()
            stream.synchronize()
            prime(stream)
            e0.record(stream)
            for _ in range(reps):
                fn()
            e1.record(stream)
            stream.synchronize()
        return e0.elapsed_time(e1) / reps

    def graphed(fn):
        g = torch.cuda.CUDAGraph()
        side.wait_stream(stream)
        with torch.cuda.graph(g, stream=stream):
            fn()
        return g

    serial_eager = timed(step_serial)
    conc_eager = timed(step_concurrent)
    g_serial, g_conc = graphed(step_serial), graphed(step_concurrent)
    serial_graph = timed(g_serial.replay)
    conc_graph = timed(g_conc.replay)
    assert int(status.item()) == 0
    dec = x.subset(npre, x.B)
    dec_bytes = decode_bytes(dec)
    nbytes = layers * (dec_bytes + store_bytes(x))
    fl = layers * prefill_flops(x.subset(0, npre))
    hbm_peak, bf16_peak, _, _ = measured_peaks()
    ideal_ms = layers * (dec_bytes + store_bytes(x)) / (hbm_peak * 1e9) * 1e3
    del pools, g_serial, g_conc
    torch.cuda.empty_cache()
    return {"workload": f"mixed_step x{layers} layers: {npre} prefill chunks ({t_pre} tokens) + "
                        f"{x.B - npre} decode seqs (kv tokens {int(dec.seq_lens.sum())}), Qwen3 heads, "
                        f"page_size 16, one KV pool per layer",
            "ms_per_step_graph": round(conc_graph, 4), "ms_per_step_eager": round(conc_eager, 4),
            "schedule": "per layer: chunks' kv_store + prefill on one stream, decode rows' fused "
                        "store + decode on another, joined before the next layer",
            "ms_per_step_graph_serial": round(serial_graph, 4),
            "ms_per_step_eager_serial": round(serial_eager, 4),
            "ideal_ms_per_step": round(ideal_ms, 4),
            "ideal": "decode + kv_store bytes at the measured HBM peak (prefill hidden under decode)",
            "tokens_per_s": round(x.Tq / (conc_graph * 1e-3), 1),
            "decode_plus_store_gbs": round(nbytes / (conc_graph * 1e-3) / 1e9, 1),
            "prefill_flops_per_step": fl, "launches_per_step": 4 * layers}


def reduce_max(v, world):
    if world <= 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ CPU oracle
def oracle_sample(x, target_s: float, threads: int):
    """Time the oracle (kv_store + attention) on the first sequences of x, growing
    the sample until it takes about target_s; returns (seconds, bytes, n_seqs)."""
    import oracle
    nseq = 1
    while True:
        sub = x.subset(0, nseq)
        t = time.perf_counter()
        oracle.run_inputs(sub, threads=threads, inplace=True)
        dt = time.perf_counter() - t
        if dt >= target_s or nseq >= x.B:
            return dt, decode_bytes(sub) + store_bytes(sub), nseq
        nseq = min(x.B, max(nseq + 1, int(nseq * min(8.0, 1.2 * target_s / max(dt, 1e-3)))))


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part")):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def cpu_baseline(x, target_s=10.0):
    """The oracle on all host cores and on one, each on a sample of about target_s."""
    import oracle
    threads = oracle.max_threads()
    dt, nbytes, nseq = oracle_sample(x, target_s, threads)
    reps = 1
    while dt < target_s and nseq == x.B:          # the whole step is quick: repeat it
        more, nb, _ = oracle_sample(x, target_s, threads)
        dt, nbytes, reps = dt + more, nbytes + nb, reps + 1
    dt1, nbytes1, nseq1 = oracle_sample(x, target_s / 2, 1)
    return {"value": round(nbytes / dt / 1e9, 4), "unit": "GB/s", "cores": threads,
            "kind": "oracle", "seconds": round(dt, 3), "cpu_model": cpu_model(),
            "sample": f"kv_store + attention of the first {nseq} of {x.B} sequences, "
                      f"{reps} time(s) ({nbytes} algorithmic bytes), float64 C, OpenMP over rows",
            "single_thread": {"value": round(nbytes1 / dt1 / 1e9, 4), "unit": "GB/s",
                              "seconds": round(dt1, 3),
                              "sample": f"kv_store + attention of the first {nseq1} of {x.B} sequences"}}


def workload_config(args, x):
    """The `config` object both arms report for the decode workload x."""
    return {
        "workload": f"{args.workload}: B={x.B}, Hq={x.Hq}, Hkv={x.Hkv}, d={x.d}, "
                    f"page_size={x.page_size}, kv tokens={int(x.seq_lens.sum())}, "
                    f"pool={x.num_pages} pages; step = kv_store + paged decode",
        "seed": args.seed,
        "bytes_per_step": decode_bytes(x) + store_bytes(x),
    }


def run_reference(args):
    """The oracle as it stands, timed on the host cores on the decode workload.
    Each step runs the same bounded sample (the first sequences of the batch),
    sized once so that the whole run takes about a minute whatever the step
    count."""
    import oracle
    from synth import make_config
    oracle.build()
    x = make_config(args.workload, seed=args.seed, **batch_override(args))
    threads = oracle.max_threads()
    per_step = min(2.0, 60.0 / (args.steps + args.warmup))
    _, _, nseq = oracle_sample(x, per_step, threads)  # size the sample once
    sub = x.subset(0, nseq)
    nb = decode_bytes(sub) + store_bytes(sub)
    for _ in range(args.warmup):
        oracle.run_inputs(sub, threads=threads, inplace=True)
    tot_t = 0.0
    for _ in range(args.steps):
        t = time.perf_counter()
        oracle.run_inputs(sub, threads=threads, inplace=True)
        tot_t += time.perf_counter() - t
    value = args.steps * nb / tot_t / 1e9
    config = workload_config(args, x)
    config["sample"] = f"first {nseq} of {x.B} sequences per step"
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * tot_t / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config,
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads,
                         "kind": "oracle",
                         "sample": f"each step: kv_store + attention of the first {nseq} of "
                                   f"{x.B} sequences"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="qwen3_decode",
                    choices=["tiny_decode", "qwen3_decode", "llama_long_decode"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--batch", type=int, default=0,
                    help="number of sequences of the decode workload (default: the workload's own)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--legs", default="all",
                    help="benchmarks run besides the headline step: all, none, or a comma list of "
                         "prefill, long_decode, mixed, page_sizes, shared_prefix")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    line = run_gpu(args, rank, world)
    if rank == 0:
        if not args.no_cpu_baseline:
            from synth import make_config
            line["cpu_baseline"] = cpu_baseline(make_config(args.workload, seed=args.seed,
                                                            **batch_override(args)))
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
