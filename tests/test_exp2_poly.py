"""The polynomial 2^x used for part of the prefill softmax: its coefficients
(read from the CUDA source) and its fp32 evaluation steps, emulated here in
numpy float32, stay within 1e-4 relative error of 2^x on the range the kernel
feeds it."""
import os
import re

import numpy as np

SRC = os.path.join(os.path.dirname(os.path.dirname(__file__)), "paged_kv_cache_out_gb300", "csrc",
                   "common.cuh")


def _coefficients():
    body = open(SRC).read().split("float exp2_poly(float x)")[1].split("}")[0]
    return [np.float32(v) for v in re.findall(r"([0-9]+\.[0-9]+)f", body) if v not in ("12582912.0",)]


def emulate(x):
    x = np.asarray(x, np.float32)
    c = _coefficients()          # c3, c2 (first fma), c1, c0
    assert len(c) == 4
    t = (x + np.float32(12582912.0)).astype(np.float32)
    j = t.view(np.int32) - np.int32(0x4B400000)
    f = (x - (t - np.float32(12582912.0))).astype(np.float32)
    p = (c[0] * f + c[1]).astype(np.float32)
    p = (p * f + c[2]).astype(np.float32)
    p = (p * f + c[3]).astype(np.float32)
    return (p.view(np.int32) + (j << 23)).astype(np.int32).view(np.float32)


def test_relative_error_bound():
    x = np.linspace(-125.0, 126.0, 2_000_001).astype(np.float32)
    got = emulate(x).astype(np.float64)
    ref = np.exp2(x.astype(np.float64))
    assert np.max(np.abs(got / ref - 1)) < 1e-4


def test_integers_and_halves():
    for v in (-3.0, -0.5, 0.0, 0.5, 1.0, 7.0, -100.0):
        got = float(emulate(np.array([v]))[0])
        assert abs(got / 2.0 ** v - 1) < 1e-4
