"""CPU oracle for paged KV-cache attention (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It loads ``pkv_oracle.c`` (plain C,
compiled with gcc on first use) through ctypes and shares no code with the
CUDA library.

The C source states the definitions it follows; this module only marshals
numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libpkv_oracle.so")
_lock = threading.Lock()
_lib = None

ERRORS = {
    0: "ok", 1: "bad argument", 2: "page id outside the pool",
    3: "seq_len beyond the page table row", 4: "bad cu_seqlens_q",
    5: "slot beyond the pool", 6: "out of memory",
}


class OracleError(RuntimeError):
    def __init__(self, code: int):
        super().__init__(f"oracle error {code}: {ERRORS.get(code, '?')}")
        self.code = code


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, OpenMP, no fast-math)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i64, i32, dbl = ctypes.c_int64, ctypes.c_int, ctypes.c_double
            lib.pkv_oracle_kv_store.argtypes = [P, P, P, i64, P, P, i64, i32, i32]
            lib.pkv_oracle_kv_store.restype = i32
            lib.pkv_oracle_attention.argtypes = [P, P, i32, P, P, i64, i32, P, i64, P,
                                                 i32, i32, i32, dbl, P, i64, P, P, i32]
            lib.pkv_oracle_attention.restype = i32
            lib.pkv_oracle_max_threads.restype = i32
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def _c(a, dtype):
    a = np.asarray(a)
    assert a.dtype == dtype, f"expected {dtype}, got {a.dtype}"
    assert a.flags.c_contiguous
    return a


def max_threads() -> int:
    return int(_load().pkv_oracle_max_threads())


def kv_store(k_new, v_new, out_loc, k_cache, v_cache) -> None:
    """Scatter new K/V rows into the pool in place (raw bf16 bits)."""
    lib = _load()
    k_new = _c(k_new, np.uint16)
    v_new = _c(v_new, np.uint16)
    out_loc = _c(out_loc, np.int32)
    k_cache = _c(k_cache, np.uint16)
    v_cache = _c(v_cache, np.uint16)
    P, ps, Hkv, d = k_cache.shape
    assert v_cache.shape == k_cache.shape
    T = out_loc.shape[0]
    assert k_new.shape == (T, Hkv, d) and v_new.shape == (T, Hkv, d)
    rc = lib.pkv_oracle_kv_store(_ptr(k_new), _ptr(v_new), _ptr(out_loc), T,
                                 _ptr(k_cache), _ptr(v_cache), P * ps, Hkv, d)
    if rc:
        raise OracleError(rc)


def attention(q, cu_seqlens_q, k_cache, v_cache, page_table, seq_lens, scale,
              rows=None, threads: int = 1, return_lse: bool = False):
    """Paged attention of the new tokens, in float64.

    Returns ``out`` shaped ``[Tq, Hq, d]`` (or ``[len(rows), d]`` when ``rows``
    lists flat ``t*Hq + h`` indices), and the natural-log LSE when asked.
    """
    lib = _load()
    q = _c(q, np.uint16)
    cu = _c(cu_seqlens_q, np.int32)
    k_cache = _c(k_cache, np.uint16)
    v_cache = _c(v_cache, np.uint16)
    pt = _c(page_table, np.int32)
    sl = _c(seq_lens, np.int32)
    Tq, Hq, d = q.shape
    P, ps, Hkv, d2 = k_cache.shape
    assert d2 == d and v_cache.shape == k_cache.shape
    B = sl.shape[0]
    assert cu.shape == (B + 1,) and pt.shape[0] == B
    pt_stride = pt.shape[1] if pt.ndim == 2 else 0
    if rows is None:
        n = Tq * Hq
        rows_arr = None
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        n = rows_arr.shape[0]
    out = np.zeros((n, d), dtype=np.float64)
    lse = np.zeros(n, dtype=np.float64) if return_lse else None
    rc = lib.pkv_oracle_attention(_ptr(q), _ptr(cu), B, _ptr(k_cache), _ptr(v_cache),
                                  P, ps, _ptr(pt), pt_stride, _ptr(sl), Hq, Hkv, d,
                                  float(scale), _ptr(rows_arr), n, _ptr(out), _ptr(lse),
                                  int(threads))
    if rc:
        raise OracleError(rc)
    if rows is None:
        out = out.reshape(Tq, Hq, d)
        if lse is not None:
            lse = lse.reshape(Tq, Hq)
    return (out, lse) if return_lse else out


def run_inputs(x, rows=None, threads: int = 1, return_lse: bool = False, inplace: bool = False):
    """kv_store of ``x``'s new tokens into copies of its pool (or into the pool
    itself when ``inplace``), then attention."""
    k_cache = x.k_cache if inplace else x.k_cache.copy()
    v_cache = x.v_cache if inplace else x.v_cache.copy()
    kv_store(x.k_new, x.v_new, x.out_loc, k_cache, v_cache)
    return attention(x.q, x.cu_seqlens_q, k_cache, v_cache, x.page_table, x.seq_lens,
                     x.scale, rows=rows, threads=threads, return_lse=return_lse)
