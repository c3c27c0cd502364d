"""The oracle's pins catch plausible slips.

Each case below plants one mistake (chosen so that it stays inside the
buffers: a planted out-of-bounds read would crash rather than fail a pin) in a copy of the oracle's C source (on the
CPU, in a temporary directory), builds it, swaps it in for the real library
and runs every pin of ``test_oracle``.  At least one pin must fail for each
planted mistake.
"""
import ctypes
import inspect
import os
import subprocess

import pytest

import oracle
import tests.test_oracle as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "pkv_oracle.c")

MUTANTS = {
    "gqa head map": ("const int g = h / (Hq / Hkv);", "const int g = h % Hkv;"),
    "no causal mask": ("const int64_t nkeys = c + i + 1;", "const int64_t nkeys = c + n;"),
    "causal off by one": ("const int64_t nkeys = c + i + 1;", "const int64_t nkeys = c + i + (i > 0);"),
    "scale dropped": ("s[j] = scale * dot;", "s[j] = dot;"),
    "page offset": ("page * page_size + j % page_size;", "page * page_size + (j + 1) % page_size;"),
    "logical page index": ("j / page_size];", "j % page_size];"),
    "max not subtracted": ("const double p = exp(s[j] - m);", "const double p = exp(s[j]);"),
    "missing normalisation": ("o[e] /= l;", "o[e] /= 1.0;"),
    "lse without max": ("*lse = m + log(l);", "*lse = log(l);"),
    "values read from the key pool": ("const uint16_t *vrow = v_cache +", "const uint16_t *vrow = k_cache +"),
    "query row ignores the head": ("q + (t * Hq + h) * (int64_t)d;", "q + (t * Hq) * (int64_t)d;"),
    "prefix length off by one": ("const int64_t c = (int64_t)seq_lens[r] - n;", "const int64_t c = (int64_t)seq_lens[r] - n - (n > 1);"),
    "page table row of another request": ("page_table[(int64_t)r * pt_stride", "page_table[(int64_t)((r + 1) % B) * pt_stride"),
    "value rows not stored": ("memcpy(v_cache + s * row", "if (0) memcpy(v_cache + s * row"),
    "store ignores the last token": ("for (int64_t t = 0; t < T; ++t) {\n        if (out_loc[t] < 0)", "for (int64_t t = 0; t + 1 < T; ++t) {\n        if (out_loc[t] < 0)"),
}


def _pin_functions():
    out = []
    for name, fn in inspect.getmembers(pins, inspect.isfunction):
        if not name.startswith("test_"):
            continue
        marks = getattr(fn, "pytestmark", [])
        params = [m for m in marks if m.name == "parametrize"]
        if params:
            argname, values = params[0].args
            for v in values:
                out.append((f"{name}[{v}]", fn, {argname: v}))
        else:
            out.append((name, fn, {}))
    return out


def _build_mutant(tmp_path, old, new):
    src = open(SRC).read()
    assert old in src, f"mutation anchor not found: {old!r}"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-o", str(lib),
                    str(path), "-lm"], check=True)
    return str(lib)


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_pins_catch_planted_mistake(mutant, tmp_path, monkeypatch):
    old, new = MUTANTS[mutant]
    lib_path = _build_mutant(tmp_path, old, new)
    real = oracle._load()
    lib = ctypes.CDLL(lib_path)
    for fname in ("pkv_oracle_kv_store", "pkv_oracle_attention", "pkv_oracle_max_threads"):
        f, g = getattr(lib, fname), getattr(real, fname)
        f.argtypes, f.restype = g.argtypes, g.restype
    monkeypatch.setattr(oracle, "_lib", lib)
    failed = []
    for name, fn, kwargs in _pin_functions():
        sig = inspect.signature(fn)
        if any(p not in kwargs for p in sig.parameters):
            continue
        try:
            fn(**kwargs)
        except Exception:
            failed.append(name)
    assert failed, f"no pin caught the planted mistake '{mutant}'"
