"""The C-ABI library loads without a GPU, exports every declared entry point,
and rejects bad host arguments before touching the device."""
import ctypes
import os
import re

import pytest

import paged_kv_cache_out_gb300 as pkv
from paged_kv_cache_out_gb300 import build as cuda_build

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "pkv.h")


@pytest.fixture(scope="module")
def lib():
    cuda_build.build()
    return pkv.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_three_operations():
    names = declared_functions()
    for n in ("pkv_kv_store", "pkv_paged_decode_attn", "pkv_paged_prefill_attn",
              "pkv_decode_workspace_size", "pkv_prefill_workspace_size", "pkv_status_string",
              "pkv_version"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in pkv.binding.SIGNATURES, f"binding lacks a signature for {name}"


def test_status_strings(lib):
    assert lib.pkv_status_string(0) == b"ok"
    assert lib.pkv_status_string(1) == b"invalid argument"
    assert lib.pkv_status_string(2) == b"unsupported shape"
    assert lib.pkv_status_string(3) == b"CUDA runtime error"
    assert lib.pkv_version() >= 100


NULL = None
FAKE = ctypes.c_void_p(0x10000)  # never dereferenced: validation fails first


def test_kv_store_rejects_bad_arguments(lib):
    # null pointers with tokens to store
    assert lib.pkv_kv_store(NULL, FAKE, FAKE, 4, FAKE, FAKE, 8, 16, 8, 128, NULL, NULL) == pkv.binding.EINVAL
    # negative sizes
    assert lib.pkv_kv_store(FAKE, FAKE, FAKE, -1, FAKE, FAKE, 8, 16, 8, 128, NULL, NULL) == pkv.binding.EINVAL
    # nothing to do is fine without a device
    assert lib.pkv_kv_store(NULL, NULL, NULL, 0, NULL, NULL, 8, 16, 8, 128, NULL, NULL) == 0
    # misaligned pointer
    bad = ctypes.c_void_p(0x10002)
    assert lib.pkv_kv_store(bad, FAKE, FAKE, 4, FAKE, FAKE, 8, 16, 8, 128, NULL, NULL) == pkv.binding.EINVAL


def _decode(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, pt=FAKE, stride=4, sl=FAKE, B=2, Hq=16, Hkv=8, d=128, ps=16,
             P=64, scale=0.088, ws=FAKE, ws_bytes=1 << 30, status=NULL, out=FAKE, stream=NULL)
    a.update(kw)
    return lib.pkv_paged_decode_attn(a["q"], a["k"], a["v"], a["pt"], a["stride"], a["sl"], a["B"],
                                     a["Hq"], a["Hkv"], a["d"], a["ps"], a["P"], a["scale"],
                                     a["ws"], a["ws_bytes"], a["status"], a["out"], a["stream"])


def test_decode_rejects_bad_arguments(lib):
    E, U = pkv.binding.EINVAL, pkv.binding.EUNSUPPORTED
    assert _decode(lib, Hq=12, Hkv=8) == E          # heads not a multiple
    assert _decode(lib, q=NULL) == E
    assert _decode(lib, B=-1) == E
    assert _decode(lib, scale=float("nan")) == E
    assert _decode(lib, d=96) == U                  # head_dim not built
    assert _decode(lib, Hq=24, Hkv=8) == U          # GQA ratio 3
    assert _decode(lib, ps=24) == U                 # not a power of two
    assert _decode(lib, ps=512) == U
    assert _decode(lib, B=5000) == U
    assert _decode(lib, B=0) == 0                   # empty batch: no-op


def _prefill(lib, **kw):
    a = dict(q=FAKE, cu=FAKE, k=FAKE, v=FAKE, pt=FAKE, stride=4, sl=FAKE, B=2, Tq=10, maxq=8,
             Hq=16, Hkv=8, d=128, ps=16, P=64, scale=0.088, ws=FAKE, ws_bytes=256, status=NULL,
             out=FAKE, stream=NULL)
    a.update(kw)
    return lib.pkv_paged_prefill_attn(a["q"], a["cu"], a["k"], a["v"], a["pt"], a["stride"], a["sl"],
                                      a["B"], a["Tq"], a["maxq"], a["Hq"], a["Hkv"], a["d"], a["ps"],
                                      a["P"], a["scale"], a["ws"], a["ws_bytes"], a["status"], a["out"],
                                      a["stream"])


def test_prefill_rejects_bad_arguments(lib):
    E, U = pkv.binding.EINVAL, pkv.binding.EUNSUPPORTED
    assert _prefill(lib, cu=NULL) == E
    assert _prefill(lib, Hq=10, Hkv=4) == E
    assert _prefill(lib, maxq=-1) == E
    assert _prefill(lib, d=256) == U
    assert _prefill(lib, Hq=48, Hkv=8) == U
    assert _prefill(lib, ps=3) == U
    assert _prefill(lib, ws=NULL) == E              # no workspace
    assert _prefill(lib, ws_bytes=8) == E           # workspace too small
    assert _prefill(lib, ws=ctypes.c_void_p(0x10008)) == E   # misaligned workspace
    assert _prefill(lib, Tq=0) == 0
    assert lib.pkv_prefill_workspace_size() >= 8


def _prefill_shared(lib, **kw):
    a = dict(q=FAKE, cu=FAKE, k=FAKE, v=FAKE, pt=FAKE, stride=4, sl=FAKE, B=2, Tq=10, maxq=8,
             Hq=16, Hkv=8, d=128, ps=16, P=64, scale=0.088, gs=FAKE, gl=FAKE, ng=1, maxg=10,
             ws=FAKE, ws_bytes=256, status=NULL, out=FAKE, stream=NULL)
    a.update(kw)
    return lib.pkv_paged_prefill_attn_shared(
        a["q"], a["cu"], a["k"], a["v"], a["pt"], a["stride"], a["sl"], a["B"], a["Tq"], a["maxq"],
        a["Hq"], a["Hkv"], a["d"], a["ps"], a["P"], a["scale"], a["gs"], a["gl"], a["ng"], a["maxg"],
        a["ws"], a["ws_bytes"], a["status"], a["out"], a["stream"])


def test_prefill_shared_rejects_bad_arguments(lib):
    """The shared-prefix entry point runs the prefill checks, plus its own:
    group arrays present when there are groups, counts not negative."""
    E, U = pkv.binding.EINVAL, pkv.binding.EUNSUPPORTED
    assert _prefill_shared(lib, cu=NULL) == E
    assert _prefill_shared(lib, gs=NULL) == E
    assert _prefill_shared(lib, gl=NULL) == E
    assert _prefill_shared(lib, ng=-1) == E
    assert _prefill_shared(lib, maxg=-1) == E
    assert _prefill_shared(lib, ws_bytes=8) == E            # workspace too small
    assert _prefill_shared(lib, ws=ctypes.c_void_p(0x10008)) == E   # misaligned workspace
    assert _prefill_shared(lib, d=256) == U
    assert _prefill_shared(lib, ps=3) == U
    assert _prefill_shared(lib, Tq=0) == 0
    # no groups: the plain prefill's checks, null group arrays allowed
    assert _prefill_shared(lib, ng=0, gs=NULL, gl=NULL, cu=NULL) == E
    assert _prefill_shared(lib, maxg=0, gs=NULL, gl=NULL, ws_bytes=8) == E


def test_workspace_size_is_zero_for_bad_sizes(lib):
    assert lib.pkv_decode_workspace_size(4, 12, 8, 128) == 0
    assert lib.pkv_decode_workspace_size(4, 16, 8, 96) == 0


def test_header_is_plain_c99(tmp_path):
    """include/pkv.h is a C header: it compiles as strict C99 with no warnings."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no gcc")
    src = tmp_path / "use_header.c"
    src.write_text('#include "pkv.h"\nint main(void) { return pkv_version() > 0 ? 0 : 1; }\n')
    inc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-fsyntax-only",
                        "-I", inc, str(src)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_noalloc_returns_the_regular_entry_points_status(lib):
    """The entry point without a workspace runs the same argument checks, in
    the same order, as pkv_paged_decode_attn (whose workspace here is large
    enough), so both return the same status for the same bad arguments."""
    cases = [dict(d=96), dict(Hq=24, Hkv=8), dict(Hq=12, Hkv=8), dict(B=-1), dict(q=NULL),
             dict(scale=float("nan")), dict(ps=24), dict(B=5000), dict(B=0, P=0), dict(B=0),
             dict(out=ctypes.c_void_p(0x10002))]
    for kw in cases:
        a = dict(q=FAKE, k=FAKE, v=FAKE, pt=FAKE, stride=4, sl=FAKE, B=2, Hq=16, Hkv=8, d=128,
                 ps=16, P=64, scale=0.088, status=NULL, out=FAKE, stream=NULL)
        a.update(kw)
        regular = _decode(lib, **kw)
        noalloc = lib.pkv_paged_decode_attn_noalloc(
            a["q"], a["k"], a["v"], a["pt"], a["stride"], a["sl"], a["B"], a["Hq"], a["Hkv"],
            a["d"], a["ps"], a["P"], a["scale"], a["status"], a["out"], a["stream"])
        assert noalloc == regular, (kw, noalloc, regular)
