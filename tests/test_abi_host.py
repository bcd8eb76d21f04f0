"""Host-side checks of the C ABI that need no GPU.

* The shared library builds, loads and exports every function that
  include/*.h declares, with the binding's signatures, and nothing else.
* Invalid arguments are rejected with the documented status code before
  anything touches a device (so these calls are safe without a GPU), and
  no-op sizes succeed without a device.
"""
import ctypes
import glob
import os
import re

import pytest

import dense_fp32_matrix_sgemm_gb300 as sg
from dense_fp32_matrix_sgemm_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return sg.load_library()


def declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        for m in re.finditer(r"\b([A-Za-z_][A-Za-z0-9_ \*]*?)\b(sgemm_[A-Za-z0-9_]+)\s*\(", text):
            names.append(m.group(2))
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ["sgemm_f32", "sgemm_f32_strided_batched", "sgemm_status_string",
                     "sgemm_last_error", "sgemm_version"]:
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"
        assert name in sg.SIGNATURES, f"{name} has no binding signature"


def test_library_exports_nothing_else(lib):
    # built with hidden visibility: the kernels and helpers stay internal
    import shutil
    import subprocess
    if shutil.which("nm") is None:
        pytest.skip("nm not available")
    out = subprocess.run(["nm", "-D", "--defined-only", sg.library_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    extra = sorted(exported - set(declared_functions()))
    assert not extra, f"exported but not declared in include/: {extra[:10]}"


def test_library_links_no_cublas(lib):
    # the product library must not depend on a vendor GEMM library
    import subprocess
    out = subprocess.run(["ldd", sg.library_path()], capture_output=True, text=True).stdout
    assert out and "cublas" not in out


def test_version_and_strings(lib):
    assert sg.version() >= 100
    assert sg.status_string(0) == "SGEMM_OK"
    for code in range(1, 8):
        assert sg.status_string(code).startswith(sg.STATUS_NAMES[code])


FAKE = 0x10000  # a 16-byte-aligned non-NULL address; never dereferenced by these calls


@pytest.mark.parametrize("args,code", [
    (dict(M=-1), 1), (dict(N=-5), 1), (dict(K=-2), 1), (dict(M=1 << 31), 1),
    (dict(transA=2), 4), (dict(transB=-1), 4),
    (dict(lda=7), 2), (dict(ldb=15), 2), (dict(ldc=15), 2),
    (dict(transA=1, lda=31), 2), (dict(transB=1, ldb=7), 2),
    (dict(C=0), 3), (dict(A=0), 3), (dict(B=0), 3), (dict(C=FAKE + 2), 3),
])
def test_invalid_arguments_rejected_on_host(lib, args, code):
    p = dict(M=32, N=16, K=8, A=FAKE, lda=8, B=FAKE, ldb=16, C=FAKE, ldc=16, transA=0, transB=0)
    p.update(args)
    st = sg.sgemm_f32(p["M"], p["N"], p["K"], p["A"], p["lda"], p["B"], p["ldb"], p["C"],
                      p["ldc"], p["transA"], p["transB"], 0, check=False)
    assert st == code, (args, st, sg.last_error())
    assert sg.last_error() != ""
    with pytest.raises(sg.SgemmError) as e:
        sg.sgemm_f32(p["M"], p["N"], p["K"], p["A"], p["lda"], p["B"], p["ldb"], p["C"],
                     p["ldc"], p["transA"], p["transB"], 0)
    assert e.value.status == code


def test_batched_argument_rules(lib):
    def call(**kw):
        p = dict(M=4, N=4, K=4, A=FAKE, lda=4, sA=16, B=FAKE, ldb=4, sB=16, C=FAKE, ldc=4,
                 sC=16, batch=3)
        p.update(kw)
        return sg.sgemm_f32_strided_batched(p["M"], p["N"], p["K"], p["A"], p["lda"], p["sA"],
                                            p["B"], p["ldb"], p["sB"], p["C"], p["ldc"], p["sC"],
                                            p["batch"], 0, 0, 0, check=False)
    assert call(batch=-1) == 5
    assert call(sC=15) == 5          # C matrices of consecutive batches would overlap
    assert call(sC=0) == 5
    assert call(sA=-4) == 5
    # a zero batch or an empty matrix is a successful no-op, with no device touched
    assert call(batch=0) == 0
    assert call(M=0) == 0 and call(N=0, A=0, B=0, C=0) == 0


def test_noop_sizes_need_no_device(lib):
    assert sg.sgemm_f32(0, 5, 7, 0, 7, 0, 5, 0, 5, 0, 0, 0) == 0
    assert sg.sgemm_f32(5, 0, 7, 0, 7, 0, 1, 0, 1, 0, 0, 0) == 0


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    # the binding never falls back to anything when the library is absent
    monkeypatch.setattr(sg, "_lib", None)
    monkeypatch.setattr(sg, "_LIB_PATH", str(tmp_path / "absent.so"))
    with pytest.raises(sg.SgemmUnavailable):
        sg.sgemm_f32(4, 4, 4, FAKE, 4, FAKE, 4, FAKE, 4)


def test_probe_arguments_rejected_on_host(lib):
    flops = ctypes.c_double(0.0)
    probe = lib.sgemm_probe_tf32_mma
    assert probe(0, ctypes.c_void_p(FAKE), ctypes.byref(flops), None) == 1
    assert probe((1 << 20) + 1, ctypes.c_void_p(FAKE), ctypes.byref(flops), None) == 1
    assert probe(10, None, ctypes.byref(flops), None) == 3
    assert probe(10, ctypes.c_void_p(FAKE), None, None) == 3
    fma = lib.sgemm_probe_fp32_fma
    assert fma(2, 10, ctypes.c_void_p(FAKE), ctypes.byref(flops), None) == 1
    assert fma(1, 0, ctypes.c_void_p(FAKE), ctypes.byref(flops), None) == 1


def test_raster_group_knob(lib):
    # returns the previous value; 0 restores the library's 8; out of range changes nothing
    assert sg.set_raster_group(3) == 8
    assert sg.set_raster_group(0) == 3
    assert lib.sgemm_set_raster_group(-1) == -1
    assert lib.sgemm_set_raster_group(65537) == -1
    assert sg.set_raster_group(0) == 8


def test_tf32x3_chunk_knob(lib):
    # returns the previous value; 0 restores 128; only multiples of 32 from 32 are taken
    assert sg.set_tf32x3_chunk_k(64) == 128
    assert sg.set_tf32x3_chunk_k(1 << 30) == 64
    assert sg.set_tf32x3_chunk_k(0) == 1 << 30
    for bad in (-32, 16, 48, 100, (1 << 30) + 32):
        assert lib.sgemm_set_tf32x3_chunk_k(bad) == -1
    assert sg.set_tf32x3_chunk_k(0) == 128


def test_extension_marshalling_matches_ctypes(lib):
    """The _calls extension (built next to the library when a C compiler and
    the Python headers are present) is bound to the same library instance as
    ctypes: host-side argument errors give the same status and detail through
    both routes, and the extension rejects malformed argument lists itself."""
    if sg.marshalling() != "extension":
        pytest.skip("the _calls extension was not built here")
    from dense_fp32_matrix_sgemm_gb300 import _calls
    cases = [
        ("sgemm_f32", (-1, 4, 4, FAKE, 4, FAKE, 4, FAKE, 4, 0, 0, 0)),
        ("sgemm_f32_strided_batched", (4, 4, 4, FAKE, 4, 16, FAKE, 4, 16, FAKE, 4, 16, -2, 0, 0, 0)),
        ("sgemm_f32_ex", (4, 4, 4, 1.0, FAKE, 2, FAKE, 4, 0.0, FAKE, 4, 0, 0, 0, 0)),
        ("sgemm_f32_ex_strided_batched", (4, 4, 4, 1.0, FAKE, 4, 16, FAKE, 4, 16, 0.0, FAKE, 4,
                                          16, 0, 2, 3, 0, 0)),
        ("sgemm_f32_tf32x3_ex", (4, 4, 4, 1.0, FAKE, 4, FAKE, 4, 0.0, FAKE, 4, 0, 0, 0, 0, 0, 0)),
        ("sgemm_f32_splitk", (4, 4, 4, FAKE, 4, FAKE, 4, FAKE, 4, 0, 0, -3, 0, 0, 0)),
        ("sgemm_f32_streamk", (4, 4, 4, FAKE, 4, FAKE, 4, FAKE, 2, 0, 0, 0, 0, 0)),
        ("sgemm_f32_tf32x3", (4, 4, 4, FAKE, 4, FAKE, 4, 0, 4, 0, 0, 0, 0, 0)),
        ("sgemm_f32_tf32x3_strided_batched", (4, 4, 4, FAKE, 4, 16, FAKE, 4, 16, FAKE, 4, 16, 1,
                                              2, 0, 0, 0, 0)),
        ("sgemm_f32_tf32", (4, -4, 4, FAKE, 4, FAKE, 4, FAKE, 4, 0, 0, 0, 0, 0)),
        ("sgemm_f32_tf32_strided_batched", (4, 4, 4, FAKE, 4, 16, FAKE, 4, 16, FAKE, 4, 0, 2, 0,
                                            0, 0, 0, 0)),
        ("sgemm_f32_tf32x3_noalloc", (4, 4, 4, FAKE, 1, FAKE, 4, FAKE, 4, 0, 0, 0)),
    ]
    assert sorted(name for name, _ in cases) == sorted(sg.FAST_ENTRIES)
    for name, args in cases:
        via_ctypes = getattr(lib, name)(*args)
        detail = sg.last_error()
        via_ext = getattr(_calls, name)(*args)
        assert via_ctypes != 0 and via_ext == via_ctypes, name
        assert sg.last_error() == detail, name
    with pytest.raises(TypeError):
        _calls.sgemm_f32(4, 4, 4)
    with pytest.raises(OverflowError):
        _calls.sgemm_f32(1 << 70, 4, 4, FAKE, 4, FAKE, 4, FAKE, 4, 0, 0, 0)
