"""Host-side checks of the C ABI (no GPU needed): the library builds and loads, exports
every function include/fp8fg.h declares with the binding's signature, and rejects
invalid arguments with FP8FG_ERR_ARG before touching the device."""
import ctypes
import os
import re
import shutil
import subprocess

import pytest

from fp8_fine_grained_cast_b300 import _lib
from fp8_fine_grained_cast_b300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp8fg.h")


@pytest.fixture(scope="module")
def lib():
    build()
    return _lib.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(fp8\w+)\s*\(", text, flags=re.M)


def test_header_declares_the_documented_entry_points():
    names = set(declared_functions())
    assert {"fp8_quant_act_1x128", "fp8_quant_w_128x128", "fp8_blockscaled_gemm", "fp8_grouped_gemm",
            "fp8fg_last_error", "fp8fg_sync_status"} <= names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in _lib.SIGNATURES, f"binding lacks {name}"


def test_binding_signatures_match_header_arity():
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    for name, (_, args) in _lib.SIGNATURES.items():
        m = re.search(name + r"\s*\(([^)]*)\)", text)
        assert m, name
        params = [p for p in m.group(1).split(",") if p.strip() and p.strip() != "void"]
        assert len(params) == len(args), (name, params)


def test_version(lib):
    assert lib.fp8fg_version() == 100


FAKE = 0x10000   # a 16-byte aligned non-null value; never dereferenced on these paths


def _rc(fn, *args):
    return fn(*args)


def test_quant_act_argument_errors(lib):
    f = lib.fp8_quant_act_1x128
    assert _rc(f, FAKE, 4, 100, 104, 0, FAKE, FAKE, None) == _lib.FP8FG_ERR_ARG        # K % 128
    assert b"multiple of 128" in lib.fp8fg_last_error()
    assert _rc(f, FAKE, 100, 256, 256, 1, FAKE, FAKE, None) == _lib.FP8FG_ERR_ARG      # M % 128 (transposed)
    assert _rc(f, FAKE, 128, 12, 12, 1, FAKE, FAKE, None) == _lib.FP8FG_ERR_ARG        # K % 8 (transposed)
    assert _rc(f, FAKE, 4, 256, 128, 0, FAKE, FAKE, None) == _lib.FP8FG_ERR_ARG        # ldx < K
    assert _rc(f, FAKE, 4, 256, 260, 0, FAKE, FAKE, None) == _lib.FP8FG_ERR_ARG        # ldx % 8
    assert _rc(f, FAKE, 4, 256, 256, 2, FAKE, FAKE, None) == _lib.FP8FG_ERR_ARG        # transposed flag
    assert _rc(f, None, 4, 256, 256, 0, FAKE, FAKE, None) == _lib.FP8FG_ERR_ARG        # null
    assert _rc(f, FAKE + 8, 4, 256, 256, 0, FAKE, FAKE, None) == _lib.FP8FG_ERR_ARG    # misaligned
    assert _rc(f, FAKE, -1, 256, 256, 0, FAKE, FAKE, None) == _lib.FP8FG_ERR_ARG       # negative
    assert _rc(f, None, 0, 256, 256, 0, None, None, None) == _lib.FP8FG_OK             # empty: no launch
    assert lib.fp8fg_last_error() == b""


def test_quant_delayed_argument_errors(lib):
    f = lib.fp8_quant_act_delayed
    ok = (FAKE, 4, 256, 256, FAKE, 16, FAKE, FAKE, None)

    def with_(i, v):
        a = list(ok)
        a[i] = v
        return _rc(f, *a)
    assert with_(2, 200) == _lib.FP8FG_ERR_ARG          # K % 128
    assert with_(5, 0) == _lib.FP8FG_ERR_ARG            # H
    assert with_(5, 1025) == _lib.FP8FG_ERR_ARG
    assert with_(4, None) == _lib.FP8FG_ERR_ARG         # history
    assert with_(4, FAKE + 4) == _lib.FP8FG_ERR_ARG     # misaligned history
    assert with_(6, None) == _lib.FP8FG_ERR_ARG         # null q


def test_quant_w_argument_errors(lib):
    f = lib.fp8_quant_w_128x128
    assert _rc(f, FAKE, 100, 128, 128, FAKE, FAKE, None) == _lib.FP8FG_ERR_ARG
    assert _rc(f, FAKE, 128, 130, 136, FAKE, FAKE, None) == _lib.FP8FG_ERR_ARG
    assert _rc(f, FAKE, 128, 128, 120, FAKE, FAKE, None) == _lib.FP8FG_ERR_ARG
    assert _rc(f, FAKE, 128, 128, 128, None, FAKE, None) == _lib.FP8FG_ERR_ARG
    assert _rc(f, None, 0, 128, 128, None, None, None) == _lib.FP8FG_OK


def test_dual_quant_argument_errors(lib):
    f = lib.fp8_quant_act_1x128_dual
    ok = (FAKE, 256, 384, 384, FAKE, FAKE, FAKE, FAKE, None)

    def with_(fn, base, i, v):
        a = list(base)
        a[i] = v
        return _rc(fn, *a)
    assert with_(f, ok, 1, 200) == _lib.FP8FG_ERR_ARG      # M % 128
    assert with_(f, ok, 2, 200) == _lib.FP8FG_ERR_ARG      # K % 128
    assert with_(f, ok, 3, 256) == _lib.FP8FG_ERR_ARG      # ldx < K
    assert with_(f, ok, 3, 388) == _lib.FP8FG_ERR_ARG      # ldx % 8
    assert with_(f, ok, 6, None) == _lib.FP8FG_ERR_ARG     # null qt
    assert with_(f, ok, 7, FAKE + 4) == _lib.FP8FG_ERR_ARG  # misaligned st
    assert with_(f, ok, 1, 0) == _lib.FP8FG_OK             # empty
    g = lib.fp8_quant_w_128x128_dual
    assert with_(g, ok, 1, 200) == _lib.FP8FG_ERR_ARG      # N % 128
    assert with_(g, ok, 2, 136) == _lib.FP8FG_ERR_ARG      # K % 128
    assert with_(g, ok, 6, None) == _lib.FP8FG_ERR_ARG     # null qt
    assert with_(g, ok, 2, 0) == _lib.FP8FG_OK             # empty


def test_gemm_argument_errors(lib):
    f = lib.fp8_blockscaled_gemm
    ok = (FAKE, FAKE, FAKE, FAKE, 0, FAKE, 1, 128, 256, 256, None)

    def with_(i, v):
        a = list(ok)
        a[i] = v
        return _rc(f, *a)
    assert with_(4, 7) == _lib.FP8FG_ERR_ARG            # sb_kind
    assert with_(6, 9) == _lib.FP8FG_ERR_ARG            # c_dtype
    assert with_(9, 200) == _lib.FP8FG_ERR_ARG          # K % 128
    assert with_(8, 100) == _lib.FP8FG_ERR_ARG          # N % 128
    assert with_(0, None) == _lib.FP8FG_ERR_ARG         # null qa
    assert with_(5, FAKE + 4) == _lib.FP8FG_ERR_ARG     # misaligned c
    assert with_(7, -5) == _lib.FP8FG_ERR_ARG           # negative M
    assert with_(7, 0) == _lib.FP8FG_OK                 # empty


def test_gemm_e4m3_argument_errors(lib):
    f = lib.fp8_blockscaled_gemm_e4m3
    ok = (FAKE, FAKE, FAKE, FAKE, 0, FAKE, FAKE, 128, 256, 256, None)

    def with_(i, v):
        a = list(ok)
        a[i] = v
        return _rc(f, *a)
    assert with_(4, 3) == _lib.FP8FG_ERR_ARG            # sb_kind
    assert with_(8, 200) == _lib.FP8FG_ERR_ARG          # N % 128
    assert with_(9, 100) == _lib.FP8FG_ERR_ARG          # K % 128
    assert with_(6, None) == _lib.FP8FG_ERR_ARG         # null scale output
    assert with_(5, FAKE + 8) == _lib.FP8FG_ERR_ARG     # misaligned codes
    assert with_(7, 0) == _lib.FP8FG_OK                 # empty


def test_gemm_ws_argument_errors(lib):
    f = lib.fp8_blockscaled_gemm_ws
    ok = [FAKE, FAKE, FAKE, FAKE, 0, FAKE, 1, 128, 256, 256, FAKE, 1 << 30, None]

    def with_(i, v):
        a = list(ok)
        a[i] = v
        return _rc(f, *a)
    assert with_(10, None) == _lib.FP8FG_ERR_ARG        # null workspace
    assert with_(10, FAKE + 8) == _lib.FP8FG_ERR_ARG    # misaligned workspace


def test_grouped_argument_errors(lib):
    f = lib.fp8_grouped_gemm
    ok = [FAKE, FAKE, FAKE, FAKE, FAKE, 4, 512, FAKE, 1, 256, 256, None]

    def with_(i, v):
        a = list(ok)
        a[i] = v
        return _rc(f, *a)
    assert with_(5, 0) == _lib.FP8FG_ERR_ARG            # E
    assert with_(5, 5000) == _lib.FP8FG_ERR_ARG
    assert with_(6, 500) == _lib.FP8FG_ERR_ARG          # Mtot % 128
    assert with_(4, None) == _lib.FP8FG_ERR_ARG         # offsets null
    assert with_(4, FAKE + 2) == _lib.FP8FG_ERR_ARG     # offsets misaligned
    assert with_(6, 0) == _lib.FP8FG_OK                 # empty


def test_binding_raises_on_error(lib):
    with pytest.raises(_lib.Fp8fgError) as ei:
        _lib.fp8_quant_w_128x128(FAKE, 100, 128, 128, FAKE, FAKE, None)
    assert ei.value.code == _lib.FP8FG_ERR_ARG


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "absent.so"))
    with pytest.raises(RuntimeError, match="missing"):
        _lib.lib()
    assert isinstance(ctypes.CDLL, type)


def test_quant_transposed_pair_argument_errors(lib):
    f = lib.fp8_quant_act_1x128_transposed_pair
    ok = [FAKE, 256, 256, FAKE, FAKE, FAKE, 512, 512, FAKE, FAKE, 384, None]

    def with_(**kw):
        names = ["x0", "K0", "ldx0", "q0", "s0", "x1", "K1", "ldx1", "q1", "s1", "M", "stream"]
        a = list(ok)
        for k, v in kw.items():
            a[names.index(k)] = v
        return _rc(f, *a)
    assert with_(M=100) == _lib.FP8FG_ERR_ARG                                   # M % 128
    assert b"multiple of 128" in lib.fp8fg_last_error()
    assert with_(K1=12) == _lib.FP8FG_ERR_ARG                                   # K % 8
    assert with_(ldx0=128) == _lib.FP8FG_ERR_ARG                                # ldx < K
    assert with_(x1=None) == _lib.FP8FG_ERR_ARG                                 # null
    assert with_(q0=FAKE + 8) == _lib.FP8FG_ERR_ARG                             # misaligned
    assert with_(K0=-1) == _lib.FP8FG_ERR_ARG                                   # negative
    assert with_(M=0, x0=None, x1=None, q0=None, q1=None, s0=None, s1=None) == _lib.FP8FG_OK   # empty
    assert lib.fp8fg_last_error() == b""


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_c_program_against_the_header_and_library(lib, tmp_path):
    """The ABI used from plain C: tests/csrc/abi_host_check.c includes include/fp8fg.h,
    links libfp8fg.so and checks argument rejection and empty problems (no GPU needed)."""
    exe = str(tmp_path / "abi_check")
    libdir = os.path.dirname(_lib.LIB_PATH)
    src = os.path.join(ROOT, "tests", "csrc", "abi_host_check.c")
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), "-o", exe, src,
                    "-L", libdir, "-l:libfp8fg.so", f"-Wl,-rpath,{libdir}"], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    checks, failures = map(int, r.stdout.split())
    assert r.returncode == 0 and failures == 0 and checks >= 19, r.stderr
