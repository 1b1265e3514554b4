"""The C-ABI library builds, loads and exports every symbol the public header
declares; argument checks that run before any CUDA call work without a GPU."""
import ctypes
import os
import re

import pytest

import nonuniform_fft_gb300 as nf
from nonuniform_fft_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nufft_gb300.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return nf.load_library()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(nufft_[a-z_]+)\s*\(", src)))


def declared_codes():
    src = open(HEADER).read()
    return {name: int(v) for name, v in re.findall(r"#define (NUFFT_ERR_[A-Z_]+|NUFFT_OK) (\d+)", src)}


def test_header_declares_the_entry_points():
    names = declared_functions()
    for required in ("nufft_makeplan", "nufft_setpts", "nufft_execute", "nufft_destroy",
                     "nufft_set_opt", "nufft_get_timings", "nufft_strerror"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_binding_mirrors_header_codes():
    codes = declared_codes()
    assert codes["NUFFT_OK"] == nf.OK
    assert codes["NUFFT_ERR_BAD_ARG"] == nf.ERR_BAD_ARG
    assert codes["NUFFT_ERR_BAD_EPS"] == nf.ERR_BAD_EPS
    assert codes["NUFFT_ERR_NO_POINTS"] == nf.ERR_NO_POINTS
    assert codes["NUFFT_ERR_BAD_POINTS"] == nf.ERR_BAD_POINTS
    assert codes["NUFFT_ERR_BAD_OPT"] == nf.ERR_BAD_OPT
    src = open(HEADER).read()
    assert len(nf.TIMING_KEYS) == int(re.search(r"#define NUFFT_T_COUNT (\d+)", src).group(1))
    assert len(nf.INFO_KEYS) == int(re.search(r"#define NUFFT_I_COUNT (\d+)", src).group(1))


def test_strerror_names_every_code(lib):
    for name, code in declared_codes().items():
        msg = nf.strerror(code)
        assert msg and msg != "unknown error code", name
    assert nf.strerror(12345) == "unknown error code"


def _makeplan(lib, type_, dim, modes, iflag, eps, dtype):
    arr = (ctypes.c_int64 * max(1, len(modes)))(*modes) if modes is not None else None
    out = ctypes.c_void_p(1234)
    rc = lib.nufft_makeplan(type_, dim, arr, iflag, eps, dtype, None, ctypes.byref(out))
    return rc, out.value


@pytest.mark.parametrize("args,code", [
    ((3, 2, [8, 8], -1, 1e-6, 0), nf.ERR_BAD_ARG),       # type
    ((1, 0, [8], -1, 1e-6, 0), nf.ERR_BAD_ARG),          # dim
    ((1, 4, [8, 8, 8, 8], -1, 1e-6, 0), nf.ERR_BAD_ARG),
    ((1, 2, [8, 0], -1, 1e-6, 0), nf.ERR_BAD_ARG),       # N < 1
    ((1, 2, None, -1, 1e-6, 0), nf.ERR_BAD_ARG),         # NULL modes
    ((1, 2, [8, 8], -1, 1e-6, 2), nf.ERR_BAD_ARG),       # dtype
    ((1, 2, [8, 8], -1, 0.0, 0), nf.ERR_BAD_EPS),
    ((1, 2, [8, 8], -1, -1e-3, 0), nf.ERR_BAD_EPS),
    ((1, 2, [8, 8], -1, float("nan"), 0), nf.ERR_BAD_EPS),
    ((1, 2, [8, 8], -1, 1.0, 0), nf.ERR_BAD_EPS),        # w = 1
    ((1, 2, [8, 8], -1, 1e-16, 1), nf.ERR_BAD_EPS),      # w = 17
])
def test_makeplan_rejects_bad_arguments(lib, args, code):
    rc, plan = _makeplan(lib, *args)
    assert rc == code
    assert plan is None


@pytest.mark.parametrize("sigma,code", [(1.0, nf.ERR_BAD_ARG), (0.5, nf.ERR_BAD_ARG),
                                        (2.5, nf.ERR_BAD_ARG), (float("nan"), nf.ERR_BAD_ARG),
                                        (-1.5, nf.ERR_BAD_ARG)])
def test_makeplan_upsampled_rejects_bad_sigma(lib, sigma, code):
    arr = (ctypes.c_int64 * 2)(8, 8)
    out = ctypes.c_void_p(1234)
    assert lib.nufft_makeplan_upsampled(1, 2, arr, -1, 1e-6, 0, sigma, None, ctypes.byref(out)) == code
    assert out.value is None


def test_makeplan_upsampled_width_limit(lib):
    """sigma = 1.25 stretches eq. (6): eps = 1e-10 needs w = ceil(10 / sqrt(0.4)) + 1
    = 17 > 16, rejected before any device work; at sigma = 2 eps = 1e-10 is fine
    in principle (w = 11) but needs a GPU, so only the rejection is checked."""
    arr = (ctypes.c_int64 * 2)(8, 8)
    out = ctypes.c_void_p(1234)
    assert lib.nufft_makeplan_upsampled(1, 2, arr, -1, 1e-10, 1, 1.25, None,
                                        ctypes.byref(out)) == nf.ERR_BAD_EPS
    assert out.value is None


def test_null_plan_calls(lib):
    assert lib.nufft_set_opt(None, b"msub", 64.0) == nf.ERR_BAD_ARG
    assert lib.nufft_setpts(None, 10, None, None, None) == nf.ERR_BAD_ARG
    assert lib.nufft_execute(None, None, None) == nf.ERR_BAD_ARG
    assert lib.nufft_execute_batch(None, 1, None, None) == nf.ERR_BAD_ARG
    assert lib.nufft_destroy(None) == nf.OK
    buf = (ctypes.c_double * 6)()
    assert lib.nufft_get_timings(None, buf, 6) == nf.ERR_BAD_ARG
    ibuf = (ctypes.c_int64 * 13)()
    assert lib.nufft_get_info(None, ibuf, 13) == nf.ERR_BAD_ARG
    assert lib.nufft_get_sort(None, None, None, None, None) == nf.ERR_BAD_ARG
    assert lib.nufft_makeplan(1, 2, (ctypes.c_int64 * 2)(8, 8), -1, 1e-6, 0, None, None) == nf.ERR_BAD_ARG


def test_binding_raises_when_library_missing(tmp_path, monkeypatch):
    monkeypatch.setattr(nf, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        nf.load_library(str(tmp_path / "nope.so"))
