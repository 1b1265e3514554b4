"""GB300 (sm_103a) nonuniform FFT: thin Python binding of the C ABI.

Every function here only marshals arguments to the CUDA library
``libnufft_gb300_<machine>.so`` (declared in ``include/nufft_gb300.h``); all
steps of the transforms run in that library's kernels and in cuFFT.  There is
no CPU fallback: if the library is missing, every call raises.

Arrays may be torch tensors (CUDA or CPU) or numpy arrays; their data pointers
are passed through unchanged (device pointers run asynchronously on the
plan's stream, host pointers are staged by the library and the call is
synchronous).  The transforms are those of "cuFINUFFT: a load-balanced GPU
library for general-purpose nonuniform FFTs" (Shih et al.), eq. (1) (type 1)
and eq. (3) (type 2).
"""
from __future__ import annotations

import ctypes
import os

from ._build import LIB_PATH

__all__ = [
    "makeplan", "set_opt", "setpts", "execute", "execute_batch", "destroy", "get_timings", "get_info",
    "get_sort", "strerror", "Plan", "NufftError", "load_library", "TIMING_KEYS", "INFO_KEYS",
]

# Error codes and result layouts mirrored from include/nufft_gb300.h.
OK = 0
ERR_BAD_ARG, ERR_BAD_EPS, ERR_ALLOC, ERR_CUDA, ERR_CUFFT = 1, 2, 3, 4, 5
ERR_NO_POINTS, ERR_BAD_POINTS, ERR_BAD_OPT, ERR_TOO_LARGE = 6, 7, 8, 9
METHOD_AUTO, METHOD_SM, METHOD_GM_SORT, METHOD_REGTILE, METHOD_GM = 0, 1, 2, 3, 4
TIMING_KEYS = ("spread_interp", "fft", "deconv_pad", "zero", "exec", "setpts")
INFO_KEYS = ("w", "n1", "n2", "n3", "M", "nbins", "nsub", "bin1", "bin2", "bin3", "msub", "method",
             "batch", "fft", "sms", "tile3d", "igroup", "bin_origin")

_lib = None


class NufftError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {strerror(code)} (code {code})")


def load_library(path: str | None = None):
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(
            f"CUDA library {path} is missing: build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'` (needs nvcc)")
    lib = ctypes.CDLL(path)
    P, I, I64, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
    lib.nufft_makeplan.argtypes = [I, I, ctypes.POINTER(I64), I, D, I, P, ctypes.POINTER(P)]
    lib.nufft_makeplan_upsampled.argtypes = [I, I, ctypes.POINTER(I64), I, D, I, D, P,
                                             ctypes.POINTER(P)]
    lib.nufft_set_opt.argtypes = [P, ctypes.c_char_p, D]
    lib.nufft_setpts.argtypes = [P, I64, P, P, P]
    lib.nufft_execute.argtypes = [P, P, P]
    lib.nufft_execute_batch.argtypes = [P, I64, P, P]
    lib.nufft_destroy.argtypes = [P]
    lib.nufft_get_timings.argtypes = [P, ctypes.POINTER(D), I]
    lib.nufft_get_info.argtypes = [P, ctypes.POINTER(I64), I]
    lib.nufft_get_sort.argtypes = [P, P, P, P, P]
    lib.nufft_strerror.argtypes = [I]
    lib.nufft_strerror.restype = ctypes.c_char_p
    for name in ("nufft_makeplan", "nufft_makeplan_upsampled", "nufft_set_opt", "nufft_setpts", "nufft_execute",
                 "nufft_execute_batch", "nufft_destroy", "nufft_get_timings", "nufft_get_info",
                 "nufft_get_sort"):
        getattr(lib, name).restype = I
    _lib = lib
    return lib


def _check(code: int, where: str):
    if code != OK:
        raise NufftError(code, where)


def _ptr(a) -> int | None:
    """Data pointer of a torch tensor or numpy array (None passes NULL)."""
    if a is None:
        return None
    if hasattr(a, "data_ptr"):
        if not a.is_contiguous():
            raise ValueError("arrays must be contiguous")
        return a.data_ptr()
    if hasattr(a, "ctypes"):
        if not a.flags["C_CONTIGUOUS"]:
            raise ValueError("arrays must be contiguous")
        return a.ctypes.data
    if isinstance(a, int):
        return a
    raise TypeError(f"unsupported array type {type(a)!r}")


def _current_stream() -> int | None:
    try:
        import torch
        if torch.cuda.is_available():
            return torch.cuda.current_stream().cuda_stream
    except ImportError:
        pass
    return None


def strerror(code: int) -> str:
    return load_library().nufft_strerror(code).decode()


def makeplan(type: int, n_modes, iflag: int, eps: float, dtype: str = "complex64",
             stream: int | None = None, sigma: float = 2.0) -> int:
    """nufft_makeplan (sigma = 2) or nufft_makeplan_upsampled: returns an
    opaque plan handle.  dtype 'complex64' or 'complex128'; stream a
    cudaStream_t value (default: torch's current)."""
    lib = load_library()
    dims = list(n_modes)
    arr = (ctypes.c_int64 * len(dims))(*dims)
    code_dtype = {"complex64": 0, "complex128": 1}[str(dtype).replace("torch.", "")]
    out = ctypes.c_void_p()
    s = _current_stream() if stream is None else stream
    sp = ctypes.c_void_p(s) if s else None
    if float(sigma) == 2.0:
        rc = lib.nufft_makeplan(int(type), len(dims), arr, int(iflag), float(eps), code_dtype, sp,
                                ctypes.byref(out))
    else:
        rc = lib.nufft_makeplan_upsampled(int(type), len(dims), arr, int(iflag), float(eps),
                                          code_dtype, float(sigma), sp, ctypes.byref(out))
    _check(rc, "makeplan")
    return out.value


def set_opt(plan: int, key: str, value: float):
    _check(load_library().nufft_set_opt(plan, key.encode(), float(value)), f"set_opt({key})")


def setpts(plan: int, M: int, x, y=None, z=None):
    _check(load_library().nufft_setpts(plan, int(M), _ptr(x), _ptr(y), _ptr(z)), "setpts")


def execute(plan: int, c, f):
    _check(load_library().nufft_execute(plan, _ptr(c), _ptr(f)), "execute")


def execute_batch(plan: int, nvec: int, c, f):
    """nufft_execute_batch: nvec vectors stored back to back in c and f."""
    _check(load_library().nufft_execute_batch(plan, int(nvec), _ptr(c), _ptr(f)), "execute_batch")


def destroy(plan: int):
    _check(load_library().nufft_destroy(plan), "destroy")


def get_timings(plan: int) -> dict:
    buf = (ctypes.c_double * len(TIMING_KEYS))()
    _check(load_library().nufft_get_timings(plan, buf, len(TIMING_KEYS)), "get_timings")
    return dict(zip(TIMING_KEYS, list(buf)))


def get_info(plan: int) -> dict:
    buf = (ctypes.c_int64 * len(INFO_KEYS))()
    _check(load_library().nufft_get_info(plan, buf, len(INFO_KEYS)), "get_info")
    return dict(zip(INFO_KEYS, list(buf)))


def get_sort(plan: int) -> dict:
    """Integer setpts results (host numpy arrays): counts, starts, perm, subproblems."""
    import numpy as np
    info = get_info(plan)
    counts = np.zeros(info["nbins"], np.int32)
    starts = np.zeros(info["nbins"], np.int32)
    perm = np.zeros(info["M"], np.int32)
    sub = np.zeros((info["nsub"], 3), np.int32)
    _check(load_library().nufft_get_sort(plan, counts.ctypes.data, starts.ctypes.data,
                                         perm.ctypes.data if perm.size else None,
                                         sub.ctypes.data if sub.size else None), "get_sort")
    return {"counts": counts, "starts": starts, "perm": perm, "subproblems": sub}


class Plan:
    """Owning wrapper: Plan(type, n_modes, iflag, eps, dtype) ... close()."""

    def __init__(self, type: int, n_modes, iflag: int, eps: float, dtype: str = "complex64",
                 stream: int | None = None, sigma: float = 2.0, **opts):
        self.type = type
        self.n_modes = tuple(int(n) for n in n_modes)
        self.dtype = dtype
        self.handle = None
        self.handle = makeplan(type, self.n_modes, iflag, eps, dtype, stream, sigma)
        for k, v in opts.items():
            set_opt(self.handle, k, v)
        self.M = 0

    def set_opt(self, key: str, value: float):
        set_opt(self.handle, key, value)

    def setpts(self, x, y=None, z=None):
        self.M = int(x.shape[0]) if hasattr(x, "shape") else len(x)
        setpts(self.handle, self.M, x, y, z)

    def execute(self, c, f):
        execute(self.handle, c, f)

    def execute_batch(self, nvec: int, c, f):
        execute_batch(self.handle, nvec, c, f)

    def timings(self) -> dict:
        return get_timings(self.handle)

    def info(self) -> dict:
        return get_info(self.handle)

    def sort(self) -> dict:
        return get_sort(self.handle)

    def close(self):
        if self.handle:
            destroy(self.handle)
            self.handle = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
