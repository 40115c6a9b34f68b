"""ctypes binding of the C ABI in include/spec_verify.h (argument marshalling only).

PyTorch supplies device memory and streams; every step of the verify path runs in the CUDA
library. There is no CPU fallback: if the library cannot be built or loaded, calls raise.
"""
from __future__ import annotations

import ctypes
import threading
from typing import Optional, Sequence

from . import build as _build

SV_OK, SV_ERR_INVALID_ARG, SV_ERR_UNSUPPORTED, SV_ERR_CUDA, SV_ERR_DEVICE_TIMEOUT = range(5)
SV_DTYPE_F32, SV_DTYPE_BF16 = 0, 1
SV_MODE_GREEDY, SV_MODE_STOCHASTIC = 0, 1

# every entry point the header declares (checked by the tests against include/*.h)
EXPORTS = ("spec_verify", "spec_verify_workspace_bytes", "spec_verify_ws", "spec_verify_debug",
           "spec_verify_host", "spec_verify_device_error", "spec_verify_status_string",
           "spec_verify_plan", "spec_verify_route", "spec_verify_noalloc", "spec_draft_sample", "spec_residual_topf",
           "spec_lmhead_stats", "spec_verify_hidden", "sv_hbm_read_probe", "sv_wait_probe",
           "spec_verify_workspace_error", "sv_wait_probe_at")
SV_PROBE_NOALLOC, SV_PROBE_WORKSPACE = 1, 2


class SvProblem(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("K", ctypes.c_int), ("V", ctypes.c_int),
                ("dtype", ctypes.c_int), ("target_row_stride", ctypes.c_longlong),
                ("draft_row_stride", ctypes.c_longlong), ("bias_k", ctypes.c_int),
                ("fanout", ctypes.POINTER(ctypes.c_int)), ("cluster_hint", ctypes.c_int)]


class SpecVerifyError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


_lock = threading.Lock()
_lib: Optional[ctypes.CDLL] = None

_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_SZ = ctypes.c_size_t
_PROB = ctypes.POINTER(SvProblem)
_COMMON = [_PROB, _P, _P, _P, _P, _P, _F, _F, _I, _P, _P, _P]


def load(build_if_needed: bool = True) -> ctypes.CDLL:
    """Load (building first if the sources changed) the verify library."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.build() if build_if_needed else _build.lib_path()
        lib = ctypes.CDLL(path)
        lib.spec_verify.argtypes = _COMMON + [_P]
        lib.spec_verify_ws.argtypes = _COMMON + [_P, _SZ, _P]
        lib.spec_verify_debug.argtypes = _COMMON + [_P, _P, _P, _P, _P]
        lib.spec_verify_host.argtypes = _COMMON + [_P]
        lib.spec_verify_noalloc.argtypes = _COMMON + [_P]
        lib.spec_verify_workspace_bytes.argtypes = [_PROB]
        lib.spec_verify_workspace_bytes.restype = _SZ
        lib.spec_verify_device_error.argtypes = [_P]
        lib.spec_verify_status_string.argtypes = [_I]
        lib.spec_verify_status_string.restype = ctypes.c_char_p
        lib.sv_hbm_read_probe.argtypes = [_P, _SZ, _P, _P]
        lib.sv_wait_probe.argtypes = [ctypes.c_uint, _P]
        lib.sv_wait_probe_at.argtypes = [ctypes.c_uint, _I, _P, _P]
        lib.spec_verify_workspace_error.argtypes = [_P, _P]
        lib.spec_verify_plan.argtypes = [_PROB, _I, _P, _P, _P]
        lib.spec_verify_route.argtypes = [_PROB, _I, _P, _P]
        lib.spec_draft_sample.argtypes = [_I, _I, _I, ctypes.c_longlong, _P, _P, _F, _F, _I,
                                          _F, _P, _P, _P, _P]
        lib.spec_residual_topf.argtypes = [_PROB, _P, _P, _P, _F, _F, _P, _P, _P, _P, _P, _P]
        lib.spec_lmhead_stats.argtypes = [_I, _I, _I, _P, ctypes.c_longlong, _P, ctypes.c_longlong,
                                          _F, _P, _P, _P, _P, _P, _P, _P]
        _LL = ctypes.c_longlong
        lib.spec_verify_hidden.argtypes = [_I, _I, _I, _I, _P, _LL, _P, _LL, _P, _LL, _P, _P, _P,
                                           _F, _F, _I, _P, _I, _P, _P, _P, _P]
        for name in EXPORTS:
            if name not in ("spec_verify_workspace_bytes", "spec_verify_status_string"):
                getattr(lib, name).restype = _I
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load().spec_verify_status_string(int(status)).decode()


def _check(status: int, where: str):
    if status != SV_OK:
        raise SpecVerifyError(status, where)


def make_problem(B: int, K: int, V: int, dtype: int, target_row_stride: int,
                 draft_row_stride: int, bias_k: int = 0,
                 fanout: Optional[Sequence[int]] = None, cluster_hint: int = 0):
    """An SvProblem plus the ctypes array that keeps ``fanout`` alive."""
    fan = None
    if fanout is not None:
        fan = (ctypes.c_int * len(fanout))(*[int(f) for f in fanout])
    prob = SvProblem(int(B), int(K), int(V), int(dtype), int(target_row_stride),
                     int(draft_row_stride), int(bias_k),
                     ctypes.cast(fan, ctypes.POINTER(ctypes.c_int)) if fan is not None else None,
                     int(cluster_hint))
    return prob, fan


def plan(prob: SvProblem, mode: int):
    """(CTAs per cluster, clusters, dynamic shared memory bytes) spec_verify would launch."""
    c, n, sm = ctypes.c_int(), ctypes.c_int(), ctypes.c_size_t()
    _check(load().spec_verify_plan(ctypes.byref(prob), int(mode), ctypes.addressof(c),
                                   ctypes.addressof(n), ctypes.addressof(sm)), "spec_verify_plan")
    return c.value, n.value, sm.value


SV_ROUTE_WALK, SV_ROUTE_GREEDY_ROWS, SV_ROUTE_SMALL = 0, 1, 2


def route(prob: SvProblem, mode: int):
    """(route, kernel launches per call) spec_verify takes for this problem."""
    r, n = ctypes.c_int(), ctypes.c_int()
    _check(load().spec_verify_route(ctypes.byref(prob), int(mode), ctypes.addressof(r),
                                    ctypes.addressof(n)), "spec_verify_route")
    return r.value, n.value


def call(name: str, prob: SvProblem, *args) -> int:
    """Raw call of entry point ``name`` with the problem and plain integer/float arguments."""
    return getattr(load(), name)(ctypes.byref(prob), *args)
