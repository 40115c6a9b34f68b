"""The C-ABI library builds, loads and exports every symbol include/*.h declares; host-side
argument checks reject bad input before any CUDA call (no GPU needed)."""
import ctypes
import glob
import math
import os
import re

import pytest

from speculative_decoding_verification_33_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for path in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(path).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(",
                             text, flags=re.M):
            if not m.group(0).lstrip().startswith(("typedef", "#", "return")):
                names.add(m.group(1))
    return names


def test_every_declared_symbol_is_exported():
    lib = _lib.load()
    names = declared_functions()
    assert {"spec_verify", "spec_verify_debug", "spec_verify_host", "sv_hbm_read_probe"} <= names
    for n in names:
        assert hasattr(lib, n), n
    assert set(_lib.EXPORTS) == names


def test_struct_layout_matches_header():
    # B, K, V, dtype (4 x int), two long long, bias_k, pointer, cluster_hint
    assert ctypes.sizeof(_lib.SvProblem) == 56
    assert _lib.SvProblem.fanout.offset == 40 and _lib.SvProblem.cluster_hint.offset == 48


def test_status_strings():
    for code in range(5):
        assert _lib.status_string(code)
    assert _lib.status_string(99) == "unknown status"


def test_workspace_bytes():
    # a fixed 256-byte header: the sequence queue counter, the finished-cluster count, the error word
    for B in (0, 1, 64, 65, 5000, 70000):
        prob, _ = _lib.make_problem(B, 1, 1, 0, 1, 1)
        assert _lib.call("spec_verify_workspace_bytes", prob) == 256


def _status(entry="spec_verify", mode=1, T=1.0, beta=1.0, ptrs=1, topf=0, extra=(), **kw):
    base = dict(B=0, K=4, V=100, dtype=1, target_row_stride=100, draft_row_stride=100,
                bias_k=0, fanout=None, cluster_hint=0)
    base.update(kw)
    prob, keep = _lib.make_problem(**base)
    p = ptrs
    args = [p, p, p, p, p, T, beta, mode, p, p, topf]
    if entry == "spec_verify_ws":
        args += list(extra)
    st = _lib.call(entry, prob, *args, 0)
    del keep
    return st


BAD_PROBLEMS = [dict(K=0), dict(K=9), dict(V=0), dict(V=262145), dict(B=-1), dict(dtype=2),
                dict(target_row_stride=99), dict(draft_row_stride=50), dict(cluster_hint=3),
                dict(cluster_hint=32), dict(bias_k=9), dict(fanout=[1, 2, 9, 0])]


@pytest.mark.parametrize("kw", BAD_PROBLEMS)
def test_bad_problem_rejected(kw):
    assert _status(**kw) == _lib.SV_ERR_INVALID_ARG


@pytest.mark.parametrize("T,beta", [(0.0, 1.0), (math.nan, 1.0), (math.inf, 1.0), (1e-5, 1.0),
                                    (1.0, 0.0), (1.0, 1.5), (1.0, math.nan)])
def test_bad_scalars_rejected(T, beta):
    assert _status(T=T, beta=beta) == _lib.SV_ERR_INVALID_ARG


def test_greedy_ignores_sampling_scalars_but_not_fanout():
    assert _status(mode=0, T=0.0, beta=7.0, bias_k=0) == _lib.SV_OK
    assert _status(mode=0, fanout=[1, 1, 1, 1], topf=1) == _lib.SV_ERR_INVALID_ARG
    assert _status(mode=3) == _lib.SV_ERR_INVALID_ARG


def test_null_pointers_rejected_when_batch_nonempty():
    assert _status(B=2, ptrs=0) == _lib.SV_ERR_INVALID_ARG
    assert _status(B=0, ptrs=0) == _lib.SV_OK  # nothing to do
    # top-F output requested without a buffer, or a buffer without fan-out
    assert _status(B=2, fanout=[1, 1, 1, 1], topf=0) == _lib.SV_ERR_INVALID_ARG
    assert _status(B=2, fanout=None, topf=1) == _lib.SV_ERR_INVALID_ARG


def test_workspace_entry_checks_workspace():
    assert _status("spec_verify_ws", extra=(0, 256)) == _lib.SV_ERR_INVALID_ARG
    assert _status("spec_verify_ws", extra=(16, 100)) == _lib.SV_ERR_INVALID_ARG
    assert _status("spec_verify_ws", extra=(8, 256)) == _lib.SV_ERR_INVALID_ARG
    assert _status("spec_verify_ws", B=64, extra=(16, 240)) == _lib.SV_ERR_INVALID_ARG


def test_error_readers_and_targeted_probe_check_arguments():
    lib = _lib.load()
    assert lib.spec_verify_workspace_error(None, None) == _lib.SV_ERR_INVALID_ARG
    assert lib.spec_verify_workspace_error(8, None) == _lib.SV_ERR_INVALID_ARG  # misaligned
    assert lib.sv_wait_probe_at(1000, 0, None, None) == _lib.SV_ERR_INVALID_ARG  # bad target
    assert lib.sv_wait_probe_at(0, _lib.SV_PROBE_NOALLOC, None, None) == _lib.SV_ERR_INVALID_ARG
    assert lib.sv_wait_probe_at(1000, _lib.SV_PROBE_WORKSPACE, None, None) == _lib.SV_ERR_INVALID_ARG
    assert lib.sv_wait_probe_at(1000, _lib.SV_PROBE_WORKSPACE, 8, None) == _lib.SV_ERR_INVALID_ARG


def test_probe_checks_arguments():
    lib = _lib.load()
    assert lib.sv_hbm_read_probe(None, 16, 16, None) == _lib.SV_ERR_INVALID_ARG
    assert lib.sv_hbm_read_probe(16, 15, 16, None) == _lib.SV_ERR_INVALID_ARG


def test_binding_refuses_host_tensors():
    torch = pytest.importorskip("torch")
    from speculative_decoding_verification_33_gb300 import api
    t = torch.zeros(1, 3, 8, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        api.verify(t, None, torch.zeros(1, 2, dtype=torch.int32), mode="greedy")


@pytest.mark.parametrize("kw", BAD_PROBLEMS[:6])
def test_route_query_checks_the_problem(kw):
    """spec_verify_route validates the problem on the host before it asks the device anything."""
    base = dict(B=2, K=4, V=1000, dtype=_lib.SV_DTYPE_BF16, target_row_stride=1000,
                draft_row_stride=1000)
    base.update(kw)
    prob, keep = _lib.make_problem(**base)
    r, n = ctypes.c_int(-7), ctypes.c_int(-7)
    st = _lib.load().spec_verify_route(ctypes.byref(prob), _lib.SV_MODE_STOCHASTIC,
                                       ctypes.addressof(r), ctypes.addressof(n))
    del keep
    assert st == _lib.SV_ERR_INVALID_ARG
    assert r.value == -7 and n.value == -7  # outputs untouched on an error
    assert _lib.load().spec_verify_route(None, _lib.SV_MODE_STOCHASTIC, None, None) == \
        _lib.SV_ERR_INVALID_ARG
