"""Python API of the verify step over torch tensors.

``spec_verify`` mirrors the C entry point argument for argument (target_logits, draft_logits,
draft_tokens, draft_lens, uniforms, temperature, beta, mode, out_accept_len, out_tokens,
out_residual_topF, stream); shapes, dtype and strides are read from the tensors. ``verify``
allocates the outputs and returns them. ``verify_host`` is the end-to-end form over host
(numpy or pinned torch) arrays.
"""
from __future__ import annotations

import ctypes
from typing import Optional, Sequence

import numpy as np
import torch

from . import _lib
from ._lib import SV_DTYPE_BF16, SV_DTYPE_F32, SV_MODE_GREEDY, SV_MODE_STOCHASTIC

_MODES = {"greedy": SV_MODE_GREEDY, "stochastic": SV_MODE_STOCHASTIC,
          SV_MODE_GREEDY: SV_MODE_GREEDY, SV_MODE_STOCHASTIC: SV_MODE_STOCHASTIC}


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return SV_DTYPE_BF16
    if t.dtype == torch.float32:
        return SV_DTYPE_F32
    raise TypeError(f"logits must be bfloat16 or float32, got {t.dtype}")


def _row_stride(t: torch.Tensor, rows: int, name: str) -> int:
    if t.dim() != 3 or t.shape[1] != rows:
        raise ValueError(f"{name} must be [B, {rows}, V], got {tuple(t.shape)}")
    if t.stride(2) != 1 or (t.shape[0] > 1 and t.stride(0) != rows * t.stride(1)):
        raise ValueError(f"{name}: rows must be contiguous with a uniform row stride")
    return t.stride(1)


def _ptr(t: Optional[torch.Tensor], name: str, dtype=None, device=True) -> int:
    if t is None:
        return 0
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if device and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous() and dtype is not None:
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _stream_handle(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _problem(target_logits, draft_logits, draft_tokens, mode, bias_k, fanout, cluster_hint):
    B, K = draft_tokens.shape
    V = target_logits.shape[2]
    ts = _row_stride(target_logits, K + 1, "target_logits")
    ds = _row_stride(draft_logits, K, "draft_logits") if draft_logits is not None else V
    if draft_logits is not None and draft_logits.dtype != target_logits.dtype:
        raise TypeError("target and draft logits must share a dtype")
    return _lib.make_problem(B, K, V, _dtype_code(target_logits), ts, ds, bias_k, fanout,
                             cluster_hint)


def spec_verify(target_logits: torch.Tensor, draft_logits: Optional[torch.Tensor],
                draft_tokens: torch.Tensor, draft_lens: Optional[torch.Tensor],
                uniforms: Optional[torch.Tensor], temperature: float, beta: float, mode,
                out_accept_len: torch.Tensor, out_tokens: torch.Tensor,
                out_residual_topF: Optional[torch.Tensor] = None, stream=None, *,
                bias_k: int = 0, fanout: Optional[Sequence[int]] = None,
                cluster_hint: int = 0, workspace: Optional[torch.Tensor] = None,
                debug: Optional[dict] = None, no_alloc: bool = False) -> None:
    """Run the verify step on the GPU (see include/spec_verify.h for the semantics).

    ``debug`` may hold float32 CUDA tensors ``lse_t`` [B, K+1], ``lse_d``, ``p_x``, ``q_x``
    [B, K]; they are filled by the diagnostic entry point. ``workspace`` selects the
    caller-owned-workspace entry point, ``no_alloc`` the one that allocates no device memory.
    """
    m = _MODES[mode]
    prob, keep = _problem(target_logits, draft_logits, draft_tokens, m, bias_k, fanout,
                          cluster_hint)
    args = [_ptr(target_logits, "target_logits"), _ptr(draft_logits, "draft_logits"),
            _ptr(draft_tokens, "draft_tokens", torch.int32),
            _ptr(draft_lens, "draft_lens", torch.int32),
            _ptr(uniforms, "uniforms", torch.float32), float(temperature), float(beta), m,
            _ptr(out_accept_len, "out_accept_len", torch.int32),
            _ptr(out_tokens, "out_tokens", torch.int32),
            _ptr(out_residual_topF, "out_residual_topF", torch.int32)]
    s = _stream_handle(stream)
    if debug is not None:
        extra = [_ptr(debug.get(k), k, torch.float32) for k in ("lse_t", "lse_d", "p_x", "q_x")]
        st = _lib.call("spec_verify_debug", prob, *args, *extra, s)
        where = "spec_verify_debug"
    elif no_alloc:
        st = _lib.call("spec_verify_noalloc", prob, *args, s)
        where = "spec_verify_noalloc"
    elif workspace is not None:
        st = _lib.call("spec_verify_ws", prob, *args, _ptr(workspace, "workspace"),
                       workspace.numel() * workspace.element_size(), s)
        where = "spec_verify_ws"
    else:
        st = _lib.call("spec_verify", prob, *args, s)
        where = "spec_verify"
    del keep
    _lib._check(st, where)


def verify(target_logits, draft_logits, draft_tokens, draft_lens=None, uniforms=None, *,
           temperature: float = 1.0, beta: float = 1.0, mode="stochastic", bias_k: int = 0,
           fanout: Optional[Sequence[int]] = None, cluster_hint: int = 0, stream=None,
           debug: bool = False):
    """Allocate the outputs, run ``spec_verify`` and return them as a dict of tensors."""
    B, K = draft_tokens.shape
    dev = target_logits.device
    out = {"accept_len": torch.empty(B, dtype=torch.int32, device=dev),
           "tokens": torch.empty(B, K + 1, dtype=torch.int32, device=dev)}
    fmax = max(fanout) if fanout else 0
    if fanout is not None:
        out["topf"] = torch.empty(B, K, max(fmax, 1), dtype=torch.int32, device=dev)
    dbg = None
    if debug:
        dbg = {"lse_t": torch.empty(B, K + 1, dtype=torch.float32, device=dev),
               "lse_d": torch.empty(B, K, dtype=torch.float32, device=dev),
               "p_x": torch.empty(B, K, dtype=torch.float32, device=dev),
               "q_x": torch.empty(B, K, dtype=torch.float32, device=dev)}
        out.update(dbg)
    spec_verify(target_logits, draft_logits, draft_tokens, draft_lens, uniforms, temperature,
                beta, mode, out["accept_len"], out["tokens"], out.get("topf"), stream,
                bias_k=bias_k, fanout=fanout, cluster_hint=cluster_hint, debug=dbg)
    return out


def draft_sample(draft_logits: torch.Tensor, uniforms: torch.Tensor, *, temperature: float = 1.0,
                 beta: float = 1.0, bias_k: int = 0, tau: float = 0.0, stream=None, out=None):
    """Draw one token per row from the beta-biased draft distribution q' and report the exit
    confidence max q (see ``spec_draft_sample`` in include/spec_verify.h).

    ``draft_logits`` is [R, V] (rows contiguous, any row stride) bf16 or f32 on the GPU,
    ``uniforms`` [R] float32. Returns {"tokens": [R] int32, "conf": [R] float32,
    "exit": [R] int32}; ``out`` may supply those tensors.
    """
    if draft_logits.dim() != 2 or draft_logits.stride(1) != 1:
        raise ValueError("draft_logits must be [R, V] with contiguous rows")
    R, V = draft_logits.shape
    if uniforms.shape != (R,):
        raise ValueError(f"uniforms must be [{R}]")
    dev = draft_logits.device
    if out is None:
        out = {"tokens": torch.empty(R, dtype=torch.int32, device=dev),
               "conf": torch.empty(R, dtype=torch.float32, device=dev),
               "exit": torch.empty(R, dtype=torch.int32, device=dev)}
    stride = draft_logits.stride(0) if R > 1 else V
    st = _lib.load().spec_draft_sample(
        int(R), int(V), _dtype_code(draft_logits), int(stride), _ptr(draft_logits, "draft_logits"),
        _ptr(uniforms, "uniforms", torch.float32), float(temperature), float(beta), int(bias_k),
        float(tau), _ptr(out["tokens"], "tokens", torch.int32),
        _ptr(out["conf"], "conf", torch.float32), _ptr(out.get("exit"), "exit", torch.int32),
        _stream_handle(stream))
    _lib._check(st, "spec_draft_sample")
    return out


def residual_topf(target_logits: torch.Tensor, draft_logits: torch.Tensor,
                  draft_lens: Optional[torch.Tensor], fanout: Sequence[int], *,
                  temperature: float = 1.0, beta: float = 1.0, bias_k: int = 0,
                  verify_out: Optional[dict] = None, stream=None):
    """Top-F ids of the exact residual max(p - q', 0) at every draft position, and (given the
    ``verify`` outputs with ``topf`` of the same call) the per-sequence cache-hit flags (see
    ``spec_residual_topf`` in include/spec_verify.h). Returns {"r2": [B, K, max F] int32} plus
    "hit": [B] int32 when ``verify_out`` is given."""
    B, K1, V = target_logits.shape
    K = K1 - 1
    ts = _row_stride(target_logits, K + 1, "target_logits")
    ds = _row_stride(draft_logits, K, "draft_logits")
    if draft_logits.dtype != target_logits.dtype:
        raise TypeError("target and draft logits must share a dtype")
    prob, keep = _lib.make_problem(B, K, V, _dtype_code(target_logits), ts, ds, bias_k, fanout)
    dev = target_logits.device
    out = {"r2": torch.empty(B, K, max(max(fanout), 1), dtype=torch.int32, device=dev)}
    acc = tok = r1 = hit = None
    if verify_out is not None:
        acc, tok, r1 = verify_out["accept_len"], verify_out["tokens"], verify_out["topf"]
        out["hit"] = hit = torch.empty(B, dtype=torch.int32, device=dev)
    st = _lib.call("spec_residual_topf", prob, _ptr(target_logits, "target_logits"),
                   _ptr(draft_logits, "draft_logits"),
                   _ptr(draft_lens, "draft_lens", torch.int32), float(temperature), float(beta),
                   _ptr(acc, "accept_len", torch.int32), _ptr(tok, "tokens", torch.int32),
                   _ptr(r1, "topf", torch.int32), _ptr(out["r2"], "r2", torch.int32),
                   _ptr(hit, "hit", torch.int32), _stream_handle(stream))
    del keep
    _lib._check(st, "spec_residual_topf")
    return out


def lmhead_stats(hidden: torch.Tensor, weight: torch.Tensor, ids: Optional[torch.Tensor] = None,
                 *, temperature: float = 1.0, logits: bool = False, stream=None):
    """Row statistics of hidden @ weight.T on the tensor cores, without writing the logits (see
    ``spec_lmhead_stats`` in include/spec_verify.h). ``hidden`` [R, d] and ``weight`` [V, d] are
    bf16 CUDA tensors with contiguous rows; ``ids`` [R] int32. Returns {"max", "lse", "argmax"
    [, "zx"][, "logits"]} (fp32; argmax int32); ``logits=True`` also writes the [R, V] logits
    (tests)."""
    for t, n in ((hidden, "hidden"), (weight, "weight")):
        if t.dtype != torch.bfloat16 or t.dim() != 2 or t.stride(1) != 1:
            raise ValueError(f"{n} must be a 2-D bf16 tensor with contiguous rows")
    R, d = hidden.shape
    V = weight.shape[0]
    if weight.shape[1] != d:
        raise ValueError("hidden and weight disagree on d")
    dev = hidden.device
    out = {"max": torch.empty(R, dtype=torch.float32, device=dev),
           "lse": torch.empty(R, dtype=torch.float32, device=dev)}
    if ids is not None:
        out["zx"] = torch.empty(R, dtype=torch.float32, device=dev)
    out["argmax"] = torch.empty(R, dtype=torch.int32, device=dev)
    if logits:
        out["logits"] = torch.empty(R, V, dtype=torch.float32, device=dev)
    st = _lib.load().spec_lmhead_stats(
        int(R), int(d), int(V), _ptr(hidden, "hidden"), int(hidden.stride(0) if R > 1 else d),
        _ptr(weight, "weight"), int(weight.stride(0) if V > 1 else d), float(temperature),
        _ptr(ids, "ids", torch.int32), _ptr(out["max"], "max"), _ptr(out["lse"], "lse"),
        _ptr(out.get("zx"), "zx"), _ptr(out["argmax"], "argmax"), _ptr(out.get("logits"), "logits"),
        _stream_handle(stream))
    _lib._check(st, "spec_lmhead_stats")
    return out


def verify_hidden(hidden_target: torch.Tensor, hidden_draft: Optional[torch.Tensor],
                  weight: torch.Tensor, draft_tokens: torch.Tensor,
                  draft_lens: Optional[torch.Tensor] = None,
                  uniforms: Optional[torch.Tensor] = None, *, temperature: float = 1.0,
                  beta: float = 1.0, bias_k: int = 0, fanout=None,
                  mode="stochastic", stream=None, out=None):
    """The verify step from hidden states (``spec_verify_hidden`` in include/spec_verify.h).

    ``hidden_target`` [B, K+1, d] and ``hidden_draft`` [B, K, d] (None in greedy mode) are bf16
    CUDA tensors whose rows are contiguous (any row stride that is a multiple of 8 elements, the
    same between positions and sequences); ``weight`` [V, d] bf16. ``beta`` and ``bias_k`` give
    the Saguaro bias set, ``fanout`` (K widths, or None) the top-F draft ids. Returns
    {"accept_len" [B], "tokens" [B, K+1]} (int32), and "topf" [B, K, max F] with a fanout."""
    B, K = draft_tokens.shape
    d = hidden_target.shape[-1]
    V = weight.shape[0]
    m = _MODES[mode]

    def stride(t, rows, name):
        if t.dtype != torch.bfloat16 or t.dim() != 3 or t.stride(2) != 1:
            raise ValueError(f"{name} must be a bf16 [B, rows, d] tensor with contiguous rows")
        if t.shape[0] != B or t.shape[1] != rows or t.shape[2] != d:
            raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {(B, rows, d)}")
        s1 = t.stride(1) if rows > 1 else d
        if B > 1 and t.stride(0) != rows * s1:
            raise ValueError(f"{name}: rows must be evenly spaced across sequences")
        return s1
    ts = stride(hidden_target, K + 1, "hidden_target")
    ds = stride(hidden_draft, K, "hidden_draft") if hidden_draft is not None else d
    if weight.dtype != torch.bfloat16 or weight.dim() != 2 or weight.stride(1) != 1 or \
            weight.shape[1] != d:
        raise ValueError("weight must be a bf16 [V, d] tensor with contiguous rows")
    dev = hidden_target.device
    fan = None
    if fanout is not None:
        if len(fanout) != K:
            raise ValueError(f"fanout needs {K} entries")
        fan = (ctypes.c_int * K)(*[int(f) for f in fanout])
    if out is None:
        out = {"accept_len": torch.empty(B, dtype=torch.int32, device=dev),
               "tokens": torch.empty(B, K + 1, dtype=torch.int32, device=dev)}
        if fanout is not None:
            out["topf"] = torch.empty(B, K, max(fanout), dtype=torch.int32, device=dev)
    st = _lib.load().spec_verify_hidden(
        int(B), int(K), int(V), int(d), _ptr(hidden_target, "hidden_target"), int(ts),
        _ptr(hidden_draft, "hidden_draft"), int(ds), _ptr(weight, "weight"),
        int(weight.stride(0) if V > 1 else d), _ptr(draft_tokens, "draft_tokens", torch.int32),
        _ptr(draft_lens, "draft_lens", torch.int32), _ptr(uniforms, "uniforms", torch.float32),
        float(temperature), float(beta), int(bias_k),
        ctypes.cast(fan, ctypes.c_void_p).value if fan is not None else 0, m,
        _ptr(out["accept_len"], "accept_len", torch.int32),
        _ptr(out["tokens"], "tokens", torch.int32),
        _ptr(out.get("topf"), "topf", torch.int32) if fanout is not None else 0,
        _stream_handle(stream))
    _lib._check(st, "spec_verify_hidden")
    return out


def _host_ptr(a) -> int:
    if a is None:
        return 0
    if isinstance(a, torch.Tensor):
        if a.is_cuda:
            raise ValueError("verify_host takes host arrays")
        return a.data_ptr()
    if not a.flags["C_CONTIGUOUS"]:
        raise ValueError("host arrays must be C-contiguous")
    return a.ctypes.data


def verify_host(target, draft, draft_tokens, draft_lens, uniforms, out_accept_len, out_tokens,
                out_topf=None, *, dtype: str, temperature: float = 1.0, beta: float = 1.0,
                mode="stochastic", bias_k: int = 0, fanout=None, cluster_hint: int = 0,
                stream=None) -> None:
    """End-to-end call over host buffers (numpy arrays or CPU torch tensors, pinned or not):
    copies the rows each sequence has to the GPU, verifies, copies the outputs back and
    synchronises. bf16 logits are passed as their 16-bit patterns."""
    B, K = draft_tokens.shape
    V = target.shape[2]
    prob, keep = _lib.make_problem(B, K, V, SV_DTYPE_BF16 if dtype == "bf16" else SV_DTYPE_F32,
                                   V, V, bias_k, fanout, cluster_hint)
    m = _MODES[mode]
    st = _lib.call("spec_verify_host", prob, _host_ptr(target), _host_ptr(draft),
                   _host_ptr(draft_tokens), _host_ptr(draft_lens), _host_ptr(uniforms),
                   float(temperature), float(beta), m, _host_ptr(out_accept_len),
                   _host_ptr(out_tokens), _host_ptr(out_topf), _stream_handle(stream))
    del keep
    _lib._check(st, "spec_verify_host")


def workspace_bytes(B: int) -> int:
    """Device bytes the caller-owned-workspace entry point needs for a batch of B sequences."""
    prob, _ = _lib.make_problem(B, 1, 1, SV_DTYPE_F32, 1, 1)
    return int(_lib.call("spec_verify_workspace_bytes", prob))


def device_error(stream=None) -> int:
    """Status of the device-side bounded waits since the last check, in calls on ``stream``
    that used the library's workspaces, and in no-alloc calls on any stream of the device."""
    return _lib.load().spec_verify_device_error(_stream_handle(stream))


def workspace_error(workspace: torch.Tensor, stream=None) -> int:
    """The same status for a caller-owned workspace of ``spec_verify_ws``."""
    return _lib.load().spec_verify_workspace_error(workspace.data_ptr(), _stream_handle(stream))


def hbm_read_probe(buf: torch.Tensor, out: torch.Tensor, stream=None) -> None:
    _lib._check(_lib.load().sv_hbm_read_probe(buf.data_ptr(), buf.numel() * buf.element_size(),
                                              out.data_ptr(), _stream_handle(stream)),
                "sv_hbm_read_probe")


def wait_probe(budget_us: int, stream=None, target: Optional[str] = None,
               workspace: Optional[torch.Tensor] = None) -> None:
    """Run one bounded wait that nothing satisfies (``sv_wait_probe``): it gives up after about
    ``budget_us`` microseconds and raises the stream's device error word, or with ``target``
    "noalloc" the no-alloc array's, or with "workspace" that of the caller's ``workspace``."""
    lib = _lib.load()
    if target is None:
        _lib._check(lib.sv_wait_probe(int(budget_us), _stream_handle(stream)), "sv_wait_probe")
        return
    t = {"noalloc": _lib.SV_PROBE_NOALLOC, "workspace": _lib.SV_PROBE_WORKSPACE}[target]
    ptr = workspace.data_ptr() if workspace is not None else None
    _lib._check(lib.sv_wait_probe_at(int(budget_us), t, ptr, _stream_handle(stream)),
                "sv_wait_probe_at")


def to_device_logits(a: np.ndarray, device="cuda") -> torch.Tensor:
    """Upload stored logits (uint16 bf16 bit patterns or float32) as a bf16/f32 tensor."""
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(a).to(device)
