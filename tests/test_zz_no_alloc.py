"""The allocation-free entry point (spec_verify_noalloc) gives the same outputs as spec_verify.

Callers that cannot allocate device memory (a serving loop that reserved all device memory up
front, a runtime whose allocations must go through its own pool) use this variant; its workspace
is a fixed array inside the library. This file is collected last so that
a failure here does not hide the other GPU tests; it must also pass on its own.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU machines too
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from speculative_decoding_verification_33_gb300 import _lib, api  # noqa: E402
from speculative_decoding_verification_33_gb300 import workloads as W  # noqa: E402


def _inputs(w):
    d = W.make_inputs(w)
    T = api.to_device_logits(d["target"])
    D = api.to_device_logits(d["draft"]) if w.mode == "stochastic" else None
    return (T, D, torch.from_numpy(d["draft_tokens"]).cuda(),
            torch.from_numpy(d["draft_lens"]).cuda(), torch.from_numpy(d["uniforms"]).cuda())


def _outputs(w):
    acc = torch.full((w.B,), -7, dtype=torch.int32, device="cuda")
    tok = torch.full((w.B, w.K + 1), -7, dtype=torch.int32, device="cuda")
    topf = (torch.full((w.B, w.K, max(w.fanout)), -7, dtype=torch.int32, device="cuda")
            if w.fanout else None)
    return acc, tok, topf


@pytest.mark.parametrize("cfg,B,V", [(4, 12, 4099), (5, 40, 9000), (2, 9, 32000)])
def test_no_alloc_matches_spec_verify_twice(cfg, B, V):
    w = W.small_variant(W.WORKLOADS[cfg], B=B, V=V)
    T, D, tok, ln, uni = _inputs(w)
    ref = _outputs(w)
    api.spec_verify(T, D, tok, ln, uni, w.temperature, w.beta, w.mode, *ref,
                    bias_k=w.bias_k, fanout=w.fanout)
    torch.cuda.synchronize()
    for _ in range(2):  # the shared array keeps the last call's contents; both calls must agree
        got = _outputs(w)
        api.spec_verify(T, D, tok, ln, uni, w.temperature, w.beta, w.mode, *got,
                        bias_k=w.bias_k, fanout=w.fanout, no_alloc=True)
        torch.cuda.synchronize()
        for a, b in zip(ref, got):
            if a is not None:
                assert np.array_equal(a.cpu().numpy(), b.cpu().numpy())
    assert api.device_error() == 0


def test_no_alloc_rejects_batches_above_its_array():
    w = W.small_variant(W.WORKLOADS[2], B=65537, V=8).replace(K=1)
    prob, keep = _lib.make_problem(w.B, w.K, w.V, _lib.SV_DTYPE_BF16, w.V, w.V)
    dummy = torch.zeros(16, dtype=torch.int32, device="cuda")
    p = dummy.data_ptr()
    st = _lib.call("spec_verify_noalloc", prob, p, 0, p, 0, 0, 0.0, 1.0, _lib.SV_MODE_GREEDY,
                   p, p, 0, torch.cuda.current_stream().cuda_stream)
    assert st == _lib.SV_ERR_UNSUPPORTED


def test_bounded_wait_gives_up_and_reports():
    """Failure detection without a GPU fault: a bounded wait that nothing satisfies runs out,
    raises the error word, the host reads SV_ERR_DEVICE_TIMEOUT once, and the context stays
    usable for a normal call."""
    from speculative_decoding_verification_33_gb300._lib import SV_ERR_DEVICE_TIMEOUT
    assert api.device_error() == 0
    api.wait_probe(2000)
    assert api.device_error() == SV_ERR_DEVICE_TIMEOUT
    assert api.device_error() == 0
    w = W.small_variant(W.WORKLOADS[3], B=4, V=4096)
    d = W.make_inputs(w)
    out = api.verify(api.to_device_logits(d["target"]), api.to_device_logits(d["draft"]),
                     torch.from_numpy(d["draft_tokens"]).cuda(),
                     torch.from_numpy(d["draft_lens"]).cuda(),
                     torch.from_numpy(d["uniforms"]).cuda(), temperature=w.temperature)
    torch.cuda.synchronize()
    assert (out["accept_len"].cpu().numpy() >= 0).all()
    assert api.device_error() == 0


def test_timeout_in_the_fixed_array_is_reported_once():
    """A bounded wait that gives up inside the no-alloc array is reported by
    spec_verify_device_error exactly once, and the next no-alloc call does not erase it first."""
    from speculative_decoding_verification_33_gb300._lib import SV_ERR_DEVICE_TIMEOUT
    assert api.device_error() == 0
    api.wait_probe(2000, target="noalloc")
    w = W.small_variant(W.WORKLOADS[3], B=6, V=4096)
    T, D, tok, ln, uni = _inputs(w)
    got = _outputs(w)
    api.spec_verify(T, D, tok, ln, uni, w.temperature, w.beta, w.mode, *got, no_alloc=True)
    torch.cuda.synchronize()
    assert (got[0].cpu().numpy() >= 0).all()
    assert api.device_error() == SV_ERR_DEVICE_TIMEOUT
    assert api.device_error() == 0


def test_timeout_in_a_caller_workspace_is_reported_once():
    """The same for a caller-owned workspace: spec_verify_workspace_error reports it once, and
    a verify call through that workspace still gives valid outcomes."""
    from speculative_decoding_verification_33_gb300._lib import SV_ERR_DEVICE_TIMEOUT
    w = W.small_variant(W.WORKLOADS[3], B=6, V=4096)
    ws = torch.zeros(api.workspace_bytes(w.B) // 4, dtype=torch.int32, device="cuda")
    assert api.workspace_error(ws) == 0
    api.wait_probe(2000, target="workspace", workspace=ws)
    assert api.workspace_error(ws) == SV_ERR_DEVICE_TIMEOUT
    assert api.workspace_error(ws) == 0
    T, D, tok, ln, uni = _inputs(w)
    got = _outputs(w)
    api.spec_verify(T, D, tok, ln, uni, w.temperature, w.beta, w.mode, *got, workspace=ws)
    torch.cuda.synchronize()
    assert (got[0].cpu().numpy() >= 0).all()
    assert api.workspace_error(ws) == 0
    assert api.device_error() == 0
