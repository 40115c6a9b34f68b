"""GPU parity of the tensor-core LM head with its softmax statistics (``spec_lmhead_stats``),
called through the C ABI, against the float64 oracle.

Tolerances. Every bf16 x bf16 product is exact in float32, so a logit summed in float32 is off
by at most ``d * 2^-23 * sum_j |h_j w_j|`` (``oracle.lmhead.logit_error_bound``, pinned against
float32 sums in the oracle's tests). The maximum moves by at most the largest logit error; the
log-sum-exp by that error over T plus the float32 rounding of the sum of exponentials (at most
``(V / 32 + 64) * 2^-23`` relative for the running sums of 32-column chunks, with ex2.approx's
two ulps) taken as 4e-6 absolute + 2e-6 relative to |lse|."""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU machines too
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from oracle import lmhead as HO  # noqa: E402
from speculative_decoding_verification_33_gb300 import api  # noqa: E402
from speculative_decoding_verification_33_gb300 import workloads as W  # noqa: E402

LSE_ABS, LSE_REL = 4e-6, 2e-6


def to_dev(bits: np.ndarray) -> "torch.Tensor":
    return torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)


def check(hb, wb, ids, T, out, rows=None, logits=True):
    rows = np.arange(hb.shape[0]) if rows is None else np.asarray(rows)
    z = HO.head_logits(hb[rows], wb)
    bound = HO.logit_error_bound(hb[rows], wb)
    st = HO.softmax_stats(z, T, ids[rows])
    if logits:
        got = out["logits"].cpu().numpy().astype(np.float64)[rows]
        err = np.abs(got - z)
        worst = np.unravel_index(np.argmax(err - bound), err.shape)
        assert np.all(err <= bound), (worst, got[worst], z[worst], bound[worst])
    zb = bound.max(axis=1)
    gm = out["max"].cpu().numpy().astype(np.float64)[rows]
    assert np.all(np.abs(gm - st.max) <= zb), np.max(np.abs(gm - st.max) - zb)
    gl = out["lse"].cpu().numpy().astype(np.float64)[rows]
    tol = zb / T + LSE_ABS + LSE_REL * np.abs(st.lse)
    assert np.all(np.abs(gl - st.lse) <= tol), np.max(np.abs(gl - st.lse) - tol)
    gx = out["zx"].cpu().numpy().astype(np.float64)[rows]
    ok = ~np.isnan(st.zx)
    assert np.array_equal(np.isnan(gx), ~ok)
    idx = np.clip(ids[rows], 0, wb.shape[0] - 1)
    xb = bound[np.arange(len(rows)), idx]
    assert np.all(np.abs(gx[ok] - st.zx[ok]) <= xb[ok])


@pytest.mark.parametrize("R,d,V,T", [
    (200, 128, 1000, 0.8),    # two row tiles (ragged), two K blocks, a ragged last column tile
    (1, 64, 1, 1.0),          # the smallest problem
    (129, 192, 5000, 1.3),    # 20 column tiles spread over many vocabulary ranges
    (300, 1024, 2304, 0.7),   # deeper K
])
def test_head_small(R, d, V, T):
    w = W.small_head(R, d, V, temperature=T)
    x = W.head_inputs(w)
    ids = x["ids"].copy()
    ids[::7] = -1         # ids outside the vocabulary give NaN
    ids[3::11] = V
    out = api.lmhead_stats(to_dev(x["hidden"]), to_dev(x["weight"]),
                           torch.from_numpy(ids).cuda(), temperature=T, logits=True)
    torch.cuda.synchronize()
    check(x["hidden"], x["weight"], ids, T, out)


def test_head_statistics_without_logits_match():
    """The statistics do not depend on whether the logits are also written."""
    w = W.small_head(256, 256, 3000, temperature=1.0)
    x = W.head_inputs(w)
    h, wt = to_dev(x["hidden"]), to_dev(x["weight"])
    ids = torch.from_numpy(x["ids"]).cuda()
    a = api.lmhead_stats(h, wt, ids, logits=True)
    b = api.lmhead_stats(h, wt, ids, logits=False)
    torch.cuda.synchronize()
    for k in ("max", "lse", "zx"):
        assert torch.equal(a[k], b[k]), k
    check(x["hidden"], x["weight"], x["ids"], 1.0, b, logits=False)


def test_head_strided_rows():
    """Hidden states and head rows read out of wider buffers (row strides > d)."""
    w = W.small_head(150, 128, 700, temperature=1.0)
    x = W.head_inputs(w)
    hw = np.zeros((150, 192), np.uint16)
    hw[:, :128] = x["hidden"]
    ww = np.zeros((700, 136), np.uint16)
    ww[:, :128] = x["weight"]
    out = api.lmhead_stats(to_dev(hw)[:, :128], to_dev(ww)[:, :128],
                           torch.from_numpy(x["ids"]).cuda(), logits=True)
    torch.cuda.synchronize()
    check(x["hidden"], x["weight"], x["ids"], 1.0, out)


def test_head_rejects_bad_arguments():
    h = torch.zeros(4, 96, dtype=torch.bfloat16, device="cuda")   # d not a multiple of 64
    wt = torch.zeros(8, 96, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(RuntimeError):
        api.lmhead_stats(h, wt)
    h = torch.zeros(4, 64, dtype=torch.bfloat16, device="cuda")
    wt = torch.zeros(8, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(RuntimeError):
        api.lmhead_stats(h, wt, temperature=0.0)
    empty = api.lmhead_stats(h[:0], wt)
    assert empty["max"].numel() == 0


@pytest.mark.parametrize("name", sorted(W.HEAD_WORKLOADS))
def test_head_full_size_sampled_rows(name):
    """The full-size heads of the bench, checked on sampled rows (statistics and logits)."""
    w = W.HEAD_WORKLOADS[name]
    x = W.head_inputs(w)
    out = api.lmhead_stats(to_dev(x["hidden"]), to_dev(x["weight"]),
                           torch.from_numpy(x["ids"]).cuda(), temperature=w.temperature,
                           logits=False)
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([np.arange(0, w.R, max(1, w.R // 12)), [w.R - 1, 127, 128]]))
    check(x["hidden"], x["weight"], x["ids"], w.temperature, out, rows=rows, logits=False)
    assert not np.isnan(out["lse"].cpu().numpy()).any()
