"""The seeded input generator: determinism, storage rounding, padding poison, drafter law."""
import math

import numpy as np
import pytest
import torch

from speculative_decoding_verification_33_gb300 import workloads as W


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.standard_normal(20000).astype(np.float32) * 7,
                        np.array([0.0, -0.0, 1e-40, 3.0e38, -np.inf, np.inf], np.float32)])
    ours = W.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    back = W.bf16_bits_to_f32(ours)
    assert np.array_equal(back, torch.from_numpy(x).to(torch.bfloat16).float().numpy())


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5])
def test_shapes_determinism_and_padding(cfg):
    w = W.small_variant(W.WORKLOADS[cfg], B=3, V=512)
    a = W.make_inputs(w, threads=2)
    b = W.make_inputs(w, threads=3)
    for k in ("target", "draft", "draft_tokens", "draft_lens", "uniforms"):
        assert np.array_equal(a[k], b[k], equal_nan=True) or (
            a[k].dtype == np.uint16 and np.array_equal(a[k], b[k]))
    B, K, V = w.B, w.K, w.V
    assert a["target"].shape == (B, K + 1, V) and a["draft"].shape == (B, K, V)
    assert a["draft_tokens"].dtype == np.int32 and a["uniforms"].dtype == np.float32
    assert ((a["draft_lens"] >= 1) & (a["draft_lens"] <= K)).all()
    for bb in range(B):
        L = int(a["draft_lens"][bb])
        assert ((a["draft_tokens"][bb, :L] >= 0) & (a["draft_tokens"][bb, :L] < V)).all()
        tgt = a["target"][bb]
        if w.dtype == "bf16":
            assert (tgt[L + 1:] == W.BF16_NAN).all() and (a["draft"][bb, L:] == W.BF16_NAN).all()
        else:
            assert np.isnan(tgt[L + 1:]).all() and np.isnan(a["draft"][bb, L:]).all()
    if not w.ragged:
        assert (a["draft_lens"] == K).all()
    u = W.uniforms(w)
    assert np.array_equal(u, np.random.default_rng(0).random((B, K + 1), dtype=np.float32))


def test_replica_offsets_differ():
    w = W.small_variant(W.WORKLOADS[5], B=2, V=256)
    a, b = W.make_inputs(w, offset=0), W.make_inputs(w, offset=1)
    assert not np.array_equal(a["target"], b["target"])


def _chi2_ok(counts, probs, n):
    exp = probs * n
    m = exp > 0
    assert counts[~m].sum() == 0
    chi2 = float(np.sum((counts[m] - exp[m]) ** 2 / exp[m]))
    dof = int(m.sum()) - 1
    return chi2 < dof + 6 * math.sqrt(2 * dof)


@pytest.mark.parametrize("beta,k", [(1.0, 0), (0.5, 2)])
def test_drafter_samples_biased_draft_law(beta, k):
    """The Gumbel-max drafter draws x with probability q'(x) (SSD page, Saguaro sampling)."""
    zd = np.array([1.0, 0.5, 0.5, -0.3, 2.0, -1.0], np.float32)
    T = 0.8
    w = W.WORKLOADS[4].replace(temperature=T, beta=beta, bias_k=k)
    rng = np.random.default_rng(0)
    n = 40000
    counts = np.bincount([W._draw_draft(zd, w, rng) for _ in range(n)], minlength=6)
    e = np.exp((zd.astype(np.float64) - zd.max()) / T)
    f = np.ones(6)
    if k:
        f[np.lexsort((np.arange(6), -zd.astype(np.float64)))[:k]] = beta
    q = e * f / np.sum(e * f)
    assert _chi2_ok(counts, q, n)
