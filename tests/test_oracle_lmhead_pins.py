"""Pins of the LM-head oracle (logits of a bf16 head and the softmax statistics of a row)
against textbook values, closed forms, algebraic laws and brute force; nothing here re-types
its formulas."""
import math
from fractions import Fraction

import numpy as np
import pytest

from oracle import lmhead as H


# ----------------------------------------------------------------------------------------------
# bf16 patterns (IEEE binary32 with the low 16 bits dropped)
# ----------------------------------------------------------------------------------------------
def test_bf16_textbook_patterns():
    pats = np.array([0x3F80, 0xC000, 0x4049, 0x0001, 0x7F80, 0x0000, 0x8000, 0x3E80], np.uint16)
    want = [1.0, -2.0, 3.140625, 2.0 ** -133, math.inf, 0.0, -0.0, 0.25]
    got = H.bf16_to_f64(pats)
    for g, w in zip(got, want):
        assert g == w
    assert math.copysign(1.0, got[6]) == -1.0


# ----------------------------------------------------------------------------------------------
# logits (Kangaroo page, section 2, "Exit 1")
# ----------------------------------------------------------------------------------------------
def test_one_hot_head_selects_hidden_units():
    """A head whose row v is the unit vector e_pi(v) yields z[r, v] = h[r, pi(v)]."""
    rng = np.random.default_rng(1)
    R, d, V = 3, 7, 5
    h = rng.integers(-20, 20, size=(R, d)).astype(np.float64) / 8.0
    pi = np.array([4, 0, 6, 2, 2])
    W = np.zeros((V, d))
    W[np.arange(V), pi] = 1.0
    z = H.head_logits(h, W)
    assert z.shape == (R, V)
    for r in range(R):
        for v in range(V):
            assert z[r, v] == h[r, pi[v]]


def test_logits_brute_force_on_tiny_integers():
    """Integer-valued bf16 entries: every logit is an exact integer, summed here term by term."""
    rng = np.random.default_rng(2)
    R, d, V = 3, 5, 4
    h = rng.integers(-9, 10, size=(R, d))
    W = rng.integers(-9, 10, size=(V, d))
    hb = np.array([[_bf16_of_int(x) for x in row] for row in h], np.uint16)
    Wb = np.array([[_bf16_of_int(x) for x in row] for row in W], np.uint16)
    z = H.head_logits(hb, Wb)
    for r in range(R):
        for v in range(V):
            acc = 0
            for j in range(d):
                acc += int(h[r, j]) * int(W[v, j])
            assert z[r, v] == acc


def _bf16_of_int(x: int) -> int:
    """bf16 pattern of a small integer, built from sign, exponent and mantissa by hand."""
    if x == 0:
        return 0
    x = int(x)
    s = 0x8000 if x < 0 else 0
    a = abs(x)
    e = a.bit_length() - 1
    mant = (a - (1 << e)) << (7 - e)  # |x| < 256: the 7 fraction bits hold it exactly
    return s | ((e + 127) << 7) | mant


def test_fraction_exact_sum_on_bf16_values():
    """Random bf16 values: the float64 logit equals the exact rational sum rounded once per
    addition at most; for d = 6 terms of 16-bit mantissas it is exact."""
    rng = np.random.default_rng(3)
    hb = rng.integers(0x3C00, 0x4100, size=(2, 6)).astype(np.uint16)
    Wb = (rng.integers(0x3C00, 0x4100, size=(3, 6)) | 0x8000 * rng.integers(0, 2, (3, 6))).astype(np.uint16)
    z = H.head_logits(hb, Wb)
    hf, wf = H.bf16_to_f64(hb), H.bf16_to_f64(Wb)
    for r in range(2):
        for v in range(3):
            exact = sum(Fraction(float(hf[r, j])) * Fraction(float(wf[v, j])) for j in range(6))
            assert Fraction(float(z[r, v])) == exact


# ----------------------------------------------------------------------------------------------
# softmax statistics (Kangaroo guide, section 3: the accept ratio p(x) / q(x))
# ----------------------------------------------------------------------------------------------
@pytest.mark.parametrize("T", [1.0, 0.8, 2.5])
def test_lse_closed_forms(T):
    V = 11
    st = H.softmax_stats(np.full((1, V), 0.75), T)
    assert st.lse[0] == pytest.approx(0.75 / T + math.log(V), rel=1e-14)
    assert st.max[0] == 0.75
    # two ids with p = 1/4, 3/4 at temperature T
    st = H.softmax_stats(np.array([[0.0, T * math.log(3.0)]]), T)
    assert st.lse[0] == pytest.approx(math.log(4.0), rel=1e-14)
    # ln p(x) = z_x / T - lse gives the probabilities back
    z = np.array([[1.0, -2.0, 0.5, 3.0]])
    st = H.softmax_stats(z, T)
    p = np.exp(z[0] / T - st.lse[0])
    e = [math.exp(v / T) for v in z[0]]
    for i in range(4):
        assert p[i] == pytest.approx(e[i] / sum(e), rel=1e-13)


def test_lse_shift_scale_and_bounds():
    rng = np.random.default_rng(4)
    z = rng.normal(0.0, 3.0, size=(5, 97))
    for T in (0.7, 1.0, 1.9):
        a = H.softmax_stats(z, T)
        b = H.softmax_stats(z + 4.25, T)
        np.testing.assert_allclose(b.lse - a.lse, 4.25 / T, rtol=1e-12)
        c = H.softmax_stats(z / T, 1.0)
        np.testing.assert_allclose(c.lse, a.lse, rtol=1e-13)
        assert np.all(a.lse >= a.max / T) and np.all(a.lse <= a.max / T + math.log(97) + 1e-12)
        np.testing.assert_array_equal(a.max, z.max(axis=1))


def test_lse_of_large_logits_stays_finite():
    st = H.softmax_stats(np.array([[1000.0, 1000.0, 990.0]]), 1.0)
    assert st.lse[0] == pytest.approx(1000.0 + math.log(2.0 + math.exp(-10.0)), rel=1e-15)
    st = H.softmax_stats(np.array([[-1000.0, -1001.0]]), 0.5)
    assert st.lse[0] == pytest.approx(-2000.0 + math.log(1.0 + math.exp(-2.0)), rel=1e-15)


def test_logit_at_id():
    z = np.arange(12, dtype=np.float64).reshape(3, 4) * 0.5 - 1.0
    st = H.softmax_stats(z, 1.0, ids=np.array([2, -1, 4]))
    assert st.zx[0] == z[0, 2]
    assert math.isnan(st.zx[1]) and math.isnan(st.zx[2])
    assert np.all(np.isnan(H.softmax_stats(z, 1.0).zx))


def test_temperature_must_be_positive():
    with pytest.raises(ValueError):
        H.softmax_stats(np.zeros((1, 3)), 0.0)


# ----------------------------------------------------------------------------------------------
# the float32 error bound used by the parity tests
# ----------------------------------------------------------------------------------------------
def test_error_bound_covers_float32_summation_orders():
    """Sequential and pairwise float32 sums of exact bf16 products stay within the bound."""
    rng = np.random.default_rng(6)
    R, d, V = 4, 512, 6
    hb = (rng.integers(0x3000, 0x4100, size=(R, d)) | 0x8000 * rng.integers(0, 2, (R, d))).astype(np.uint16)
    Wb = (rng.integers(0x3000, 0x4100, size=(V, d)) | 0x8000 * rng.integers(0, 2, (V, d))).astype(np.uint16)
    z = H.head_logits(hb, Wb)
    bound = H.logit_error_bound(hb, Wb)
    h32 = H.bf16_to_f64(hb).astype(np.float32)
    w32 = H.bf16_to_f64(Wb).astype(np.float32)
    for r in range(R):
        for v in range(V):
            prods = h32[r] * w32[v]  # exact in float32 (8-bit x 8-bit significands)
            s = np.float32(0.0)
            for t in prods:
                s = np.float32(s + t)
            assert abs(float(s) - z[r, v]) <= bound[r, v]
            pw = prods.copy()
            while pw.size > 1:
                pw = (pw[0::2] + pw[1::2]).astype(np.float32)
            assert abs(float(pw[0]) - z[r, v]) <= bound[r, v]
    assert np.all(bound > 0)


# ----------------------------------------------------------------------------------------------
# the verify step from hidden states (Kangaroo guide, section 3)
# ----------------------------------------------------------------------------------------------
@pytest.mark.parametrize("mode", ["stochastic", "greedy"])
def test_identity_head_reduces_to_the_verify_step(mode):
    """With W = I (V = d) the logits are the hidden states, so the outcome must be the verify
    step's on those rows read as logits (a transposed or shifted head, or rows scored at the
    wrong position, would change it)."""
    from oracle import verify as O
    rng = np.random.default_rng(9)
    B, K, d = 6, 3, 7
    ht = rng.normal(0.0, 1.5, size=(B, K + 1, d))
    hd = ht[:, :K] + rng.normal(0.0, 0.6, size=(B, K, d))
    W = np.eye(d)
    lens = np.array([3, 1, 2, 3, 2, 1], np.int32)
    x = rng.integers(0, d, size=(B, K)).astype(np.int32)
    if mode == "greedy":
        x[:, 0] = ht[:, 0].argmax(axis=1)  # so that some drafts are accepted
    u = rng.random((B, K + 1)).astype(np.float32)
    got = H.verify_hidden_batch(ht, hd if mode == "stochastic" else None, W, x, lens, u,
                                temperature=0.9, mode=mode)
    tgt = np.where(np.arange(K + 1)[None, :, None] <= lens[:, None, None], ht, np.nan)
    dft = np.where(np.arange(K)[None, :, None] < lens[:, None, None], hd, np.nan)
    want = O.verify_batch(tgt, dft if mode == "stochastic" else None, x, lens, u,
                          temperature=0.9, mode=mode)
    accepted = 0
    for g, w in zip(got, want):
        assert g.accept_len == w.accept_len
        assert np.array_equal(g.tokens, w.tokens)
        accepted += g.accept_len
    assert accepted > 0


def test_identity_head_carries_the_bias_set_and_top_f():
    """With W = I the bias set and the top-F ids of the verify step from hidden states are those
    of the verify step on the hidden states read as logits: the ids of the largest draft hidden
    units (a head that scored the target rows, or transposed ids, would give others)."""
    from oracle import verify as O
    rng = np.random.default_rng(11)
    B, K, d = 8, 4, 24
    ht = rng.normal(0.0, 1.0, size=(B, K + 1, d))
    hd = ht[:, :K] + rng.normal(0.0, 0.8, size=(B, K, d))
    lens = np.array([4, 1, 2, 3, 4, 2, 1, 3], np.int32)
    x = rng.integers(0, d, size=(B, K)).astype(np.int32)
    u = rng.random((B, K + 1)).astype(np.float32)
    fan = (5, 3, 2, 1)
    got = H.verify_hidden_batch(ht, hd, np.eye(d), x, lens, u, temperature=1.1, mode="stochastic",
                                beta=0.4, bias_k=6, fanout=fan)
    tgt = np.where(np.arange(K + 1)[None, :, None] <= lens[:, None, None], ht, np.nan)
    dft = np.where(np.arange(K)[None, :, None] < lens[:, None, None], hd, np.nan)
    want = O.verify_batch(tgt, dft, x, lens, u, temperature=1.1, mode="stochastic", beta=0.4,
                          bias_k=6, fanout=fan)
    for b, (g, w) in enumerate(zip(got, want)):
        assert g.accept_len == w.accept_len
        assert np.array_equal(g.tokens, w.tokens)
        assert np.array_equal(g.topf, w.topf)
        for i in range(lens[b]):  # the top-F ids are the largest draft hidden units of row i
            f = fan[i]
            assert list(g.topf[i, :f]) == list(np.argsort(-hd[b, i], kind="stable")[:f])
    base = H.verify_hidden_batch(ht, hd, np.eye(d), x, lens, u, temperature=1.1,
                                 mode="stochastic")
    assert any(g.accept_len != h.accept_len or not np.array_equal(g.tokens, h.tokens)
               for g, h in zip(got, base))  # the bias set changes some outcome


def test_head_stats_of_a_one_hot_head():
    """A head whose row v is the unit vector e_pi(v) scores z[r, v] = h[r, pi(v)], so the row
    statistics are those of the selected hidden units: max, ln sum exp(h / T) term by term, and
    the logit of the requested id (a transposed head or a dropped temperature changes them)."""
    rng = np.random.default_rng(11)
    R, d, V, T = 3, 6, 5, 0.6
    h = rng.integers(-16, 17, size=(R, d)).astype(np.float64) / 8.0
    pi = np.array([5, 1, 1, 3, 0])
    W = np.zeros((V, d))
    W[np.arange(V), pi] = 1.0
    ids = np.array([2, 4, 7])
    st = H.head_stats(h, W, T, ids)
    for r in range(R):
        sel = [h[r, pi[v]] for v in range(V)]
        assert st.max[r] == max(sel)
        assert st.lse[r] == pytest.approx(math.log(math.fsum(math.exp(s / T) for s in sel)),
                                          rel=1e-14)
    assert st.zx[0] == h[0, pi[2]] and st.zx[1] == h[1, pi[4]] and math.isnan(st.zx[2])
