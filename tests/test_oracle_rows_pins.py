"""Pins of the row-step oracle (draft draw, exit confidence, exact-residual top-F, cache hit)
against closed forms, exact enumeration and brute force; nothing here re-types its formulas."""
import math

import numpy as np
import pytest

from oracle import rows as R
from tests.test_oracle_pins import biased_probs_of, logits_for, probs_of


# ----------------------------------------------------------------------------------------------
# exit confidence (Kangaroo page, section 2, "Exit 2")
# ----------------------------------------------------------------------------------------------
def test_confidence_closed_forms():
    z1 = np.float32(math.log(3.0))
    row = np.array([0.0, z1], np.float32)
    # two logits: max softmax = logistic(z1 / T)
    for T in (1.0, 2.0, 0.5):
        d = R.draft_sample(row, 0.3, temperature=T)
        assert d.conf == pytest.approx(1.0 / (1.0 + math.exp(-float(z1) / T)), rel=1e-14)
    # flat row: 1 / V
    d = R.draft_sample(np.zeros(7, np.float32), 0.5, temperature=1.3)
    assert d.conf == pytest.approx(1.0 / 7.0, rel=1e-14)
    # two tied maxima and one e-fold smaller entry
    d = R.draft_sample(np.array([1.0, 1.0, 0.0], np.float32), 0.5, temperature=1.0)
    assert d.conf == pytest.approx(math.e / (2.0 * math.e + 1.0), rel=1e-14)
    # -inf entries carry no mass
    d = R.draft_sample(np.array([-np.inf, 0.0, -np.inf, 0.0], np.float32), 0.5, temperature=1.0)
    assert d.conf == 0.5


def test_confidence_ignores_the_bias_and_sets_the_exit_flag():
    row = np.array([0.0, np.float32(math.log(3.0))], np.float32)
    c = 1.0 / (1.0 + 1.0 / 3.0)
    d = R.draft_sample(row, 0.1, temperature=1.0, beta=0.5, bias_k=1, tau=0.0)
    assert d.conf == pytest.approx(c, rel=1e-7)  # q = [1/4, 3/4], not q' = [0.4, 0.6]
    assert R.draft_sample(row, 0.1, temperature=1.0, tau=c + 1e-6).exit == 1
    assert R.draft_sample(row, 0.1, temperature=1.0, tau=c - 1e-6).exit == 0
    assert R.draft_sample(row, 0.1, temperature=1.0, tau=0.0).exit == 0


# ----------------------------------------------------------------------------------------------
# the draw from q' (SSD page, "Method")
# ----------------------------------------------------------------------------------------------
@pytest.mark.parametrize("T,beta,k", [(1.0, 1.0, 0), (0.7, 1.0, 0), (1.0, 0.5, 2), (1.4, 0.2, 1)])
def test_draw_frequencies_by_exact_enumeration(T, beta, k):
    """Over a fine grid of uniforms the share of each token equals q'(v) up to the grid step."""
    rng = np.random.default_rng(5)
    p = rng.dirichlet(np.ones(6))
    p[4] = 0.0
    p /= p.sum()
    z = logits_for(p)
    q = probs_of(z, T)
    qb = biased_probs_of(q, z, beta, k)
    N = 1 << 13
    counts = np.zeros(6)
    for j in range(N):
        d = R.draft_sample(z, (j + 0.5) / N, temperature=T, beta=beta, bias_k=k)
        counts[d.token] += 1
    assert counts[4] == 0
    assert np.all(np.abs(counts / N - qb) <= 1.5 / N)


def test_draw_bin_edges_hand_example():
    row = np.array([0.0, np.float32(math.log(3.0))], np.float32)  # q = [1/4, 3/4]
    assert R.draft_sample(row, 0.0, temperature=1.0).token == 0
    assert R.draft_sample(row, 0.2499, temperature=1.0).token == 0
    assert R.draft_sample(row, 0.2501, temperature=1.0).token == 1
    assert R.draft_sample(row, 0.9999, temperature=1.0).token == 1
    # beta = 0.5 on the top id: q' = [0.25, 0.375] / 0.625 = [0.4, 0.6]
    kw = dict(temperature=1.0, beta=0.5, bias_k=1)
    assert R.draft_sample(row, 0.3999, **kw).token == 0
    assert R.draft_sample(row, 0.4001, **kw).token == 1
    d = R.draft_sample(row, 0.4, **kw)
    assert d.margin < 1e-6


def test_bad_rows_and_uniforms():
    nan = np.array([0.0, np.nan, 1.0], np.float32)
    d = R.draft_sample(nan, 0.5, temperature=1.0)
    assert (d.token, d.exit) == (-1, -1) and math.isnan(d.conf)
    assert R.draft_sample(np.array([0.0, np.inf], np.float32), 0.5, temperature=1.0).token == -1
    d = R.draft_sample(np.full(4, -np.inf, np.float32), 0.5, temperature=1.0)
    assert d.token == -1 and math.isnan(d.conf)
    ok = np.array([0.0, 1.0], np.float32)
    for u in (1.0, -0.25, float("nan")):
        d = R.draft_sample(ok, u, temperature=1.0, tau=0.9)
        assert d.token == -1 and d.exit == 1
        assert d.conf == pytest.approx(1.0 / (1.0 + math.exp(-1.0)))


# ----------------------------------------------------------------------------------------------
# exact-residual order (SSD page, "Key claims")
# ----------------------------------------------------------------------------------------------
def test_residual_order_hand_examples():
    p = logits_for([0.5, 0.3, 0.2])
    q = logits_for([0.2, 0.5, 0.3])
    _, ids = R.residual_order(p, q, temperature=1.0)
    assert ids.tolist() == [0]
    p = logits_for([0.1, 0.2, 0.4, 0.3])
    q = logits_for([0.1, 0.1, 0.4, 0.4])
    _, ids = R.residual_order(p, q, temperature=1.0)
    assert ids.tolist() == [1]  # r = [0, 0.1, 0, 0]
    # beta = 0.5 on the top draft id (a tie between ids 2 and 3 goes to 2):
    # q' = [0.1, 0.1, 0.2, 0.4] / 0.8, r = [0, 0.075, 0.15, 0]
    r, ids = R.residual_order(p, q, temperature=1.0, beta=0.5, bias_k=1)
    assert ids.tolist() == [2, 1]
    assert r[2] == pytest.approx(0.15, abs=1e-7) and r[1] == pytest.approx(0.075, abs=1e-7)
    # planted tie: ids 1 and 3 have identical rows, r = [0, 0.2, 0, 0.2] -> lower id first
    p = logits_for([0.2, 0.3, 0.2, 0.3])
    q = logits_for([0.4, 0.1, 0.4, 0.1])
    _, ids = R.residual_order(p, q, temperature=1.0)
    assert ids.tolist() == [1, 3]


def test_residual_order_brute_force():
    rng = np.random.default_rng(23)
    for trial in range(30):
        V = 10
        zt = (rng.standard_normal(V) * 2).astype(np.float32)
        zd = (zt + rng.standard_normal(V)).astype(np.float32)
        T = [1.0, 0.6, 1.7][trial % 3]
        beta, k = [(1.0, 0), (0.5, 3), (0.1, 1)][trial % 3]
        p = probs_of(zt, T)
        qb = biased_probs_of(probs_of(zd, T), zd, beta, k)
        r = [max(a - b, 0.0) for a, b in zip(p, qb)]
        ref = [v for v in sorted(range(V), key=lambda v: (-r[v], v)) if r[v] > 1e-15]
        _, ids = R.residual_order(zt, zd, temperature=T, beta=beta, bias_k=k)
        assert ids.tolist() == ref


def test_residual_topf_widths_lengths_and_bad_rows():
    rng = np.random.default_rng(3)
    B, K, V = 3, 4, 9
    tgt = rng.standard_normal((B, K + 1, V)).astype(np.float32)
    dft = (tgt[:, :K] + rng.standard_normal((B, K, V))).astype(np.float32)
    lens = np.array([2, 0, 4], np.int32)
    dft[2, 3, 1] = np.nan
    fan = (4, 2, 1, 1)
    out = R.residual_topf(tgt, dft, lens, temperature=1.0, fanout=fan)
    assert out.shape == (B, K, 4)
    assert (out[1] == -1).all()  # L = 0: no residual anywhere
    assert (out[0, 2:] == -1).all()  # positions at or after L
    assert (out[2, 3] == -1).all()  # bad draft row
    for b, i in ((0, 0), (0, 1), (2, 0), (2, 2)):
        _, ids = R.residual_order(tgt[b, i], dft[b, i], temperature=1.0)
        f = min(fan[i], len(ids))
        assert out[b, i, :f].tolist() == ids[:f].tolist()
        assert (out[b, i, f:] == -1).all()


# ----------------------------------------------------------------------------------------------
# cache hit
# ----------------------------------------------------------------------------------------------
def test_cache_hit_hand_examples():
    fan = (3, 2, 1)
    topf = np.array([[5, 6, 7], [8, 9, -1], [4, -1, -1]], np.int32)
    tok = np.array([6, 0, 0, 0], np.int32)
    assert R.cache_hit(0, tok, topf, 3, fan) == 1  # 6 is the second of the three keys
    assert R.cache_hit(0, np.array([4, 0, 0, 0]), topf, 3, fan) == 0
    assert R.cache_hit(1, np.array([1, 9, 0, 0]), topf, 3, fan) == 1
    assert R.cache_hit(2, np.array([1, 2, 5, 0]), topf, 3, fan) == 0  # F_2 = 1: only id 4
    assert R.cache_hit(2, np.array([1, 2, 4, 0]), topf, 3, fan) == 1
    assert R.cache_hit(3, np.array([1, 2, 3, 9]), topf, 3, fan) == -1  # bonus draw
    assert R.cache_hit(1, np.array([1, 2, 3, 9]), topf, 1, fan) == -1  # a == L
    assert R.cache_hit(-1, tok, topf, 3, fan) == -1  # invalid sequence
    assert R.cache_hit(0, tok, topf, 0, fan) == -1  # L outside [1, K]
