"""Pins of the float64 oracle against what the pages and the mathematics fix.

Nothing here re-types the oracle's formulas: the checks are closed forms, brute force on tiny
inputs, hand-worked examples, independent library routines and the exact output law found by
bisection on the oracle itself (losslessness, glossary page "Why It Produces Identical Outputs";
Kangaroo page section 3).
"""
import math
import os

import numpy as np
import pytest

from oracle import verify as O
from tests._law import output_law

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------------------------------------
# helpers that build rows from probabilities (test side, independent routines)
# ----------------------------------------------------------------------------------------------
def logits_for(p, T=1.0):
    """float32 logits whose softmax at temperature T is (close to) p; zeros map to -inf."""
    p = np.asarray(p, dtype=np.float64)
    with np.errstate(divide="ignore"):
        return (T * np.log(p)).astype(np.float32)


def probs_of(z32, T):
    """softmax of stored float32 logits by math.exp + math.fsum (independent of numpy sums)."""
    z = [float(v) for v in z32]
    m = max(z)
    e = [math.exp((v - m) / T) if v != -math.inf else 0.0 for v in z]
    s = math.fsum(e)
    return np.array([x / s for x in e])


def biased_probs_of(q, zd, beta, k):
    """q' built as f*q / fsum(f*q) with f = beta on the k largest draft logits (ties: lower id)."""
    if beta >= 1.0 or k <= 0:
        return q
    order = sorted(range(len(zd)), key=lambda v: (-float(zd[v]), v))[:k]
    f = np.ones(len(q))
    f[order] = beta
    fq = [float(a) * float(b) for a, b in zip(f, q)]
    s = math.fsum(fq)
    return np.array([x / s for x in fq])


def runner(tgt, dft, T, beta=1.0, bias_k=0):
    """run(x, u) -> (accept_len, tokens) of the oracle on fixed rows."""
    L = dft.shape[0]

    def run(x, u):
        r = O.verify_sequence(tgt, dft, np.array(x), L, u, temperature=T, mode="stochastic",
                              beta=beta, bias_k=bias_k)
        return r.accept_len, r.tokens
    return run


def random_probs(rng, V, zero_frac=0.0):
    p = rng.dirichlet(np.ones(V) * 0.8)
    if zero_frac > 0:
        mask = rng.random(V) < zero_frac
        if mask.all():
            mask[rng.integers(V)] = False
        p[mask] = 0.0
        p /= p.sum()
    return p


# ----------------------------------------------------------------------------------------------
# softmax / log-sum-exp
# ----------------------------------------------------------------------------------------------
@pytest.mark.parametrize("T", [1.0, 0.8, 2.5])
@pytest.mark.parametrize("store", ["f32", "bf16"])
def test_softmax_against_fsum(T, store):
    rng = np.random.default_rng(7)
    z32 = (rng.standard_normal(4099) * 3).astype(np.float32)
    if store == "bf16":
        from speculative_decoding_verification_33_gb300.workloads import f32_to_bf16_bits
        row = f32_to_bf16_bits(z32)
        z = [float(v) for v in (row.astype(np.uint32) << 16).view(np.float32)]
    else:
        row = z32
        z = [float(v) for v in z32]
    p, lse = O.softmax(O.row_to_f64(row), T)
    m = max(z) / T
    s = math.fsum(math.exp(v / T - m) for v in z)
    assert abs(lse - (m + math.log(s))) < 1e-12 * max(1.0, abs(lse))
    assert abs(math.fsum(p.tolist()) - 1.0) < 1e-13
    i = int(rng.integers(len(z)))
    assert abs(p[i] - math.exp(z[i] / T - m) / s) < 1e-15 + 1e-12 * p[i]


def test_softmax_closed_forms():
    # uniform row: p = 1/V, lse = z/T + ln V
    p, lse = O.softmax(np.full(1000, 2.0), 0.5)
    assert np.allclose(p, 1e-3, rtol=0, atol=1e-16)
    assert abs(lse - (4.0 + math.log(1000))) < 1e-12
    # two-point row: p_0 = sigmoid((z0 - z1)/T)
    p, _ = O.softmax(np.array([1.5, -0.5]), 2.0)
    assert abs(p[0] - 1.0 / (1.0 + math.exp(-1.0))) < 1e-15
    # -inf entries carry zero mass
    p, lse = O.softmax(np.array([0.0, -np.inf, 0.0]), 1.0)
    assert p[1] == 0.0 and abs(p[0] - 0.5) < 1e-16 and abs(lse - math.log(2)) < 1e-15


def test_row_validity():
    assert O.row_is_bad(np.array([0.0, np.nan]))
    assert O.row_is_bad(np.array([0.0, np.inf]))
    assert O.row_is_bad(np.array([-np.inf, -np.inf]))
    assert not O.row_is_bad(np.array([-np.inf, 3.0]))


# ----------------------------------------------------------------------------------------------
# top-k ids and the Saguaro bias
# ----------------------------------------------------------------------------------------------
def test_top_ids_planted_ties():
    z = np.array([1.0, 3.0, 3.0, 2.0, 3.0, -np.inf, 2.0])
    assert O.top_ids(z, 3).tolist() == [1, 2, 4]
    assert O.top_ids(z, 5).tolist() == [1, 2, 4, 3, 6]
    assert O.top_ids(z, 9).tolist() == [1, 2, 4, 3, 6, 0, 5]
    assert O.top_ids(z, 0).tolist() == []


def test_top_ids_against_lexsort():
    rng = np.random.default_rng(3)
    for _ in range(20):
        z = rng.integers(-4, 4, size=300).astype(np.float64)  # many ties
        ref = np.lexsort((np.arange(300), -z))[:8]
        assert O.top_ids(z, 8).tolist() == ref.tolist()


def test_biased_draft_hand_example():
    # q = (0.4, 0.3, 0.2, 0.1); down-weight the top-1 by beta = 1/2:
    # (0.2, 0.3, 0.2, 0.1) / 0.8 = (0.25, 0.375, 0.25, 0.125)
    q = np.array([0.4, 0.3, 0.2, 0.1])
    zd = np.log(q)
    qb, S = O.biased_draft(q, zd, 0.5, 1)
    assert S.tolist() == [0]
    assert np.allclose(qb, [0.25, 0.375, 0.25, 0.125], rtol=0, atol=1e-15)
    # top-2: (0.2, 0.15, 0.2, 0.1) / 0.65
    qb, S = O.biased_draft(q, zd, 0.5, 2)
    assert np.allclose(qb, np.array([0.2, 0.15, 0.2, 0.1]) / 0.65, rtol=0, atol=1e-15)
    # beta = 1 is the unbiased draft
    qb, S = O.biased_draft(q, zd, 1.0, 8)
    assert qb is q and len(S) == 0


# ----------------------------------------------------------------------------------------------
# inverse CDF
# ----------------------------------------------------------------------------------------------
def _brute_icdf(w, u):
    W = math.fsum(w)
    t = u * W
    c = 0.0
    for v, x in enumerate(w):
        c += x
        if c > t:
            return v
    return max(v for v, x in enumerate(w) if x > 0)


def test_inverse_cdf_brute_force_and_searchsorted():
    rng = np.random.default_rng(11)
    for _ in range(300):
        V = int(rng.integers(1, 40))
        w = rng.random(V) * (rng.random(V) < 0.7)
        if w.sum() == 0:
            w[0] = 1.0
        u = float(rng.random())
        v, margin = O.inverse_cdf(w, u)
        assert v == _brute_icdf(list(w), u)
        C = np.cumsum(w)
        assert v == int(np.searchsorted(C, u * C[-1], side="right"))
        assert w[v] > 0 and 0.0 <= margin <= 0.5 + 1e-12


def test_inverse_cdf_special_cases():
    w = np.array([0.0, 0.0, 2.0, 0.0, 1.0])
    assert O.inverse_cdf(w, 0.0)[0] == 2  # u = 0 -> first id with mass
    assert O.inverse_cdf(w, 0.6666)[0] == 2
    assert O.inverse_cdf(w, 0.6667)[0] == 4
    assert O.inverse_cdf(w, np.nextafter(1.0, 0.0))[0] == 4
    assert O.inverse_cdf(np.array([0.0, 5.0, 0.0]), 0.999)[0] == 1  # one-hot
    # margin is the distance to the nearest edge, relative to W
    v, m = O.inverse_cdf(np.array([1.0, 1.0, 2.0]), 0.3)
    assert v == 1 and abs(m - 0.05) < 1e-15


# ----------------------------------------------------------------------------------------------
# losslessness by exact enumeration
# ----------------------------------------------------------------------------------------------
LAW_CASES = [
    # V, L, T, beta, bias_k, zero_frac, seed
    (2, 1, 1.0, 1.0, 0, 0.0, 1),
    (2, 3, 1.0, 1.0, 0, 0.0, 2),
    (3, 2, 0.7, 1.0, 0, 0.0, 3),
    (3, 3, 1.0, 0.5, 1, 0.0, 4),
    (5, 1, 1.0, 1.0, 0, 0.3, 5),
    (5, 2, 1.3, 0.5, 2, 0.0, 6),
    (4, 2, 1.0, 1.0, 0, 0.4, 7),
]


def _law_setup(V, L, T, beta, bias_k, zero_frac, seed):
    rng = np.random.default_rng(seed)
    K = L
    tgt = np.stack([logits_for(random_probs(rng, V, zero_frac), T) for _ in range(K + 1)])
    dft = np.stack([logits_for(random_probs(rng, V, zero_frac), T) for _ in range(K)])
    p = [probs_of(tgt[i], T) for i in range(K + 1)]
    qb = [biased_probs_of(probs_of(dft[i], T), dft[i], beta, bias_k) for i in range(K)]
    return tgt, dft, p, qb


@pytest.mark.parametrize("case", LAW_CASES)
def test_losslessness_exact_enumeration(case):
    V, L, T, beta, bias_k, zero_frac, seed = case
    tgt, dft, p, qb = _law_setup(*case)
    run = runner(tgt, dft, T, beta, bias_k)
    law = output_law(run, L, L, V, lambda xs: float(np.prod([qb[i][x] for i, x in enumerate(xs)])))
    # closed-form outcome law: prod_{i<a} min(p_i(x_i), q'_i(x_i)) * (residual or bonus)
    expect = {}
    import itertools
    for a in range(L + 1):
        for pre in itertools.product(range(V), repeat=a):
            base = float(np.prod([min(p[i][x], qb[i][x]) for i, x in enumerate(pre)]))
            for y in range(V):
                tail = max(p[a][y] - qb[a][y], 0.0) if a < L else p[L][y]
                if base * tail > 0:
                    expect[tuple(pre) + (y,)] = base * tail
    keys = set(law) | set(expect)
    err = max(abs(law.get(k, 0.0) - expect.get(k, 0.0)) for k in keys)
    assert err < 1e-11, err
    assert abs(sum(law.values()) - 1.0) < 1e-11
    # consequence: every emitted position j is distributed as the target p_j
    alpha = [float(np.sum(np.minimum(p[i], qb[i]))) for i in range(L)]
    for j in range(L + 1):
        reach = float(np.prod(alpha[:j]))
        for v in range(V):
            got = sum(pr for k, pr in law.items() if len(k) > j and k[j] == v)
            assert abs(got - reach * p[j][v]) < 1e-11


@pytest.mark.parametrize("case", LAW_CASES[:4])
def test_expected_accept_len_closed_form(case):
    V, L, T, beta, bias_k, zero_frac, seed = case
    tgt, dft, p, qb = _law_setup(*case)
    law = output_law(runner(tgt, dft, T, beta, bias_k), L, L, V,
                     lambda xs: float(np.prod([qb[i][x] for i, x in enumerate(xs)])))
    e_a = sum(pr * (len(k) - 1) for k, pr in law.items())
    alpha = [float(np.sum(np.minimum(p[i], qb[i]))) for i in range(L)]
    assert abs(e_a - O.expected_accept_len(alpha)) < 1e-11


def test_expected_accept_len_monte_carlo():
    """Random drafts and uniforms on a wider row set: the mean accept length within 5 sigma."""
    rng = np.random.default_rng(21)
    V, K, T, n = 64, 4, 1.0, 4000
    zt = (rng.standard_normal((K + 1, V)) * 1.5).astype(np.float32)
    zd = (zt[:K] + rng.standard_normal((K, V)) * 0.6).astype(np.float32)
    p = [probs_of(zt[i], T) for i in range(K + 1)]
    q = [probs_of(zd[i], T) for i in range(K)]
    alpha = [float(np.sum(np.minimum(p[i], q[i]))) for i in range(K)]
    acc = []
    for _ in range(n):
        x = np.array([rng.choice(V, p=q[i]) for i in range(K)])
        u = rng.random(K + 1)
        acc.append(O.verify_sequence(zt, zd, x, K, u, temperature=T, mode="stochastic").accept_len)
    acc = np.array(acc, dtype=np.float64)
    mean, sd = acc.mean(), acc.std(ddof=1) / math.sqrt(n)
    assert abs(mean - O.expected_accept_len(alpha)) < 5 * sd


# ----------------------------------------------------------------------------------------------
# page values (tests/golden)
# ----------------------------------------------------------------------------------------------
def _read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if "=" in line:
                k, v = line.split("=", 1)
                vals[k.strip()] = v.strip()
    return vals


def _two_token_chain(alpha, L):
    """Rows with per-position acceptance exactly alpha: p = (1/2, 1/2), q = (1 - alpha + 1/2...)"""
    # min(p, q) sums to alpha when q = (1.5 - alpha, alpha - 0.5) for alpha in [0.5, 1]
    p = np.array([0.5, 0.5])
    q = np.array([1.5 - alpha, alpha - 0.5])
    tgt = np.stack([logits_for(p)] * (L + 1))
    dft = np.stack([logits_for(q)] * L)
    qq = probs_of(dft[0], 1.0)
    pp = probs_of(tgt[0], 1.0)
    return tgt, dft, pp, qq


@pytest.mark.parametrize("fixture", ["glossary_speedup_analysis.txt",
                                     "kangaroo_verification_chain.txt"])
def test_golden_acceptance_chain(fixture):
    g = _read_golden(fixture)
    alpha, L = float(g["alpha"]), int(g["draft_len"])
    tgt, dft, pp, qq = _two_token_chain(alpha, L)
    law = output_law(runner(tgt, dft, 1.0), L, L, 2,
                     lambda xs: float(np.prod([qq[x] for x in xs])))
    e_a = sum(pr * (len(k) - 1) for k, pr in law.items())
    a_real = float(np.sum(np.minimum(pp, qq)))  # alpha after float32 logit rounding
    assert abs(a_real - alpha) < 1e-6
    assert abs(e_a - O.expected_accept_len([a_real] * L)) < 1e-11
    assert abs(e_a - float(g["expected_accepted"])) < 1e-4
    assert abs(e_a + 1 - float(g["expected_tokens_per_round"])) < 1e-4
    if "page_claim_tokens" in g:  # the page's ~3.5 is alpha*K, which ignores the stop rule
        assert abs(float(g["page_claim_tokens"]) - alpha * L) < 1e-9
        assert e_a + 1 < float(g["page_claim_tokens"])


def test_golden_layerskip_greedy_trace():
    g = _read_golden("layerskip_greedy_trace.txt")
    V = int(g["vocab"])
    cases = [k for k in g if k.startswith("case")]
    assert cases
    for c in cases:
        drafts, preds, acc, toks = [s.strip() for s in g[c].split("|")]
        drafts = [int(v) for v in drafts.split()]
        preds = [int(v) for v in preds.split()]
        K = len(drafts)
        tgt = np.full((K + 1, V), -1.0, np.float32)
        for i, t in enumerate(preds):
            tgt[i, t] = 4.0  # planted unique argmax
        r = O.verify_sequence(tgt, None, np.array(drafts), K, np.zeros(K + 1, np.float32),
                              temperature=0.0, mode="greedy")
        assert r.accept_len == int(acc)
        assert r.tokens[: r.accept_len + 1].tolist() == [int(v) for v in toks.split()]


# ----------------------------------------------------------------------------------------------
# greedy and special cases
# ----------------------------------------------------------------------------------------------
def test_greedy_ties_and_prefix():
    V, K = 16, 3
    tgt = np.zeros((K + 1, V), np.float32)
    tgt[0, [3, 7]] = 5.0  # tie -> 3
    tgt[1, [9]] = 2.0
    tgt[2, [0, 15]] = 1.0  # tie -> 0
    tgt[3, [12, 13]] = 8.0  # bonus tie -> 12
    run = lambda x: O.verify_sequence(tgt, None, np.array(x), K, None, temperature=0,
                                      mode="greedy")
    r = run([3, 9, 0])
    assert r.accept_len == 3 and r.tokens.tolist() == [3, 9, 0, 12]
    r = run([7, 9, 0])
    assert r.accept_len == 0 and r.tokens.tolist() == [3, -1, -1, -1]
    r = run([3, 9, 15])
    assert r.accept_len == 2 and r.tokens.tolist() == [3, 9, 0, -1]


def test_q_equals_p_always_accepts():
    rng = np.random.default_rng(5)
    V, K, T = 50, 4, 0.9
    rows = (rng.standard_normal((K + 1, V)) * 2).astype(np.float32)
    for _ in range(50):
        x = rng.integers(0, V, size=K)
        u = rng.random(K + 1).astype(np.float32)
        r = O.verify_sequence(rows, rows[:K], x, K, u, temperature=T, mode="stochastic")
        assert r.accept_len == K
        # the bonus is the inverse-CDF draw from p_K
        assert r.tokens[K] == _brute_icdf(list(probs_of(rows[K], T)), float(u[K]))


def test_disjoint_one_hot_rejects_at_zero():
    V, K = 10, 3
    tgt = np.full((K + 1, V), -np.inf, np.float32)
    dft = np.full((K, V), -np.inf, np.float32)
    tgt[:, 2] = 0.0
    dft[:, 5] = 0.0
    for u0 in [0.0, 0.3, 0.999]:
        u = np.array([u0, 0.5, 0.5, 0.7], np.float32)
        r = O.verify_sequence(tgt, dft, np.array([5, 5, 5]), K, u, temperature=1.0,
                              mode="stochastic")
        assert r.accept_len == 0 and r.tokens.tolist() == [2, -1, -1, -1]


def test_zero_draft_probability_accepts():
    # q(x) = 0 < p(x): ratio is +inf, the draft is kept whatever u is
    tgt = np.array([[0.0, 0.0], [0.0, 0.0]], np.float32)
    dft = np.array([[0.0, -np.inf]], np.float32)
    r = O.verify_sequence(tgt, dft, np.array([1]), 1, np.array([0.99, 0.1], np.float32),
                          temperature=1.0, mode="stochastic")
    assert r.accept_len == 1


def test_beta_one_equals_unbiased():
    rng = np.random.default_rng(9)
    V, K = 40, 3
    zt = rng.standard_normal((K + 1, V)).astype(np.float32)
    zd = (zt[:K] + rng.standard_normal((K, V)) * 0.5).astype(np.float32)
    for _ in range(30):
        x = rng.integers(0, V, K)
        u = rng.random(K + 1).astype(np.float32)
        a = O.verify_sequence(zt, zd, x, K, u, temperature=1.0, mode="stochastic")
        b = O.verify_sequence(zt, zd, x, K, u, temperature=1.0, mode="stochastic", beta=1.0,
                              bias_k=8)
        assert a.accept_len == b.accept_len and a.tokens.tolist() == b.tokens.tolist()


def test_topf_is_prefix_of_top8():
    rng = np.random.default_rng(13)
    V, K = 200, 5
    zt = rng.integers(-3, 3, (K + 1, V)).astype(np.float32)  # heavy ties
    zd = rng.integers(-3, 3, (K, V)).astype(np.float32)
    x = rng.integers(0, V, K)
    r = O.verify_sequence(zt, zd, x, K, rng.random(K + 1).astype(np.float32), temperature=1.0,
                          mode="stochastic", beta=0.5, bias_k=8, fanout=(8, 4, 2, 1, 1))
    for i, F in enumerate((8, 4, 2, 1, 1)):
        ref = np.lexsort((np.arange(V), -zd[i].astype(np.float64)))[:8]
        assert r.topf[i, :F].tolist() == ref[:F].tolist()
        assert (r.topf[i, F:] == -1).all()


# ----------------------------------------------------------------------------------------------
# validity
# ----------------------------------------------------------------------------------------------
def test_invalid_sequences():
    V, K = 8, 3
    zt = np.zeros((K + 1, V), np.float32)
    zd = np.zeros((K, V), np.float32)
    u = np.full(K + 1, 0.5, np.float32)
    kw = dict(temperature=1.0, mode="stochastic")
    assert O.verify_sequence(zt, zd, np.array([1, 2, 3]), 0, u, **kw).accept_len == -1
    assert O.verify_sequence(zt, zd, np.array([1, 2, 3]), 4, u, **kw).accept_len == -1
    assert O.verify_sequence(zt, zd, np.array([1, 8, 3]), 3, u, **kw).accept_len == -1
    bad_u = u.copy()
    bad_u[K] = 1.0
    assert O.verify_sequence(zt, zd, np.array([1, 2, 3]), 3, bad_u, **kw).accept_len == -1
    nan_t = zt.copy()
    nan_t[0, 4] = np.nan
    r = O.verify_sequence(nan_t, zd, np.array([1, 2, 3]), 3, u, **kw)
    assert r.accept_len == -1 and (r.tokens == -1).all()
    # q == p accepts everything: a NaN in a padding row past L is never read
    pad = zt.copy()
    pad[K] = np.nan
    r = O.verify_sequence(pad, zd, np.array([1, 2, 3]), 2, u, **kw)
    assert r.valid and r.accept_len == 2
    # a row after the rejection is not needed either
    zt2 = np.zeros((K + 1, V), np.float32)
    zt2[0, 1] = -30.0  # p(x_0) ~ 0 -> reject at 0
    zt2[1:] = np.nan
    zd2 = zd.copy()
    zd2[1:] = np.nan
    r = O.verify_sequence(zt2, zd2, np.array([1, 2, 3]), 3, u, **kw)
    assert r.valid and r.accept_len == 0
    # ... unless top-F ids are requested, which need every draft row below L
    r = O.verify_sequence(zt2, zd2, np.array([1, 2, 3]), 3, u, fanout=(2, 2, 2), **kw)
    assert r.accept_len == -1
    # an all -inf row is invalid, a single -inf entry is fine
    ninf = zt.copy()
    ninf[0] = -np.inf
    assert O.verify_sequence(ninf, zd, np.array([1, 2, 3]), 3, u, **kw).accept_len == -1
    one = zt.copy()
    one[0, 0] = -np.inf
    assert O.verify_sequence(one, zd, np.array([1, 2, 3]), 3, u, **kw).valid


def test_residual_top_ids_brute_force():
    """Diagnostic top-f of the exact residual: brute force over a tiny row (SSD page, Method)."""
    rng = np.random.default_rng(17)
    for _ in range(20):
        V = 12
        zt = (rng.standard_normal(V) * 2).astype(np.float32)
        zd = (zt + rng.standard_normal(V)).astype(np.float32)
        p, q = probs_of(zt, 1.0), probs_of(zd, 1.0)
        r = [max(a - b, 0.0) for a, b in zip(p, q)]
        ref = [v for v in sorted(range(V), key=lambda v: (-r[v], v)) if r[v] > 0][:4]
        got = O.residual_top_ids(zt, zd, temperature=1.0, f=4).tolist()
        assert got == ref
