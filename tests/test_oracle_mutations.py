"""The pins must catch plausible mistakes: each test plants one in the oracle (CPU only, via
monkeypatch) and checks that a pin from test_oracle_pins.py then fails."""
import math

import numpy as np
import pytest

from oracle import verify as O
from tests import test_oracle_pins as P


def _fails(fn, *args):
    with pytest.raises(AssertionError):
        fn(*args)


def test_inverted_ratio_is_caught(monkeypatch):
    monkeypatch.setattr(O, "accept_ratio", lambda px, qx: (qx / px) if px > 0 else math.inf)
    _fails(P.test_losslessness_exact_enumeration, P.LAW_CASES[1])


def test_ratio_without_draft_probability_is_caught(monkeypatch):
    monkeypatch.setattr(O, "accept_ratio", lambda px, qx: px)
    _fails(P.test_losslessness_exact_enumeration, P.LAW_CASES[2])


def test_missing_bias_renormalisation_is_caught(monkeypatch):
    real = O.biased_draft

    def wrong(q, zd, beta, k):
        qb, S = real(q, zd, beta, k)
        if len(S) == 0:
            return qb, S
        f = np.ones_like(q)
        f[S] = beta
        return q * f, S
    monkeypatch.setattr(O, "biased_draft", wrong)
    _fails(P.test_losslessness_exact_enumeration, P.LAW_CASES[3])


def test_dropped_temperature_is_caught(monkeypatch):
    real = O.softmax
    monkeypatch.setattr(O, "softmax", lambda z, T: real(z, 1.0))
    _fails(P.test_losslessness_exact_enumeration, P.LAW_CASES[2])


def test_unclamped_residual_is_caught(monkeypatch):
    monkeypatch.setattr(O, "residual_weights", lambda p, qb: p - qb + 0.0)
    _fails(P.test_losslessness_exact_enumeration, P.LAW_CASES[5])


def test_swapped_residual_is_caught(monkeypatch):
    monkeypatch.setattr(O, "residual_weights", lambda p, qb: np.maximum(qb - p, 0.0))
    _fails(P.test_losslessness_exact_enumeration, P.LAW_CASES[1])


def test_last_occurrence_argmax_is_caught(monkeypatch):
    monkeypatch.setattr(O, "argmax_first", lambda z: int(len(z) - 1 - np.argmax(z[::-1])))
    _fails(P.test_greedy_ties_and_prefix)


def test_non_strict_cdf_edge_is_caught(monkeypatch):
    def wrong(w, u):
        C = np.cumsum(w)
        t = u * C[-1]
        v = int(np.argmax(C >= t))
        return v, 0.5
    monkeypatch.setattr(O, "inverse_cdf", wrong)
    _fails(P.test_inverse_cdf_special_cases)


def test_descending_cdf_is_caught(monkeypatch):
    real = O.inverse_cdf

    def wrong(w, u):
        v, m = real(w[::-1], u)
        return len(w) - 1 - v, m
    monkeypatch.setattr(O, "inverse_cdf", wrong)
    _fails(P.test_inverse_cdf_brute_force_and_searchsorted)


def test_higher_id_tie_break_is_caught(monkeypatch):
    def wrong(z, k):
        order = sorted(range(len(z)), key=lambda v: (-z[v], -v))
        return np.asarray(order[:k], dtype=np.int64)
    monkeypatch.setattr(O, "top_ids", wrong)
    _fails(P.test_top_ids_planted_ties)
