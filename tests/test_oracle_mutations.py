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


# ---- row steps (oracle/rows.py) ----
from oracle import rows as RO  # noqa: E402
from tests import test_oracle_rows_pins as RP  # noqa: E402


def test_confidence_from_biased_draft_is_caught(monkeypatch):
    real = RO.draft_sample

    def wrong(row, u, *, temperature, beta=1.0, bias_k=0, tau=0.0):
        d = real(row, u, temperature=temperature, beta=beta, bias_k=bias_k, tau=tau)
        z = O.row_to_f64(np.asarray(row))
        if O.row_is_bad(z):
            return d
        q, _ = O.softmax(z, temperature)
        qb, _ = O.biased_draft(q, z, beta, bias_k)
        d.conf = float(np.max(qb))
        return d
    monkeypatch.setattr(RO, "draft_sample", wrong)
    _fails(RP.test_confidence_ignores_the_bias_and_sets_the_exit_flag)


def test_draw_from_unbiased_draft_is_caught(monkeypatch):
    monkeypatch.setattr(O, "biased_draft", lambda q, zd, beta, k: (q, np.zeros(0, np.int64)))
    _fails(RP.test_draw_frequencies_by_exact_enumeration, 1.0, 0.5, 2)


def test_residual_against_unbiased_draft_is_caught(monkeypatch):
    monkeypatch.setattr(O, "biased_draft", lambda q, zd, beta, k: (q, np.zeros(0, np.int64)))
    _fails(RP.test_residual_order_hand_examples)


def test_residual_ties_to_higher_id_are_caught(monkeypatch):
    real = RO.residual_order

    def wrong(t, d, **kw):
        r, ids = real(t, d, **kw)
        return r, np.asarray(sorted(ids.tolist(), key=lambda v: (-round(r[v], 12), -v)))
    monkeypatch.setattr(RO, "residual_order", wrong)
    _fails(RP.test_residual_order_hand_examples)


def test_hit_at_the_bonus_position_is_caught(monkeypatch):
    def wrong(a, tokens, topf, L, fanout):
        if a < 0:
            return -1
        a = min(a, L - 1)
        return 1 if int(tokens[a]) in [int(v) for v in topf[a, :fanout[a]]] else 0
    monkeypatch.setattr(RO, "cache_hit", wrong)
    _fails(RP.test_cache_hit_hand_examples)


# ----------------------------------------------------------------------------------------------
# LM-head oracle
# ----------------------------------------------------------------------------------------------
from oracle import lmhead as HO  # noqa: E402
from tests import test_oracle_lmhead_pins as HP  # noqa: E402


def test_transposed_head_is_caught(monkeypatch):
    real = HO.head_logits
    # the head read column-wise: z[r, v] = sum_j h[r, j] W[j', v] for the square part
    monkeypatch.setattr(HO, "head_logits", lambda h, w: real(h, np.asarray(w)[::-1]))
    _fails(HP.test_one_hot_head_selects_hidden_units)


def test_lse_without_temperature_is_caught(monkeypatch):
    real = HO.softmax_stats
    monkeypatch.setattr(HO, "softmax_stats", lambda z, T, ids=None: real(z, 1.0, ids))
    _fails(HP.test_lse_closed_forms, 0.8)


def test_log2_sum_is_caught(monkeypatch):
    real = HO.softmax_stats

    def wrong(z, T, ids=None):
        st = real(z, T, ids)
        st.lse = st.max / T + (st.lse - st.max / T) / math.log(2.0)
        return st
    monkeypatch.setattr(HO, "softmax_stats", wrong)
    _fails(HP.test_lse_closed_forms, 1.0)


def test_unshifted_exponentials_are_caught(monkeypatch):
    def wrong(z, T, ids=None):
        z = np.asarray(z, np.float64)
        with np.errstate(over="ignore", divide="ignore"):
            lse = np.log(np.exp(z / T).sum(axis=1))
        return HO.HeadStats(z.max(axis=1), lse, np.full(z.shape[0], math.nan))
    monkeypatch.setattr(HO, "softmax_stats", wrong)
    _fails(HP.test_lse_of_large_logits_stays_finite)


def test_off_by_one_logit_at_id_is_caught(monkeypatch):
    real = HO.softmax_stats

    def wrong(z, T, ids=None):
        return real(z, T, None if ids is None else np.asarray(ids) + 1)
    monkeypatch.setattr(HO, "softmax_stats", wrong)
    _fails(HP.test_logit_at_id)


def test_too_tight_error_bound_is_caught(monkeypatch):
    real = HO.logit_error_bound
    monkeypatch.setattr(HO, "logit_error_bound", lambda h, w: real(h, w) / 4096.0)
    _fails(HP.test_error_bound_covers_float32_summation_orders)
