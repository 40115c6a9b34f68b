"""Float64 CPU oracle for the batched speculative-sampling verify step.

TEST INFRASTRUCTURE. Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline /
reference legs of ``bench.py`` may import this module. The product path (the CUDA library and
its binding) never calls it, and it shares no code with that path.

It is a plain, slow, row-at-a-time restatement of what the pages define, in float64:

* Accept / reject (Kangaroo page, section "3. Lossless Speculative Verification"; glossary page
  "speculative decoding llm", "How Speculative Decoding Works" step 3 and "Why It Produces
  Identical Outputs"): draft token ``x_i`` is kept when ``u_i < min(1, p_i(x_i) / q_i(x_i))``;
  verification stops at the first rejection.
* Correction sample (same passages; SSD page "Key claims" on the bonus token): after a rejection
  at position ``a`` the emitted token is drawn from ``max(p_a - q_a, 0)`` normalised.
* Bonus sample (SSD page "Method": the outcome is the accepted-prefix length plus a bonus id;
  Kangaroo simulation's guaranteed bonus token): when every draft is accepted the token is drawn
  from ``p_L`` of the target row after the last draft.
* Greedy verification (LayerSkip page, "Systems Mechanics", Verification Phase and Prefix
  Acceptance): accept while the draft equals the target argmax, then emit the target argmax.
* Temperature-scaled full-vocabulary softmax (Kangaroo page, "Exit 1", the ``Softmax(W h)``
  draft head; SSD page on temperature).
* Saguaro biasing (SSD page, "Key claims" and "Method"): the ``bias_k`` most likely draft tokens
  have their draft probability scaled by ``beta`` and the distribution is renormalised; the same
  ``q'`` is used to draft and to verify.
* Top-F speculation-cache keys (SSD page, "Key claims", geometric fan-out; "Method"): for each
  position ``i < L`` the first ``F_i`` ids of the draft row ordered by logit (descending, ties to
  the lower id).

Readings where the pages are silent (each is listed with its reason in the design notes):
strict ``<`` in the accept test; ``q'(x) = 0`` gives ratio ``+inf`` if ``p(x) > 0`` else 0;
one temperature for both models; the final sample is an inverse CDF over ascending ids
(smallest ``v`` with ``C(v) > u W``); argmax ties go to the lower id; a zero residual mass falls
back to sampling ``p_a``; the greedy path emits a bonus argmax when every draft matches.

Validity: a sequence is invalid (accept length -1, all tokens -1) when ``L`` is outside
``[1, K]``, a draft id ``x_i`` (``i < L``) is outside ``[0, V)``, a used uniform is outside
``[0, 1)``, or a row the outcome needs holds NaN or ``+inf`` or is entirely ``-inf``. The rows
an outcome needs are read in order: target rows ``0..a`` and draft rows ``0..min(a, L-1)``
(plus every draft row ``i < L`` when top-F ids are requested).

Parity pins: every function here is checked in ``tests/test_oracle_pins.py`` against closed
forms, brute force and exact enumeration (losslessness), not against itself.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional, Sequence

import numpy as np

MARGIN = 1e-6  # decisions closer than this to their threshold are flagged, not compared


# --------------------------------------------------------------------------------------------
# element conversion
# --------------------------------------------------------------------------------------------
def row_to_f64(row: np.ndarray) -> np.ndarray:
    """Exact widening of one stored logit row (bf16 bit patterns as uint16, or float32)."""
    if row.dtype == np.uint16:
        return (row.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    return row.astype(np.float64)


def row_is_bad(z: np.ndarray) -> bool:
    """NaN or +inf anywhere, or every entry -inf: the row defines no distribution."""
    if np.isnan(z).any() or np.isposinf(z).any():
        return True
    return bool(np.isneginf(z).all())


# --------------------------------------------------------------------------------------------
# distributions
# --------------------------------------------------------------------------------------------
def softmax(z: np.ndarray, T: float):
    """p = softmax(z / T) over the whole vocabulary, and its log-normaliser lse(z / T).

    Returns (p, lse). Subtracting the maximum first is the usual overflow guard; it changes
    nothing mathematically.
    """
    y = z / T
    m = float(np.max(y))
    e = np.exp(y - m)
    s = float(np.sum(e))
    return e / s, m + math.log(s)


def top_ids(z: np.ndarray, k: int) -> np.ndarray:
    """The k ids with the largest logit, ordered by logit descending, ties to the lower id."""
    V = z.shape[0]
    k = min(k, V)
    if k <= 0:
        return np.zeros(0, dtype=np.int64)
    kth = np.partition(z, V - k)[V - k]  # k-th largest value
    cand = np.nonzero(z >= kth)[0]
    order = sorted(cand.tolist(), key=lambda v: (-z[v], v))
    return np.asarray(order[:k], dtype=np.int64)


def biased_draft(q: np.ndarray, zd: np.ndarray, beta: float, bias_k: int):
    """Saguaro-style draft: q'(v) = q(v) f(v) / (1 - (1 - beta) sum_{u in S} q(u)).

    S is the set of the ``bias_k`` ids with the largest draft logit, f = beta on S and 1 off it.
    beta == 1 or bias_k == 0 returns q unchanged (no renormalisation).
    Returns (q', S).
    """
    if beta >= 1.0 or bias_k <= 0:
        return q, np.zeros(0, dtype=np.int64)
    S = top_ids(zd, bias_k)
    f = np.ones_like(q)
    f[S] = beta
    return q * f / (1.0 - (1.0 - beta) * float(np.sum(q[S]))), S


def residual_weights(p: np.ndarray, qb: np.ndarray) -> np.ndarray:
    """Unnormalised corrected distribution max(p - q', 0) (Kangaroo page, section 3)."""
    return np.maximum(p - qb, 0.0)


def argmax_first(z: np.ndarray) -> int:
    """Index of the largest logit; ties go to the lower id."""
    return int(np.argmax(z))


def accept_ratio(px: float, qx: float) -> float:
    """p(x)/q'(x), with q'(x) = 0 read as +inf when p(x) > 0 and 0 otherwise."""
    if qx > 0.0:
        return px / qx
    return math.inf if px > 0.0 else 0.0


def inverse_cdf(w: np.ndarray, u: float):
    """Smallest id v with C(v) > u W, C the ascending-id cumulative sum of w, W = C(V-1).

    Returns (v, margin) with margin = min(t - C(v-1), C(v) - t) / W and t = u W, the relative
    distance of the draw to the nearest bin edge. If rounding leaves no such v, the largest id
    with w > 0 is taken.
    """
    C = np.cumsum(w)
    W = float(C[-1])
    t = u * W
    above = C > t
    if above.any():
        v = int(np.argmax(above))
    else:
        v = int(np.nonzero(w > 0)[0][-1])
    lo = float(C[v - 1]) if v > 0 else 0.0
    margin = min(t - lo, float(C[v]) - t) / W
    return v, margin


# --------------------------------------------------------------------------------------------
# one sequence
# --------------------------------------------------------------------------------------------
@dataclass
class SeqResult:
    accept_len: int
    tokens: np.ndarray  # [K+1] int32, -1 padded
    topf: np.ndarray  # [K, F_max] int32, -1 padded
    valid: bool = True
    # the decision chain, in order: ("acc", i, margin) for accept tests, ("cdf", a, margin)
    decisions: List[tuple] = field(default_factory=list)
    # diagnostics per position (NaN where not computed)
    lse_t: Optional[np.ndarray] = None  # [K+1]
    lse_d: Optional[np.ndarray] = None  # [K]
    p_x: Optional[np.ndarray] = None  # [K]
    q_x: Optional[np.ndarray] = None  # [K]
    alpha: Optional[np.ndarray] = None  # [K]
    residual_mass: float = math.nan
    used_fallback: bool = False

    def first_flag(self, margin: float = MARGIN):
        """Index into ``decisions`` of the first decision closer than ``margin``, or None."""
        for j, d in enumerate(self.decisions):
            if d[2] < margin:
                return j
        return None


def _invalid(K: int, fmax: int) -> SeqResult:
    return SeqResult(-1, np.full(K + 1, -1, np.int32), np.full((K, fmax), -1, np.int32),
                     valid=False)


def verify_sequence(target, draft, x, L, u, *, temperature: float, mode: str,
                    beta: float = 1.0, bias_k: int = 0,
                    fanout: Optional[Sequence[int]] = None, all_rows: bool = False):
    """Verify one sequence.

    target: [K+1, V] stored rows (uint16 bf16 bits or float32); draft: [K, V] or None (greedy).
    x: [K] draft ids; L: draft length; u: [K+1] float32 uniforms (u[i] accept test i, u[K] the
    final sample). ``all_rows`` also fills the diagnostics of rows after the decision; it never
    changes the outputs or the validity.
    """
    K = len(x)
    V = target.shape[1]
    fmax = max(fanout) if fanout else 0
    res = _invalid(K, fmax)
    res.lse_t = np.full(K + 1, np.nan)
    res.lse_d = np.full(K, np.nan)
    res.p_x = np.full(K, np.nan)
    res.q_x = np.full(K, np.nan)
    res.alpha = np.full(K, np.nan)
    bad = _invalid(K, fmax)
    if not (1 <= L <= K):
        return bad
    xs = [int(v) for v in x[:L]]
    if any(v < 0 or v >= V for v in xs):
        return bad
    greedy = mode == "greedy"
    if not greedy:
        used_u = [float(u[i]) for i in range(L)] + [float(u[K])]
        if any(not (0.0 <= uu < 1.0) for uu in used_u):
            return bad

    tokens = np.full(K + 1, -1, np.int32)
    topf = np.full((K, fmax), -1, np.int32)

    if greedy:
        a = None
        for i in range(L + 1):
            zt = row_to_f64(target[i])
            if row_is_bad(zt):
                return bad
            g = argmax_first(zt)
            if i < L and xs[i] == g:
                continue
            a, tok = i, g
            break
        res.accept_len = a
        tokens[:a] = xs[:a]
        tokens[a] = tok
        res.tokens, res.topf, res.valid = tokens, topf, True
        return res

    T = float(temperature)
    a = None
    w = None
    for i in range(L):
        zt, zd = row_to_f64(target[i]), row_to_f64(draft[i])
        if row_is_bad(zt) or row_is_bad(zd):
            return bad
        p, lse_t = softmax(zt, T)
        q, lse_d = softmax(zd, T)
        qb, _ = biased_draft(q, zd, beta, bias_k)
        px, qx = float(p[xs[i]]), float(qb[xs[i]])
        ratio = accept_ratio(px, qx)
        res.lse_t[i], res.lse_d[i], res.p_x[i], res.q_x[i] = lse_t, lse_d, px, qx
        res.alpha[i] = float(np.sum(np.minimum(p, qb)))
        res.decisions.append(("acc", i, abs(float(u[i]) - ratio)))
        if float(u[i]) < ratio:
            continue
        a = i
        w = residual_weights(p, qb)
        res.residual_mass = float(np.sum(w))
        if not res.residual_mass > 0.0:
            w = p
            res.used_fallback = True
        break
    if a is None:
        a = L
        zt = row_to_f64(target[L])
        if row_is_bad(zt):
            return bad
        w, res.lse_t[L] = softmax(zt, T)
    if fanout:
        for i in range(L):
            zd = row_to_f64(draft[i])
            if row_is_bad(zd):
                return bad
            f = min(int(fanout[i]), 8)
            ids = top_ids(zd, f)
            topf[i, :len(ids)] = ids
    tok, margin = inverse_cdf(w, float(u[K]))
    res.decisions.append(("cdf", a, margin))
    res.accept_len = a
    tokens[:a] = xs[:a]
    tokens[a] = tok
    res.tokens, res.topf, res.valid = tokens, topf, True

    if all_rows:  # diagnostics of the rows after the decision; outputs are already fixed
        for i in range(a + 1, L + 1):
            zt = row_to_f64(target[i])
            if not row_is_bad(zt):
                p, res.lse_t[i] = softmax(zt, T)
            if i < L:
                zd = row_to_f64(draft[i])
                if not row_is_bad(zd) and not row_is_bad(zt):
                    q, res.lse_d[i] = softmax(zd, T)
                    qb, _ = biased_draft(q, zd, beta, bias_k)
                    res.p_x[i], res.q_x[i] = float(p[xs[i]]), float(qb[xs[i]])
                    res.alpha[i] = float(np.sum(np.minimum(p, qb)))
    return res


def residual_top_ids(target_row, draft_row, *, temperature, beta=1.0, bias_k=0, f=8):
    """Diagnostic: the top-f ids of the exact residual max(p - q', 0) (ties to the lower id),
    restricted to ids with positive residual."""
    zt, zd = row_to_f64(target_row), row_to_f64(draft_row)
    p, _ = softmax(zt, temperature)
    q, _ = softmax(zd, temperature)
    qb, _ = biased_draft(q, zd, beta, bias_k)
    r = np.maximum(p - qb, 0.0)
    ids = top_ids(r, f)
    return ids[r[ids] > 0]


# --------------------------------------------------------------------------------------------
# a batch
# --------------------------------------------------------------------------------------------
def verify_batch(target, draft, draft_tokens, draft_lens, uniforms, *, temperature: float,
                 mode: str, beta: float = 1.0, bias_k: int = 0,
                 fanout: Optional[Sequence[int]] = None, all_rows: bool = False,
                 seqs: Optional[Sequence[int]] = None):
    """Verify every sequence (or the listed ``seqs``). Returns a list of SeqResult."""
    B, K = draft_tokens.shape
    idx = range(B) if seqs is None else seqs
    out = []
    for b in idx:
        L = int(draft_lens[b]) if draft_lens is not None else K
        u = uniforms[b] if uniforms is not None else np.zeros(K + 1, np.float32)
        out.append(verify_sequence(target[b], None if draft is None else draft[b],
                                   draft_tokens[b], L, u, temperature=temperature, mode=mode,
                                   beta=beta, bias_k=bias_k, fanout=fanout, all_rows=all_rows))
    return out


def expected_accept_len(alphas: Sequence[float]) -> float:
    """Closed form E[a] = sum_{j=1..L} prod_{i<j} alpha_i for per-position acceptance alpha_i.

    The glossary page's speedup analysis uses alpha ~ 0.7 and K = 5; acceptance stops at the
    first rejection, so the count is geometric-like rather than alpha * K.
    """
    total, run = 0.0, 1.0
    for al in alphas:
        run *= al
        total += run
    return total
