"""Float64 CPU oracle for the row steps beside the verify step: drawing a draft token from the
biased draft distribution (with the draft head's exit confidence), the exact-residual top-F ids
and the speculation-cache hit flag.

TEST INFRASTRUCTURE. Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline /
reference legs of ``bench.py`` may import this module. The product path never calls it and it
shares no code with that path.

* Draft draw (SSD page, "Method": the drafter samples from the Saguaro-biased ``q'``, the same
  distribution the verifier divides by): ``x ~ q'`` by the inverse CDF over ascending ids that
  the verify step's final draw uses.
* Exit confidence (Kangaroo page, section 2, "Exit 2"): ``c = max_v q(v)`` of the draft head's
  unbiased softmax; drafting stops once ``c < tau``. The pages give the confidence of the draft
  head's own distribution, so the biased ``q'`` plays no part in it (a reading; the design notes
  list it).
* Exact-residual top-F (SSD page, "Key claims" and "Method"): after a rejection at position
  ``i`` the emitted token follows ``max(p_i - q'_i, 0)``; its ``F_i`` most likely ids (ties to the
  lower id, ids with zero residual left out) are what a cache keyed by the exact residual would
  prepare, next to the draft-row top-F keys the verify step reports.
* Cache hit: whether the token drawn at the decided position ``a < L`` is among the top-F keys
  prepared for position ``a``; undefined (-1) when every draft was accepted (the bonus draw
  from ``p_L`` is no residual) or the sequence is invalid.

Parity pins: ``tests/test_oracle_rows_pins.py`` (closed forms, exact enumeration of the draw,
brute force of the residual order, hand-worked hit flags).
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Optional, Sequence

import numpy as np

from . import verify as _v


@dataclass
class DraftDraw:
    token: int     # -1 for a bad row or a uniform outside [0, 1)
    margin: float  # relative distance of u W to the nearest CDF edge (inf when token is -1)
    conf: float    # max_v q(v) of the unbiased softmax (NaN for a bad row)
    exit: int      # 1 if conf < tau, 0 if not, -1 for a bad row


def draft_sample(row, u: float, *, temperature: float, beta: float = 1.0, bias_k: int = 0,
                 tau: float = 0.0) -> DraftDraw:
    """One draft step on one stored logit row (uint16 bf16 bits or float32)."""
    z = _v.row_to_f64(np.asarray(row))
    if _v.row_is_bad(z):
        return DraftDraw(-1, math.inf, math.nan, -1)
    q, _ = _v.softmax(z, float(temperature))
    conf = float(np.max(q))
    ex = 1 if conf < float(tau) else 0
    if not (0.0 <= float(u) < 1.0):
        return DraftDraw(-1, math.inf, conf, ex)
    qb, _ = _v.biased_draft(q, z, float(beta), int(bias_k))
    tok, margin = _v.inverse_cdf(qb, float(u))
    return DraftDraw(int(tok), float(margin), conf, ex)


def residual_order(target_row, draft_row, *, temperature: float, beta: float = 1.0,
                   bias_k: int = 0):
    """(r, ids): the exact residual max(p - q', 0) of one position and its positive ids ordered
    by residual descending, ties to the lower id."""
    zt, zd = _v.row_to_f64(np.asarray(target_row)), _v.row_to_f64(np.asarray(draft_row))
    p, _ = _v.softmax(zt, float(temperature))
    q, _ = _v.softmax(zd, float(temperature))
    qb, _ = _v.biased_draft(q, zd, float(beta), int(bias_k))
    r = _v.residual_weights(p, qb)
    pos = np.nonzero(r > 0.0)[0]
    ids = pos[np.lexsort((pos, -r[pos]))]
    return r, ids


def residual_topf(target, draft, draft_lens, *, temperature: float, fanout: Sequence[int],
                  beta: float = 1.0, bias_k: int = 0, seqs: Optional[Sequence[int]] = None):
    """[n, K, max F] int32: the first F_i ids of ``residual_order`` for every position i < L of
    the listed sequences, -1 padded; all -1 for L outside [1, K] and for a position whose target
    or draft row is bad (NaN, +inf, or all -inf)."""
    B, K = draft.shape[0], draft.shape[1]
    fmax = max(max(fanout), 1)
    idx = list(range(B)) if seqs is None else list(seqs)
    out = np.full((len(idx), K, fmax), -1, np.int32)
    for n, b in enumerate(idx):
        L = int(draft_lens[b]) if draft_lens is not None else K
        if not 1 <= L <= K:
            continue
        for i in range(L):
            zt, zd = _v.row_to_f64(target[b, i]), _v.row_to_f64(draft[b, i])
            if _v.row_is_bad(zt) or _v.row_is_bad(zd):
                continue
            _, ids = residual_order(target[b, i], draft[b, i], temperature=temperature,
                                    beta=beta, bias_k=bias_k)
            f = min(int(fanout[i]), 8, len(ids))
            out[n, i, :f] = ids[:f]
    return out


def cache_hit(accept_len: int, tokens, topf, L: int, fanout: Sequence[int]) -> int:
    """1 if the token drawn at the decided position a < L is among the first F_a entries of
    ``topf[a]``, 0 if not, -1 when a == L (every draft accepted) or the sequence is invalid."""
    a = int(accept_len)
    if a < 0 or not 1 <= L <= len(fanout) or a >= L:
        return -1
    f = min(int(fanout[a]), topf.shape[1])
    return 1 if int(tokens[a]) in [int(v) for v in topf[a, :f]] else 0
