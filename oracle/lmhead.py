"""Float64 CPU oracle for the LM head of the verify step and its softmax statistics.

TEST INFRASTRUCTURE. Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline /
reference legs of ``bench.py`` may import this module. The product path never calls it and it
shares no code with that path.

* Logits (Kangaroo page, section 2, "Exit 1": the head maps a hidden state ``h`` to
  ``Softmax(W h)``; LayerSkip page: the early exit reuses the full model's head): ``z = h W^T``
  for bf16 ``h`` [R, d] and ``W`` [V, d], every product and sum taken in float64 (a bf16 x bf16
  product is exact there; the sum of ``d`` such terms carries one float64 rounding each).
* Statistics of the temperature softmax ``p = softmax(z / T)`` that the verify step needs per
  row (Kangaroo guide, section 3, and glossary, "Why It Produces Identical Outputs": the accept
  ratio ``p(x) / q(x)``): the largest logit ``max_v z_v``, the natural log-sum-exp
  ``ln sum_v exp(z_v / T)`` (so that ``ln p(x) = z_x / T - lse``), and the logit ``z_x`` of a
  requested id (NaN for an id outside ``[0, V)``). The log-sum-exp is taken about the maximum,
  ``M / T + ln sum exp((z - M) / T)``.

* The verify step from hidden states (Kangaroo guide, section 3, with the logits of "Exit 1";
  LayerSkip guide, "Verification Phase": the early-exit draft and the full model share the
  head): the logits of each sequence's rows are ``h W^T`` as above, and the outcome (with the
  Saguaro bias set and the top-F draft ids when asked for) is the one
  ``oracle.verify.verify_sequence`` gives for those float64 rows.

Parity pins: ``tests/test_oracle_lmhead_pins.py`` (one-hot heads, closed-form sums, shift and
scale laws, brute-force products on tiny inputs, and an identity head under which the verify
step from hidden states is the verify step of the hidden states read as logits).
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Optional, Sequence

import numpy as np

from . import verify as _v


def bf16_to_f64(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) to float64, exactly: the pattern is the top half of a float32."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def head_logits(hidden, weight) -> np.ndarray:
    """z = h W^T in float64 for ``hidden`` [R, d] and ``weight`` [V, d] (bf16 bits or floats)."""
    h = bf16_to_f64(hidden) if np.asarray(hidden).dtype == np.uint16 else np.asarray(hidden, np.float64)
    w = bf16_to_f64(weight) if np.asarray(weight).dtype == np.uint16 else np.asarray(weight, np.float64)
    if h.shape[-1] != w.shape[-1]:
        raise ValueError("hidden and weight disagree on d")
    return h @ w.T


@dataclass
class HeadStats:
    max: np.ndarray  # [R] largest logit
    lse: np.ndarray  # [R] ln sum_v exp(z_v / T)
    zx: np.ndarray   # [R] logit of the requested id (NaN when out of range or not asked)


def softmax_stats(z, temperature: float, ids: Optional[np.ndarray] = None) -> HeadStats:
    """The row statistics of ``softmax(z / T)`` for a float64 logit matrix ``z`` [R, V]."""
    z = np.asarray(z, dtype=np.float64)
    T = float(temperature)
    if not (T > 0.0):
        raise ValueError("temperature must be positive")
    R, V = z.shape
    M = z.max(axis=1)
    lse = M / T + np.log(np.exp((z - M[:, None]) / T).sum(axis=1))
    zx = np.full(R, math.nan)
    if ids is not None:
        ids = np.asarray(ids, dtype=np.int64)
        ok = (ids >= 0) & (ids < V)
        zx[ok] = z[np.nonzero(ok)[0], ids[ok]]
    return HeadStats(M, lse, zx)


def head_stats(hidden, weight, temperature: float, ids=None) -> HeadStats:
    """Logits of the head and their softmax statistics, in one call."""
    return softmax_stats(head_logits(hidden, weight), temperature, ids)


def logit_error_bound(hidden, weight) -> np.ndarray:
    """Bound on |fl32(z) - z| for logits summed in float32 from exact bf16 products, per
    (row, id): d * 2^-23 * sum_j |h_j w_j| (the classical bound for a sum of d terms, with a
    unit roundoff of 2^-23 so that truncating adders are covered too), times 1.01."""
    h = np.abs(bf16_to_f64(hidden))
    w = np.abs(bf16_to_f64(weight))
    d = h.shape[-1]
    return (d * 2.0 ** -23 * 1.01) * (h @ w.T)


def verify_hidden_batch(hidden_target, hidden_draft, weight, draft_tokens, draft_lens, uniforms,
                        *, temperature: float, mode: str, beta: float = 1.0, bias_k: int = 0,
                        fanout: Optional[Sequence[int]] = None,
                        seqs: Optional[Sequence[int]] = None):
    """The verify step on logits computed from hidden states: ``hidden_target`` [B, K+1, d],
    ``hidden_draft`` [B, K, d] (None in greedy mode) and ``weight`` [V, d], bf16 bits or floats.
    Only rows 0..L_b (target) and 0..L_b-1 (draft) are scored; the others are NaN rows the verify
    step never reads. ``beta``, ``bias_k`` (the Saguaro bias set of the draft rows) and ``fanout``
    (top-F draft ids) mean what they mean for ``oracle.verify.verify_sequence``, on those logits.
    Returns a list of ``oracle.verify.SeqResult``."""
    B, K = np.asarray(draft_tokens).shape
    V = np.asarray(weight).shape[0]
    out = []
    for b in (range(B) if seqs is None else seqs):
        L = int(draft_lens[b])
        zt = np.full((K + 1, V), np.nan)
        zd = np.full((K, V), np.nan) if hidden_draft is not None else None
        if 1 <= L <= K:
            zt[:L + 1] = head_logits(np.asarray(hidden_target)[b, :L + 1], weight)
            if zd is not None:
                zd[:L] = head_logits(np.asarray(hidden_draft)[b, :L], weight)
        out.append(_v.verify_sequence(zt, zd, draft_tokens[b], L, uniforms[b],
                                      temperature=temperature, mode=mode, beta=beta,
                                      bias_k=bias_k, fanout=fanout))
    return out
