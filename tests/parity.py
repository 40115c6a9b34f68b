"""Comparison of GPU verify outputs with the float64 oracle (shared by the GPU tests, smoke()
and bench.py's full-size check).

Accept lengths, token ids and top-F ids must match exactly, except that a decision whose oracle
margin is below 1e-6 (|u - p/q'| for an accept test, the relative CDF gap for the final draw)
is flagged: that decision and everything after it in the sequence are counted, not compared.
Diagnostics (log-normalisers, p(x), q'(x)) must agree within 1e-5 relative.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

from oracle import verify as O

REL_TOL = 1e-5


@dataclasses.dataclass
class Report:
    sequences: int = 0
    invalid: int = 0
    flagged: int = 0
    mismatches: list = dataclasses.field(default_factory=list)
    diag_checked: int = 0
    diag_bad: list = dataclasses.field(default_factory=list)

    def ok(self) -> bool:
        return not self.mismatches and not self.diag_bad

    def summary(self) -> str:
        return (f"{self.sequences} sequences, {self.invalid} invalid, {self.flagged} flagged, "
                f"{len(self.mismatches)} mismatches, {self.diag_checked} diagnostics checked, "
                f"{len(self.diag_bad)} out of tolerance")


def _close(a: float, b: float) -> bool:
    if math.isnan(a) or math.isnan(b):
        return math.isnan(a) and math.isnan(b)
    return abs(a - b) <= REL_TOL * max(1.0, abs(b)) if abs(b) >= 1.0 else \
        abs(a - b) <= REL_TOL * abs(b) + 1e-30


def compare(results, seqs, gpu_acc, gpu_tok, gpu_topf=None, dbg=None, x=None,
            margin: float = O.MARGIN) -> Report:
    """results: oracle SeqResults for sequences ``seqs``; gpu_*: numpy arrays over all B.
    ``margin``: decisions closer than this are flagged (1e-6 unless the inputs call for more)."""
    rep = Report()
    for r, b in zip(results, seqs):
        rep.sequences += 1
        ga, gt = int(gpu_acc[b]), gpu_tok[b]
        if not r.valid:
            rep.invalid += 1
            if ga != -1 or (gt != -1).any():
                rep.mismatches.append((b, "invalid", r.accept_len, ga))
            continue
        j = r.first_flag(margin)
        if j is None:
            if ga != r.accept_len or not np.array_equal(gt, r.tokens):
                rep.mismatches.append((b, "tokens", r.accept_len, ga, r.tokens.tolist(),
                                       gt.tolist()))
        else:
            rep.flagged += 1
            kind, pos, _ = r.decisions[j]
            if kind == "acc":
                if ga < pos or not np.array_equal(gt[:pos], r.tokens[:pos]):
                    rep.mismatches.append((b, "flagged-acc", pos, ga))
            else:
                a = r.accept_len
                if ga != a or not np.array_equal(gt[:a], r.tokens[:a]) or (gt[a + 1:] != -1).any():
                    rep.mismatches.append((b, "flagged-cdf", a, ga))
        if gpu_topf is not None and r.topf.shape[1] > 0:
            if not np.array_equal(gpu_topf[b][:, :r.topf.shape[1]], r.topf):
                rep.mismatches.append((b, "topf", r.topf.tolist(), gpu_topf[b].tolist()))
        if dbg is not None:
            for name, ref in (("lse_t", r.lse_t), ("lse_d", r.lse_d), ("p_x", r.p_x),
                              ("q_x", r.q_x)):
                got = dbg[name][b]
                for i, v in enumerate(ref):
                    if math.isnan(v):
                        continue
                    rep.diag_checked += 1
                    if not _close(float(got[i]), float(v)):
                        rep.diag_bad.append((b, name, i, float(got[i]), float(v)))
    return rep
