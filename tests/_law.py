"""Exact output law of a verify function, found by treating it as a black box.

For fixed logits and a fixed draft string, the verify outcome is a piecewise-constant function
of the uniforms: accept test ``i`` depends only on ``u[i]`` (given that tests ``0..i-1`` passed)
and the final token is a non-decreasing step function of ``u[K]`` (inverse CDF over ascending
ids). The edges of those pieces are located by bisection on the function itself, so the law
returned here is the function's own law, to ~1e-14, and never uses the formulas it is checked
against.
"""
from __future__ import annotations

import itertools
from collections import defaultdict

import numpy as np

BISECT_STEPS = 48


def _edge(pred, lo=0.0, hi=1.0):
    """Boundary r of a predicate that is True on [0, r) and False on [r, 1)."""
    top = np.nextafter(1.0, 0.0)
    if not pred(0.0):
        return 0.0
    if pred(top):
        return 1.0
    a, b = lo, hi
    for _ in range(BISECT_STEPS):
        m = 0.5 * (a + b)
        if pred(m):
            a = m
        else:
            b = m
    return 0.5 * (a + b)


def _final_cells(tok_of):
    """[(token, length)] pieces of the non-decreasing step function u -> token on [0, 1)."""
    cells = []
    start = 0.0
    top = np.nextafter(1.0, 0.0)
    while start < 1.0:
        tok = tok_of(start)
        if tok_of(top) == tok:
            cells.append((tok, 1.0 - start))
            break
        a, b = start, 1.0
        for _ in range(BISECT_STEPS):
            m = 0.5 * (a + b)
            if tok_of(m) == tok:
                a = m
            else:
                b = m
        cells.append((tok, b - start))
        start = b
    return cells


def output_law(run, K, L, V, draft_law):
    """Law of the emitted outcome ``(x_0..x_{a-1}, y)``.

    run(x, u) -> (accept_len, tokens) for a draft string x (length K) and float64 uniforms u
    (length K+1). ``draft_law(x)`` is the probability of the draft string (the drafter's law).
    Returns {outcome tuple: probability}.
    """
    law = defaultdict(float)
    for xs in itertools.product(range(V), repeat=L):
        px = draft_law(xs)
        if px <= 0.0:
            continue
        x = list(xs) + [0] * (K - L)

        def rec(i, us, wt):
            if wt <= 0.0:
                return
            if i == L:
                _final(us, wt, i)
                return

            def acc(v):
                u = np.array(us + [v] + [0.5] * (K - i - 1) + [0.5])
                return run(x, u)[0] > i

            r = _edge(acc)
            if r > 0.0:
                rec(i + 1, us + [0.5 * r], wt * r)
            if r < 1.0:
                _final(us + [0.5 * (1.0 + r)], wt * (1.0 - r), i)

        def _final(us, wt, a):
            pad = [0.5] * (K - len(us))

            def tok_of(v):
                acc_len, toks = run(x, np.array(us + pad + [v]))
                assert acc_len == a, (acc_len, a)
                return int(toks[a])

            for tok, ln in _final_cells(tok_of):
                law[tuple(xs[:a]) + (tok,)] += px * wt * ln

        rec(0, [], 1.0)
    return dict(law)
