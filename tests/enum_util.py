"""Exact enumeration of a verification round's outcomes (test helper).

For one sequence with fixed logits and draft tokens, the outcome is a
deterministic function of the uniforms: accept test i passes for
u_accept[i] < theta_i, and the draw is a nondecreasing step function of
u_resample.  Finding the thresholds and the draw's breakpoints by bisection on
the *outputs alone* gives every outcome's exact probability (the product of
the cell widths), without trusting any internal quantity of the implementation
under test.
"""
from __future__ import annotations

import numpy as np

ONE_MINUS = 1.0 - 2.0 ** -53


def threshold(accepts, iters: int = 64) -> float:
    """theta such that accepts(u) holds for u < theta and fails above."""
    if not accepts(0.0):
        return 0.0
    if accepts(ONE_MINUS):
        return 1.0
    lo, hi = 0.0, 1.0
    for _ in range(iters):
        mid = 0.5 * (lo + hi)
        if mid <= lo or mid >= hi:
            break
        if accepts(mid):
            lo = mid
        else:
            hi = mid
    return hi


def draw_cells(token_of, iters: int = 64):
    """[(token, width)] for a nondecreasing step function on [0, 1)."""
    out = []

    def rec(lo, hi, tlo, thi, depth):
        if tlo == thi:
            out.append((tlo, lo, hi))
            return
        if depth >= iters or hi - lo <= 1e-17:
            # a breakpoint inside [lo, hi]; split it at its midpoint
            mid = 0.5 * (lo + hi)
            out.append((tlo, lo, mid))
            out.append((thi, mid, hi))
            return
        mid = 0.5 * (lo + hi)
        tm = token_of(mid)
        rec(lo, mid, tlo, tm, depth + 1)
        rec(mid, hi, tm, thi, depth + 1)

    rec(0.0, 1.0, token_of(0.0), token_of(ONE_MINUS), 0)
    # intervals come out in order and contiguous: merge runs of one token
    merged = []
    for tok, lo, hi in out:
        if merged and merged[-1][0] == tok:
            merged[-1] = (tok, merged[-1][1], hi)
        else:
            merged.append((tok, lo, hi))
    return [(tok, hi - lo) for tok, lo, hi in merged]


def enumerate_round(run, k: int):
    """All outcomes of one round and their probabilities.

    run(u_accept: list[float], u_resample: float) -> (n_acc, out_tokens list).
    Returns {emitted tuple: probability}.
    """
    outcomes = {}

    def add(key, prob):
        if prob > 0.0:
            outcomes[key] = outcomes.get(key, 0.0) + prob

    def rec(i, ua, prob):
        # positions < i are accepted with the uniforms in ua
        if i == k:
            cells = draw_cells(lambda u: tuple(run(ua, u)[1]))
            for toks, w in cells:
                add(tuple(t for t in toks if t >= 0), prob * w)
            return
        th = threshold(lambda u: run(ua + [u] + [0.0] * (k - i - 1), 0.5)[0] > i)
        if th < 1.0:
            mid = 0.5 * (th + 1.0)
            pre = ua + [mid] + [0.0] * (k - i - 1)
            cells = draw_cells(lambda u: tuple(run(pre, u)[1]))
            for toks, w in cells:
                add(tuple(t for t in toks if t >= 0), prob * (1.0 - th) * w)
        if th > 0.0:
            rec(i + 1, ua + [0.5 * th], prob * th)

    rec(0, [], 1.0)
    return outcomes


def softmax64(logits, T: float = 1.0):
    from scipy.special import softmax
    return softmax(np.asarray(logits, np.float64) / T)


def enumerate_leaves(run, k: int):
    """Like enumerate_round, but returns the cells themselves:
    [(u_accept midpoints list, u_resample midpoint, probability, draw width,
    emitted tuple)].  Used to replay every cell through another
    implementation at its midpoint."""
    leaves = []

    def draw_leaves(pre, prob):
        out = []

        def tok(u):
            return tuple(run(pre, u)[1])
        # breakpoints of the draw as a function of u_resample
        cells = []
        acc = 0.0
        for toks, w in draw_cells(tok):
            cells.append((toks, acc, acc + w))
            acc += w
        for toks, lo, hi in cells:
            out.append((list(pre), 0.5 * (lo + hi), prob * (hi - lo), hi - lo,
                        tuple(t for t in toks if t >= 0)))
        return out

    def rec(i, ua, prob):
        if i == k:
            leaves.extend(draw_leaves(ua, prob))
            return
        th = threshold(lambda u: run(ua + [u] + [0.0] * (k - i - 1), 0.5)[0] > i)
        if th < 1.0:
            pre = ua + [0.5 * (th + 1.0)] + [0.0] * (k - i - 1)
            leaves.extend(draw_leaves(pre, prob * (1.0 - th)))
        if th > 0.0:
            rec(i + 1, ua + [0.5 * th], prob * th)

    rec(0, [], 1.0)
    return leaves
