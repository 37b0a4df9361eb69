"""Comparison of CUDA outputs with the oracle's, with the exemption band.

Integer outputs must match exactly.  The only allowed difference is a
sequence whose first diverging decision had the oracle's uniform within
BAND of its threshold (accept test: |u - min(1, P/Q)|) or of its draw cell's
boundary (|u - C(x-1)/R| or |C(x)/R - u|); such sequences are counted, and
the count must stay under MAX_EXEMPT_FRACTION (0.01 %) of the decisions
(check_bound).  Greedy decisions are exact comparisons and get no band.
"""
from __future__ import annotations

import numpy as np

BAND = 1e-5
MAX_EXEMPT_FRACTION = 1e-4


def check_bound(rep, accept_allowance=1):
    """Exempt mismatches against the 0.01 % bound, per call.  Draw mismatches:
    at most MAX_EXEMPT_FRACTION of the call's decisions, so none in a call of
    fewer than 1e4 decisions (draws within ~1e-6 of a cell edge are recomputed
    exactly, leaving only uniforms within ~1e-12 of an edge).  Accept-test
    mismatches: at most max(accept_allowance, the same fraction) per call; the
    fp32 ratio p/q is good to ~1e-6, and about 2e-6 of accept decisions have a
    uniform that close to it, so one per call is tolerated and the aggregate
    rate is checked over >1e5 decisions in tests/test_exact_draw_gpu.py."""
    kinds = [m[1] for m in rep["mismatched"]]
    draws = sum(1 for k in kinds if k != "accept")
    accepts = sum(1 for k in kinds if k == "accept")
    cap = MAX_EXEMPT_FRACTION * rep["decisions"]
    assert draws <= cap, f"{draws} draw mismatches in {rep['decisions']} decisions: {rep}"
    assert accepts <= max(accept_allowance, cap), \
        f"{accepts} accept-test mismatches in {rep['decisions']} decisions: {rep}"


def decisions_of(n_ref, k, greedy):
    """Decisions the oracle took for one sequence: accept tests plus one draw."""
    if n_ref < 0:
        return 1
    tests = min(n_ref + 1, k)
    return tests + 1


def compare(case, g_tokens, g_n, r_tokens, r_n, trace, band=BAND):
    """Returns a report dict; raises AssertionError on a non-exempt mismatch.
    `band` widens the exemption where the GPU's inputs to the decisions carry
    a known extra rounding (the fused LM head's fp32 logits)."""
    B, k = case.B, case.k
    g_tokens = np.asarray(g_tokens)
    g_n = np.asarray(g_n)
    report = dict(sequences=B, decisions=0, exempt=0, near_band=0, mismatched=[])
    for b in range(B):
        greedy = case.temperature[b] == 0
        report["decisions"] += decisions_of(int(r_n[b]), k, greedy)
        if not greedy and r_n[b] >= 0:
            tested = min(int(r_n[b]) + 1, k)
            th = trace[b, :tested]
            report["near_band"] += int(np.sum(np.abs(case.u_accept[b, :tested] - th) < band))
            lo, hi = trace[b, k], trace[b, k + 1]
            u = float(case.u_resample[b])
            if min(u - lo, hi - u) < band:
                report["near_band"] += 1
        if g_n[b] == r_n[b] and np.array_equal(g_tokens[b], r_tokens[b]):
            continue
        why = f"b={b} T={case.temperature[b]} gpu n={g_n[b]} {g_tokens[b].tolist()} " \
              f"oracle n={r_n[b]} {r_tokens[b].tolist()}"
        if greedy or g_n[b] < 0 or r_n[b] < 0:
            raise AssertionError("mismatch without exemption: " + why)
        if g_n[b] != r_n[b]:
            pos = int(min(g_n[b], r_n[b]))
            margin = abs(float(case.u_accept[b, pos]) - trace[b, pos])
            kind = "accept"
        else:
            lo, hi = trace[b, k], trace[b, k + 1]
            u = float(case.u_resample[b])
            margin = min(u - lo, hi - u)
            kind = "bonus" if r_n[b] == k else "residual"
        if not margin < band:
            raise AssertionError(f"mismatch outside the {band} band (margin {margin:.3g}): " + why)
        report["exempt"] += 1
        report["mismatched"].append((b, kind, float(margin)))
    report["draws"] = int(np.sum(np.asarray(r_n) >= 0))
    return report


def check_invariants(case, g_tokens, g_n):
    """Properties of any correct output: counts in range, accepted prefix is
    the drafts, one emitted token in range, -1 padding after it."""
    g_tokens = np.asarray(g_tokens)
    g_n = np.asarray(g_n)
    k, V = case.k, case.V
    assert g_n.shape == (case.B,) and g_tokens.shape == (case.B, k + 1)
    ok = g_n >= 0
    assert np.all((g_n[ok] >= 0) & (g_n[ok] <= k))
    for b in np.flatnonzero(ok):
        n = g_n[b]
        assert np.array_equal(g_tokens[b, :n], case.tokens[b, :n]), b
        assert 0 <= g_tokens[b, n] < V, b
        assert np.all(g_tokens[b, n + 1:] == -1), b
    assert np.all(g_tokens[~ok] == -1)
