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
    `band` is a scalar, or per decision an array [B, k+1] (accept test i in
    column i, the draw in column k): it widens the exemption where the GPU's
    inputs to the decisions carry a known extra rounding (the fused LM head's
    fp32 logits)."""
    B, k = case.B, case.k
    g_tokens = np.asarray(g_tokens)
    g_n = np.asarray(g_n)
    bands = np.broadcast_to(np.asarray(band, np.float64), (B, k + 1))
    report = dict(sequences=B, decisions=0, exempt=0, near_band=0, mismatched=[])
    for b in range(B):
        greedy = case.temperature[b] == 0
        report["decisions"] += decisions_of(int(r_n[b]), k, greedy)
        if not greedy and r_n[b] >= 0:
            tested = min(int(r_n[b]) + 1, k)
            th = trace[b, :tested]
            report["near_band"] += int(np.sum(np.abs(case.u_accept[b, :tested] - th)
                                              < bands[b, :tested]))
            lo, hi = trace[b, k], trace[b, k + 1]
            u = float(case.u_resample[b])
            if min(u - lo, hi - u) < bands[b, k]:
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
            bd = float(bands[b, pos])
        else:
            lo, hi = trace[b, k], trace[b, k + 1]
            u = float(case.u_resample[b])
            margin = min(u - lo, hi - u)
            kind = "bonus" if r_n[b] == k else "residual"
            bd = float(bands[b, k])
        if not margin < bd:
            raise AssertionError(f"mismatch outside the {bd:.3g} band (margin {margin:.3g}): " + why)
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


def compare_tree(tc, g_tokens, g_nodes, g_n, r_tokens, r_nodes, r_n, trace, band=BAND):
    """Tree-verification outputs against the oracle's.  Decisions per
    sequence: the sibling tests the oracle traced plus its one draw (greedy:
    one argmax comparison per visited node).  A mismatch is allowed only at
    a sampled sequence's first differing decision with the oracle's uniform
    within `band` of it: the sibling test one side accepted and the other
    rejected (|u - threshold|), or the draw (distance to the cell's edges).
    Returns the report of compare()."""
    g_tokens, g_nodes, g_n = map(np.asarray, (g_tokens, g_nodes, g_n))
    N = tc.N
    report = dict(sequences=tc.B, decisions=0, exempt=0, mismatched=[])
    for b in range(tc.B):
        greedy = tc.temperature[b] == 0
        rn = int(r_n[b])
        if rn < 0:
            report["decisions"] += 1
        elif greedy:
            report["decisions"] += rn + 1
        else:
            report["decisions"] += int(np.count_nonzero(~np.isnan(trace[b, 1:N]))) + 1
        same = (g_n[b] == r_n[b] and np.array_equal(g_tokens[b], r_tokens[b])
                and np.array_equal(g_nodes[b], r_nodes[b]))
        if same:
            continue
        why = (f"b={b} T={tc.temperature[b]} gpu n={g_n[b]} nodes {g_nodes[b][:max(0, g_n[b])].tolist()} "
               f"tokens {g_tokens[b][:max(0, g_n[b]) + 1].tolist()} oracle n={rn} "
               f"nodes {r_nodes[b][:max(0, rn)].tolist()} tokens {r_tokens[b][:max(0, rn) + 1].tolist()}")
        if greedy or g_n[b] < 0 or rn < 0:
            raise AssertionError("mismatch without exemption: " + why)
        gn = int(g_n[b])
        i = 0
        while i < min(gn, rn) and g_nodes[b, i] == r_nodes[b, i]:
            i += 1
        if i == gn == rn:
            lo, hi = trace[b, N], trace[b, N + 1]
            u = float(tc.u_resample[b])
            margin = min(u - lo, hi - u)
            kind = "draw"
        else:
            g = int(g_nodes[b, i]) if i < gn else 1 << 30
            o = int(r_nodes[b, i]) if i < rn else 1 << 30
            x = min(g, o)
            assert x < N and not np.isnan(trace[b, x]), "first differing test not traced: " + why
            margin = abs(float(tc.u_accept[b, x]) - trace[b, x])
            kind = "accept"
        if not margin < band:
            raise AssertionError(f"mismatch outside the {band} band (margin {margin:.3g}): " + why)
        report["exempt"] += 1
        report["mismatched"].append((b, kind, float(margin)))
    return report


def check_tree_invariants(tc, g_tokens, g_nodes, g_n):
    """Properties of any correct tree output: the path descends from the
    root through children, its tokens are the nodes' tokens, one emitted
    token in range, -1 padding after it."""
    g_tokens, g_nodes, g_n = map(np.asarray, (g_tokens, g_nodes, g_n))
    for b in range(tc.B):
        n = int(g_n[b])
        if n < 0:
            assert np.all(g_tokens[b] == -1) and np.all(g_nodes[b] == -1), b
            continue
        prev = 0
        for i in range(n):
            x = int(g_nodes[b, i])
            assert 0 < x < tc.n_nodes[b] and tc.parent[b, x] == prev, (b, i)
            assert g_tokens[b, i] == tc.tokens[b, x], (b, i)
            prev = x
        assert 0 <= g_tokens[b, n] < tc.V, b
        assert np.all(g_tokens[b, n + 1:] == -1) and np.all(g_nodes[b, n:] == -1), b
