"""Pins of the fp64 oracle to what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: a value the
pages print (tests/golden/), a closed form, an exact enumeration of outcome
probabilities (the exactness theorem), a library routine (scipy softmax,
numpy searchsorted / argmax), or a Monte-Carlo chi-square.  A dropped term, a
wrong sign, a swapped p/q or a non-strict comparison in the oracle fails at
least one of them.
"""
import json
import os

import numpy as np
import pytest
from scipy import stats
from scipy.special import softmax as sp_softmax

import oracle
from tests.enum_util import enumerate_round, softmax64, threshold


def _one(target_rows, draft_rows, tokens, T=1.0, dtype=np.float32):
    """Bind a single sequence's inputs; returns run(u_accept list, u_resample)."""
    t = np.asarray(target_rows, dtype)[None]
    d = np.asarray(draft_rows, dtype)[None]
    g = np.asarray(tokens, np.int32)[None]
    k = g.shape[1]

    def run(ua, ur):
        toks, n, _ = oracle.verify(t, d, g, np.asarray(ua, np.float64)[None],
                                   np.asarray([ur], np.float64), np.asarray([T]))
        return int(n[0]), [int(x) for x in toks[0]]
    run.k = k
    return run


# ------------------------------------------------------------ building blocks

def test_softmax_matches_scipy():
    rng = np.random.default_rng(0)
    for V in (2, 3, 17, 1000):
        for T in (0.3, 1.0, 2.5):
            l = (rng.standard_normal(V) * 3).astype(np.float32).astype(np.float64)
            p = oracle.softmax(l, T)
            np.testing.assert_allclose(p, sp_softmax(l / T), rtol=1e-13, atol=1e-300)


def test_softmax_masked_entries_are_zero():
    p = oracle.softmax(np.array([0.0, -np.inf, 1.0, -np.inf]), 1.0)
    assert p[1] == 0.0 and p[3] == 0.0
    np.testing.assert_allclose(p[[0, 2]], sp_softmax([0.0, 1.0]), rtol=1e-15)


def test_residual_split_identity():
    """min(p,q) + max(0,p-q) = p for every x, and the rejection mass
    sum max(0,p-q) = 1 - sum min(p,q): "Speculative Decoding and the Art of
    Fast LLM Inference", "Why It Stays Exact"; the interview page's proof."""
    rng = np.random.default_rng(1)
    for V in (2, 3, 10, 1000):
        for _ in range(20):
            p = rng.dirichlet(np.ones(V) * 0.5)
            q = rng.dirichlet(np.ones(V) * 0.5)
            w, R = oracle.residual(p, q)
            np.testing.assert_allclose(np.minimum(p, q) + w, p, rtol=0, atol=1e-15)
            assert abs(R - (1.0 - np.minimum(p, q).sum())) < 1e-14
            assert np.all(w >= 0)
            assert np.all(w[p <= q] == 0)


def test_inverse_cdf_matches_searchsorted():
    """smallest x with C(x) > u*R equals numpy's searchsorted(side='right') on
    the running sum; zero-weight tokens are never drawn."""
    rng = np.random.default_rng(2)
    for V in (2, 5, 64, 777):
        w = rng.random(V) * (rng.random(V) < 0.6)
        if w.sum() == 0:
            w[0] = 1.0
        C = np.cumsum(w)
        for u in np.concatenate([rng.random(200), [0.0, ONE_MINUS_F32, 1 - 2 ** -53]]):
            x, cell = oracle.inverse_cdf(w, u)
            exp = int(np.searchsorted(C, u * C[-1], side="right"))
            if exp >= V:  # rounding clamp: largest positive-weight token
                exp = int(np.flatnonzero(w > 0)[-1])
            assert x == exp
            assert w[x] > 0
            assert cell[0] - 1e-15 <= u < cell[1] + 1e-15
            assert u * C[-1] < C[-1]  # u < 1 keeps u*R below R, so the clamp never fires


ONE_MINUS_F32 = float(np.nextafter(np.float32(1), np.float32(0)))


def test_accept_is_strict_less_than():
    """accept_token: `random.random() < target_prob / draft_prob` -- a uniform
    equal to the ratio rejects.  p = 1/4 everywhere, q = (1/2, 1/2, 0, 0): the
    ratio at token 0 is exactly 1/2."""
    run = _one([[0, 0, 0, 0], [0, 0, 0, 0]], [[0, 0, -np.inf, -np.inf]], [0])
    assert run([0.5], 0.5)[0] == 0
    assert run([np.nextafter(0.5, 0)], 0.5)[0] == 1


def test_accept_when_target_at_least_draft():
    """target_prob >= draft_prob accepts whatever the uniform."""
    run = _one([[1.0, 0.0], [0.0, 0.0]], [[0.0, 0.0]], [0])
    assert run([1 - 2 ** -53], 0.5)[0] == 1


def test_zero_target_probability_always_rejects():
    run = _one([[-np.inf, 0.0], [0.0, 0.0]], [[0.0, 0.0]], [0])
    n, toks = run([0.0], 0.3)
    assert n == 0 and toks[0] == 1  # the residual puts all mass on token 1


# ------------------------------------------------------------ worked example

def test_red_blue_example(golden_dir):
    """The red/blue example: draft 0.8/0.2, target 0.5/0.5 -> emitted 50/50;
    accepted red 0.5, blue 0.2, the rejected 0.3 all resampled to blue."""
    g = json.load(open(os.path.join(golden_dir, "red_blue.json")))
    q = np.array(g["draft_probs"])
    p = np.array(g["target_probs"])
    d_logits = np.log(q).astype(np.float32)
    t_logits = np.log(p).astype(np.float32)
    qf = softmax64(d_logits)
    pf = softmax64(t_logits)
    emitted = np.zeros(2)
    accepted = np.zeros(2)
    resampled = np.zeros(2)
    for tok in (0, 1):
        run = _one([t_logits, [0.0, 0.0]], [d_logits], [tok])
        out = enumerate_round(run, 1)
        for seq, prob in out.items():
            emitted[seq[0]] += qf[tok] * prob
            if len(seq) == 2:
                accepted[tok] += qf[tok] * prob
            else:
                resampled[seq[0]] += qf[tok] * prob
    # exact in the fp32-rounded distributions, and equal to the printed values
    np.testing.assert_allclose(emitted, pf, atol=1e-12)
    np.testing.assert_allclose(emitted, g["emitted"], atol=1e-7)
    assert abs(accepted[0] - g["accepted_red_mass"]) < 1e-7
    assert abs(accepted[1] - g["accepted_blue_mass"]) < 1e-7
    assert abs(resampled.sum() - g["resampled_mass"]) < 1e-7
    assert resampled[0] < 1e-12 and abs(resampled[1] - g["resampled_mass"]) < 1e-7


def test_trace_thresholds_match_bisection():
    """The oracle's trace (used for parity margins) agrees with thresholds
    found from its outputs alone."""
    rng = np.random.default_rng(3)
    for _ in range(10):
        t = rng.standard_normal((3, 5)).astype(np.float32)
        d = rng.standard_normal((2, 5)).astype(np.float32)
        g = rng.integers(0, 5, 2)
        run = _one(t, d, g)
        th = threshold(lambda u: run([u, 0.0], 0.5)[0] >= 1)
        _, _, tr = oracle.verify(t[None], d[None], g[None].astype(np.int32),
                                 np.array([[0.5 * th, 0.0]]), np.array([0.5]), np.array([1.0]))
        assert abs(tr[0, 0] - th) < 1e-12


# ------------------------------------------------------- sequence exactness

@pytest.mark.parametrize("seed", [11, 12, 13])
def test_exact_enumeration_V3_k2(seed):
    """Emitted-sequence probabilities equal the target's autoregressive
    distribution: per-position exactness carries over to whole generated
    sequences (thelatentsource page, 'The correction that keeps the target in
    charge').  V=3, k=2; every draft sequence g in V^2 weighted
    by q, every accept/draw cell by its width.  Emitted prefixes shorter than
    k+1 are completed with the target's own conditionals."""
    V, k = 3, 2
    rng = np.random.default_rng(seed)
    f = lambda *s: (rng.standard_normal(s) * 1.5).astype(np.float32)
    t0, t1, t2 = f(V), f(V, V), f(V, V, V)
    d0, d1 = f(V), f(V, V)
    p0, p1, p2 = softmax64(t0), np.array([softmax64(r) for r in t1]), \
        np.array([[softmax64(r) for r in rr] for rr in t2])
    q0, q1 = softmax64(d0), np.array([softmax64(r) for r in d1])
    joint = np.zeros((V, V, V))
    for g1 in range(V):
        for g2 in range(V):
            wg = q0[g1] * q1[g1, g2]
            run = _one([t0, t1[g1], t2[g1, g2]], [d0, d1[g1]], [g1, g2])
            for seq, prob in enumerate_round(run, k).items():
                pr = wg * prob
                if len(seq) == 3:
                    joint[seq] += pr
                elif len(seq) == 2:
                    joint[seq[0], seq[1], :] += pr * p2[seq[0], seq[1]]
                else:
                    joint[seq[0]] += pr * p1[seq[0]][:, None] * p2[seq[0]]
    target = p0[:, None, None] * p1[:, :, None] * p2
    np.testing.assert_allclose(joint, target, atol=1e-12)
    assert abs(joint.sum() - 1.0) < 1e-12


def test_enumeration_detects_a_planted_mistake():
    """The enumeration is sensitive: sampling the correction from p instead of
    norm(max(0, p-q)) (the page's warning that this biases the result) gives
    a visibly different emitted distribution for the red/blue example."""
    q = np.array([0.8, 0.2])
    p = np.array([0.5, 0.5])
    theta = np.minimum(1, p / q)
    right = q * theta + (1 - (q * theta).sum()) * np.maximum(0, p - q) / np.maximum(0, p - q).sum()
    wrong = q * theta + (1 - (q * theta).sum()) * p
    np.testing.assert_allclose(right, p, atol=1e-15)
    assert np.abs(wrong - p).max() > 0.1


# --------------------------------------------------------- accept-count law

def _constant_alpha_law(p, q, k):
    """Exact distribution of the number of accepted drafts when every position
    has the same target p and draft q (V=2): enumeration over g in {0,1}^k."""
    tl = np.log(np.asarray(p, np.float64)).astype(np.float32)
    dl = np.log(np.asarray(q, np.float64)).astype(np.float32)
    qf = softmax64(dl)
    law = np.zeros(k + 1)
    for code in range(2 ** k):
        g = [(code >> i) & 1 for i in range(k)]
        wg = float(np.prod([qf[x] for x in g]))
        run = _one([tl] * (k + 1), [dl] * k, g)
        prob_reach = 1.0
        ua = []
        for i in range(k):
            th = threshold(lambda u: run(ua + [u] + [0.0] * (k - i - 1), 0.5)[0] > i)
            law[i] += wg * prob_reach * (1 - th)
            prob_reach *= th
            ua.append(0.5 * th)
            if th == 0.0:
                break
        law[k] += wg * prob_reach
    alpha = float(np.minimum(softmax64(tl), qf).sum())
    return law, alpha


@pytest.mark.parametrize("p,q,k,golden_alpha", [
    ((0.7, 0.3), (0.5, 0.5), 5, 0.8),
    ((0.7, 0.3), (0.5, 0.5), 4, 0.8),
    ((0.9, 0.1), (0.5, 0.5), 4, 0.6),
    ((0.6, 0.4), (0.5, 0.5), 6, 0.9),
])
def test_expected_tokens_closed_form(golden_dir, p, q, k, golden_alpha):
    """E[tokens] = (1 - alpha^(k+1)) / (1 - alpha) under constant alpha
    (alpha = sum min(p,q)): the full law P(n=a) = alpha^a (1-alpha), a<k, and
    alpha^k at a=k, and the printed values 3.68928, ~3.4, ~2.3, ~5.2."""
    law, alpha = _constant_alpha_law(p, q, k)
    exp_law = np.array([alpha ** a * (1 - alpha) for a in range(k)] + [alpha ** k])
    np.testing.assert_allclose(law, exp_law, atol=1e-12)
    E = float(np.dot(np.arange(1, k + 2), law))
    assert abs(E - (1 - alpha ** (k + 1)) / (1 - alpha)) < 1e-12
    g = json.load(open(os.path.join(golden_dir, "expected_tokens.json")))
    case = [c for c in g["cases"] if c["alpha"] == golden_alpha and c["k"] == k][0]
    # alpha differs from the page's value only by fp32 rounding of log p
    assert abs(alpha - golden_alpha) < 1e-7
    assert abs(E - case["printed"]) <= case["abs_tol"] + 1e-6


def test_expected_tokens_alpha_one(golden_dir):
    """p == q bit-identical: every draft is accepted, k+1 = 6 tokens at K=5."""
    rng = np.random.default_rng(5)
    k, V = 5, 50
    t = (rng.standard_normal((64, k + 1, V)) * 2).astype(np.float32)
    d = np.ascontiguousarray(t[:, :k])
    g = rng.integers(0, V, (64, k)).astype(np.int32)
    toks, n, _ = oracle.verify(t, d, g, rng.random((64, k)), rng.random(64), np.ones(64))
    assert np.all(n == k)
    case = [c for c in json.load(open(os.path.join(golden_dir, "expected_tokens.json")))["cases"]
            if c["alpha"] == 1.0][0]
    assert float(np.mean(n + 1)) == case["printed"]


# ------------------------------------------------------------- Monte Carlo

def test_chi_square_tiny_vocab():
    """First emitted token ~ p_1 and the first two tokens ~ p(y1) p(y2|y1):
    V=4, k=3, 200000 seeded rounds, chi-square p-value > 1e-3."""
    V, k, N = 4, 3, 200_000
    rng = np.random.default_rng(42)
    f = lambda *s: (rng.standard_normal(s) * 1.2).astype(np.float32)
    T0, T1, T2, T3 = f(V), f(V, V), f(V, V, V), f(V, V, V, V)
    D0, D1, D2 = f(V), f(V, V), f(V, V, V)
    q0 = softmax64(D0)
    q1 = sp_softmax(D1.astype(np.float64), axis=-1)
    q2 = sp_softmax(D2.astype(np.float64), axis=-1)
    srng = np.random.default_rng(7)
    cdf = lambda pr, u: (u[..., None] < np.cumsum(pr, -1)).argmax(-1)
    g1 = cdf(np.broadcast_to(q0, (N, V)), srng.random(N))
    g2 = cdf(q1[g1], srng.random(N))
    g3 = cdf(q2[g1, g2], srng.random(N))
    tgt = np.stack([np.broadcast_to(T0, (N, V)), T1[g1], T2[g1, g2], T3[g1, g2, g3]], 1)
    dft = np.stack([np.broadcast_to(D0, (N, V)), D1[g1], D2[g1, g2]], 1)
    toks, n, _ = oracle.verify(np.ascontiguousarray(tgt), np.ascontiguousarray(dft),
                               np.stack([g1, g2, g3], 1), srng.random((N, k)), srng.random(N),
                               np.ones(N), nthreads=os.cpu_count() or 1, want_trace=False)
    p0 = softmax64(T0)
    p1 = sp_softmax(T1.astype(np.float64), axis=-1)
    y1 = toks[:, 0]
    assert stats.chisquare(np.bincount(y1, minlength=V), N * p0).pvalue > 1e-3
    y2 = np.where(n >= 1, toks[:, 1], cdf(p1[y1], srng.random(N)))
    obs = np.bincount(y1 * V + y2, minlength=V * V)
    exp = N * (p0[:, None] * p1).ravel()
    assert stats.chisquare(obs, exp).pvalue > 1e-3
    # a draft-distributed first token (the plausible bug: accepting everything)
    # is rejected by the same test
    assert stats.chisquare(np.bincount(g1, minlength=V), N * p0).pvalue < 1e-6


# ------------------------------------------------------------------ greedy

def test_greedy_reduces_to_argmax():
    """T = 0: accept while the target's argmax equals the draft token
    (interview page, 'Deep dive'); correction/bonus = target argmax; ties go
    to the lowest index (numpy's argmax convention)."""
    rng = np.random.default_rng(8)
    B, k, V = 300, 4, 9
    t = rng.integers(-3, 3, (B, k + 1, V)).astype(np.float32)  # many ties
    d = rng.standard_normal((B, k, V)).astype(np.float32)
    am = np.argmax(t, -1)
    g = np.where(rng.random((B, k)) < 0.8, am[:, :k], rng.integers(0, V, (B, k))).astype(np.int32)
    toks, n, _ = oracle.verify(t, d, g, rng.random((B, k)), rng.random(B), np.zeros(B))
    for b in range(B):
        mism = np.flatnonzero(g[b] != am[b, :k])
        j = int(mism[0]) if mism.size else k
        assert n[b] == j
        assert list(toks[b, :j]) == list(g[b, :j])
        assert toks[b, j] == am[b, j]
        assert np.all(toks[b, j + 1:] == -1)


def test_greedy_ignores_draft_logits():
    rng = np.random.default_rng(9)
    t = rng.standard_normal((2, 3, 6)).astype(np.float32)
    d = np.full((2, 2, 6), np.nan, np.float32)  # never read when T == 0
    g = np.argmax(t[:, :2], -1).astype(np.int32)
    toks, n, _ = oracle.verify(t, d, g, np.zeros((2, 2)), np.zeros(2), np.zeros(2))
    assert list(n) == [2, 2]


# -------------------------------------------------------------- invariants

def test_temperature_divides_logits():
    """softmax(l/T): (l, T=0.5) and (2l, T=1) are the same distributions, so
    every output and every threshold agree exactly; (l, T) vs (l*T, 1) does not
    hold in general, which a multiply-by-T mistake would show."""
    rng = np.random.default_rng(10)
    B, k, V = 50, 3, 40
    t = (rng.standard_normal((B, k + 1, V)) * 2).astype(np.float32)
    d = (t[:, :k] + rng.standard_normal((B, k, V)) * 0.5).astype(np.float32)
    g = rng.integers(0, V, (B, k)).astype(np.int32)
    ua, ur = rng.random((B, k)), rng.random(B)
    a = oracle.verify(t, d, g, ua, ur, np.full(B, 0.5))
    b = oracle.verify(2 * t, 2 * d, g, ua, ur, np.ones(B))
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])
    np.testing.assert_array_equal(np.nan_to_num(a[2], nan=-7), np.nan_to_num(b[2], nan=-7))
    c = oracle.verify(0.5 * t, 0.5 * d, g, ua, ur, np.ones(B))
    assert not np.array_equal(np.nan_to_num(a[2], nan=-7), np.nan_to_num(c[2], nan=-7))


def test_probs_match_scipy():
    rng = np.random.default_rng(12)
    B, k, V = 5, 3, 33
    t = (rng.standard_normal((B, k + 1, V)) * 2).astype(np.float32)
    d = (rng.standard_normal((B, k, V)) * 2).astype(np.float32)
    g = rng.integers(0, V, (B, k)).astype(np.int32)
    T = np.array([0.7, 1.0, 1.3, 0.0, 2.0])
    pq = oracle.probs(t, d, g, T)
    for b in range(B):
        for i in range(k):
            if T[b] == 0:
                assert np.isnan(pq[b, i]).all()
                continue
            assert abs(pq[b, i, 0] / softmax64(t[b, i], T[b])[g[b, i]] - 1) < 1e-13
            assert abs(pq[b, i, 1] / softmax64(d[b, i], T[b])[g[b, i]] - 1) < 1e-13


def test_thread_count_does_not_change_results():
    from speculative_decoding_verification_65_gb300 import synth
    c = synth.make_config(2, B=12)
    a = oracle.verify(c.target, c.draft, c.tokens, c.u_accept, c.u_resample, c.temperature, 1)
    b = oracle.verify(c.target, c.draft, c.tokens, c.u_accept, c.u_resample, c.temperature, 5)
    for x, y in zip(a[:2], b[:2]):
        np.testing.assert_array_equal(x, y)


def test_output_shape_invariant():
    """Each round emits between 1 and k+1 tokens: the accepted prefix, one
    correction or bonus, then -1 padding."""
    from speculative_decoding_verification_65_gb300 import synth
    c = synth.make_config(4, B=16, V=2000)
    toks, n, _ = oracle.verify(c.target, c.draft, c.tokens, c.u_accept, c.u_resample,
                               c.temperature)
    for b in range(c.B):
        assert 0 <= n[b] <= c.k
        assert list(toks[b, :n[b]]) == list(c.tokens[b, :n[b]])
        assert 0 <= toks[b, n[b]] < c.V
        assert np.all(toks[b, n[b] + 1:] == -1)


# ------------------------------------------------------------ error rows

def _err_case():
    rng = np.random.default_rng(13)
    B, k, V = 8, 3, 16
    t = rng.standard_normal((B, k + 1, V)).astype(np.float32)
    d = rng.standard_normal((B, k, V)).astype(np.float32)
    g = rng.integers(0, V, (B, k)).astype(np.int32)
    return t, d, g, rng.random((B, k)), rng.random(B), np.ones(B)


@pytest.mark.parametrize("what", ["T_neg", "T_nan", "T_inf", "T_denormal", "tok_hi", "tok_neg",
                                  "nan_target_bonus", "posinf_draft_last", "all_neginf_target",
                                  "q_zero_first"])
def test_error_rows(what):
    t, d, g, ua, ur, T = _err_case()
    b = 3
    if what == "T_neg":
        T[b] = -1.0
    elif what == "T_nan":
        T[b] = np.nan
    elif what == "T_inf":
        T[b] = np.inf
    elif what == "T_denormal":
        T[b] = 1e-40
    elif what == "tok_hi":
        g[b, 2] = t.shape[2]
    elif what == "tok_neg":
        g[b, 1] = -5
    elif what == "nan_target_bonus":
        t[b, -1, 7] = np.nan
    elif what == "posinf_draft_last":
        d[b, -1, 0] = np.inf
    elif what == "all_neginf_target":
        t[b, 1, :] = -np.inf
    elif what == "q_zero_first":
        d[b, 0, g[b, 0]] = -np.inf
    toks, n, _ = oracle.verify(t, d, g, ua, ur, T)
    assert n[b] == -1 and np.all(toks[b] == -1)
    others = [x for x in range(len(n)) if x != b]
    assert np.all(n[others] >= 0)


def test_q_zero_after_rejection_is_not_an_error():
    """Positions after the first rejection are discarded, so their draft
    probabilities are never tested."""
    t, d, g, ua, ur, T = _err_case()
    b = 2
    t[b, 0, g[b, 0]] = -np.inf   # p(g_1) = 0: rejection at position 1
    d[b, 1, g[b, 1]] = -np.inf   # q(g_2) = 0, never reached
    toks, n, _ = oracle.verify(t, d, g, ua, ur, T)
    assert n[b] == 0 and toks[b, 0] >= 0
