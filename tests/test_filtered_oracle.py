"""Pins of the top-k / top-p filtered oracle (oracle.verify_filtered,
oracle.filtered_softmax).

Reading (the pages name top-p among the sampling parameters that draft and
target must share -- "Speculative Decoding and the Art of Fast LLM Inference",
"Why It Stays Exact", key limitation -- but do not define the filters):
tokens ranked by logit descending, ties by index ascending; top-k keeps the
first K; top-p keeps, among those, a token while the mass ranked before it is
below P times the top-k mass; both distributions are renormalised over their
kept sets before the accept test, the residual and the bonus draw.

The pins: hand-computed kept sets; with the filters off the result is the
unfiltered oracle's, exactly; top-k = 1 reduces sampling to the greedy rule;
the method's exactness carries over to the filtered target (exact enumeration
of the uniforms); bad filter parameters and a draft token outside the draft's
kept set are sequence errors.
"""
import math

import numpy as np
import pytest

import oracle
from speculative_decoding_verification_65_gb300 import synth
from tests.enum_util import enumerate_round

L7 = np.array([3.0, 1.0, 3.0, 2.0, 0.5, -np.inf, 2.0])


def _e(x):
    return math.exp(x)


@pytest.mark.parametrize("K,P,n_kept,kept", [
    (0, 1.0, 7, [0, 1, 2, 3, 4, 6]),   # no filter (the -inf entry is kept, without mass)
    (2, 1.0, 2, [0, 2]),
    (3, 1.0, 3, [0, 2, 3]),            # the tie at 2.0 goes to the lower index
    (4, 1.0, 4, [0, 2, 3, 6]),
    (0, 0.5, 2, [0, 2]),               # masses 1, 1, e^-1, e^-1, ...: 2 of 2.95 covers 0.5
    (0, 0.9, 4, [0, 2, 3, 6]),
    (4, 0.6, 2, [0, 2]),               # 0.6 of the top-4 mass 2.74 is 1.64 < 2
    (1, 0.01, 1, [0]),
    (0, 1e-9, 1, [0]),                 # at least one token is kept
])
def test_kept_sets_by_hand(K, P, n_kept, kept):
    p, n, mg = oracle.filtered_softmax(L7, 1.0, K, P)
    assert n == n_kept
    assert sorted(np.nonzero(p)[0].tolist()) == kept
    w = np.array([_e(L7[i] - 3.0) for i in kept])
    np.testing.assert_allclose(p[kept], w / w.sum(), rtol=1e-15)
    assert math.isnan(mg) == (P >= 1.0)


def test_temperature_applies_before_the_nucleus():
    # at T = 0.25 the mass concentrates: 0.9 of it is the two 3.0 tokens alone
    p, n, _ = oracle.filtered_softmax(L7, 0.25, 0, 0.9)
    assert n == 2 and sorted(np.nonzero(p)[0].tolist()) == [0, 2]


def _case(seed, B=24, k=4, V=700, dtype="f32", T=(0.0, 0.7, 1.0)):
    return synth.gauss_case(B=B, k=k, V=V, dtype=dtype, seed=seed, T=T)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_filters_off_equal_the_unfiltered_oracle(dtype):
    c = _case(3, dtype=dtype)
    args = (c.target, c.draft, c.tokens, c.u_accept, c.u_resample, c.temperature)
    rt, rn, rtr = oracle.verify(*args)
    for top_k, top_p in [(None, None), (np.zeros(c.B, np.int32), np.ones(c.B)),
                         (np.full(c.B, c.V, np.int32), np.full(c.B, 1.5))]:
        ft, fn, ftr = oracle.verify_filtered(*args, top_k, top_p)
        assert np.array_equal(ft, rt) and np.array_equal(fn, rn)
        np.testing.assert_array_equal(ftr[:, :c.k + 3], rtr)
        assert np.all(np.isnan(ftr[:, c.k + 3]))


def test_top_k_one_is_the_greedy_rule():
    # with K = 1 both distributions are one-hot at their argmax: a draft token
    # equal to the draft argmax is accepted iff it is the target argmax, and
    # the correction / bonus token is the target argmax -- the greedy rule
    c = _case(5, T=(0.8,))
    g = np.argmax(synth.decode(c.draft), axis=2).astype(np.int32)
    args = (c.target, c.draft, g, c.u_accept, c.u_resample)
    ft, fn, _ = oracle.verify_filtered(*args, c.temperature, np.ones(c.B, np.int32), None)
    gt, gn, _ = oracle.verify(*args, np.zeros(c.B))
    assert np.array_equal(ft, gt) and np.array_equal(fn, gn)


@pytest.mark.parametrize("what", ["k_neg", "p_nan", "p_zero", "p_neg"])
def test_bad_filter_parameters_are_sequence_errors(what):
    c = _case(7, B=3, T=(1.0,))
    top_k = np.zeros(3, np.int32)
    top_p = np.ones(3)
    if what == "k_neg":
        top_k[1] = -2
    elif what == "p_nan":
        top_p[1] = np.nan
    elif what == "p_zero":
        top_p[1] = 0.0
    else:
        top_p[1] = -0.3
    ft, fn, _ = oracle.verify_filtered(c.target, c.draft, c.tokens, c.u_accept, c.u_resample,
                                       c.temperature, top_k, top_p)
    assert fn[1] == -1 and np.all(ft[1] == -1)
    assert fn[0] >= 0 and fn[2] >= 0


def test_draft_token_outside_the_draft_kept_set_is_an_error():
    c = _case(9, B=1, k=1, T=(1.0,))
    d = synth.decode(c.draft)[0, 0]
    worst = np.argsort(-d, kind="stable")[-1]          # the draft's least likely token
    g = np.array([[worst]], np.int32)
    ft, fn, _ = oracle.verify_filtered(c.target, c.draft, g, c.u_accept, c.u_resample,
                                       c.temperature, np.array([5], np.int32), None)
    assert fn[0] == -1


def _filtered64(row, T, K, P):
    return oracle.filtered_softmax(np.asarray(row, np.float64), T, K, P)[0]


@pytest.mark.parametrize("K,P,seed", [(3, 1.0, 0), (0, 0.8, 1), (4, 0.7, 2), (2, 0.95, 3)])
def test_exactness_carries_over_to_the_filtered_target(K, P, seed):
    """V = 5, k = 1: draft token g weighted by the filtered q, every accept and
    draw cell by its width.  The emitted pair (a, b) -- b the bonus, or the
    target's next token after a correction -- must have probability
    p~_0(a) * p~_1[a](b), the filtered target's own autoregressive law."""
    V, T = 5, 0.9
    rng = np.random.default_rng(seed)
    t0 = (rng.standard_normal(V) * 1.5).astype(np.float32)
    t1 = (rng.standard_normal((V, V)) * 1.5).astype(np.float32)
    d0 = (rng.standard_normal(V) * 1.5).astype(np.float32)
    p0 = _filtered64(t0, T, K, P)
    p1 = np.array([_filtered64(r, T, K, P) for r in t1])
    q0 = _filtered64(d0, T, K, P)
    joint = np.zeros((V, V))
    for g in range(V):
        if q0[g] == 0.0:
            continue

        def run(ua, ur, g=g):
            tgt = np.stack([t0, t1[g]])[None]
            ft, fn, _ = oracle.verify_filtered(tgt, d0[None, None], np.array([[g]], np.int32),
                                               np.array([ua]), np.array([ur]), np.array([T]),
                                               np.array([K], np.int32), np.array([P]))
            assert fn[0] >= 0
            return int(fn[0]), [int(x) for x in ft[0]]

        for seq, prob in enumerate_round(run, 1).items():
            if len(seq) == 2:
                joint[seq] += q0[g] * prob
            else:
                joint[seq[0], :] += q0[g] * prob * p1[seq[0]]
    np.testing.assert_allclose(joint, p0[:, None] * p1, atol=1e-12)
