"""Pins of the sampling oracle (oracle.sample) to things other than itself.

The operation is the draft model's sampling step ("Speculative Decoding and
the Art of Fast LLM Inference", "The Algorithm, Step by Step", the drafting
step): one token per row from softmax(l / T) by inverse CDF with the row's
uniform, argmax at T = 0.  Each pin would catch a different plausible mistake:
a shifted cell boundary (<= vs <), a temperature applied as a multiplier, a
cumulative sum over the wrong axis or order, a greedy tie resolved to the last
index, a masked entry given mass, a bf16 pattern decoded wrongly.
"""
import math

import numpy as np
import pytest

import oracle

scipy_special = pytest.importorskip("scipy.special")


def _bf16_bits(x):
    """Round-to-nearest-even fp32 -> bf16 bit patterns (uint16)."""
    b = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return b.astype(np.uint16)


def test_cells_of_a_closed_form_distribution():
    # logits ln(1..4) at T = 1: p = (0.1, 0.2, 0.3, 0.4), cells
    # [0, .1), [.1, .3), [.3, .6), [.6, 1)
    l = np.log(np.array([[1, 2, 3, 4]], np.float64)).astype(np.float32)
    for u, want in [(0.0, 0), (0.0999, 0), (0.1001, 1), (0.2999, 1), (0.3001, 2),
                    (0.5999, 2), (0.6001, 3), (0.999999, 3)]:
        tok, tr = oracle.sample(l, [u], [1.0])
        assert tok[0] == want, (u, tok[0])
        assert tr[0, 0] <= u < tr[0, 1]


def test_a_uniform_on_a_cell_boundary_takes_the_next_token():
    # equal logits give C = (1/4, 1/2, 3/4, 1) exactly; "the smallest x with
    # C(x) > u*R" puts u = 1/4 in token 1, not 0
    l = np.zeros((1, 4), np.float32)
    for u, want in [(0.0, 0), (0.25, 1), (0.5, 2), (0.75, 3)]:
        assert oracle.sample(l, [u], [1.0])[0][0] == want


def test_temperature_divides_the_logits():
    # logits T * ln(w) at temperature T give p proportional to w for every T
    w = np.array([5.0, 1.0, 2.0, 2.0], np.float64)
    cdf = np.cumsum(w) / w.sum()          # 0.5, 0.6, 0.8, 1.0
    for T in (0.25, 0.7, 1.0, 3.0):
        l = (T * np.log(w)).astype(np.float32)[None, :]
        for u, want in [(0.49, 0), (0.51, 1), (0.59, 1), (0.61, 2), (0.79, 2), (0.81, 3)]:
            tok, _ = oracle.sample(l, [u], [T])
            assert tok[0] == want, (T, u, tok[0], cdf)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_matches_scipy_softmax_and_searchsorted(dtype):
    rng = np.random.default_rng(7)
    R, V = 40, 3000
    l32 = (rng.standard_normal((R, V)) * 2.5).astype(np.float32)
    if dtype == "bf16":
        bits = _bf16_bits(l32)
        l_in = bits
        l64 = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    else:
        l_in = l32
        l64 = l32.astype(np.float64)
    u = rng.random(R)
    T = rng.choice([0.3, 0.7, 1.0, 1.6], size=R)
    tok, tr = oracle.sample(l_in, u, T)
    checked = 0
    for r in range(R):
        p = scipy_special.softmax(l64[r] / T[r])
        C = np.cumsum(p)
        want = int(np.searchsorted(C, u[r] * C[-1], side="right"))
        # skip the (unlikely) rows whose uniform sits within rounding of a boundary
        if want > 0 and abs(u[r] * C[-1] - C[want - 1]) < 1e-12:
            continue
        if abs(u[r] * C[-1] - C[want]) < 1e-12:
            continue
        assert tok[r] == want, (r, tok[r], want)
        assert tr[r, 0] <= u[r] < tr[r, 1]
        checked += 1
    assert checked >= R - 2


def test_frequencies_by_quadrature():
    # uniforms on a fine midpoint grid: the share of draws of each token equals
    # its probability within one grid step (a deterministic chi-square)
    l = np.array([[0.0, 1.5, -2.0, 0.7, 3.1, -np.inf, 0.2, 1.0]], np.float32)
    T = 0.8
    p = scipy_special.softmax(np.where(np.isinf(l[0]), -np.inf, l[0] / T))
    N = 20000
    u = (np.arange(N) + 0.5) / N
    toks, _ = oracle.sample(np.repeat(l, N, axis=0), u, np.full(N, T))
    freq = np.bincount(toks, minlength=l.shape[1]) / N
    assert np.all(np.abs(freq - p) <= 1.0 / N + 1e-12)
    assert freq[5] == 0.0  # the masked entry is never drawn


def test_greedy_is_the_first_argmax():
    rng = np.random.default_rng(3)
    l = rng.integers(-3, 4, size=(50, 200)).astype(np.float32)  # many ties
    tok, tr = oracle.sample(l, rng.random(50), np.zeros(50))
    assert np.array_equal(tok, np.argmax(l, axis=1))  # numpy: first occurrence
    assert np.all(np.isnan(tr))


def test_greedy_ignores_the_uniform():
    l = np.array([[1.0, 4.0, 4.0, 2.0]], np.float32)
    for u in (0.0, 0.5, 0.9999):
        assert oracle.sample(l, [u], [0.0])[0][0] == 1


@pytest.mark.parametrize("what", ["nan", "posinf", "all_neginf", "T_neg", "T_nan", "T_inf",
                                  "T_denormal"])
def test_error_rows(what):
    l = np.zeros((3, 16), np.float32)
    T = np.ones(3)
    if what == "nan":
        l[1, 5] = np.nan
    elif what == "posinf":
        l[1, 5] = np.inf
    elif what == "all_neginf":
        l[1, :] = -np.inf
    elif what == "T_neg":
        T[1] = -0.5
    elif what == "T_nan":
        T[1] = np.nan
    elif what == "T_inf":
        T[1] = np.inf
    elif what == "T_denormal":
        T[1] = 1e-40
    tok, _ = oracle.sample(l, [0.3, 0.3, 0.3], T)
    assert tok[1] == -1
    assert tok[0] >= 0 and tok[2] >= 0


def test_masked_entries_are_never_drawn():
    rng = np.random.default_rng(11)
    R, V = 200, 64
    l = rng.standard_normal((R, V)).astype(np.float32)
    mask = rng.random((R, V)) < 0.5
    mask[:, 0] = False
    l[mask] = -np.inf
    tok, _ = oracle.sample(l, rng.random(R), np.full(R, 1.0))
    assert not np.any(mask[np.arange(R), tok])


def test_bf16_patterns_decode_to_their_values():
    rng = np.random.default_rng(5)
    l = rng.standard_normal((30, 500)).astype(np.float32)
    bits = _bf16_bits(l)
    widened = (bits.astype(np.uint32) << 16).view(np.float32)
    u, T = rng.random(30), np.full(30, 0.9)
    assert np.array_equal(oracle.sample(bits, u, T)[0], oracle.sample(widened, u, T)[0])


def test_thread_count_does_not_change_results():
    rng = np.random.default_rng(9)
    l = rng.standard_normal((64, 700)).astype(np.float32)
    u, T = rng.random(64), rng.choice([0.0, 0.5, 1.0], size=64)
    a = oracle.sample(l, u, T, nthreads=1)[0]
    b = oracle.sample(l, u, T, nthreads=7)[0]
    assert np.array_equal(a, b)


def test_one_token_vocabulary_edge():
    # V = 2 with one entry masked: every uniform draws the other entry
    l = np.array([[-np.inf, 0.3]], np.float32)
    for u in (0.0, 0.5, 0.999999):
        assert oracle.sample(l, [u], [1.0])[0][0] == 1
    assert math.isclose(oracle.sample(l, [0.5], [1.0])[1][0, 2], 1.0)
