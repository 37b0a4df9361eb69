"""Pins of the tree-verification oracle (oracle.verify_tree), on the CPU.

The rule (a reading: the pages name tree verification -- "Speculative
Decoding and the Art of Fast LLM Inference", "Where the Draft Comes From",
EAGLE-2/3; techaiinterview, "Drafts and limits" -- without an acceptance rule
among siblings): each child is one accept test against the target's current
distribution, and a rejection replaces that distribution by the normalised
residual norm(max(0, p - q)) before the next sibling.  What pins it:

  - a worked example in exact rational arithmetic, with the residuals taken
    by the recursive definition (not the oracle's running constants);
  - the exactness theorem ("Why It Stays Exact"; techaiinterview, "Deep dive:
    correctness and speedup"): exact enumeration of every draft tree and
    every accept/draw outcome at V = 3 gives the target's own law for the
    emitted tokens; greedy trees emit a prefix of the target's argmax path;
  - the chain is the special case of one child per node: the tree oracle
    equals the chain oracle there;
  - a chi-square test of sampled trees against the target law;
  - mutated copies of the oracle (no residual update; no renormalisation)
    fail the enumeration, so the pin can see those mistakes.
"""
from __future__ import annotations

import ctypes
import itertools
import os
import subprocess
from fractions import Fraction

import numpy as np
import pytest

import oracle
from speculative_decoding_verification_65_gb300 import synth


def _logits_of(p):
    return np.log(np.asarray(p, np.float64)).astype(np.float32)


def _run(target, draft, parent, tokens, n_nodes, ua, ur, T, fn=None):
    fn = fn or oracle.verify_tree
    return fn(target, draft, parent, tokens, n_nodes, ua, ur, T)


# --------------------------------------------------------- worked example

def _residual_exact(p, q):
    w = [max(Fraction(0), a - b) for a, b in zip(p, q)]
    s = sum(w)
    return [x / s for x in w]


def test_worked_example_three_siblings():
    """V = 4, p = (.4, .3, .2, .1), q = (.1, .2, .3, .4); the root's three
    children carry tokens 2, 3, 1 (leaves).  By the definition: child 1 tests
    p(2)/q(2) = 2/3; after its rejection the target is r1 = norm(max(0, p-q))
    = (3/4, 1/4, 0, 0); child 2 tests r1(3)/q(3) = 0; then r2 = norm(max(0,
    r1 - q)) = (13/14, 1/14, 0, 0); child 3 tests r2(1)/q(1) = 5/14; after a
    third rejection r3 = norm(max(0, r2 - q)) = (1, 0, 0, 0)."""
    F = Fraction
    p = [F(4, 10), F(3, 10), F(2, 10), F(1, 10)]
    q = [F(1, 10), F(2, 10), F(3, 10), F(4, 10)]
    r1 = _residual_exact(p, q)
    r2 = _residual_exact(r1, q)
    r3 = _residual_exact(r2, q)
    assert r1 == [F(3, 4), F(1, 4), 0, 0]
    assert r2 == [F(13, 14), F(1, 14), 0, 0]
    assert r3 == [1, 0, 0, 0]
    ratios = [p[2] / q[2], r1[3] / q[3], r2[1] / q[1]]
    assert ratios == [F(2, 3), 0, F(5, 14)]

    V, N = 4, 4
    t = np.zeros((1, N, V), np.float32)
    d = np.zeros((1, N, V), np.float32)
    t[0, 0] = _logits_of([float(x) for x in p])
    d[0, 0] = _logits_of([float(x) for x in q])
    leaf = [0.1, 0.2, 0.3, 0.4]  # the children's own target rows (bonus draws)
    for n in range(1, N):
        t[0, n] = _logits_of(leaf)
        d[0, n] = _logits_of(leaf)
    parent = np.array([[-1, 0, 0, 0]], np.int32)
    tokens = np.array([[-1, 2, 3, 1]], np.int32)
    nn = np.array([N], np.int32)
    T = np.array([1.0])

    # u = 0.9, 0.5, 0.3: reject, reject, accept child 3 (5/14 = 0.357 > 0.3);
    # the bonus draw from the leaf row with u = 0.35 lands in token 2's cell
    # [0.3, 0.6).
    ot, on, na, tr = _run(t, d, parent, tokens, nn, np.array([[0, .9, .5, .3]]),
                          np.array([0.35]), T)
    assert na[0] == 1 and on[0, 0] == 3 and ot[0, :2].tolist() == [1, 2]
    np.testing.assert_allclose(tr[0, 1:4], [float(r) for r in ratios], atol=1e-6)
    np.testing.assert_allclose(tr[0, N:N + 2], [0.3, 0.6], atol=1e-6)

    # u_3 = 0.4: all rejected; the draw is from r3 = (1, 0, 0, 0) whatever u.
    for ur in (0.0, 0.5, 0.999):
        ot, on, na, tr = _run(t, d, parent, tokens, nn, np.array([[0, .9, .5, .4]]),
                              np.array([ur]), T)
        assert na[0] == 0 and ot[0, 0] == 0 and ot[0, 1:].tolist() == [-1] * 3
        np.testing.assert_allclose(tr[0, N:N + 2], [0.0, 1.0], atol=1e-12)
        # total mass of max(0, p - C q) at C = 1 + 2/5 + 7/25 = 42/25
        np.testing.assert_allclose(tr[0, N + 2], float(F(4, 10) - F(42, 25) * F(1, 10)),
                                   rtol=1e-6)

    # child 2 with token 0 instead: r1(0)/q(0) = 7.5 >= 1, accepted whatever u.
    tokens2 = np.array([[-1, 2, 0, 1]], np.int32)
    ot, on, na, tr = _run(t, d, parent, tokens2, nn, np.array([[0, .9, .999, .0]]),
                          np.array([0.5]), T)
    assert na[0] == 1 and on[0, 0] == 2 and ot[0, 0] == 0
    assert tr[0, 2] == 1.0 and np.isnan(tr[0, 3])


# ------------------------------------------------------ exact enumeration

SHAPE = synth.tree_shape((2, 1))  # root; nodes 1, 2; node 3 below 1, node 4 below 2
V3 = 3


def _prefix_tables(seed, V=V3, depth=3):
    """Random target and draft logits for every token prefix up to `depth`."""
    rng = np.random.default_rng(seed)
    tl, dl = {}, {}
    for L in range(depth):
        for pre in itertools.product(range(V), repeat=L):
            tl[pre] = (rng.standard_normal(V) * 1.5).astype(np.float32)
            dl[pre] = (tl[pre] + rng.standard_normal(V) * 1.0).astype(np.float32)
    return tl, dl


def _softmax(l, T):
    x = np.asarray(l, np.float64) / T
    e = np.exp(x - x.max())
    return e / e.sum()


def _paths(shape, toks):
    out = {0: ()}
    for n in range(1, shape.size):
        out[n] = out[int(shape[n])] + (int(toks[n]),)
    return out


def _rows_for(shape, toks, tl, dl, V):
    N = shape.size
    paths = _paths(shape, toks)
    t = np.zeros((1, N, V), np.float32)
    d = np.zeros((1, N, V), np.float32)
    for n in range(N):
        t[0, n] = tl[paths[n]]
        d[0, n] = dl.get(paths[n], tl[paths[n]])
    return t, d


def _walk_law(shape, toks, tl, dl, T, fn):
    """Exact law of the emitted sequence for one draft tree: follow every
    accept/reject branch (u placed inside each side of the oracle's traced
    threshold, the decision checked on the re-run) and every draw cell."""
    N, V = shape.size, len(tl[()])
    t, d = _rows_for(shape, toks, tl, dl, V)
    parent = shape.reshape(1, N).astype(np.int32)
    tokens = np.asarray(toks, np.int32).reshape(1, N)
    nn = np.array([N], np.int32)
    TT = np.array([T])
    law = {}
    stack = [({}, 1.0)]
    while stack:
        fixed, prob = stack.pop()
        ua = np.full((1, N), 0.5)
        for n, u in fixed.items():
            ua[0, n] = u
        ot, on, na, tr = _run(t, d, parent, tokens, nn, ua, np.array([0.0]), TT, fn)
        assert na[0] >= 0
        tested = [n for n in range(1, N) if not np.isnan(tr[0, n])]
        free = [n for n in tested if n not in fixed]
        if free:
            n = free[0]
            r = float(tr[0, n])
            if r > 0:
                stack.append(({**fixed, n: r / 2}, prob * r))
            if r < 1:
                stack.append(({**fixed, n: (1 + r) / 2}, prob * (1 - r)))
            continue
        # the decisions are fixed: check them against the thresholds
        path = [int(x) for x in on[0, :na[0]]]
        for n in tested:
            assert (n in path) == (ua[0, n] < tr[0, n] or tr[0, n] == 1.0)
        emitted = tuple(int(x) for x in ot[0, :na[0]])
        # every draw cell: u at the lower edge of each cell in turn
        u, total = 0.0, 0.0
        while u < 1.0:
            ot2, on2, na2, tr2 = _run(t, d, parent, tokens, nn, ua, np.array([u]), TT, fn)
            assert na2[0] == na[0]
            lo, hi = float(tr2[0, N]), float(tr2[0, N + 1])
            assert lo <= u + 1e-12 and hi > u
            key = emitted + (int(ot2[0, na2[0]]),)
            law[key] = law.get(key, 0.0) + prob * (hi - u)
            total += hi - u
            u = hi + 1e-13 if hi < 1.0 else 1.0
        assert abs(total - 1.0) < 1e-9
    return law


def _extended_law(law, tl, T, L):
    """Law of the first L tokens when the emitted sequence is continued by
    sampling the target itself (defined for any emitted length <= L)."""
    out = {}
    for seq, pr in law.items():
        todo = [(seq, pr)]
        while todo:
            s, w = todo.pop()
            if len(s) >= L:
                out[s[:L]] = out.get(s[:L], 0.0) + w
                continue
            p = _softmax(tl[s], T)
            for x in range(len(p)):
                todo.append((s + (x,), w * p[x]))
    return out


def _target_law(tl, T, L, V=V3):
    out = {}
    for seq in itertools.product(range(V), repeat=L):
        w = 1.0
        for i in range(L):
            w *= _softmax(tl[seq[:i]], T)[seq[i]]
        out[seq] = w
    return out


def _tree_law(tl, dl, T, fn=None, shape=SHAPE):
    """Law of the emitted tokens over all draft trees (children drawn
    independently from the parent's draft distribution) and all outcomes."""
    fn = fn or oracle.verify_tree
    N = shape.size
    total = {}
    for assign in itertools.product(range(V3), repeat=N - 1):
        toks = (-1,) + assign
        paths = _paths(shape, toks)
        pa = 1.0
        for n in range(1, N):
            pa *= _softmax(dl[paths[int(shape[n])]], T)[toks[n]]
        if pa == 0.0:
            continue
        for seq, w in _walk_law(shape, toks, tl, dl, T, fn).items():
            total[seq] = total.get(seq, 0.0) + pa * w
    return total


@pytest.mark.parametrize("seed,T", [(1, 1.0), (2, 0.7), (3, 1.6)])
def test_enumeration_exactness(seed, T):
    """Every outcome of every draft tree at V = 3: the emitted tokens, continued
    by the target, have exactly the target's law (to fp64 rounding)."""
    tl, dl = _prefix_tables(seed)
    law = _tree_law(tl, dl, T)
    assert abs(sum(law.values()) - 1.0) < 1e-12
    ext = _extended_law(law, tl, T, 3)
    ref = _target_law(tl, T, 3)
    for seq, w in ref.items():
        assert abs(ext.get(seq, 0.0) - w) < 1e-12, (seq, ext.get(seq), w)
    # the first token alone is the root's target distribution
    first = np.zeros(V3)
    for seq, w in law.items():
        first[seq[0]] += w
    np.testing.assert_allclose(first, _softmax(tl[()], T), atol=1e-13)


def test_enumeration_greedy():
    """T = 0: for every token assignment, the emitted tokens are the target's
    argmax path, and the walk stops only where no child holds the argmax."""
    tl, dl = _prefix_tables(4)
    N = SHAPE.size
    for assign in itertools.product(range(V3), repeat=N - 1):
        toks = (-1,) + assign
        t, d = _rows_for(SHAPE, toks, tl, dl, V3)
        ot, on, na, _ = oracle.verify_tree(t, d, SHAPE.reshape(1, N), np.array([toks]),
                                           np.array([N]), np.full((1, N), 0.5),
                                           np.array([0.5]), np.array([0.0]))
        n = int(na[0])
        seq = tuple(int(x) for x in ot[0, :n + 1])
        for i in range(n + 1):
            assert seq[i] == int(np.argmax(tl[seq[:i]]))
        last = 0 if n == 0 else int(on[0, n - 1])
        kids = [c for c in range(1, N) if SHAPE[c] == last]
        assert all(toks[c] != seq[n] for c in kids)


# ------------------------------------------------------- planted mistakes

def _mutant(tmp_path, old, new):
    """A copy of the oracle with one line replaced, compiled on the side."""
    src = open(os.path.join(os.path.dirname(oracle.__file__), "spec_ref.c")).read()
    assert src.count(old) == 1
    path = tmp_path / "mut.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / "libmut.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                    "-o", str(so), str(path), "-lm", "-lpthread"], check=True)
    lib = ctypes.CDLL(str(so))
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    lib.spec_verify_tree_ref_mt.argtypes = [vp, vp, i32, vp, vp, vp, vp, vp, vp,
                                            i64, i64, i64, vp, vp, vp, vp, i32]
    lib.spec_verify_tree_ref_mt.restype = i32
    lib._tree_ready = True

    def fn(*args):
        real = oracle._lib
        oracle._lib = lib
        try:
            return oracle.verify_tree(*args)
        finally:
            oracle._lib = real
    oracle._load()
    return fn


@pytest.mark.parametrize("old,new", [
    # every sibling tested against p itself (no residual between siblings)
    ("C += M;\n                    M = ref_tree_residual",
     "C += 0.0;\n                    M = ref_tree_residual"),
    # the residual not renormalised between siblings
    ("const double ratio = num / (M * Q);", "const double ratio = num / Q;"),
], ids=["no-residual-update", "no-renormalisation"])
def test_enumeration_sees_mistakes(tmp_path, old, new):
    fn = _mutant(tmp_path, old, new)
    tl, dl = _prefix_tables(1)
    law = _tree_law(tl, dl, 1.0, fn=fn)
    ext = _extended_law(law, tl, 1.0, 3)
    ref = _target_law(tl, 1.0, 3)
    err = max(abs(ext.get(s, 0.0) - w) for s, w in ref.items())
    assert err > 1e-3, err


# ------------------------------------------------------------ chain case

@pytest.mark.parametrize("dtype", [synth.F32, synth.BF16])
def test_chain_tree_equals_chain_oracle(dtype):
    """A tree with one child per node is the chain of spec_verify: same tokens,
    accepted counts, thresholds and draw cells."""
    case = synth.gauss_case(B=64, k=5, V=300, dtype=dtype, seed=17, T=(0.0, 0.6, 1.0, 1.4))
    B, k, V = case.B, case.k, case.V
    N = k + 1
    t = case.target
    d = np.zeros_like(t)
    d[:, :k] = case.draft
    parent = np.tile(np.arange(-1, k, dtype=np.int32), (B, 1))
    tokens = np.concatenate([np.full((B, 1), -1, np.int32), case.tokens], axis=1)
    ua = np.concatenate([np.zeros((B, 1), np.float32), case.u_accept], axis=1)
    ot, on, na, tr = oracle.verify_tree(t, d, parent, tokens, np.full(B, N, np.int32), ua,
                                        case.u_resample, case.temperature)
    rt, rn, rtr = oracle.verify(case.target, case.draft, case.tokens, case.u_accept,
                                case.u_resample, case.temperature)
    np.testing.assert_array_equal(na, rn)
    np.testing.assert_array_equal(ot, rt)
    for b in range(B):
        assert on[b, :na[b]].tolist() == list(range(1, na[b] + 1))
    np.testing.assert_array_equal(tr[:, 1:N], rtr[:, :k])
    np.testing.assert_array_equal(tr[:, N:], rtr[:, k:])


# ------------------------------------------------------------ chi-square

def test_chi_square_sampled_trees():
    """200 000 sampled trees (V = 6, three first-level candidates, two below
    each): the first two emitted tokens (the second drawn from the target when
    only one was emitted) against the target's law."""
    from scipy.stats import chisquare
    V, T, B = 6, 1.0, 200_000
    shape = synth.tree_shape((3, 2))
    N = shape.size
    rng = np.random.default_rng(99)
    tl, dl = {}, {}
    for L in range(3):
        for pre in itertools.product(range(V), repeat=L):
            tl[pre] = (rng.standard_normal(V) * 1.2).astype(np.float32)
            dl[pre] = (tl[pre] + rng.standard_normal(V) * 0.9).astype(np.float32)
    gum = lambda l, size: np.argmax(np.asarray(l, np.float64) / T
                                    - np.log(rng.standard_exponential((size, V))), axis=1)
    toks = np.full((B, N), -1, np.int32)
    for n in range(1, N):
        par = int(shape[n])
        if par == 0:
            toks[:, n] = gum(dl[()], B)
        else:
            for x in range(V):
                sel = toks[:, par] == x
                toks[sel, n] = gum(dl[(x,)], int(sel.sum()))
    t = np.empty((B, N, V), np.float32)
    d = np.empty((B, N, V), np.float32)
    t[:, 0] = tl[()]
    d[:, 0] = dl[()]
    for n in range(1, N):
        par = int(shape[n])
        for b_pre in itertools.product(range(V), repeat=1 if par == 0 else 2):
            if par == 0:
                sel = toks[:, n] == b_pre[0]
            else:
                sel = (toks[:, par] == b_pre[0]) & (toks[:, n] == b_pre[1])
            t[sel, n] = tl[b_pre]
            d[sel, n] = dl.get(b_pre, tl[b_pre])
    ua = rng.random((B, N))
    ur = rng.random(B)
    ot, on, na, _ = oracle.verify_tree(t, d, np.tile(shape, (B, 1)), toks,
                                       np.full(B, N, np.int32), ua, ur, np.full(B, T),
                                       nthreads=8, want_trace=False)
    assert np.all(na >= 0)
    y1 = ot[:, 0]
    y2 = np.where(na >= 1, ot[:, 1], -1)
    for x in range(V):
        sel = y2 == -1
        sel &= y1 == x
        y2[sel] = rng.choice(V, size=int(sel.sum()), p=_softmax(tl[(x,)], T))
    obs = np.bincount(y1 * V + y2, minlength=V * V)
    p1 = _softmax(tl[()], T)
    exp = np.array([p1[a] * _softmax(tl[(a,)], T)[b] for a in range(V) for b in range(V)]) * B
    stat, pval = chisquare(obs, exp)
    assert pval > 1e-3, (stat, pval)


# ---------------------------------------------------------- sequence errors

def test_errors_and_unvisited_rows():
    tc = synth.make_tree_case(dict(synth.TREE_CONFIGS[1], ragged=False, temps=(1.0,)), seed=31)
    B, N = tc.B, tc.N
    base = oracle.verify_tree(tc.target, tc.draft, tc.parent, tc.tokens, tc.n_nodes,
                              tc.u_accept, tc.u_resample, tc.temperature)
    b = 0
    assert base[2][b] >= 0

    def run(**over):
        a = dict(target=tc.target.copy(), draft=tc.draft.copy(), parent=tc.parent.copy(),
                 tokens=tc.tokens.copy(), n_nodes=tc.n_nodes.copy(),
                 u_accept=tc.u_accept, u_resample=tc.u_resample,
                 temperature=tc.temperature.copy())
        for k_, f in over.items():
            f(a[k_])
        return oracle.verify_tree(**a)

    def expect_error(res):
        ot, on, na, _ = res
        assert na[b] == -1 and np.all(ot[b] == -1) and np.all(on[b] == -1)
        others = np.arange(B) != b
        np.testing.assert_array_equal(na[others], base[2][others])

    expect_error(run(n_nodes=lambda a: a.__setitem__(b, 0)))
    expect_error(run(n_nodes=lambda a: a.__setitem__(b, N + 1)))
    expect_error(run(parent=lambda a: a.__setitem__((b, 5), 5)))
    expect_error(run(parent=lambda a: a.__setitem__((b, 3), -1)))
    expect_error(run(tokens=lambda a: a.__setitem__((b, 4), tc.V)))
    expect_error(run(temperature=lambda a: a.__setitem__(b, np.nan)))
    expect_error(run(target=lambda a: a.__setitem__((b, 0, 7), np.inf)))
    visited = {0} | set(int(x) for x in base[1][b, :base[2][b]])
    unvisited = [n for n in range(N) if n not in visited]
    # a NaN in a row the walk never reads changes nothing
    res = run(target=lambda a: a.__setitem__((b, unvisited[0], 3), np.nan))
    np.testing.assert_array_equal(res[0], base[0])
    np.testing.assert_array_equal(res[2], base[2])
    # a zero draft probability at a tested child is an error
    tok = int(tc.tokens[b, 1])
    expect_error(run(draft=lambda a: a.__setitem__((b, 0, tok), -np.inf)))
    # a root-only tree at T > 0 is the bonus draw from the root's target row
    one = run(n_nodes=lambda a: a.__setitem__(b, 1), temperature=lambda a: a.__setitem__(b, 1.0))
    assert one[2][b] == 0
    ref_tok, _ = oracle.sample(tc.target[b, :1], tc.u_resample[b:b + 1], np.array([1.0]))
    assert one[0][b, 0] == ref_tok[0]
