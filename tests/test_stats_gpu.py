"""Distributional pins run through the CUDA path: chi-square at tiny V with
10^6 rounds in one call, the accept-count law under constant alpha, and the
exact V=3, k=2 enumeration replayed at every cell's midpoint."""
import numpy as np
import pytest
from scipy import stats
from scipy.special import softmax as sp_softmax

import oracle
from tests.enum_util import enumerate_leaves, softmax64

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import speculative_decoding_verification_65_gb300 as sv  # noqa: E402


def gpu_verify(t, d, g, ua, ur, T):
    dev = "cuda"
    to = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a, dtype=dt)).to(dev)
    toks, n = sv.spec_verify(to(t, np.float32), to(d, np.float32), to(g, np.int32),
                             to(ua, np.float32), to(ur, np.float32), to(T, np.float32))
    torch.cuda.synchronize()
    return toks.cpu().numpy(), n.cpu().numpy()


def test_chi_square_one_million_rounds():
    V, k, N = 4, 3, 1_000_000
    rng = np.random.default_rng(77)
    f = lambda *s: (rng.standard_normal(s) * 1.2).astype(np.float32)
    T0, T1, T2, T3 = f(V), f(V, V), f(V, V, V), f(V, V, V, V)
    D0, D1, D2 = f(V), f(V, V), f(V, V, V)
    q0 = softmax64(D0)
    q1 = sp_softmax(D1.astype(np.float64), axis=-1)
    q2 = sp_softmax(D2.astype(np.float64), axis=-1)
    srng = np.random.default_rng(8)
    cdf = lambda pr, u: (u[..., None] < np.cumsum(pr, -1)).argmax(-1)
    g1 = cdf(np.broadcast_to(q0, (N, V)), srng.random(N))
    g2 = cdf(q1[g1], srng.random(N))
    g3 = cdf(q2[g1, g2], srng.random(N))
    tgt = np.stack([np.broadcast_to(T0, (N, V)), T1[g1], T2[g1, g2], T3[g1, g2, g3]], 1)
    dft = np.stack([np.broadcast_to(D0, (N, V)), D1[g1], D2[g1, g2]], 1)
    toks, n = gpu_verify(tgt, dft, np.stack([g1, g2, g3], 1),
                         srng.random((N, k), dtype=np.float32),
                         srng.random(N, dtype=np.float32), np.ones(N))
    p0 = softmax64(T0)
    p1 = sp_softmax(T1.astype(np.float64), axis=-1)
    y1 = toks[:, 0]
    assert stats.chisquare(np.bincount(y1, minlength=V), N * p0).pvalue > 1e-3
    y2 = np.where(n >= 1, toks[:, 1], cdf(p1[y1], srng.random(N)))
    obs = np.bincount(y1 * V + y2, minlength=V * V)
    assert stats.chisquare(obs, N * (p0[:, None] * p1).ravel()).pvalue > 1e-3


@pytest.mark.parametrize("p,k", [((0.7, 0.3), 5), ((0.9, 0.1), 4), ((0.6, 0.4), 6)])
def test_accept_count_law_monte_carlo(p, k):
    """Constant alpha = sum min(p, q) with q = (1/2, 1/2): P(n=a) = alpha^a
    (1-alpha) for a < k, alpha^k for a = k; mean tokens per round
    (1 - alpha^(k+1)) / (1 - alpha) (3.69 at alpha=0.8, K=5)."""
    N, V = 1_000_000, 2
    tl = np.log(np.asarray(p)).astype(np.float32)
    dl = np.log([0.5, 0.5]).astype(np.float32)
    alpha = float(np.minimum(softmax64(tl), softmax64(dl)).sum())
    rng = np.random.default_rng(int(1000 * p[0]) + k)
    g = rng.integers(0, 2, (N, k)).astype(np.int32)
    t = np.broadcast_to(tl, (N, k + 1, V))
    d = np.broadcast_to(dl, (N, k, V))
    toks, n = gpu_verify(t, d, g, rng.random((N, k), dtype=np.float32),
                         rng.random(N, dtype=np.float32), np.ones(N))
    law = np.array([alpha ** a * (1 - alpha) for a in range(k)] + [alpha ** k])
    assert stats.chisquare(np.bincount(n, minlength=k + 1), N * law).pvalue > 1e-3
    E = (1 - alpha ** (k + 1)) / (1 - alpha)
    tokens = n + 1
    assert abs(tokens.mean() - E) < 4 * tokens.std() / np.sqrt(N)


@pytest.mark.parametrize("seed", [11, 12, 13])
def test_exact_enumeration_replayed_on_gpu(seed):
    """Every accept/draw cell of the V=3, k=2 enumeration, evaluated by the
    GPU at the cell's midpoint, gives the oracle's outcome; the emitted joint
    (completed with the target's conditionals) equals the target's
    autoregressive distribution to 1e-6."""
    V, k = 3, 2
    rng = np.random.default_rng(seed)
    f = lambda *s: (rng.standard_normal(s) * 1.5).astype(np.float32)
    t0, t1, t2 = f(V), f(V, V), f(V, V, V)
    d0, d1 = f(V), f(V, V)
    p0 = softmax64(t0)
    p1 = np.array([softmax64(r) for r in t1])
    p2 = np.array([[softmax64(r) for r in rr] for rr in t2])
    q0 = softmax64(d0)
    q1 = np.array([softmax64(r) for r in d1])
    rows_t, rows_d, toks_g, UA, UR, W, EXP = [], [], [], [], [], [], []
    for g1 in range(V):
        for g2 in range(V):
            tr = np.stack([t0, t1[g1], t2[g1, g2]])
            dr = np.stack([d0, d1[g1]])

            def run(ua, ur, tr=tr, dr=dr, g=(g1, g2)):
                o_t, o_n, _ = oracle.verify(tr[None], dr[None], np.array([g], np.int32),
                                            np.array([ua]), np.array([ur]), np.array([1.0]))
                return int(o_n[0]), [int(x) for x in o_t[0]]
            for ua, ur, prob, width, emitted in enumerate_leaves(run, k):
                rows_t.append(tr)
                rows_d.append(dr)
                toks_g.append((g1, g2))
                UA.append(ua)
                UR.append(ur)
                W.append(q0[g1] * q1[g1, g2] * prob)
                EXP.append(emitted)
    UA32 = np.asarray(UA, np.float32)
    UR32 = np.asarray(UR, np.float32)
    out_t, out_n = gpu_verify(np.stack(rows_t), np.stack(rows_d), np.asarray(toks_g),
                              UA32, UR32, np.ones(len(W)))
    joint = np.zeros((V, V, V))
    for i, (w, emitted) in enumerate(zip(W, EXP)):
        got = tuple(int(x) for x in out_t[i] if x >= 0)
        if got != emitted:
            # only a cell too narrow for its fp32 midpoint may differ
            assert w < 1e-6, (i, got, emitted, w)
        seq = got
        if len(seq) == 3:
            joint[seq] += w
        elif len(seq) == 2:
            joint[seq[0], seq[1], :] += w * p2[seq[0], seq[1]]
        else:
            joint[seq[0]] += w * p1[seq[0]][:, None] * p2[seq[0]]
    target = p0[:, None, None] * p1[:, :, None] * p2
    np.testing.assert_allclose(joint, target, atol=1e-6)
