"""Parity of top-k / top-p filtered verification (spec_verify_filtered) with
the fp64 oracle (oracle.verify_filtered).

Integer outputs must equal the oracle's.  Exempt, and counted: a sequence
whose oracle decision had its uniform within BAND of a threshold or draw-cell
boundary (as for the unfiltered path, and held to the same 0.01 % bound by
parity_util.check_bound), or whose top-p cut had a running mass within BAND
of P times the top-k mass (the kept set is decided from masses in 2^-40 fixed
point of ex2.approx weights, so a cut that close may keep a different last
token; mismatches among such sequences are counted apart, at most one per
call or 0.01 % of its decisions).
Draft tokens are drawn from the filtered draft distribution, as a draft model
sampling with the same parameters would.
"""
import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
import speculative_decoding_verification_65_gb300 as sv  # noqa: E402
from speculative_decoding_verification_65_gb300 import synth  # noqa: E402
from tests.parity_util import MAX_EXEMPT_FRACTION, check_bound, compare  # noqa: E402

BAND = 1e-5
NTHREADS = os.cpu_count() or 1


def filtered_tokens(case, top_k, top_p, seed):
    """Draft tokens g_i ~ the filtered q_i (greedy sequences: the draft argmax)."""
    rng = np.random.default_rng(seed)
    d = synth.decode(case.draft)
    g = np.empty((case.B, case.k), np.int32)
    for b in range(case.B):
        T = float(case.temperature[b])
        for i in range(case.k):
            if T == 0.0:
                g[b, i] = int(np.argmax(d[b, i]))
                continue
            K = 0 if top_k is None else int(top_k[b])
            P = 1.0 if top_p is None else float(top_p[b])
            q, _, _ = oracle.filtered_softmax(d[b, i].astype(np.float64), T, max(K, 0),
                                              P if P > 0 else 1.0)
            g[b, i] = int(rng.choice(case.V, p=q / q.sum()))
    return g


def run_gpu(case, tokens, top_k, top_p, want_probs=False, ws=None):
    d = sv.to_device(case)
    d["tokens"] = torch.from_numpy(tokens).cuda()
    tk = None if top_k is None else torch.from_numpy(np.asarray(top_k, np.int32)).cuda()
    tp = None if top_p is None else torch.from_numpy(np.asarray(top_p, np.float32)).cuda()
    out = sv.spec_verify_filtered(**d, top_k=tk, top_p=tp, want_probs=want_probs, ws=ws)
    torch.cuda.synchronize()
    return tuple(x.cpu().numpy() for x in out)


def window_ws(case):
    """A workspace without room for group maxima: every row takes the
    streaming (window / radix) filter."""
    dt = sv.SPEC_F32 if case.dtype == synth.F32 else sv.SPEC_BF16
    need = sv.spec_verify_workspace_size(case.B, case.k, case.V, dt)
    return torch.zeros(need, dtype=torch.uint8, device="cuda")


def check(case, tokens, top_k, top_p, ws=None):
    gt, gn = run_gpu(case, tokens, top_k, top_p, ws=ws)
    rt, rn, tr = oracle.verify_filtered(case.target, case.draft, tokens, case.u_accept,
                                        case.u_resample, case.temperature, top_k, top_p,
                                        nthreads=NTHREADS)
    near = np.nan_to_num(tr[:, case.k + 3], nan=1.0) < BAND
    keep = np.nonzero(~near)[0]
    sub = case.subset(keep)
    sub.tokens = tokens[keep]
    rep = compare(sub, gt[keep], gn[keep], rt[keep], rn[keep], tr[keep][:, :case.k + 3])
    check_bound(rep)
    cut = int(np.sum(near & ((gn != rn) | np.any(gt != rt, axis=1))))
    assert cut <= max(1, MAX_EXEMPT_FRACTION * rep["decisions"]), (cut, rep["decisions"])
    return gn, rn


PARAMS = {
    "topk50": lambda B, rng: (np.full(B, 50, np.int32), None),
    "topp0.9": lambda B, rng: (None, np.full(B, 0.9, np.float32)),
    "both": lambda B, rng: (np.full(B, 20, np.int32), np.full(B, 0.8, np.float32)),
    "mixed": lambda B, rng: (rng.choice([0, 1, 5, 50, 1000], B).astype(np.int32),
                             rng.choice([1.0, 0.5, 0.9, 0.99], B).astype(np.float32)),
}


@pytest.mark.parametrize("path", ["group", "window"])
@pytest.mark.parametrize("params", list(PARAMS))
@pytest.mark.parametrize("cfg,B", [(2, 12), (3, 8), (4, 8), (5, 24)])
def test_workloads(cfg, B, params, path):
    """Both cuts of top-k rows: from group maxima (the default workspace of the
    binding) and by the streaming filter (a workspace without their room)."""
    case = synth.make_config(cfg, B=B)
    top_k, top_p = PARAMS[params](B, np.random.default_rng(cfg))
    tokens = filtered_tokens(case, top_k, top_p, seed=cfg + 17)
    gn, rn = check(case, tokens, top_k, top_p, ws=window_ws(case) if path == "window" else None)
    assert np.all(rn[case.temperature > 0] >= 0)  # drawn from the filtered q: no errors


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("V", [37, 1000, 40000])
def test_group_cut_equals_streaming_cut(dtype, V):
    """The cut from group maxima and the streaming cut compute the same exact
    record (fixed-point masses, the same sort and cut), so the outputs are
    identical; K spans 1 .. 256 (the group cut's limit) and 257 (streaming)."""
    rng = np.random.default_rng(V)
    B, k = 24, 3
    case = synth.gauss_case(B=B, k=k, V=V, dtype=dtype, seed=V + 1, T=(0.6, 1.0, 1.4))
    top_k = rng.choice([1, 2, 7, 50, 255, 256, 257], B).astype(np.int32)
    top_k = np.minimum(top_k, V - 1)
    top_p = rng.choice([1.0, 0.9, 0.5], B).astype(np.float32)
    tokens = filtered_tokens(case, top_k, top_p, seed=3)
    g = run_gpu(case, tokens, top_k, top_p)
    w = run_gpu(case, tokens, top_k, top_p, ws=window_ws(case))
    assert np.array_equal(g[0], w[0]) and np.array_equal(g[1], w[1])
    check(case, tokens, top_k, top_p)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_group_cut_with_massive_ties(dtype):
    """Integer-valued logits: thousands of tokens share the K-th key, more than
    the group cut's buffers hold, so the radix kernel finishes those rows."""
    B, k, V = 6, 2, 40000
    rng = np.random.default_rng(21)
    case = synth.gauss_case(B=B, k=k, V=V, dtype=dtype, seed=22, T=(1.0,))
    for arr in (case.target, case.draft):
        vals = np.round(rng.normal(0.0, 0.3, arr.shape)).astype(np.float32)  # ~5 % are 1
        arr[...] = synth.f32_to_bf16_bits(vals) if dtype == "bf16" else vals
    top_k = np.full(B, 100, np.int32)
    tokens = filtered_tokens(case, top_k, None, seed=6)
    check(case, tokens, top_k, None)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_group_cut_far_maximum_and_negative_rows(dtype):
    """The group cut's first histogram covers the 256 16-bit key prefixes at
    and below the row maximum's (two binades).  Rows with three logits far
    above the rest hold fewer than K group keys there, so tau comes from the
    radix search from the top; rows of only negative logits run the window
    pass on negative keys.  Both must give the streaming cut's records."""
    rng = np.random.default_rng(31)
    B, k, V = 12, 2, 30000
    case = synth.gauss_case(B=B, k=k, V=V, dtype=dtype, seed=32, T=(0.8, 1.0))
    for arr in (case.target, case.draft):
        vals = rng.normal(0.0, 1.0, arr.shape).astype(np.float32)
        far = rng.integers(0, V, size=(B, arr.shape[1], 3))
        for b in range(B // 2):
            for i in range(arr.shape[1]):
                vals[b, i, far[b, i]] = 40.0
        vals[B // 2:] -= 30.0
        arr[...] = synth.f32_to_bf16_bits(vals) if dtype == "bf16" else vals
    top_k = rng.choice([2, 5, 50, 256], B).astype(np.int32)
    top_p = rng.choice([1.0, 0.9], B).astype(np.float32)
    tokens = filtered_tokens(case, top_k, top_p, seed=8)
    g = run_gpu(case, tokens, top_k, top_p)
    w = run_gpu(case, tokens, top_k, top_p, ws=window_ws(case))
    assert np.array_equal(g[0], w[0]) and np.array_equal(g[1], w[1])
    check(case, tokens, top_k, top_p)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_kept_set_draws_stored_and_gathered(dtype):
    """The kept-set draws read a row's kept tokens back as the group cut
    stored them, or gather them when the cut left the row to the streaming
    filter.  Draft rows of integer logits (ties past the cut's buffers) next
    to gaussian target rows make both happen within one sequence; K spans 1
    to 256; both cuts must give the oracle's tokens and the streaming cut's."""
    rng = np.random.default_rng(41)
    B, k, V = 16, 3, 20000
    case = synth.gauss_case(B=B, k=k, V=V, dtype=dtype, seed=42, T=(0.7, 1.0))
    vals = np.round(rng.normal(0.0, 0.3, case.draft.shape)).astype(np.float32)
    vals[B // 2:] = rng.normal(0.0, 2.0, vals[B // 2:].shape).astype(np.float32)
    case.draft[...] = synth.f32_to_bf16_bits(vals) if dtype == "bf16" else vals
    top_k = rng.choice([1, 3, 40, 200, 256], B).astype(np.int32)
    top_p = rng.choice([1.0, 0.95, 0.6], B).astype(np.float32)
    tokens = filtered_tokens(case, top_k, top_p, seed=9)
    g = run_gpu(case, tokens, top_k, top_p)
    w = run_gpu(case, tokens, top_k, top_p, ws=window_ws(case))
    assert np.array_equal(g[0], w[0]) and np.array_equal(g[1], w[1])
    check(case, tokens, top_k, top_p)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_filters_off_equal_spec_verify(dtype):
    case = synth.gauss_case(B=16, k=4, V=5000, dtype=dtype, seed=3, T=(0.0, 0.7, 1.2))
    d = sv.to_device(case)
    t0, n0 = sv.spec_verify(**d)
    zk = torch.zeros(case.B, dtype=torch.int32, device="cuda")
    op = torch.ones(case.B, dtype=torch.float32, device="cuda")
    for tk, tp in ((None, None), (zk, op), (zk + case.V, op * 2)):
        t1, n1 = sv.spec_verify_filtered(**d, top_k=tk, top_p=tp)
        torch.cuda.synchronize()
        assert torch.equal(t0, t1) and torch.equal(n0, n1)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_wide_nucleus_and_massive_ties(dtype):
    # flat rows: the top-p end sits deep in the ranking (several narrowing
    # passes); integer-valued logits: one key value holds thousands of ties,
    # past the sort buffer, so the index-order tie pass decides
    rng = np.random.default_rng(11)
    B, k, V = 6, 2, 40000
    case = synth.gauss_case(B=B, k=k, V=V, dtype=dtype, seed=12, T=(1.0,), sigma_d=0.05,
                            sigma_n=0.02)
    top_p = np.full(B, 0.97, np.float32)
    tokens = filtered_tokens(case, None, top_p, seed=5)
    check(case, tokens, None, top_p)
    ints = rng.integers(-2, 3, size=(B, k + 1, V)).astype(np.float32)
    intd = rng.integers(-2, 3, size=(B, k, V)).astype(np.float32)
    if dtype == "bf16":
        ints, intd = synth.f32_to_bf16_bits(ints), synth.f32_to_bf16_bits(intd)
    case2 = synth.Case(ints, intd, case.tokens, case.u_accept, case.u_resample,
                       case.temperature, dtype)
    top_k = np.array([9000, 12000, 30000, 100, 1, 20000], np.int32)
    tokens2 = filtered_tokens(case2, top_k, None, seed=6)
    check(case2, tokens2, top_k, None)
    check(case2, tokens2, top_k, np.full(B, 0.6, np.float32))


def test_bad_parameters_fail_the_sequence():
    case = synth.gauss_case(B=5, k=3, V=3000, seed=4, T=(1.0,))
    top_k = np.array([0, -1, 0, 0, 0], np.int32)
    top_p = np.array([1.0, 1.0, np.nan, 0.0, -0.5], np.float32)
    case.temperature[:] = np.array([1.0, 0.0, 1.0, 1.0, 0.0], np.float32)
    gt, gn = run_gpu(case, case.tokens, top_k, top_p)
    rt, rn, _ = oracle.verify_filtered(case.target, case.draft, case.tokens, case.u_accept,
                                       case.u_resample, case.temperature, top_k, top_p)
    assert np.array_equal(gn, rn) and np.array_equal(gt, rt)
    assert np.all(gn[1:] == -1)


@pytest.mark.parametrize("cfg", [5, 4])
def test_filtered_intermediates_within_tolerance(cfg):
    """The filtered P, Q at the full vocabulary of workloads 5 (bf16) and 4
    (fp32, temperatures 0, 0.5, 1, 1.3), on 12 sequences of each recipe."""
    case = synth.make_config(cfg, B=12)
    if cfg == 4:
        case.temperature[:] = np.array([0.5, 1.0, 1.3, 0.0] * 3, np.float32)
    top_k = np.full(case.B, 40, np.int32)
    top_p = np.full(case.B, 0.9, np.float32)
    tokens = filtered_tokens(case, top_k, top_p, seed=8)
    _, _, probs = run_gpu(case, tokens, top_k, top_p, want_probs=True)
    d = synth.decode(case.target), synth.decode(case.draft)
    for b in range(case.B):
        T = float(case.temperature[b])
        if T == 0.0:
            assert np.all(np.isnan(probs[b]))  # greedy sequences have no P, Q
            continue
        for i in range(case.k):
            p, _, mp = oracle.filtered_softmax(d[0][b, i].astype(np.float64), T, 40, 0.9)
            q, _, mq = oracle.filtered_softmax(d[1][b, i].astype(np.float64), T, 40, 0.9)
            if min(mp, mq) < BAND:
                continue
            g = tokens[b, i]
            for got, want in ((probs[b, i, 0], p[g]), (probs[b, i, 1], q[g])):
                if want == 0.0:
                    assert got == 0.0
                else:
                    assert abs(got - want) <= 1e-5 * want, (b, i, got, want)


def test_deterministic_with_garbage_workspace():
    case = synth.make_config(3, B=8)
    top_k = np.full(case.B, 30, np.int32)
    top_p = np.full(case.B, 0.85, np.float32)
    tokens = filtered_tokens(case, top_k, top_p, seed=9)
    need = sv.spec_verify_workspace_size(case.B, case.k, case.V, sv.SPEC_BF16)
    ws = torch.randint(0, 256, (need,), dtype=torch.uint8, device="cuda")
    ws[:256] = 0
    a = run_gpu(case, tokens, top_k, top_p, ws=ws)
    b = run_gpu(case, tokens, top_k, top_p, ws=ws)
    assert all(np.array_equal(x, y) for x, y in zip(a, b))
    assert sv.spec_verify_read_status(ws) == sv.SPEC_DEV_OK
