"""CUDA path vs the fp64 oracle, through the C ABI (ctypes binding).

Integer outputs (accept counts, tokens) must match exactly; the only
exemption is a decision whose uniform lies within 1e-5 of the oracle's
threshold or draw-cell boundary (tests/parity_util.py).  Exempt mismatches
are counted and held to 0.01 % of decisions by parity_util.check_bound: no
draw mismatch in a call under 1e4 decisions, at most one accept-test
mismatch per call (the aggregate rate over >1e5 decisions is checked in
tests/test_exact_draw_gpu.py).  Intermediate probabilities P = p(g),
Q = q(g) must agree with the oracle within 1e-5 relative.
"""
import os

import numpy as np
import pytest

import oracle
from tests import parity_util as pu

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import speculative_decoding_verification_65_gb300 as sv  # noqa: E402
from speculative_decoding_verification_65_gb300 import synth  # noqa: E402

NTHR = os.cpu_count() or 1


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    sv.library()


def run_gpu(case, ws=None):
    d = sv.to_device(case)
    toks, n = sv.spec_verify(**d, ws=ws)
    torch.cuda.synchronize()
    return toks.cpu().numpy(), n.cpu().numpy()


def run_oracle(case):
    return oracle.verify(case.target, case.draft, case.tokens, case.u_accept, case.u_resample,
                         case.temperature, nthreads=NTHR)


def check(case, tag=None):
    g_t, g_n = run_gpu(case)
    r_t, r_n, tr = run_oracle(case)
    pu.check_invariants(case, g_t, g_n)
    rep = pu.compare(case, g_t, g_n, r_t, r_n, tr)
    out = os.environ.get("PARITY_REPORT_DIR")
    if out and tag:
        import json
        os.makedirs(out, exist_ok=True)
        with open(os.path.join(out, f"parity_{tag}.json"), "w") as f:
            json.dump(rep, f)
    pu.check_bound(rep)
    return rep, g_t, g_n


# ----------------------------------------------------------------- workloads

@pytest.mark.parametrize("cfg", [1, 2, 3])
def test_workload_full_oracle(cfg):
    case = synth.make_config(cfg)
    rep, _, g_n = check(case, f"cfg{cfg}")
    print(f"cfg{cfg}: {rep['decisions']} decisions, exempt {rep['exempt']}, "
          f"near-band {rep['near_band']}, mean accepted {np.mean(g_n):.3f}")


@pytest.mark.parametrize("cfg", [4, 5])
def test_workload_full_size(cfg):
    """The full-size workloads, as the benchmark launches them: every sequence
    against the oracle (the oracle is threaded over sequences)."""
    case = synth.make_config(cfg)
    rep, g_t, g_n = check(case, f"cfg{cfg}")
    if cfg == 5:
        cls0 = np.arange(case.B) % 3 == 0  # target == draft bit for bit: always accepted
        assert np.all(g_n[cls0] == case.k)
    if cfg == 4:
        greedy = case.temperature == 0
        tgt = torch.from_numpy(case.target[greedy]).cuda()
        am = torch.argmax(tgt, dim=-1).cpu().numpy()  # first maximal index
        for row, b in enumerate(np.flatnonzero(greedy)):
            mism = np.flatnonzero(case.tokens[b] != am[row, :case.k])
            j = int(mism[0]) if mism.size else case.k
            assert g_n[b] == j and g_t[b, j] == am[row, j]
    print(f"cfg{cfg}: {rep}")


def test_recipes_small_sizes_many_seeds():
    for cfg in (2, 3, 4, 5):
        for off in (11, 12):
            case = synth.make_config(cfg, B=24, V=5000 + 37 * off, seed_offset=off)
            check(case)


# ---------------------------------------------------------------- edge cases

@pytest.mark.parametrize("V", [2, 3, 5, 33, 1023, 8191, 8193, 16385, 40001])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_ragged_vocab(V, dtype):
    case = synth.gauss_case(B=7, k=3, V=V, dtype=dtype, seed=V, T=(0.0, 0.5, 1.0, 2.0))
    check(case)


@pytest.mark.parametrize("k", [1, 2, 8, 32])
def test_draft_lengths(k):
    case = synth.gauss_case(B=9, k=k, V=777, dtype="bf16", seed=k, T=(0.0, 0.8, 1.0),
                            sigma_n=0.3)
    check(case)


def test_single_sequence_large_vocab():
    case = synth.gauss_case(B=1, k=4, V=1 << 20, dtype="f32", seed=3, sigma_n=0.2)
    check(case)


def test_zero_batch():
    z = torch.empty(0, device="cuda")
    toks, n = sv.spec_verify(torch.empty((0, 3, 5), device="cuda"),
                             torch.empty((0, 2, 5), device="cuda"),
                             torch.empty((0, 2), dtype=torch.int32, device="cuda"),
                             torch.empty((0, 2), device="cuda"), z, z)
    assert toks.shape == (0, 3) and n.shape == (0,)


def test_identical_rows_always_accept():
    for V, dt in ((33, "f32"), (1000, "bf16"), (50000, "f32")):
        case = synth.gauss_case(B=16, k=5, V=V, dtype=dt, seed=V, T=(0.5, 1.0, 1.7))
        case.target[:, :case.k] = case.draft
        g_t, g_n = run_gpu(case)
        assert np.all(g_n == case.k)
        check(case)


def test_greedy_ties():
    rng = np.random.default_rng(4)
    B, k, V = 64, 4, 3000
    case = synth.gauss_case(B=B, k=k, V=V, dtype="bf16", seed=4, T=0.0)
    bits = synth.f32_to_bf16_bits(rng.integers(-2, 3, (B, k + 1, V)).astype(np.float32))
    case.target[:] = bits
    am = np.argmax(synth.bf16_bits_to_f32(case.target), -1)
    case.tokens[:] = np.where(rng.random((B, k)) < 0.7, am[:, :k], rng.integers(0, V, (B, k)))
    check(case)


@pytest.mark.parametrize("what", ["T_neg", "T_nan", "T_inf", "T_denormal", "tok_hi", "tok_neg",
                                  "nan_target_bonus", "posinf_draft_last", "all_neginf_target",
                                  "q_zero_first", "nan_draft_greedy_ok", "q_zero_after_reject"])
def test_error_rows(what):
    case = synth.gauss_case(B=8, k=3, V=300, dtype="f32", seed=21, T=1.0)
    b = 3
    t, d, g, T = case.target, case.draft, case.tokens, case.temperature
    if what == "T_neg":
        T[b] = -1.0
    elif what == "T_nan":
        T[b] = np.nan
    elif what == "T_inf":
        T[b] = np.inf
    elif what == "T_denormal":
        T[b] = np.float32(1e-40)
    elif what == "tok_hi":
        g[b, 2] = case.V
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
    elif what == "nan_draft_greedy_ok":
        T[b] = 0.0
        d[b, :, :] = np.nan
    elif what == "q_zero_after_reject":
        t[b, 0, g[b, 0]] = -np.inf
        d[b, 1, g[b, 1]] = -np.inf
    g_t, g_n = run_gpu(case)
    r_t, r_n, tr = run_oracle(case)
    np.testing.assert_array_equal(g_n, r_n)
    np.testing.assert_array_equal(g_t, r_t)
    expect_err = what not in ("nan_draft_greedy_ok", "q_zero_after_reject")
    assert (g_n[b] == -1) == expect_err


# ----------------------------------------------------------- intermediates

@pytest.mark.parametrize("cfg", [1, 2, 3])
def test_intermediate_probabilities(cfg):
    case = synth.make_config(cfg, B=min(synth.CONFIGS[cfg]["B"], 32))
    d = sv.to_device(case)
    toks, n, probs = sv.spec_verify_probs(**d)
    torch.cuda.synchronize()
    ref = oracle.probs(case.target, case.draft, case.tokens, case.temperature)
    got = probs.cpu().numpy().astype(np.float64)
    ok = np.isfinite(ref)
    assert np.all(np.isfinite(got[ok]))
    rel = np.abs(got[ok] - ref[ok]) / np.maximum(ref[ok], 1e-300)
    big = ref[ok] > 1e-30  # fp32 flushes values below its normal range
    assert rel[big].max() < 1e-5, rel[big].max()


@pytest.mark.parametrize("cfg", [4, 5])
def test_intermediate_probabilities_full_size(cfg):
    """The two largest workloads at full size, as the benchmark launches them
    (fp32 V = 151936 with T in {0, 0.5, 1, 1.3}; bf16 V = 128256 with its three
    classes): the GPU runs the whole batch, and the fp64 oracle checks a sample
    of 12 sequences of every sampling temperature (workload 4) or class
    (workload 5), every drafted position.  Greedy sequences have no P, Q."""
    case = synth.make_config(cfg)
    d = sv.to_device(case)
    _, _, probs = sv.spec_verify_probs(**d)
    torch.cuda.synchronize()
    rng = np.random.default_rng(100 + cfg)
    if cfg == 4:
        groups = [np.flatnonzero(case.temperature == T) for T in (0.5, 1.0, 1.3)]
    else:
        groups = [np.arange(c, case.B, 3) for c in range(3)]
    assert all(g.size for g in groups)
    idx = np.sort(np.concatenate([rng.choice(g, size=min(12, g.size), replace=False)
                                  for g in groups]))
    sub = case.subset(idx)
    ref = oracle.probs(sub.target, sub.draft, sub.tokens, sub.temperature)
    got = probs.cpu().numpy()[idx].astype(np.float64)
    ok = np.isfinite(ref)
    assert ok.sum() == idx.size * case.k * 2
    assert np.all(np.isfinite(got[ok]))
    rel = np.abs(got[ok] - ref[ok]) / np.maximum(ref[ok], 1e-300)
    big = ref[ok] > 1e-30  # fp32 flushes values below its normal range
    print(f"cfg{cfg}: {idx.size} sequences, max relative error {rel[big].max():.3g}")
    assert rel[big].max() < 1e-5, rel[big].max()


# ---------------------------------------------------- determinism, workspace

def test_deterministic_across_calls_and_workspaces():
    case = synth.make_config(2)
    d = sv.to_device(case)
    ws = sv.workspace(case.B, case.k, case.V, sv.SPEC_BF16)
    outs = []
    for i in range(3):
        if i == 2:  # a workspace full of garbage gives the same answer: nothing carries over
            ws = torch.randint(0, 255, (ws.numel(),), dtype=torch.uint8, device="cuda")
            ws[:256] = 0
        t, n = sv.spec_verify(**d, ws=ws)
        outs.append((t.clone(), n.clone()))
    torch.cuda.synchronize()
    for t, n in outs[1:]:
        assert torch.equal(t, outs[0][0]) and torch.equal(n, outs[0][1])
    assert sv.spec_verify_read_status(ws) == sv.SPEC_DEV_OK


def test_workspace_reuse_across_shapes():
    """One workspace serves calls of different shapes back to back."""
    a = synth.gauss_case(B=4, k=8, V=20000, dtype="f32", seed=1)
    b = synth.gauss_case(B=40, k=4, V=20000, dtype="bf16", seed=2)
    need = max(sv.spec_verify_workspace_size(4, 8, 20000, 0),
               sv.spec_verify_workspace_size(40, 4, 20000, 1))
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    for case in (a, b, a, b):
        d = sv.to_device(case)
        t, n = sv.spec_verify(**d, ws=ws)
        torch.cuda.synchronize()
        pu.compare(case, t.cpu().numpy(), n.cpu().numpy(), *run_oracle(case))


def test_streams_and_workspaces_are_independent():
    a = synth.make_config(1)
    b = synth.make_config(2)
    da, db = sv.to_device(a), sv.to_device(b)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    with torch.cuda.stream(s1):
        ta, na = sv.spec_verify(**da)
    with torch.cuda.stream(s2):
        tb, nb = sv.spec_verify(**db)
    torch.cuda.synchronize()
    ra = run_oracle(a)
    rb = run_oracle(b)
    pu.compare(a, ta.cpu().numpy(), na.cpu().numpy(), *ra)
    pu.compare(b, tb.cpu().numpy(), nb.cpu().numpy(), *rb)


def test_host_entry_matches_device_entry():
    case = synth.make_config(2)
    g_t, g_n = run_gpu(case)
    B, k, V = case.B, case.k, case.V
    arena = torch.zeros(sv.spec_verify_host_arena_size(B, k, V, sv.SPEC_BF16),
                        dtype=torch.uint8, device="cuda")
    pin = lambda a: torch.from_numpy(a).pin_memory()
    tgt = pin(case.target.view(np.int16)).view(torch.bfloat16)
    dft = pin(case.draft.view(np.int16)).view(torch.bfloat16)
    t, n = sv.spec_verify_host(tgt, dft, pin(case.tokens), pin(case.u_accept),
                               pin(case.u_resample), pin(case.temperature), arena)
    np.testing.assert_array_equal(t.numpy(), g_t)
    np.testing.assert_array_equal(n.numpy(), g_n)


def test_host_entry_leaves_greedy_draft_rows_on_the_host():
    """spec_verify_host copies draft rows only for sequences with T != 0: NaN
    in a greedy sequence's host draft rows (never copied, never read) changes
    nothing, and a run pattern with greedy sequences at both ends and between
    runs gives the oracle's outputs."""
    case = synth.gauss_case(B=11, k=3, V=3001, dtype=synth.F32, seed=61, T=(0.0, 1.0))
    case.temperature[:] = np.array([0, 1, 1, 0, 0.7, 0, 1.3, 1, 1, 0, 0], np.float32)
    B, k, V = case.B, case.k, case.V
    dft = case.draft.copy()
    dft[case.temperature == 0] = np.nan
    arena = torch.zeros(sv.spec_verify_host_arena_size(B, k, V, sv.SPEC_F32),
                        dtype=torch.uint8, device="cuda")
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
    t, n = sv.spec_verify_host(pin(case.target), pin(dft), pin(case.tokens), pin(case.u_accept),
                               pin(case.u_resample), pin(case.temperature), arena)
    r_t, r_n, tr = run_oracle(case)
    pu.compare(case, t.numpy(), n.numpy(), r_t, r_n, tr)
    assert np.all(n.numpy() >= 0)
