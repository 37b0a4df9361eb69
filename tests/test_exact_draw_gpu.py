"""The exact draw (csrc/resolve.cuh) against the fp64 oracle, on the GPU.

The fp32 draw lists a sequence for the exact draw when its u * R lies within
a guard of the chosen cell's edges.  Two properties are checked:

* with every draw listed (spec_verify_trace(resolve_all=True)) the exact
  draw alone decides every token, and it must equal the oracle's except where
  the oracle's uniform lies within 1e-10 of a cell edge (float-float weights
  and exact fixed-point sums: about 1e-12 of R);
* in the default mode, over more than 1e5 decisions of the two largest
  workloads, mismatches with the oracle (all of them inside the 1e-5 band)
  stay under 0.01 % of the decisions, the bound the verification must meet.
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
EXACT_BAND = 1e-10     # where the exact draw may still differ from fp64
MAX_EXEMPT_FRACTION = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    sv.library()


def run_trace(case, resolve_all):
    d = sv.to_device(case)
    toks, n, draw, _ = sv.spec_verify_trace(**d, resolve_all=resolve_all)
    torch.cuda.synchronize()
    return toks.cpu().numpy(), n.cpu().numpy(), draw.cpu().numpy()


def run_oracle(case):
    return oracle.verify(case.target, case.draft, case.tokens, case.u_accept, case.u_resample,
                         case.temperature, nthreads=NTHR)


def draw_margins(case, r_n, trace):
    """The oracle's distance of u to its draw cell's nearer edge, per sequence
    (inf where nothing is drawn from a distribution)."""
    k = case.k
    m = np.full(case.B, np.inf)
    for b in range(case.B):
        if case.temperature[b] == 0 or r_n[b] < 0:
            continue
        lo, hi = trace[b, k], trace[b, k + 1]
        u = float(case.u_resample[b])
        m[b] = min(u - lo, hi - u)
    return m


def check_exact(case, band=EXACT_BAND):
    g_t, g_n, draw = run_trace(case, resolve_all=True)
    r_t, r_n, tr = run_oracle(case)
    pu.check_invariants(case, g_t, g_n)
    rep = pu.compare(case, g_t, g_n, r_t, r_n, tr)
    # every exempt mismatch must be a draw within `band`, or an accept test
    for b, kind, margin in rep["mismatched"]:
        if kind != "accept":
            assert margin < band, (b, kind, margin)
    drawn = draw[:, 1] == 1
    # every drawing sequence was listed, and the token written is the exact one
    for b in np.flatnonzero(drawn):
        j = g_n[b]
        assert g_t[b, j] == draw[b, 2], b
    fp32_wrong = np.flatnonzero(drawn & (draw[:, 0] != draw[:, 2]))
    m = draw_margins(case, r_n, tr)
    worst = float(np.max(m[fp32_wrong])) if fp32_wrong.size else 0.0
    # the fp32 search's error: its distance to the nearer cell edge against
    # the oracle's, where both chose the same cell
    gap = draw[:, 3].astype(np.int32).view(np.float32).astype(np.float64)
    same = drawn & (draw[:, 0] == draw[:, 2]) & (g_t[np.arange(case.B), np.maximum(g_n, 0)] ==
                                                   r_t[np.arange(case.B), np.maximum(r_n, 0)])
    same &= np.isfinite(m) & (gap > 0)
    err = np.abs(gap[same] - m[same])
    rep["fp32_gap_err_max"] = float(err.max()) if err.size else 0.0
    return rep, int(drawn.sum()), fp32_wrong.size, worst


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5])
def test_exact_draw_every_sequence(cfg):
    """resolve_all: the exact draw decides every token on the full workload."""
    case = synth.make_config(cfg)
    rep, listed, n_wrong, worst = check_exact(case)
    print(f"cfg{cfg}: {listed} draws listed, fp32 token differed on {n_wrong} "
          f"(largest oracle margin among them {worst:.3g}); {rep['exempt']} exempt; "
          f"fp32 edge error up to {rep['fp32_gap_err_max']:.3g} of R")
    # the fp32 draw's own errors must sit well inside its guard: a listing
    # guard of 4e-6 needs the fp32 error well below it
    assert worst < 1e-6, worst


@pytest.mark.parametrize("V,dtype", [(2, "f32"), (3, "bf16"), (2047, "f32"), (2049, "bf16"),
                                     (40001, "f32"), (100003, "bf16")])
def test_exact_draw_ragged(V, dtype):
    case = synth.gauss_case(B=16, k=3, V=V, dtype=dtype, seed=V + 5, T=(0.0, 0.5, 1.0, 2.0))
    check_exact(case)


@pytest.mark.parametrize("k", [1, 2, 8, 32])
def test_exact_draw_lengths(k):
    case = synth.gauss_case(B=12, k=k, V=5000, dtype="bf16", seed=40 + k, T=(0.8, 1.0),
                            sigma_n=0.3)
    check_exact(case)


def test_exact_draw_near_identical_rows():
    """Target = draft + noise of 1e-6: nearly every element's p/q is within
    2^-14 of 1, the list of undecided elements overflows and the exact draw
    takes its slow path (every chunk again with the exact mass ratio).  The
    residual is then ~1e-6 of the mass, so the weights' 1e-13 relative error
    is ~1e-7 of R and the ordinary 1e-5 band applies to the draws."""
    case = synth.gauss_case(B=8, k=2, V=20000, dtype="f32", seed=77, T=(1.0,), sigma_n=1e-6)
    # make rejections likely: the largest uniform below 1
    case.u_accept[:] = np.nextafter(np.float32(1), np.float32(0))
    rep, listed, _, _ = check_exact(case, band=pu.BAND)
    assert listed > 0


def test_exact_draw_large_vocab():
    case = synth.gauss_case(B=2, k=2, V=1 << 20, dtype="f32", seed=9, sigma_n=0.5)
    check_exact(case)


def test_exempt_rate_below_bound():
    """Default mode (fp32 draws, the exact draw for listed sequences only) on
    workloads 4 and 5 at full size over several seeds: more than 1e5
    decisions, exempt mismatches at most 0.01 % of them."""
    n4 = int(os.environ.get("EXACT_SEEDS_4", "10"))
    n5 = int(os.environ.get("EXACT_SEEDS_5", "26"))
    total = dict(decisions=0, exempt=0, draws=0, listed=0)
    for cfg, n in ((4, n4), (5, n5)):
        for off in range(n):
            case = synth.make_config(cfg, seed_offset=off) if off else synth.make_config(cfg)
            g_t, g_n, draw = run_trace(case, resolve_all=False)
            r_t, r_n, tr = run_oracle(case)
            pu.check_invariants(case, g_t, g_n)
            rep = pu.compare(case, g_t, g_n, r_t, r_n, tr)
            total["decisions"] += rep["decisions"]
            total["exempt"] += rep["exempt"]
            total["draws"] += rep["draws"]
            total["listed"] += int((draw[:, 1] == 1).sum())
    print(f"exempt rate: {total}")
    if n4 + n5 >= 36:
        assert total["decisions"] >= 100_000, total
    assert total["exempt"] <= MAX_EXEMPT_FRACTION * total["decisions"], total
