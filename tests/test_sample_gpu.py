"""Parity of the CUDA sampler (spec_sample) with the fp64 oracle.

Tokens must match exactly, except a sampled row whose uniform sits within
BAND = 1e-5 of its oracle draw cell's boundary (|u - C(x-1)/R| or
|C(x)/R - u|).  Such rows are counted and held to 0.01 % of the draws: the
fp32 pick lists every row within 1.2e-6 of R of an edge for the exact draw, so
a mismatch needs a uniform within ~1e-12 of an edge.  Greedy rows (T = 0) and
error rows get no band.
"""
import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
import speculative_decoding_verification_65_gb300 as sv  # noqa: E402
from speculative_decoding_verification_65_gb300 import synth  # noqa: E402

BAND = 1e-5
MAX_EXEMPT = 1e-4
NTHREADS = os.cpu_count() or 1


def gpu_sample(sc, ws=None):
    d = sv.sample_to_device(sc)
    tok = sv.spec_sample(d["logits"], d["u"], d["temperature"], ws=ws)
    torch.cuda.synchronize()
    return tok.cpu().numpy()


def compare(sc, g):
    r, tr = oracle.sample(sc.logits, sc.u.astype(np.float64), sc.temperature.astype(np.float64),
                          nthreads=NTHREADS)
    exempt = []
    for i in np.nonzero(g != r)[0]:
        why = f"row {i} T={sc.temperature[i]} gpu {g[i]} oracle {r[i]}"
        assert sc.temperature[i] > 0 and r[i] >= 0 and g[i] >= 0, "mismatch without band: " + why
        lo, hi = tr[i, 0], tr[i, 1]
        margin = min(float(sc.u[i]) - lo, hi - float(sc.u[i]))
        assert margin < BAND, f"mismatch outside the band (margin {margin:.3g}): " + why
        exempt.append(int(i))
    draws = int(np.count_nonzero((sc.temperature > 0) & (r >= 0)))
    assert len(exempt) <= MAX_EXEMPT * draws, (len(exempt), draws)
    return r, exempt


@pytest.mark.parametrize("cfg,B", [(1, None), (2, None), (3, 16), (4, 16), (5, 48)])
def test_workload_rows(cfg, B):
    sc = synth.make_sample_config(cfg, B=B)
    g = gpu_sample(sc)
    r, _ = compare(sc, g)
    assert np.all(g[sc.temperature > 0] >= 0)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("V", [2, 3, 7, 100, 1023, 2049, 4097, 100003])
def test_ragged_vocabularies(dtype, V):
    case = synth.gauss_case(B=6, k=3, V=V, dtype=dtype, seed=V, T=(0.0, 0.6, 1.0, 1.7))
    sc = synth.sample_case_from(case, seed=V + 1)
    compare(sc, gpu_sample(sc))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_largest_vocabulary(dtype):
    case = synth.gauss_case(B=2, k=2, V=sv.SPEC_MAX_V, dtype=dtype, seed=3, T=(0.0, 1.0))
    sc = synth.sample_case_from(case, seed=4)
    compare(sc, gpu_sample(sc))


def test_full_size_workload_rows():
    # the benchmark's sampling workload: the 4096 draft rows of the
    # B1024/k4/V128256 bf16 workload, every row checked
    sc = synth.make_sample_config(5)
    compare(sc, gpu_sample(sc))


def test_greedy_ties_take_the_lowest_index():
    rng = np.random.default_rng(1)
    for dtype in ("f32", "bf16"):
        l = rng.integers(-3, 4, size=(64, 5000)).astype(np.float32)
        logits = synth.f32_to_bf16_bits(l) if dtype == "bf16" else l
        sc = synth.SampleCase(logits, rng.random(64, dtype=np.float32),
                              np.zeros(64, np.float32), dtype)
        assert np.array_equal(gpu_sample(sc), np.argmax(l, axis=1))


def test_error_rows_and_masked_entries():
    rng = np.random.default_rng(2)
    R, V = 12, 3000
    l = rng.standard_normal((R, V)).astype(np.float32)
    T = np.ones(R, np.float32)
    l[1, 77] = np.nan
    l[2, 5] = np.inf
    l[3, :] = -np.inf
    T[4] = -1.0
    T[5] = np.nan
    T[6] = np.inf
    T[7] = 1e-40
    mask = rng.random(V) < 0.7
    mask[0] = False
    l[8, mask] = -np.inf
    l[9, mask] = -np.inf
    T[9] = 0.0
    sc = synth.SampleCase(l, rng.random(R, dtype=np.float32), T, "f32")
    g = gpu_sample(sc)
    assert np.all(g[1:8] == -1)
    assert not mask[g[8]] and not mask[g[9]]
    compare(sc, g)


@pytest.mark.parametrize("V", [4, 4096, 40000])
def test_uniform_on_a_cell_boundary(V):
    # equal logits: every running sum is an exact integer on both sides, so a
    # uniform on a boundary has one right answer: the next token
    R = 4
    sc = synth.SampleCase(np.zeros((R, V), np.float32),
                          np.array([0.0, 0.25, 0.5, 0.75], np.float32),
                          np.ones(R, np.float32), "f32")
    g = gpu_sample(sc)
    assert np.array_equal(g, np.array([0, V // 4, V // 2, 3 * V // 4]))
    assert np.array_equal(g, oracle.sample(sc.logits, sc.u, sc.temperature)[0])


def test_no_rows_is_a_no_op():
    d = sv.sample_to_device(synth.SampleCase(np.zeros((0, 8), np.float32),
                                             np.zeros(0, np.float32), np.zeros(0, np.float32),
                                             "f32"))
    out = sv.spec_sample(d["logits"], d["u"], d["temperature"])
    torch.cuda.synchronize()
    assert out.numel() == 0


def test_garbage_workspace_and_repeat_calls_agree():
    sc = synth.make_sample_config(3, B=8)
    need = sv.spec_sample_workspace_size(sc.R, sc.V, sv.SPEC_BF16)
    ws = torch.randint(0, 256, (need,), dtype=torch.uint8, device="cuda")
    ws[:256] = 0  # only the status word must start at zero
    a = gpu_sample(sc, ws=ws)
    b = gpu_sample(sc, ws=ws)
    assert np.array_equal(a, b)
    assert sv.spec_verify_read_status(ws) == sv.SPEC_DEV_OK
    compare(sc, a)


def test_interleaved_with_verification_on_one_workspace():
    case = synth.make_config(2, B=8)
    sc = synth.sample_case_from(case, seed=5)
    d = sv.to_device(case)
    t1, n1 = sv.spec_verify(**d)
    s1 = gpu_sample(sc)
    t2, n2 = sv.spec_verify(**d)
    s2 = gpu_sample(sc)
    torch.cuda.synchronize()
    assert torch.equal(t1, t2) and torch.equal(n1, n2)
    assert np.array_equal(s1, s2)


def test_draw_frequencies_chi_square():
    stats = pytest.importorskip("scipy.stats")
    rng = np.random.default_rng(13)
    V, N, T = 64, 400000, 0.9
    row = (rng.standard_normal(V) * 1.5).astype(np.float32)
    p = np.exp((row.astype(np.float64) - row.max()) / T)
    p /= p.sum()
    sc = synth.SampleCase(np.repeat(row[None, :], N, axis=0), rng.random(N, dtype=np.float32),
                          np.full(N, T, np.float32), "f32")
    g = gpu_sample(sc)
    counts = np.bincount(g, minlength=V)
    keep = p * N >= 5
    obs, exp = counts[keep], p[keep] * N
    if not keep.all():  # pool the rare tokens into one bucket
        obs = np.append(obs, counts[~keep].sum())
        exp = np.append(exp, p[~keep].sum() * N)
    assert stats.chisquare(obs, exp * (obs.sum() / exp.sum())).pvalue > 1e-4
