"""Parity of the LM-head-fused verification (spec_verify_lmhead) and of its
tensor-core product (spec_lmhead_logits) with the fp64 oracle.

On the grid recipe every partial sum of h.W is exact in fp32, so the GPU's
logits equal the oracle's and the integer outputs must match with the usual
1e-5 exemption band, the exempt count held to 0.01 % of the decisions.  On the
gauss recipe the fp32 accumulation rounds: the product is checked against a
bound on that rounding, and each decision gets its own band, the effect of
its row's per-logit bounds on the threshold or on the draw's cell edges.
Every mismatch must lie inside its band.  Accept-test mismatches stay under
the 0.01 % cap; draw mismatches are counted and held to 8 % of the draws: the
GPU's logits are a different fp32 rounding of the same dot products (about
1e-6), and on a 128256-token row of this spread that moves u * R across a
cell edge in a few percent of the draws (9 of 256 measured at full size).
"""
import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
import speculative_decoding_verification_65_gb300 as sv  # noqa: E402
from speculative_decoding_verification_65_gb300 import synth  # noqa: E402
from tests.parity_util import (BAND, MAX_EXEMPT_FRACTION, check_bound,  # noqa: E402
                               check_invariants, compare)

NTHREADS = os.cpu_count() or 1


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _bf16(a):
    return _dev(a).view(torch.bfloat16)


def to_device(c):
    draft = _bf16(c.draft) if c.dtype == "bf16" else _dev(c.draft)
    return dict(hidden=_bf16(c.hidden), lm_head=_bf16(c.lm_head), draft=draft,
                tokens=_dev(c.tokens), u_accept=_dev(c.u_accept), u_resample=_dev(c.u_resample),
                temperature=_dev(c.temperature))


def run(c, ws=None, want_probs=False):
    out = sv.spec_verify_lmhead(**to_device(c), ws=ws, want_probs=want_probs)
    torch.cuda.synchronize()
    return tuple(x.cpu().numpy() for x in out)


def rounding_bound(hidden_bits, w_bits):
    """A bound on |fp32 tensor-core sum - exact sum| per logit: the accumulator
    takes d/16 MMA steps of 16 products each, every addition rounding by at
    most 2^-24 of a partial sum no larger than sum_j |h_j w_j|; 16 more units
    cover the rounding inside one step."""
    h = np.abs(oracle._bf16_to_f64(hidden_bits))
    w = np.abs(oracle._bf16_to_f64(w_bits))
    d = h.shape[-1]
    return (d / 16 + 16) * 2.0 ** -24 * (h.reshape(-1, d) @ w.T)


@pytest.mark.parametrize("M,V,d", [(1, 2, 64), (128, 256, 64), (129, 257, 128),
                                   (300, 1000, 256), (257, 5003, 512)])
def test_product_within_the_fp32_bound(M, V, d):
    rng = np.random.default_rng(M + V)
    hb = synth.f32_to_bf16_bits(rng.standard_normal((M, d)).astype(np.float32))
    wb = synth.f32_to_bf16_bits((rng.standard_normal((V, d)) / np.sqrt(d)).astype(np.float32))
    out, status = sv.spec_lmhead_logits(_bf16(hb), _bf16(wb))
    torch.cuda.synchronize()
    got = out.cpu().numpy().astype(np.float64)
    want = oracle.lmhead_logits(hb, wb)
    assert int(status.item()) == sv.SPEC_DEV_OK
    assert np.all(np.abs(got - want) <= rounding_bound(hb, wb))


def test_grid_product_is_exact():
    c = synth.make_lmhead_case(B=20, k=4, V=3001, d=1024, recipe="grid", seed=3)
    out, _ = sv.spec_lmhead_logits(_bf16(c.hidden.reshape(-1, c.d)), _bf16(c.lm_head))
    torch.cuda.synchronize()
    want = oracle.lmhead_logits(c.hidden, c.lm_head).reshape(-1, c.V)
    assert np.array_equal(out.cpu().numpy().astype(np.float64), want)


@pytest.mark.parametrize("B,k,V,d,dtype,T", [
    (24, 4, 3000, 256, "bf16", (1.0,)),
    (40, 3, 32000, 512, "bf16", (0.7, 1.0, 1.3)),
    (33, 5, 5003, 128, "f32", (0.0, 0.5, 1.0)),      # rows past a 128-row tile, a ragged V
    (8, 1, 257, 64, "f32", (1.0,)),
    (6, 31, 1000, 64, "bf16", (1.0, 0.0)),            # the largest k
])
def test_parity_grid(B, k, V, d, dtype, T):
    c = synth.make_lmhead_case(B, k, V, d, dtype, recipe="grid", seed=B + V, T=T)
    gt, gn = run(c)
    rt, rn, tr = oracle.verify_lmhead(c.hidden, c.lm_head, c.draft, c.tokens, c.u_accept,
                                      c.u_resample, c.temperature, nthreads=NTHREADS)
    check_invariants(c, gt, gn)
    rep = compare(c, gt, gn, rt, rn, tr)
    check_bound(rep)


def test_probs_equal_the_oracle_on_the_grid():
    c = synth.make_lmhead_case(16, 4, 4000, 512, "bf16", recipe="grid", seed=9, T=(0.8, 1.0))
    _, _, probs = run(c, want_probs=True)
    t = oracle.lmhead_logits(c.hidden, c.lm_head).astype(np.float32)
    d32 = synth.bf16_bits_to_f32(c.draft)
    PQ = oracle.probs(t, d32, c.tokens, c.temperature)
    np.testing.assert_allclose(probs[..., 0], PQ[..., 0], rtol=1e-5, atol=1e-30)
    np.testing.assert_allclose(probs[..., 1], PQ[..., 1], rtol=1e-5, atol=1e-30)


def _softmax(t, T):
    x = t / T
    e = np.exp(x - x.max())
    return e / e.sum()


def logit_bounds(hidden_bits, w_bits):
    """rounding_bound with |h|.|W| taken in float32, scaled by 1 + 1e-3 to
    cover that product's own rounding (all its terms are positive)."""
    h = np.abs(synth.bf16_bits_to_f32(hidden_bits))
    w = np.abs(synth.bf16_bits_to_f32(w_bits))
    d = h.shape[-1]
    return (d / 16 + 16) * 2.0 ** -24 * (h.reshape(-1, d) @ w.T).astype(np.float64) * (1 + 1e-3)


def decision_bands(c, t64, eps, rn, tr):
    """Per decision, how far the logits' fp32 rounding can move it.  Logits
    perturbed by |delta_x| <= eps_x move log p(g) by at most
    (eps_g + E_p[eps]) / T to first order (the numerator and the normaliser),
    so an accept threshold min(1, P/Q) by min(1, r) (exp(that) - 1); they
    move the total variation sum |dp| by at most 2 E_p[eps] / T, so a draw
    cell edge C/R by at most twice that over R.  A factor 1.25 covers the
    second order; the floor is the usual 1e-5."""
    B, k = c.B, c.k
    band = np.full((B, k + 1), BAND)
    for b in range(B):
        T = float(c.temperature[b])
        if T == 0 or rn[b] < 0:
            continue
        for i in range(min(int(rn[b]) + 1, k)):
            p = _softmax(t64[b, i], T)
            g = int(c.tokens[b, i])
            delta = (eps[b, i, g] + p @ eps[b, i]) / T
            band[b, i] = max(BAND, 1.25 * min(1.0, tr[b, i]) * np.expm1(delta))
        j = int(rn[b])
        p = _softmax(t64[b, j], T)
        R = 1.0 if j == k else tr[b, k + 2]
        band[b, k] = max(BAND, 1.25 * 4.0 * float(p @ eps[b, j]) / (T * R))
    return band


def _check_gauss(c, gt, gn, idx, max_draw_fraction=0.08):
    """Parity of sequences `idx` of a gauss-recipe call with per-decision
    bands: every mismatch inside its band, accept-test mismatches under the
    0.01 % cap, draw mismatches under `max_draw_fraction` of the draws."""
    s = synth.LmheadCase(c.hidden[idx], c.lm_head, c.draft[idx], c.tokens[idx],
                         c.u_accept[idx], c.u_resample[idx], c.temperature[idx], c.dtype, c.name)
    rt, rn, tr = oracle.verify_lmhead(s.hidden, s.lm_head, s.draft, s.tokens, s.u_accept,
                                      s.u_resample, s.temperature, nthreads=NTHREADS)
    t64 = oracle.lmhead_logits(s.hidden, s.lm_head).astype(np.float32).astype(np.float64)
    eps = logit_bounds(s.hidden, s.lm_head).reshape(s.B, s.k + 1, s.V)
    band = decision_bands(s, t64, eps, rn, tr)
    check_invariants(s, gt[idx], gn[idx])
    rep = compare(s, gt[idx], gn[idx], rt, rn, tr, band=band)
    kinds = [m[1] for m in rep["mismatched"]]
    accepts = kinds.count("accept")
    draws = len(kinds) - accepts
    assert accepts <= max(1, MAX_EXEMPT_FRACTION * rep["decisions"]), rep
    assert draws <= max(1, max_draw_fraction * rep["draws"]), rep
    print(f"{c.name}: {rep['decisions']} decisions, {accepts} accept and {draws} draw "
          f"mismatches inside their bands (median draw band {np.median(band[:, s.k]):.2g})")
    return rep


def test_parity_gauss_per_logit_band():
    B, k, V, d = 32, 4, 8000, 1024
    c = synth.make_lmhead_case(B, k, V, d, "bf16", recipe="gauss", seed=21, T=(0.7, 1.0, 1.3))
    gt, gn = run(c)
    _check_gauss(c, gt, gn, np.arange(B))


def test_parity_gauss_full_size():
    """The benchmarked shape, B1024 k4 V128256 d4096 on gaussian inputs: the
    GEMM runs over every row; the first 256 sequences are checked against
    the oracle."""
    B, k, V, d = 1024, 4, 128256, 4096
    c = synth.make_lmhead_case(B, k, V, d, "bf16", recipe="gauss", seed=6, T=(0.7, 1.0, 1.3),
                               draft_product="f32")
    gt, gn = run(c)
    _check_gauss(c, gt, gn, np.arange(256))


def test_parity_grid_full_size():
    """The benchmarked shape on the grid recipe (exact fp32 logits): the
    first 256 sequences against the oracle, held to the 0.01 % cap."""
    B, k, V, d = 1024, 4, 128256, 4096
    c = synth.make_lmhead_case(B, k, V, d, "bf16", recipe="grid", seed=5, T=(0.7, 1.0, 1.3),
                               draft_product="f32")
    gt, gn = run(c)
    idx = np.arange(256)
    s = synth.LmheadCase(c.hidden[idx], c.lm_head, c.draft[idx], c.tokens[idx],
                         c.u_accept[idx], c.u_resample[idx], c.temperature[idx], c.dtype, c.name)
    rt, rn, tr = oracle.verify_lmhead(s.hidden, s.lm_head, s.draft, s.tokens, s.u_accept,
                                      s.u_resample, s.temperature, nthreads=NTHREADS)
    check_invariants(s, gt[idx], gn[idx])
    check_bound(compare(s, gt[idx], gn[idx], rt, rn, tr))


def test_error_sequences():
    c = synth.make_lmhead_case(6, 3, 700, 64, "f32", recipe="grid", seed=4, T=(1.0,))
    c.temperature[1] = np.nan
    c.tokens[2, 1] = 700                       # token out of range
    c.hidden[3, 2, 5] = 0x7FC0                 # NaN in a target hidden state
    c.draft[4, 0, 17] = np.inf                 # +inf in a draft row
    gt, gn = run(c)
    rt, rn, _ = oracle.verify_lmhead(c.hidden, c.lm_head, c.draft, c.tokens, c.u_accept,
                                     c.u_resample, c.temperature)
    assert np.array_equal(gn, rn) and np.array_equal(gt, rt)
    assert list(gn[1:5]) == [-1, -1, -1, -1] and gn[0] >= 0 and gn[5] >= 0


def test_deterministic_with_garbage_workspace():
    c = synth.make_lmhead_case(12, 4, 2000, 256, "bf16", recipe="gauss", seed=8, T=(1.0, 0.0))
    need = sv.spec_verify_lmhead_workspace_size(c.B, c.k, c.V, c.d, sv.SPEC_BF16)
    ws = torch.randint(0, 256, (need,), dtype=torch.uint8, device="cuda")
    ws[:256] = 0
    a = run(c, ws=ws)
    b = run(c, ws=ws)
    assert all(np.array_equal(x, y) for x, y in zip(a, b))
    assert sv.spec_verify_read_status(ws) == sv.SPEC_DEV_OK


def test_bad_sizes_are_rejected():
    c = synth.make_lmhead_case(2, 2, 300, 64, "f32", recipe="grid", seed=1)
    dev = to_device(c)
    bad = dict(dev, hidden=torch.zeros((2, 3, 96), dtype=torch.bfloat16, device="cuda"),
               lm_head=torch.zeros((300, 96), dtype=torch.bfloat16, device="cuda"))
    with pytest.raises(sv.SpecVerifyError):
        sv.spec_verify_lmhead(**bad)  # d = 96 is not a multiple of 64
    assert sv.spec_verify_lmhead_workspace_size(2, 32, 300, 64, sv.SPEC_F32) == 0


def test_explicit_side_stream():
    """Called on a stream other than the current one, with no workspace given:
    the binding zero-fills its workspace (and the product's status word) on
    that stream, so the kernels see them zeroed."""
    c = synth.make_lmhead_case(20, 3, 3000, 256, "bf16", recipe="grid", seed=13, T=(0.0, 1.0))
    d = to_device(c)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    out = sv.spec_verify_lmhead(**d, stream=side)
    logits, status = sv.spec_lmhead_logits(d["hidden"].view(-1, c.d), d["lm_head"], stream=side)
    side.synchronize()
    gt, gn = (x.cpu().numpy() for x in out)
    rt, rn, tr = oracle.verify_lmhead(c.hidden, c.lm_head, c.draft, c.tokens, c.u_accept,
                                      c.u_resample, c.temperature, nthreads=NTHREADS)
    check_invariants(c, gt, gn)
    check_bound(compare(c, gt, gn, rt, rn, tr))
    # grid inputs: every logit is exact in fp32
    want = oracle.lmhead_logits(c.hidden, c.lm_head).reshape(-1, c.V)
    assert int(status.item()) == 0
    assert np.array_equal(logits.cpu().numpy().astype(np.float64), want)
