"""Parity of the LM-head-fused verification (spec_verify_lmhead) and of its
tensor-core product (spec_lmhead_logits) with the fp64 oracle.

On the grid recipe every partial sum of h.W is exact in fp32, so the GPU's
logits equal the oracle's and the integer outputs must match with the usual
1e-5 exemption band.  On the gauss recipe the fp32 accumulation rounds: the
product is checked against a bound on that rounding, and the decisions get a
band widened by its effect on the probabilities.
"""
import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
import speculative_decoding_verification_65_gb300 as sv  # noqa: E402
from speculative_decoding_verification_65_gb300 import synth  # noqa: E402
from tests.parity_util import compare, check_invariants  # noqa: E402

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
    assert rep["exempt"] <= max(1, rep["decisions"] // 1000), rep


def test_probs_equal_the_oracle_on_the_grid():
    c = synth.make_lmhead_case(16, 4, 4000, 512, "bf16", recipe="grid", seed=9, T=(0.8, 1.0))
    _, _, probs = run(c, want_probs=True)
    t = oracle.lmhead_logits(c.hidden, c.lm_head).astype(np.float32)
    d32 = synth.bf16_bits_to_f32(c.draft)
    PQ = oracle.probs(t, d32, c.tokens, c.temperature)
    np.testing.assert_allclose(probs[..., 0], PQ[..., 0], rtol=1e-5, atol=1e-30)
    np.testing.assert_allclose(probs[..., 1], PQ[..., 1], rtol=1e-5, atol=1e-30)


def test_parity_gauss_with_widened_band():
    # fp32 rounding of the logits moves P and Q by at most about 2 log(2) c
    # times the rounding bound (numerator and normaliser); the band is that
    # relative change, taken over the batch's largest bound
    B, k, V, d = 32, 4, 8000, 1024
    c = synth.make_lmhead_case(B, k, V, d, "bf16", recipe="gauss", seed=21, T=(1.0,))
    gt, gn = run(c)
    rt, rn, tr = oracle.verify_lmhead(c.hidden, c.lm_head, c.draft, c.tokens, c.u_accept,
                                      c.u_resample, c.temperature, nthreads=NTHREADS)
    eps = float(rounding_bound(c.hidden.reshape(-1, d), c.lm_head).max())
    band = max(1e-5, 4.0 * eps / float(np.min(c.temperature)))
    assert band < 0.01
    check_invariants(c, gt, gn)
    rep = compare(c, gt, gn, rt, rn, tr, band=band)
    assert rep["exempt"] <= max(1, rep["draws"] // 50), rep


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
    rep = compare(c, gt, gn, rt, rn, tr)
    assert rep["exempt"] <= max(1, rep["decisions"] // 1000), rep
    # grid inputs: every logit is exact in fp32
    want = oracle.lmhead_logits(c.hidden, c.lm_head).reshape(-1, c.V)
    assert int(status.item()) == 0
    assert np.array_equal(logits.cpu().numpy().astype(np.float64), want)
