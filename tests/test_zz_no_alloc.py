"""spec_verify_noalloc: the entry point for callers that cannot allocate device
memory when they verify (a plugin given no memory by its host runtime, a
loop that must not call cudaMalloc).  It runs the same kernels on the
library's own fixed scratch array instead of a caller workspace.

Its outputs must equal spec_verify's exactly (integers), on consecutive calls
whose shapes differ, so that whatever the previous call left in the shared
scratch cannot leak into the next one, and they must agree with the fp64
oracle like spec_verify's.  A kernel that gave up on a bounded wait must be
visible through spec_verify_noalloc_read_status (the caller has no workspace
pointer to read).  Kept in a file of its own, collected last, and independent
of every other test: it passes alone or after them.
"""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
import speculative_decoding_verification_65_gb300 as sv  # noqa: E402
from speculative_decoding_verification_65_gb300 import synth  # noqa: E402
from tests import parity_util as pu  # noqa: E402


def _both(case):
    d = sv.to_device(case)
    ref_t, ref_n = sv.spec_verify(**d)
    out_t = torch.full((case.B, case.k + 1), -7, dtype=torch.int32, device="cuda")
    out_n = torch.full((case.B,), -7, dtype=torch.int32, device="cuda")
    sv.spec_verify_noalloc(**d, out_tokens=out_t, out_num_accepted=out_n)
    torch.cuda.synchronize()
    return (ref_t.cpu().numpy(), ref_n.cpu().numpy()), (out_t.cpu().numpy(), out_n.cpu().numpy())


def test_noalloc_matches_spec_verify_on_consecutive_calls():
    assert torch.cuda.is_available()
    cases = [
        synth.make_config(2),                                            # bf16, B=32, k=5, V=32000
        synth.gauss_case(B=6, k=8, V=151936, dtype="f32", seed=5, T=(0.0, 0.7, 1.3)),
    ]
    for case in cases:  # two calls in a row through the shared scratch
        (rt, rn), (gt, gn) = _both(case)
        np.testing.assert_array_equal(gn, rn)
        np.testing.assert_array_equal(gt, rt)
        assert np.all(gn >= 0)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    lib = sv.library()
    cap = sv.spec_verify_noalloc_max_bytes()
    assert cap == 8 << 20
    B, k, V = 8192, 32, 151936  # needs far more than the fixed scratch
    assert sv.spec_verify_workspace_size(B, k, V, sv.SPEC_F32) > cap
    fake = [ctypes.c_void_p(0x100000 * (i + 1)) for i in range(8)]
    rc = lib.spec_verify_noalloc(*fake, B, k, V, sv.SPEC_F32, None)
    assert rc == sv.SPEC_ENOSPACE


def _noalloc(case):
    d = sv.to_device(case)
    out_t = torch.full((case.B, case.k + 1), -7, dtype=torch.int32, device="cuda")
    out_n = torch.full((case.B,), -7, dtype=torch.int32, device="cuda")
    sv.spec_verify_noalloc(**d, out_tokens=out_t, out_num_accepted=out_n)
    torch.cuda.synchronize()
    return out_t.cpu().numpy(), out_n.cpu().numpy()


def test_noalloc_matches_the_oracle():
    """The scratch-array path against the fp64 oracle directly, with the same
    exemption bound as spec_verify (workloads 1 and 3: fp32 and bf16)."""
    for case in (synth.make_config(1), synth.make_config(3, B=24)):
        g_t, g_n = _noalloc(case)
        r_t, r_n, tr = oracle.verify(case.target, case.draft, case.tokens, case.u_accept,
                                     case.u_resample, case.temperature)
        pu.check_invariants(case, g_t, g_n)
        rep = pu.compare(case, g_t, g_n, r_t, r_n, tr)
        pu.check_bound(rep)
        assert sv.spec_verify_noalloc_read_status() == sv.SPEC_DEV_OK


def test_noalloc_status_reports_a_timed_out_wait():
    """The bounded wait of the rings, run on the noalloc scratch with a 1 ms
    limit on an mbarrier nothing arrives at: the status reads
    SPEC_DEV_WAIT_TIMEOUT until the next spec_verify_noalloc call, which clears
    it and verifies normally (no fault, the context stays usable)."""
    sv.spec_selftest_wait_timeout_noalloc(1_000_000)
    torch.cuda.synchronize()
    assert sv.spec_verify_noalloc_read_status() == sv.SPEC_DEV_WAIT_TIMEOUT
    case = synth.make_config(1)
    g_t, g_n = _noalloc(case)
    assert sv.spec_verify_noalloc_read_status() == sv.SPEC_DEV_OK
    r_t, r_n, _ = oracle.verify(case.target, case.draft, case.tokens, case.u_accept,
                                case.u_resample, case.temperature)
    np.testing.assert_array_equal(g_n, r_n)
    np.testing.assert_array_equal(g_t, r_t)
