"""spec_verify_noalloc: the entry point for callers that cannot allocate device
memory when they verify (a plugin given no memory by its host runtime, a
loop that must not call cudaMalloc).  It runs the same kernels on the
library's own fixed scratch array instead of a caller workspace.

Its outputs must equal spec_verify's exactly (integers), on consecutive calls
whose shapes differ, so that whatever the previous call left in the shared
scratch cannot leak into the next one.  Kept in a file of its own, collected
last, and independent of every other test: it passes alone or after them.
"""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import speculative_decoding_verification_65_gb300 as sv  # noqa: E402
from speculative_decoding_verification_65_gb300 import synth  # noqa: E402


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
