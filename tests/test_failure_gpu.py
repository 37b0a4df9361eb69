"""Failure detection without a GPU fault: the bounded wait every ring uses
gives up, records SPEC_DEV_WAIT_TIMEOUT in the workspace status word, and
leaves the context usable.

spec_selftest_wait_timeout runs the rings' own bounded wait on an mbarrier
that nothing arrives at (a flag that nothing sets), with a 1 ms limit.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
import speculative_decoding_verification_65_gb300 as sv  # noqa: E402
from speculative_decoding_verification_65_gb300 import synth  # noqa: E402


def test_wait_times_out_records_status_and_context_survives():
    case = synth.make_config(1)
    d = sv.to_device(case)
    need = sv.spec_verify_workspace_size(case.B, case.k, case.V, sv.SPEC_F32)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    assert sv.spec_verify_read_status(ws) == sv.SPEC_DEV_OK

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    sv.spec_selftest_wait_timeout(ws, 1_000_000)  # 1 ms
    e1.record()
    torch.cuda.synchronize()
    waited_ms = e0.elapsed_time(e1)
    assert 0.9 <= waited_ms < 100.0, waited_ms
    assert sv.spec_verify_read_status(ws) == sv.SPEC_DEV_WAIT_TIMEOUT

    # the status word stays set until the caller resets it; the context is fine
    sv.spec_verify_workspace_reset(ws)
    toks, n = sv.spec_verify(**d, ws=ws)
    torch.cuda.synchronize()
    assert sv.spec_verify_read_status(ws) == sv.SPEC_DEV_OK
    rt, rn, _ = oracle.verify(case.target, case.draft, case.tokens, case.u_accept,
                              case.u_resample, case.temperature)
    assert np.array_equal(n.cpu().numpy(), rn) and np.array_equal(toks.cpu().numpy(), rt)
