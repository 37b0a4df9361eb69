"""The Python binding's argument checks, on the CPU.

The binding passes raw pointers and sizes to the C library, so it checks
every tensor first. Inputs must have the shapes and dtypes the call
implies. Caller-supplied outputs must be contiguous, of the call's shape and
dtype, and on the inputs' device, because the kernels write every element.
The workspace and the host-path arena must be contiguous uint8 device
tensors. Any mismatch raises ValueError before the library is called.
"""
import pytest

torch = pytest.importorskip("torch")

import speculative_decoding_verification_65_gb300 as sv  # noqa: E402


def _host_inputs(B=3, k=2, V=50):
    return dict(target=torch.zeros((B, k + 1, V)), draft=torch.zeros((B, k, V)),
                tokens=torch.zeros((B, k), dtype=torch.int32),
                u_accept=torch.zeros((B, k)), u_resample=torch.zeros(B),
                temperature=torch.ones(B))


@pytest.mark.parametrize("name,bad", [
    ("draft", torch.zeros((3, 3, 50))), ("tokens", torch.zeros((3, 1), dtype=torch.int32)),
    ("tokens", torch.zeros((3, 2), dtype=torch.int64)), ("u_accept", torch.zeros((3, 3))),
    ("u_resample", torch.zeros(4)), ("temperature", torch.ones(2)),
])
def test_host_entry_rejects_mismatched_inputs(name, bad):
    x = _host_inputs()
    x[name] = bad
    with pytest.raises(ValueError):
        sv.spec_verify_host(**x, arena=torch.zeros(1, dtype=torch.uint8))


class _FakeCuda:
    """Stands in for a CUDA tensor in the binding's argument checks."""

    def __init__(self, shape, dtype, device="cuda:0", contiguous=True):
        self.shape, self.dtype = torch.Size(shape), dtype
        self.device, self.is_cuda = torch.device(device), True
        self._contiguous = contiguous

    def is_contiguous(self):
        return self._contiguous

    def data_ptr(self):
        return 0x10000

    def dim(self):
        return len(self.shape)

    def numel(self):
        n = 1
        for x in self.shape:
            n *= int(x)
        return n


ARENA = _FakeCuda((1 << 20,), torch.uint8)


@pytest.mark.parametrize("out_t,out_n", [
    (torch.zeros((3, 2), dtype=torch.int32), torch.zeros(3, dtype=torch.int32)),
    (torch.zeros((3, 3), dtype=torch.int32), torch.zeros(3, dtype=torch.int64)),
    (torch.zeros((3, 3), dtype=torch.int32), torch.zeros(4, dtype=torch.int32)),
    (_FakeCuda((3, 3), torch.int32), torch.zeros(3, dtype=torch.int32)),
])
def test_host_entry_rejects_mismatched_outputs(out_t, out_n):
    with pytest.raises(ValueError):
        sv.spec_verify_host(**_host_inputs(), arena=ARENA, out_tokens=out_t,
                            out_num_accepted=out_n)


def test_host_entries_need_a_device_arena():
    with pytest.raises(ValueError):
        sv.spec_verify_host(**_host_inputs(), arena=torch.zeros(1 << 20, dtype=torch.uint8))
    with pytest.raises(ValueError):
        sv.spec_sample_host(torch.zeros((4, 50)), torch.zeros(4), torch.ones(4),
                            arena=torch.zeros(1 << 20, dtype=torch.uint8))
    with pytest.raises(ValueError):  # u of the wrong length
        sv.spec_sample_host(torch.zeros((4, 50)), torch.zeros(5), torch.ones(4), arena=ARENA)
    with pytest.raises(ValueError):  # an output of the wrong length
        sv.spec_sample_host(torch.zeros((4, 50)), torch.zeros(4), torch.ones(4), arena=ARENA,
                            out=torch.zeros(3, dtype=torch.int32))


def test_output_and_workspace_checks():
    dev = torch.device("cuda:0")
    sv._dev_out("out", _FakeCuda((4, 3), torch.int32), (4, 3), torch.int32, dev)
    for bad in (_FakeCuda((4, 2), torch.int32), _FakeCuda((4, 3), torch.int64),
                _FakeCuda((4, 3), torch.int32, "cuda:1"),
                _FakeCuda((4, 3), torch.int32, contiguous=False),
                torch.zeros((4, 3), dtype=torch.int32)):
        with pytest.raises(ValueError):
            sv._dev_out("out", bad, (4, 3), torch.int32, dev)
    sv._check_ws(_FakeCuda((1 << 20,), torch.uint8), dev)
    for bad in (_FakeCuda((1 << 20,), torch.float32), _FakeCuda((1 << 20,), torch.uint8, "cuda:1"),
                torch.zeros(1 << 20, dtype=torch.uint8)):
        with pytest.raises(ValueError):
            sv._check_ws(bad, dev)


def test_library_calls_run_with_the_tensors_device_current(monkeypatch):
    """The C library takes the device from the CUDA runtime's current device
    (its per-device caches and the noalloc scratch address are keyed by it),
    so the binding makes every call with the tensors' device current: here a
    call on cuda:1 tensors enters that device around the library call."""
    seen = []

    class Rec:
        def __init__(self, dev):
            self.dev = str(dev)

        def __enter__(self):
            seen.append(("enter", self.dev))

        def __exit__(self, *exc):
            seen.append(("exit", self.dev))

    class Lib:
        def spec_verify(self, *args):
            seen.append(("call", None))
            return sv.SPEC_OK

    monkeypatch.setattr(sv, "_on", lambda d: Rec(d))
    monkeypatch.setattr(sv, "library", lambda: Lib())
    monkeypatch.setattr(sv, "_stream_handle", lambda s, d: None)
    B, k, V, dev = 3, 2, 50, "cuda:1"
    x = dict(target=_FakeCuda((B, k + 1, V), torch.float32, dev),
             draft=_FakeCuda((B, k, V), torch.float32, dev),
             tokens=_FakeCuda((B, k), torch.int32, dev),
             u_accept=_FakeCuda((B, k), torch.float32, dev),
             u_resample=_FakeCuda((B,), torch.float32, dev),
             temperature=_FakeCuda((B,), torch.float32, dev))
    sv.spec_verify(**x, out_tokens=_FakeCuda((B, k + 1), torch.int32, dev),
                   out_num_accepted=_FakeCuda((B,), torch.int32, dev),
                   ws=_FakeCuda((1 << 20,), torch.uint8, dev))
    assert seen == [("enter", "cuda:1"), ("call", None), ("exit", "cuda:1")]
