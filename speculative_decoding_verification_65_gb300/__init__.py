"""GB300-native batched speculative-sampling verification.

Thin Python binding over the C ABI of ``libspecverify.so`` (declared in
``include/spec_verify.h``, ``include/spec_sample.h`` and
``include/spec_lmhead.h``, ``include/spec_tree.h``).  Every function here only checks and marshals
arguments (shapes, dtypes, device pointers, the current CUDA stream) and calls
the function of the same name in the library; all arithmetic runs in the CUDA
kernels.  PyTorch is used for device memory and streams only.

If the library has not been built the first call raises: there is no CPU
fallback.  Build it with ``__graft_entry__.build()`` (or
``python -m speculative_decoding_verification_65_gb300.build``).
"""
from __future__ import annotations

import ctypes
import os
import threading

SPEC_F32 = 0
SPEC_BF16 = 1
SPEC_OK = 0
SPEC_EINVAL = 1
SPEC_ECUDA = 2
SPEC_ENOSPACE = 3
SPEC_DEV_OK = 0
SPEC_DEV_WAIT_TIMEOUT = 1
SPEC_MAX_K = 32
SPEC_MAX_V = 1 << 20
SPEC_STAGES = 5
SPEC_SAMPLE_STAGES = 3
SPEC_FILTERED_STAGES = 6
SPEC_LMHEAD_STAGES = 5
SPEC_TREE_MAX_NODES = 1024

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libspecverify.so")
_lib = None
_lock = threading.Lock()


class SpecVerifyError(RuntimeError):
    pass


def library():
    """The loaded ctypes library (raises if it was never built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise SpecVerifyError(
                f"{LIB_PATH} is missing: build the CUDA library first "
                "(__graft_entry__.build()); there is no fallback")
        lib = ctypes.CDLL(LIB_PATH)
        vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
        lib.spec_verify_abi_version.restype = i32
        lib.spec_verify_abi_version.argtypes = []
        lib.spec_verify_strerror.restype = ctypes.c_char_p
        lib.spec_verify_strerror.argtypes = [i32]
        lib.spec_verify_workspace_size.restype = sz
        lib.spec_verify_workspace_size.argtypes = [i32, i32, i32, i32]
        lib.spec_verify_workspace_reset.restype = i32
        lib.spec_verify_workspace_reset.argtypes = [vp, sz, vp]
        lib.spec_verify.restype = i32
        lib.spec_verify.argtypes = [vp] * 8 + [i32] * 4 + [vp, sz, vp]
        lib.spec_verify_probs.restype = i32
        lib.spec_verify_probs.argtypes = [vp] * 9 + [i32] * 4 + [vp, sz, vp]
        lib.spec_verify_trace.restype = i32
        lib.spec_verify_trace.argtypes = [vp] * 10 + [i32] * 5 + [vp, sz, vp]
        lib.spec_verify_timed.restype = i32
        lib.spec_verify_timed.argtypes = [vp] * 8 + [i32] * 4 + [vp, sz, vp, vp]
        lib.spec_verify_filtered.restype = i32
        lib.spec_verify_filtered.argtypes = [vp] * 11 + [i32] * 4 + [vp, sz, vp]
        lib.spec_verify_filtered_timed.restype = i32
        lib.spec_verify_filtered_timed.argtypes = [vp] * 10 + [i32] * 4 + [vp, sz, vp, vp]
        lib.spec_verify_noalloc.restype = i32
        lib.spec_verify_noalloc.argtypes = [vp] * 8 + [i32] * 4 + [vp]
        lib.spec_verify_noalloc_max_bytes.restype = sz
        lib.spec_verify_noalloc_max_bytes.argtypes = []
        lib.spec_verify_read_status.restype = i32
        lib.spec_verify_read_status.argtypes = [vp, vp, vp]
        lib.spec_verify_host_arena_size.restype = sz
        lib.spec_verify_host_arena_size.argtypes = [i32, i32, i32, i32]
        lib.spec_verify_host.restype = i32
        lib.spec_verify_host.argtypes = [vp] * 8 + [i32] * 4 + [vp, sz, vp]
        lib.spec_sample_workspace_size.restype = sz
        lib.spec_sample_workspace_size.argtypes = [i32, i32, i32]
        lib.spec_sample.restype = i32
        lib.spec_sample.argtypes = [vp] * 4 + [i32] * 3 + [vp, sz, vp]
        lib.spec_sample_timed.restype = i32
        lib.spec_sample_timed.argtypes = [vp] * 4 + [i32] * 3 + [vp, sz, vp, vp]
        lib.spec_sample_host_arena_size.restype = sz
        lib.spec_sample_host_arena_size.argtypes = [i32, i32, i32]
        lib.spec_sample_host.restype = i32
        lib.spec_sample_host.argtypes = [vp] * 4 + [i32] * 3 + [vp, sz, vp]
        lib.spec_bench_read.restype = i32
        lib.spec_bench_read.argtypes = [vp, sz, vp, vp]
        lib.spec_bench_read_sink_words.restype = i32
        lib.spec_bench_read_sink_words.argtypes = []
        lib.spec_selftest_wait_timeout.restype = i32
        lib.spec_selftest_wait_timeout.argtypes = [vp, ctypes.c_uint64, vp]
        lib.spec_selftest_wait_timeout_noalloc.restype = i32
        lib.spec_selftest_wait_timeout_noalloc.argtypes = [ctypes.c_uint64, vp]
        lib.spec_verify_noalloc_read_status.restype = i32
        lib.spec_verify_noalloc_read_status.argtypes = [vp, vp]
        lib.spec_verify_lmhead_workspace_size.restype = sz
        lib.spec_verify_lmhead_workspace_size.argtypes = [i32] * 5
        lib.spec_verify_lmhead.restype = i32
        lib.spec_verify_lmhead.argtypes = [vp] * 9 + [i32] * 5 + [vp, sz, vp]
        lib.spec_verify_lmhead_timed.restype = i32
        lib.spec_verify_lmhead_timed.argtypes = [vp] * 10 + [i32] * 5 + [vp, sz, vp, vp]
        lib.spec_lmhead_logits.restype = i32
        lib.spec_lmhead_logits.argtypes = [vp, vp, vp, i32, i32, i32, vp, vp]
        lib.spec_verify_filtered_workspace_size.restype = sz
        lib.spec_verify_filtered_workspace_size.argtypes = [i32, i32, i32, i32]
        lib.spec_verify_tree.restype = i32
        lib.spec_verify_tree.argtypes = [vp] * 11 + [i32] * 4 + [vp]
        _lib = lib
        return lib


def _check(rc: int, what: str):
    if rc != SPEC_OK:
        msg = library().spec_verify_strerror(rc).decode()
        raise SpecVerifyError(f"{what} failed: {msg} (status {rc})")


def _torch():
    import torch
    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.float32:
        return SPEC_F32
    if t.dtype == torch.bfloat16:
        return SPEC_BF16
    raise TypeError(f"logits must be float32 or bfloat16, got {t.dtype}")


def _on(device):
    """The library takes the device from the CUDA runtime's current device, so
    every call is made with the tensors' device current."""
    return _torch().cuda.device(device)


def _stream_handle(stream, device):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def spec_verify_abi_version() -> int:
    return int(library().spec_verify_abi_version())


def spec_verify_workspace_size(B: int, k: int, V: int, dtype: int) -> int:
    return int(library().spec_verify_workspace_size(B, k, V, dtype))


def spec_verify_host_arena_size(B: int, k: int, V: int, dtype: int) -> int:
    return int(library().spec_verify_host_arena_size(B, k, V, dtype))


_ws_cache = {}


def workspace(B: int, k: int, V: int, dtype: int, device=None, stream=None):
    """A zeroed workspace tensor big enough for these sizes, cached per
    (device, stream): calls in flight on one stream run in order, so they can
    share it."""
    torch = _torch()
    device = torch.device(device if device is not None else "cuda")
    if device.index is None:
        device = torch.device("cuda", torch.cuda.current_device())
    s = stream if stream is not None else torch.cuda.current_stream(device)
    need = spec_verify_workspace_size(B, k, V, dtype)
    if need == 0:
        raise ValueError(f"sizes out of range: B={B} k={k} V={V} dtype={dtype}")
    return _cached_workspace(need, device, s)


def spec_verify_filtered_workspace_size(B: int, k: int, V: int, dtype: int) -> int:
    return int(library().spec_verify_filtered_workspace_size(B, k, V, dtype))


def filtered_workspace(B: int, k: int, V: int, dtype: int, device=None, stream=None):
    """workspace() with room for the top-k cut from group maxima
    (spec_verify_filtered_workspace_size)."""
    torch = _torch()
    device = torch.device(device if device is not None else "cuda")
    if device.index is None:
        device = torch.device("cuda", torch.cuda.current_device())
    s = stream if stream is not None else torch.cuda.current_stream(device)
    need = spec_verify_filtered_workspace_size(B, k, V, dtype)
    if need == 0:
        raise ValueError(f"sizes out of range: B={B} k={k} V={V} dtype={dtype}")
    return _cached_workspace(need, device, s)


def _cached_workspace(need: int, device, s):
    torch = _torch()
    key = (device.index, s.cuda_stream)
    ws = _ws_cache.get(key)
    if ws is None or ws.numel() < need:
        with torch.cuda.stream(s):
            ws = torch.zeros(max(need, 1 << 20), dtype=torch.uint8, device=device)
        _ws_cache[key] = ws
    return ws


def spec_verify_workspace_reset(ws, stream=None):
    with _on(ws.device):
        _check(library().spec_verify_workspace_reset(_ptr(ws), ws.numel(),
                                                     _stream_handle(stream, ws.device)),
               "spec_verify_workspace_reset")


def spec_verify_read_status(ws, stream=None) -> int:
    st = ctypes.c_int32(-99)
    with _on(ws.device):
        _check(library().spec_verify_read_status(_ptr(ws), ctypes.byref(st),
                                                 _stream_handle(stream, ws.device)),
               "spec_verify_read_status")
    return int(st.value)


def _shapes(target, draft, tokens, u_accept, u_resample, temperature):
    """Shapes and dtypes of the verification inputs: (B, k, V, dtype code)."""
    torch = _torch()
    if target.dim() != 3 or draft.dim() != 3:
        raise ValueError("target must be [B,k+1,V] and draft [B,k,V]")
    B, k1, V = target.shape
    k = k1 - 1
    if tuple(draft.shape) != (B, k, V):
        raise ValueError(f"draft shape {tuple(draft.shape)} != {(B, k, V)}")
    dt = _dtype_code(target)
    if draft.dtype != target.dtype:
        raise TypeError("target and draft must share a dtype")
    for name, t, shape, dtype in (("draft_tokens", tokens, (B, k), torch.int32),
                                  ("u_accept", u_accept, (B, k), torch.float32),
                                  ("u_resample", u_resample, (B,), torch.float32),
                                  ("temperature", temperature, (B,), torch.float32)):
        if tuple(t.shape) != shape or t.dtype != dtype:
            raise ValueError(f"{name} must be {dtype} {shape}, got {t.dtype} {tuple(t.shape)}")
    return B, k, V, dt


def _check_out(name, t, shape, dtype):
    if tuple(t.shape) != shape or t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {dtype} {shape} tensor, "
                         f"got {t.dtype} {tuple(t.shape)}")


def _dev_out(name, t, shape, dtype, dev):
    """A caller-supplied output: contiguous, of the call's shape and dtype, on
    the inputs' device (the kernels write every element of it)."""
    _check_out(name, t, shape, dtype)
    if not t.is_cuda or t.device != dev:
        raise ValueError(f"{name} must be on {dev}, got {t.device}")


def _check_ws(ws, dev):
    torch = _torch()
    if not ws.is_cuda or ws.device != dev or ws.dtype != torch.uint8 or not ws.is_contiguous():
        raise ValueError(f"ws must be a contiguous uint8 tensor on {dev}")


def _marshal(target, draft, tokens, u_accept, u_resample, temperature):
    B, k, V, dt = _shapes(target, draft, tokens, u_accept, u_resample, temperature)
    for t in (target, draft, tokens, u_accept, u_resample, temperature):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("all inputs must be contiguous CUDA tensors")
        if t.device != target.device:
            raise ValueError("all inputs must be on one device")
    return B, k, V, dt


def spec_verify(target, draft, tokens, u_accept, u_resample, temperature,
                out_tokens=None, out_num_accepted=None, ws=None, stream=None):
    """Run the verification step on the current (or given) stream.

    target [B,k+1,V] and draft [B,k,V]: float32 or bfloat16 CUDA tensors;
    tokens int32 [B,k]; u_accept float32 [B,k]; u_resample, temperature
    float32 [B].  Returns (out_tokens int32 [B,k+1], out_num_accepted int32
    [B]); asynchronous like any CUDA op."""
    torch = _torch()
    B, k, V, dt = _marshal(target, draft, tokens, u_accept, u_resample, temperature)
    dev = target.device
    if out_tokens is None:
        out_tokens = torch.empty((B, k + 1), dtype=torch.int32, device=dev)
    if out_num_accepted is None:
        out_num_accepted = torch.empty((B,), dtype=torch.int32, device=dev)
    _dev_out("out_tokens", out_tokens, (B, k + 1), torch.int32, dev)
    _dev_out("out_num_accepted", out_num_accepted, (B,), torch.int32, dev)
    if ws is None:
        ws = workspace(B, k, V, dt, dev, stream)
    _check_ws(ws, dev)
    with _on(dev):
        rc = library().spec_verify(_ptr(target), _ptr(draft), _ptr(tokens), _ptr(u_accept),
                                   _ptr(u_resample), _ptr(temperature), _ptr(out_tokens),
                                   _ptr(out_num_accepted), B, k, V, dt, _ptr(ws), ws.numel(),
                                   _stream_handle(stream, dev))
    _check(rc, "spec_verify")
    return out_tokens, out_num_accepted


def _filters(B, dev, top_k, top_p):
    torch = _torch()
    for name, t, dtype in (("top_k", top_k, torch.int32), ("top_p", top_p, torch.float32)):
        if t is not None and (tuple(t.shape) != (B,) or t.dtype != dtype or not t.is_cuda
                              or not t.is_contiguous() or t.device != dev):
            raise ValueError(f"{name} must be a contiguous {dtype} CUDA tensor of shape ({B},)")


def spec_verify_filtered(target, draft, tokens, u_accept, u_resample, temperature,
                         top_k=None, top_p=None, out_tokens=None, out_num_accepted=None,
                         want_probs=False, ws=None, stream=None):
    """spec_verify with top-k / top-p filtered distributions (see
    include/spec_verify.h): top_k int32 [B] (0 = none), top_p float32 [B]
    (>= 1 = none), either may be None.  Returns (out_tokens, out_num_accepted)
    and, with want_probs, the filtered P, Q [B, k, 2] as a third value."""
    torch = _torch()
    B, k, V, dt = _marshal(target, draft, tokens, u_accept, u_resample, temperature)
    dev = target.device
    _filters(B, dev, top_k, top_p)
    if out_tokens is None:
        out_tokens = torch.empty((B, k + 1), dtype=torch.int32, device=dev)
    if out_num_accepted is None:
        out_num_accepted = torch.empty((B,), dtype=torch.int32, device=dev)
    _dev_out("out_tokens", out_tokens, (B, k + 1), torch.int32, dev)
    _dev_out("out_num_accepted", out_num_accepted, (B,), torch.int32, dev)
    probs = torch.empty((B, k, 2), dtype=torch.float32, device=dev) if want_probs else None
    if ws is None:
        ws = filtered_workspace(B, k, V, dt, dev, stream)
    _check_ws(ws, dev)
    with _on(dev):
        rc = library().spec_verify_filtered(_ptr(target), _ptr(draft), _ptr(tokens), _ptr(u_accept),
                                            _ptr(u_resample), _ptr(temperature), _ptr(top_k),
                                            _ptr(top_p), _ptr(out_tokens), _ptr(out_num_accepted),
                                            _ptr(probs), B, k, V, dt, _ptr(ws), ws.numel(),
                                            _stream_handle(stream, dev))
    _check(rc, "spec_verify_filtered")
    if want_probs:
        return out_tokens, out_num_accepted, probs
    return out_tokens, out_num_accepted


def spec_verify_filtered_timed(target, draft, tokens, u_accept, u_resample, temperature,
                               top_k, top_p, out_tokens, out_num_accepted, ws, stage_events,
                               stream=None):
    """spec_verify_filtered recording SPEC_FILTERED_STAGES events: after the
    statistics, the filter (all of its kernels), the accept scan, the draw
    tiles, the final search and the exact draws."""
    torch = _torch()
    B, k, V, dt = _marshal(target, draft, tokens, u_accept, u_resample, temperature)
    dev = target.device
    _filters(B, dev, top_k, top_p)
    _dev_out("out_tokens", out_tokens, (B, k + 1), torch.int32, dev)
    _dev_out("out_num_accepted", out_num_accepted, (B,), torch.int32, dev)
    _check_ws(ws, dev)
    handles = (ctypes.c_void_p * SPEC_FILTERED_STAGES)(
        *[ctypes.c_void_p(e.cuda_event) for e in stage_events])
    with _on(target.device):
        rc = library().spec_verify_filtered_timed(
            _ptr(target), _ptr(draft), _ptr(tokens), _ptr(u_accept), _ptr(u_resample),
            _ptr(temperature), _ptr(top_k), _ptr(top_p), _ptr(out_tokens), _ptr(out_num_accepted),
            B, k, V, dt, _ptr(ws), ws.numel(), _stream_handle(stream, target.device), handles)
    _check(rc, "spec_verify_filtered_timed")
    return out_tokens, out_num_accepted


def spec_verify_timed(target, draft, tokens, u_accept, u_resample, temperature,
                      out_tokens, out_num_accepted, ws, stage_events, stream=None):
    """spec_verify recording the given torch.cuda.Event objects (SPEC_STAGES of
    them, recorded once beforehand so that they exist) after each stage:
    statistics, accept scan, draw tiles, final search, exact draws."""
    torch = _torch()
    B, k, V, dt = _marshal(target, draft, tokens, u_accept, u_resample, temperature)
    dev = target.device
    _dev_out("out_tokens", out_tokens, (B, k + 1), torch.int32, dev)
    _dev_out("out_num_accepted", out_num_accepted, (B,), torch.int32, dev)
    _check_ws(ws, dev)
    handles = (ctypes.c_void_p * SPEC_STAGES)(*[ctypes.c_void_p(e.cuda_event) for e in stage_events])
    with _on(target.device):
        rc = library().spec_verify_timed(_ptr(target), _ptr(draft), _ptr(tokens), _ptr(u_accept),
                                         _ptr(u_resample), _ptr(temperature), _ptr(out_tokens),
                                         _ptr(out_num_accepted), B, k, V, dt, _ptr(ws), ws.numel(),
                                         _stream_handle(stream, target.device), handles)
    _check(rc, "spec_verify_timed")
    return out_tokens, out_num_accepted


def spec_verify_noalloc(target, draft, tokens, u_accept, u_resample, temperature,
                        out_tokens, out_num_accepted, stream=None):
    """spec_verify without a workspace, for callers that cannot allocate device
    memory when they verify: the library's own fixed scratch array is used
    instead (see include/spec_verify.h).  The output tensors are supplied by
    the caller, so this wrapper allocates nothing either.  Calls that overlap
    on the GPU share that scratch and race."""
    torch = _torch()
    B, k, V, dt = _marshal(target, draft, tokens, u_accept, u_resample, temperature)
    _dev_out("out_tokens", out_tokens, (B, k + 1), torch.int32, target.device)
    _dev_out("out_num_accepted", out_num_accepted, (B,), torch.int32, target.device)
    with _on(target.device):
        rc = library().spec_verify_noalloc(_ptr(target), _ptr(draft), _ptr(tokens), _ptr(u_accept),
                                           _ptr(u_resample), _ptr(temperature), _ptr(out_tokens),
                                           _ptr(out_num_accepted), B, k, V, dt,
                                           _stream_handle(stream, target.device))
    _check(rc, "spec_verify_noalloc")
    return out_tokens, out_num_accepted


def spec_verify_noalloc_read_status(stream=None, device=None) -> int:
    """The device status word of spec_verify_noalloc's scratch (SPEC_DEV_*)."""
    torch = _torch()
    dev = torch.device(device if device is not None else "cuda")
    if dev.index is None:
        dev = torch.device("cuda", torch.cuda.current_device())
    st = ctypes.c_int32(-99)
    with torch.cuda.device(dev):
        _check(library().spec_verify_noalloc_read_status(ctypes.byref(st),
                                                         _stream_handle(stream, dev)),
               "spec_verify_noalloc_read_status")
    return int(st.value)


def spec_selftest_wait_timeout_noalloc(limit_ns: int, stream=None, device=None):
    """spec_selftest_wait_timeout on spec_verify_noalloc's scratch."""
    torch = _torch()
    dev = torch.device(device if device is not None else "cuda")
    if dev.index is None:
        dev = torch.device("cuda", torch.cuda.current_device())
    with torch.cuda.device(dev):
        _check(library().spec_selftest_wait_timeout_noalloc(int(limit_ns),
                                                            _stream_handle(stream, dev)),
               "spec_selftest_wait_timeout_noalloc")


def spec_verify_noalloc_max_bytes() -> int:
    return int(library().spec_verify_noalloc_max_bytes())


def spec_verify_probs(target, draft, tokens, u_accept, u_resample, temperature,
                      ws=None, stream=None):
    """spec_verify plus the fp32 intermediates P = p_i(g_i), Q = q_i(g_i):
    returns (out_tokens, out_num_accepted, probs [B,k,2])."""
    torch = _torch()
    B, k, V, dt = _marshal(target, draft, tokens, u_accept, u_resample, temperature)
    dev = target.device
    out_tokens = torch.empty((B, k + 1), dtype=torch.int32, device=dev)
    out_n = torch.empty((B,), dtype=torch.int32, device=dev)
    probs = torch.empty((B, k, 2), dtype=torch.float32, device=dev)
    if ws is None:
        ws = workspace(B, k, V, dt, dev, stream)
    _check_ws(ws, dev)
    with _on(dev):
        rc = library().spec_verify_probs(_ptr(target), _ptr(draft), _ptr(tokens), _ptr(u_accept),
                                         _ptr(u_resample), _ptr(temperature), _ptr(out_tokens),
                                         _ptr(out_n), _ptr(probs), B, k, V, dt, _ptr(ws),
                                         ws.numel(), _stream_handle(stream, dev))
    _check(rc, "spec_verify_probs")
    return out_tokens, out_n, probs


def spec_verify_trace(target, draft, tokens, u_accept, u_resample, temperature,
                      resolve_all=False, want_probs=False, ws=None, stream=None):
    """spec_verify with the trace of each draw (include/spec_verify.h):
    returns (out_tokens, out_num_accepted, draw [B,4] int32, probs or None).
    draw[b] = (fp32 token, listed for the exact draw, token written, the fp32
    distance of u to its cell's nearer edge as float32 bits);
    sequences that draw nothing keep -2 everywhere.  resolve_all lists every
    draw."""
    torch = _torch()
    B, k, V, dt = _marshal(target, draft, tokens, u_accept, u_resample, temperature)
    dev = target.device
    out_tokens = torch.empty((B, k + 1), dtype=torch.int32, device=dev)
    out_n = torch.empty((B,), dtype=torch.int32, device=dev)
    draw = torch.full((B, 4), -2, dtype=torch.int32, device=dev)
    probs = torch.empty((B, k, 2), dtype=torch.float32, device=dev) if want_probs else None
    if ws is None:
        ws = workspace(B, k, V, dt, dev, stream)
    _check_ws(ws, dev)
    with _on(dev):
        rc = library().spec_verify_trace(_ptr(target), _ptr(draft), _ptr(tokens), _ptr(u_accept),
                                         _ptr(u_resample), _ptr(temperature), _ptr(out_tokens),
                                         _ptr(out_n), _ptr(probs), _ptr(draw),
                                         1 if resolve_all else 0, B, k, V, dt, _ptr(ws),
                                         ws.numel(), _stream_handle(stream, dev))
    _check(rc, "spec_verify_trace")
    return out_tokens, out_n, draw, probs


def spec_verify_host(target, draft, tokens, u_accept, u_resample, temperature,
                     arena, out_tokens=None, out_num_accepted=None, stream=None):
    """End-to-end call on HOST tensors (CPU, ideally pinned): the library copies
    the inputs into the device `arena` (a CUDA uint8 tensor of at least
    spec_verify_host_arena_size bytes), verifies, copies the outputs back and
    synchronises.  Returns host (out_tokens, out_num_accepted)."""
    torch = _torch()
    B, k, V, dt = _shapes(target, draft, tokens, u_accept, u_resample, temperature)
    for t in (target, draft, tokens, u_accept, u_resample, temperature):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("host inputs must be contiguous CPU tensors")
    if not arena.is_cuda or arena.dtype != torch.uint8 or not arena.is_contiguous():
        raise ValueError("arena must be a contiguous uint8 CUDA tensor")
    for name, t, shape in (("out_tokens", out_tokens, (B, k + 1)),
                           ("out_num_accepted", out_num_accepted, (B,))):
        if t is not None:
            _check_out(name, t, shape, torch.int32)
            if t.is_cuda:
                raise ValueError(f"{name} must be a host tensor")
    if out_tokens is None:
        out_tokens = torch.empty((B, k + 1), dtype=torch.int32, pin_memory=True)
    if out_num_accepted is None:
        out_num_accepted = torch.empty((B,), dtype=torch.int32, pin_memory=True)
    with _on(arena.device):
        rc = library().spec_verify_host(_ptr(target), _ptr(draft), _ptr(tokens), _ptr(u_accept),
                                        _ptr(u_resample), _ptr(temperature), _ptr(out_tokens),
                                        _ptr(out_num_accepted), B, k, V, dt, _ptr(arena),
                                        arena.numel(), _stream_handle(stream, arena.device))
    _check(rc, "spec_verify_host")
    return out_tokens, out_num_accepted


def spec_sample_workspace_size(R: int, V: int, dtype: int) -> int:
    return int(library().spec_sample_workspace_size(R, V, dtype))


def sample_workspace(R: int, V: int, dtype: int, device=None, stream=None):
    """A zeroed workspace for spec_sample, shared with spec_verify's cache for
    the same (device, stream)."""
    torch = _torch()
    device = torch.device(device if device is not None else "cuda")
    if device.index is None:
        device = torch.device("cuda", torch.cuda.current_device())
    s = stream if stream is not None else torch.cuda.current_stream(device)
    need = spec_sample_workspace_size(R, V, dtype)
    if need == 0:
        raise ValueError(f"sizes out of range: R={R} V={V} dtype={dtype}")
    return _cached_workspace(need, device, s)


def _sample_shapes(logits, u, temperature):
    """Shapes and dtypes of the sampling inputs: (R, V, dtype code)."""
    torch = _torch()
    if logits.dim() != 2:
        raise ValueError("logits must be [R, V]")
    R, V = logits.shape
    dt = _dtype_code(logits)
    for name, t in (("u", u), ("temperature", temperature)):
        if tuple(t.shape) != (R,) or t.dtype != torch.float32:
            raise ValueError(f"{name} must be float32 ({R},), got {t.dtype} {tuple(t.shape)}")
    return R, V, dt


def _marshal_sample(logits, u, temperature):
    R, V, dt = _sample_shapes(logits, u, temperature)
    for t in (logits, u, temperature):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("all inputs must be contiguous CUDA tensors")
        if t.device != logits.device:
            raise ValueError("all inputs must be on one device")
    return R, V, dt


def spec_sample(logits, u, temperature, out=None, ws=None, stream=None):
    """One token per row of logits [R, V] (float32 or bfloat16 CUDA tensor)
    from softmax(logits / T) by inverse CDF with the row's uniform u (float32
    [R] in [0, 1)); temperature float32 [R], 0 = argmax.  Returns int32 [R]
    (-1 on a row error); asynchronous like any CUDA op."""
    torch = _torch()
    R, V, dt = _marshal_sample(logits, u, temperature)
    dev = logits.device
    if out is None:
        out = torch.empty((R,), dtype=torch.int32, device=dev)
    _dev_out("out", out, (R,), torch.int32, dev)
    if ws is None:
        ws = sample_workspace(R, V, dt, dev, stream)
    _check_ws(ws, dev)
    with _on(dev):
        rc = library().spec_sample(_ptr(logits), _ptr(u), _ptr(temperature), _ptr(out), R, V, dt,
                                   _ptr(ws), ws.numel(), _stream_handle(stream, dev))
    _check(rc, "spec_sample")
    return out


def spec_sample_timed(logits, u, temperature, out, ws, stage_events, stream=None):
    """spec_sample recording the given torch.cuda.Event objects
    (SPEC_SAMPLE_STAGES of them, recorded once beforehand) after each stage:
    chunk records, pick, exact draws."""
    torch = _torch()
    R, V, dt = _marshal_sample(logits, u, temperature)
    _dev_out("out", out, (R,), torch.int32, logits.device)
    _check_ws(ws, logits.device)
    handles = (ctypes.c_void_p * SPEC_SAMPLE_STAGES)(
        *[ctypes.c_void_p(e.cuda_event) for e in stage_events])
    with _on(logits.device):
        rc = library().spec_sample_timed(_ptr(logits), _ptr(u), _ptr(temperature), _ptr(out), R, V,
                                         dt, _ptr(ws), ws.numel(),
                                         _stream_handle(stream, logits.device), handles)
    _check(rc, "spec_sample_timed")
    return out


def to_device(case, device="cuda"):
    """Copy a synth.Case's host arrays to device tensors (bf16 bit patterns
    become torch.bfloat16)."""
    import numpy as np
    torch = _torch()

    def logits(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)
        return torch.from_numpy(a).to(device)

    return dict(target=logits(case.target), draft=logits(case.draft),
                tokens=torch.from_numpy(case.tokens).to(device),
                u_accept=torch.from_numpy(case.u_accept).to(device),
                u_resample=torch.from_numpy(case.u_resample).to(device),
                temperature=torch.from_numpy(case.temperature).to(device))


def spec_sample_host_arena_size(R: int, V: int, dtype: int) -> int:
    return int(library().spec_sample_host_arena_size(R, V, dtype))


def spec_sample_host(logits, u, temperature, arena, out=None, stream=None):
    """End-to-end call on HOST tensors (CPU, ideally pinned): the library copies
    the inputs into the device `arena` (a CUDA uint8 tensor of at least
    spec_sample_host_arena_size bytes), samples, copies the tokens back and
    synchronises.  Returns the host int32 [R] tokens."""
    torch = _torch()
    R, V, dt = _sample_shapes(logits, u, temperature)
    for t in (logits, u, temperature):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("host inputs must be contiguous CPU tensors")
    if not arena.is_cuda or arena.dtype != torch.uint8 or not arena.is_contiguous():
        raise ValueError("arena must be a contiguous uint8 CUDA tensor")
    if out is not None:
        _check_out("out", out, (R,), torch.int32)
        if out.is_cuda:
            raise ValueError("out must be a host tensor")
    else:
        out = torch.empty((R,), dtype=torch.int32, pin_memory=True)
    with _on(arena.device):
        rc = library().spec_sample_host(_ptr(logits), _ptr(u), _ptr(temperature), _ptr(out), R, V,
                                        dt, _ptr(arena), arena.numel(),
                                        _stream_handle(stream, arena.device))
    _check(rc, "spec_sample_host")
    return out


def spec_bench_read(buf, sink, stream=None):
    """The benchmark's read-only probe over a CUDA tensor `buf` (16-byte
    aligned, size a multiple of 16 bytes); `sink` is an int32 CUDA tensor of
    at least spec_bench_read_sink_words() elements."""
    with _on(buf.device):
        rc = library().spec_bench_read(_ptr(buf), buf.numel() * buf.element_size(), _ptr(sink),
                                       _stream_handle(stream, buf.device))
    _check(rc, "spec_bench_read")


def spec_selftest_wait_timeout(ws, limit_ns: int, stream=None):
    """Launch the bounded-wait self-test on workspace `ws` (see
    include/spec_bench.h); read its outcome with spec_verify_read_status."""
    with _on(ws.device):
        _check(library().spec_selftest_wait_timeout(_ptr(ws), int(limit_ns),
                                                    _stream_handle(stream, ws.device)),
               "spec_selftest_wait_timeout")


def spec_bench_read_sink_words() -> int:
    return int(library().spec_bench_read_sink_words())


def sample_to_device(sc, device="cuda"):
    """Copy a synth.SampleCase's host arrays to device tensors."""
    import numpy as np
    torch = _torch()
    a = sc.logits
    if a.dtype == np.uint16:
        logits = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)
    else:
        logits = torch.from_numpy(a).to(device)
    return dict(logits=logits, u=torch.from_numpy(sc.u).to(device),
                temperature=torch.from_numpy(sc.temperature).to(device))


# ------------------------------------------------ LM-head-fused verification

def spec_verify_lmhead_workspace_size(B: int, k: int, V: int, d: int, draft_dtype: int) -> int:
    return int(library().spec_verify_lmhead_workspace_size(B, k, V, d, draft_dtype))


def _marshal_lmhead(hidden, lm_head, draft, tokens, u_accept, u_resample, temperature):
    torch = _torch()
    if hidden.dtype != torch.bfloat16 or lm_head.dtype != torch.bfloat16:
        raise TypeError("hidden and lm_head must be bfloat16")
    if hidden.dim() != 3 or lm_head.dim() != 2 or draft.dim() != 3:
        raise ValueError("hidden [B,k+1,d], lm_head [V,d], draft [B,k,V] expected")
    B, k1, d = hidden.shape
    V = lm_head.shape[0]
    k = k1 - 1
    if lm_head.shape[1] != d or tuple(draft.shape) != (B, k, V):
        raise ValueError("shape mismatch between hidden, lm_head and draft")
    for name, t, shape, dtype in (("tokens", tokens, (B, k), torch.int32),
                                  ("u_accept", u_accept, (B, k), torch.float32),
                                  ("u_resample", u_resample, (B,), torch.float32),
                                  ("temperature", temperature, (B,), torch.float32)):
        if tuple(t.shape) != shape or t.dtype != dtype:
            raise ValueError(f"{name} must be {dtype} {shape}, got {t.dtype} {tuple(t.shape)}")
    for t in (hidden, lm_head, draft, tokens, u_accept, u_resample, temperature):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("all tensors must be contiguous CUDA tensors")
    return B, k, V, d, _dtype_code(draft)


def _zeros_on(stream, device, n, dtype):
    """A zero-filled device tensor whose fill is ordered before later work on
    `stream` (the current stream when None)."""
    torch = _torch()
    device = torch.device(device if device is not None else "cuda")
    s = stream if stream is not None else torch.cuda.current_stream(device)
    with torch.cuda.stream(s):
        return torch.zeros(n, dtype=dtype, device=device)


def lmhead_workspace(B: int, k: int, V: int, d: int, draft_dtype: int, device=None,
                     stream=None):
    """A zeroed workspace for spec_verify_lmhead, zero-filled on `stream`."""
    torch = _torch()
    need = spec_verify_lmhead_workspace_size(B, k, V, d, draft_dtype)
    if need == 0:
        raise SpecVerifyError("sizes out of range for spec_verify_lmhead")
    return _zeros_on(stream, device, need, torch.uint8)


def spec_verify_lmhead(hidden, lm_head, draft, tokens, u_accept, u_resample, temperature,
                       out_tokens=None, out_num_accepted=None, ws=None, want_probs=False,
                       stream=None):
    """Verification with the target's LM head fused in: target logits
    t = hidden @ lm_head^T are formed on the tensor cores and never stored.
    hidden bf16 [B,k+1,d], lm_head bf16 [V,d], draft [B,k,V] f32 or bf16.
    Returns (out_tokens, out_num_accepted) or, with want_probs, also the fp32
    P = p_i(g_i), Q = q_i(g_i) as [B,k,2]."""
    torch = _torch()
    B, k, V, d, ddt = _marshal_lmhead(hidden, lm_head, draft, tokens, u_accept, u_resample,
                                      temperature)
    dev = hidden.device
    if out_tokens is None:
        out_tokens = torch.empty((B, k + 1), dtype=torch.int32, device=dev)
    if out_num_accepted is None:
        out_num_accepted = torch.empty((B,), dtype=torch.int32, device=dev)
    _dev_out("out_tokens", out_tokens, (B, k + 1), torch.int32, dev)
    _dev_out("out_num_accepted", out_num_accepted, (B,), torch.int32, dev)
    if ws is None:
        ws = lmhead_workspace(B, k, V, d, ddt, dev, stream)
    _check_ws(ws, dev)
    probs = torch.empty((B, k, 2), dtype=torch.float32, device=dev) if want_probs else None
    h = _stream_handle(stream, dev)
    with _on(dev):
        if want_probs:
            rc = library().spec_verify_lmhead_timed(
                _ptr(hidden), _ptr(lm_head), _ptr(draft), _ptr(tokens), _ptr(u_accept),
                _ptr(u_resample), _ptr(temperature), _ptr(out_tokens), _ptr(out_num_accepted),
                _ptr(probs), B, k, V, d, ddt, _ptr(ws), ws.numel(), h, None)
        else:
            rc = library().spec_verify_lmhead(
                _ptr(hidden), _ptr(lm_head), _ptr(draft), _ptr(tokens), _ptr(u_accept),
                _ptr(u_resample), _ptr(temperature), _ptr(out_tokens), _ptr(out_num_accepted),
                B, k, V, d, ddt, _ptr(ws), ws.numel(), h)
    _check(rc, "spec_verify_lmhead")
    if want_probs:
        return out_tokens, out_num_accepted, probs
    return out_tokens, out_num_accepted


def spec_verify_lmhead_timed(hidden, lm_head, draft, tokens, u_accept, u_resample, temperature,
                             out_tokens, out_num_accepted, ws, stage_events, stream=None):
    """spec_verify_lmhead recording SPEC_LMHEAD_STAGES events, one after each
    kernel (draft chunk records, statistics GEMM, accept scan, draw GEMM,
    final search)."""
    torch = _torch()
    B, k, V, d, ddt = _marshal_lmhead(hidden, lm_head, draft, tokens, u_accept, u_resample,
                                      temperature)
    dev = hidden.device
    _dev_out("out_tokens", out_tokens, (B, k + 1), torch.int32, dev)
    _dev_out("out_num_accepted", out_num_accepted, (B,), torch.int32, dev)
    _check_ws(ws, dev)
    handles = (ctypes.c_void_p * SPEC_LMHEAD_STAGES)(
        *[ctypes.c_void_p(e.cuda_event) for e in stage_events])
    with _on(hidden.device):
        rc = library().spec_verify_lmhead_timed(
            _ptr(hidden), _ptr(lm_head), _ptr(draft), _ptr(tokens), _ptr(u_accept), _ptr(u_resample),
            _ptr(temperature), _ptr(out_tokens), _ptr(out_num_accepted), None, B, k, V, d, ddt,
            _ptr(ws), ws.numel(), _stream_handle(stream, hidden.device), handles)
    _check(rc, "spec_verify_lmhead_timed")
    return out_tokens, out_num_accepted


def spec_lmhead_logits(hidden, lm_head, out=None, stream=None):
    """The fused GEMM alone, storing out[r][x] = sum_j hidden[r][j] lm_head[x][j]
    (fp32) for checking the tensor-core product.  hidden bf16 [M,d]."""
    torch = _torch()
    if hidden.dtype != torch.bfloat16 or lm_head.dtype != torch.bfloat16:
        raise TypeError("hidden and lm_head must be bfloat16")
    if hidden.dim() != 2 or lm_head.dim() != 2 or lm_head.shape[1] != hidden.shape[1]:
        raise ValueError("hidden [M,d] and lm_head [V,d] expected")
    for t in (hidden, lm_head):
        if not t.is_cuda or not t.is_contiguous() or t.device != hidden.device:
            raise ValueError("hidden and lm_head must be contiguous CUDA tensors on one device")
    M, d = hidden.shape
    V = lm_head.shape[0]
    if out is None:
        out = torch.empty((M, V), dtype=torch.float32, device=hidden.device)
    _dev_out("out", out, (M, V), torch.float32, hidden.device)
    status = _zeros_on(stream, hidden.device, 1, torch.int32)
    with _on(hidden.device):
        rc = library().spec_lmhead_logits(_ptr(hidden), _ptr(lm_head), _ptr(out), M, V, d,
                                          _ptr(status), _stream_handle(stream, hidden.device))
    _check(rc, "spec_lmhead_logits")
    return out, status


# ------------------------------------------------------- tree verification

def spec_verify_tree(target, draft, parent, tokens, n_nodes, u_accept, u_resample, temperature,
                     out_tokens=None, out_nodes=None, out_num_accepted=None, stream=None):
    """Tree verification (include/spec_tree.h) on the current (or given)
    stream.  target and draft [B, N, V]: float32 or bfloat16 CUDA tensors;
    parent, tokens int32 [B, N]; n_nodes int32 [B]; u_accept float32 [B, N];
    u_resample, temperature float32 [B].  Returns (out_tokens int32 [B, N],
    out_nodes int32 [B, N], out_num_accepted int32 [B]); asynchronous like
    any CUDA op."""
    torch = _torch()
    if target.dim() != 3 or tuple(draft.shape) != tuple(target.shape):
        raise ValueError("target and draft must both be [B, N, V]")
    B, N, V = target.shape
    dt = _dtype_code(target)
    if draft.dtype != target.dtype:
        raise TypeError("target and draft must share a dtype")
    dev = target.device
    for name, t, shape, dtype in (("parent", parent, (B, N), torch.int32),
                                  ("tokens", tokens, (B, N), torch.int32),
                                  ("n_nodes", n_nodes, (B,), torch.int32),
                                  ("u_accept", u_accept, (B, N), torch.float32),
                                  ("u_resample", u_resample, (B,), torch.float32),
                                  ("temperature", temperature, (B,), torch.float32)):
        if tuple(t.shape) != shape or t.dtype != dtype:
            raise ValueError(f"{name} must be {dtype} {shape}, got {t.dtype} {tuple(t.shape)}")
    for t in (target, draft, parent, tokens, n_nodes, u_accept, u_resample, temperature):
        if not t.is_cuda or not t.is_contiguous() or t.device != dev:
            raise ValueError(f"all inputs must be contiguous CUDA tensors on {dev}")
    if out_tokens is None:
        out_tokens = torch.empty((B, N), dtype=torch.int32, device=dev)
    if out_nodes is None:
        out_nodes = torch.empty((B, N), dtype=torch.int32, device=dev)
    if out_num_accepted is None:
        out_num_accepted = torch.empty((B,), dtype=torch.int32, device=dev)
    _dev_out("out_tokens", out_tokens, (B, N), torch.int32, dev)
    _dev_out("out_nodes", out_nodes, (B, N), torch.int32, dev)
    _dev_out("out_num_accepted", out_num_accepted, (B,), torch.int32, dev)
    with _on(dev):
        rc = library().spec_verify_tree(_ptr(target), _ptr(draft), _ptr(parent), _ptr(tokens),
                                        _ptr(n_nodes), _ptr(u_accept), _ptr(u_resample),
                                        _ptr(temperature), _ptr(out_tokens), _ptr(out_nodes),
                                        _ptr(out_num_accepted), B, N, V, dt,
                                        _stream_handle(stream, dev))
    _check(rc, "spec_verify_tree")
    return out_tokens, out_nodes, out_num_accepted


def tree_to_device(tc, device="cuda"):
    """Copy a synth.TreeCase's host arrays to device tensors."""
    import numpy as np
    torch = _torch()

    def logits(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)
        return torch.from_numpy(a).to(device)

    return dict(target=logits(tc.target), draft=logits(tc.draft),
                parent=torch.from_numpy(tc.parent).to(device),
                tokens=torch.from_numpy(tc.tokens).to(device),
                n_nodes=torch.from_numpy(tc.n_nodes).to(device),
                u_accept=torch.from_numpy(tc.u_accept).to(device),
                u_resample=torch.from_numpy(tc.u_resample).to(device),
                temperature=torch.from_numpy(tc.temperature).to(device))
