"""Plain fp64 CPU oracle for batched speculative-sampling verification.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / reference arm may import this package.  The
product path (the CUDA library and its binding) never imports it, and it
imports nothing from the product.

The arithmetic lives in ``spec_ref.c`` (plain C, fp64, sequential loops); this
module only compiles it with gcc and marshals numpy arrays through ctypes.
Every function there cites the passage of the pages it follows.

Parity pins for each function are in ``tests/test_oracle_pins.py`` (and, per
path, ``tests/test_sample_oracle.py``, ``tests/test_filtered_oracle.py``,
``tests/test_lmhead_oracle.py``, ``tests/test_tree_oracle.py``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "spec_ref.c")
_LIB = os.path.join(_HERE, "libspecref.so")
_lock = threading.Lock()
_lib = None

F32 = 0
BF16 = 1


def build(force: bool = False) -> str:
    """Compile spec_ref.c into libspecref.so (gcc, strict IEEE: no fast-math,
    no FMA contraction, so x86 and Arm hosts give identical results)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-Wall", "-Wextra", "-Wno-unused-parameter",
           "-o", tmp, _SRC, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB)
        vp, i64, i32, dp = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
        lib.spec_verify_ref_mt.argtypes = [vp, vp, i32, vp, dp, dp, dp, i64, i64, i64,
                                           vp, vp, dp, i32]
        lib.spec_verify_ref_mt.restype = i32
        lib.spec_ref_probs.argtypes = [vp, vp, i32, vp, dp, i64, i64, i64, dp]
        lib.spec_ref_probs.restype = i32
        lib.spec_ref_softmax.argtypes = [dp, i64, ctypes.c_double, dp]
        lib.spec_ref_softmax.restype = i32
        lib.spec_ref_residual.argtypes = [dp, dp, i64, dp]
        lib.spec_ref_residual.restype = ctypes.c_double
        lib.spec_ref_inverse_cdf.argtypes = [dp, i64, ctypes.c_double, dp]
        lib.spec_ref_inverse_cdf.restype = i64
        lib.spec_sample_ref_mt.argtypes = [vp, i32, dp, dp, i64, i64, vp, dp, i32]
        lib.spec_verify_ref_filtered_mt.argtypes = [vp, vp, i32, vp, dp, dp, dp, vp, dp,
                                                    i64, i64, i64, vp, vp, dp, i32]
        lib.spec_verify_ref_filtered_mt.restype = i32
        lib.spec_ref_filtered_softmax.argtypes = [dp, i64, ctypes.c_double, i64,
                                                  ctypes.c_double, dp, dp]
        lib.spec_ref_filtered_softmax.restype = i64
        lib.spec_sample_ref_mt.restype = i32
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _logits_and_dtype(arr: np.ndarray):
    arr = np.ascontiguousarray(arr)
    if arr.dtype == np.float32:
        return arr, F32
    if arr.dtype == np.uint16:  # bf16 bit patterns
        return arr, BF16
    raise TypeError(f"logits must be float32 or uint16 (bf16 bits), got {arr.dtype}")


def verify(target, draft, tokens, u_accept, u_resample, temperature,
           nthreads: int = 1, want_trace: bool = True):
    """Run the oracle.  Logits: float32 or uint16 (bf16 bits), [B,k+1,V] and
    [B,k,V].  Uniforms and temperature may be float32 (the product's input
    type) or float64.  Returns (out_tokens [B,k+1] int32, num_accepted [B]
    int32, trace [B,k+3] float64 or None)."""
    lib = _load()
    target, dt = _logits_and_dtype(target)
    draft, dd = _logits_and_dtype(draft)
    if dt != dd:
        raise TypeError("target and draft must share a dtype")
    B, k1, V = target.shape
    k = k1 - 1
    if draft.shape != (B, k, V):
        raise ValueError(f"draft shape {draft.shape} != {(B, k, V)}")
    tokens = np.ascontiguousarray(tokens, dtype=np.int32).reshape(B, k)
    ua = np.ascontiguousarray(u_accept, dtype=np.float64).reshape(B, k)
    ur = np.ascontiguousarray(u_resample, dtype=np.float64).reshape(B)
    tt = np.ascontiguousarray(temperature, dtype=np.float64).reshape(B)
    out_tokens = np.empty((B, k + 1), np.int32)
    out_n = np.empty((B,), np.int32)
    trace = np.empty((B, k + 3), np.float64) if want_trace else None
    rc = lib.spec_verify_ref_mt(_ptr(target), _ptr(draft), dt, _ptr(tokens), _ptr(ua),
                                _ptr(ur), _ptr(tt), B, k, V, _ptr(out_tokens),
                                _ptr(out_n), _ptr(trace) if trace is not None else None,
                                int(nthreads))
    if rc != 0:
        raise RuntimeError(f"spec_verify_ref failed with status {rc}")
    return out_tokens, out_n, trace


def probs(target, draft, tokens, temperature):
    """P = p_i(g_i) and Q = q_i(g_i) at every position: [B,k,2] float64."""
    lib = _load()
    target, dt = _logits_and_dtype(target)
    draft, _ = _logits_and_dtype(draft)
    B, k1, V = target.shape
    k = k1 - 1
    tokens = np.ascontiguousarray(tokens, dtype=np.int32).reshape(B, k)
    tt = np.ascontiguousarray(temperature, dtype=np.float64).reshape(B)
    out = np.empty((B, k, 2), np.float64)
    rc = lib.spec_ref_probs(_ptr(target), _ptr(draft), dt, _ptr(tokens), _ptr(tt),
                            B, k, V, _ptr(out))
    if rc != 0:
        raise RuntimeError(f"spec_ref_probs failed with status {rc}")
    return out


def verify_filtered(target, draft, tokens, u_accept, u_resample, temperature, top_k, top_p,
                    nthreads: int = 1, want_trace: bool = True):
    """verify() with top-k / top-p filtered distributions (top_k int [B], 0 =
    none; top_p float [B], >= 1 = none; either may be None).  The trace has a
    last column: the smallest top-p margin over the rows read."""
    lib = _load()
    target, dt = _logits_and_dtype(target)
    draft, _ = _logits_and_dtype(draft)
    B, k1, V = target.shape
    k = k1 - 1
    tokens = np.ascontiguousarray(tokens, dtype=np.int32).reshape(B, k)
    ua = np.ascontiguousarray(u_accept, dtype=np.float64).reshape(B, k)
    ur = np.ascontiguousarray(u_resample, dtype=np.float64).reshape(B)
    tt = np.ascontiguousarray(temperature, dtype=np.float64).reshape(B)
    tk = None if top_k is None else np.ascontiguousarray(top_k, dtype=np.int32).reshape(B)
    tp = None if top_p is None else np.ascontiguousarray(top_p, dtype=np.float64).reshape(B)
    out_tokens = np.empty((B, k + 1), np.int32)
    out_n = np.empty((B,), np.int32)
    trace = np.empty((B, k + 4), np.float64) if want_trace else None
    rc = lib.spec_verify_ref_filtered_mt(
        _ptr(target), _ptr(draft), dt, _ptr(tokens), _ptr(ua), _ptr(ur), _ptr(tt),
        _ptr(tk) if tk is not None else None, _ptr(tp) if tp is not None else None,
        B, k, V, _ptr(out_tokens), _ptr(out_n), _ptr(trace) if trace is not None else None,
        int(nthreads))
    if rc != 0:
        raise RuntimeError(f"spec_verify_ref_filtered failed with status {rc}")
    return out_tokens, out_n, trace


def filtered_softmax(logits, T: float, K: int, P: float):
    """Top-k / top-p filtered softmax of one row (fp64): (p, kept count, margin)."""
    lib = _load()
    l = np.ascontiguousarray(logits, dtype=np.float64)
    p = np.empty_like(l)
    mg = np.empty(1, np.float64)
    n = lib.spec_ref_filtered_softmax(_ptr(l), l.size, float(T), int(K), float(P), _ptr(p),
                                      _ptr(mg))
    if n < 0:
        raise ValueError("bad arguments")
    return p, int(n), float(mg[0])


def sample(logits, u, temperature, nthreads: int = 1, want_trace: bool = True):
    """One token per row of logits [R, V] (float32, or uint16 bf16 bit
    patterns) from softmax(logits / T) by inverse CDF with u, argmax at T = 0.
    Returns (tokens int32 [R] with -1 on a row error, trace [R, 3] float64 =
    the chosen cell [lo, hi) in u-units and the total, or None)."""
    lib = _load()
    logits, dt = _logits_and_dtype(logits)
    if logits.ndim != 2:
        raise ValueError("logits must be [R, V]")
    R, V = logits.shape
    uu = np.ascontiguousarray(u, dtype=np.float64).reshape(R)
    tt = np.ascontiguousarray(temperature, dtype=np.float64).reshape(R)
    out = np.empty((R,), np.int32)
    trace = np.empty((R, 3), np.float64) if want_trace else None
    rc = lib.spec_sample_ref_mt(_ptr(logits), dt, _ptr(uu), _ptr(tt), R, V, _ptr(out),
                                _ptr(trace) if trace is not None else None, int(nthreads))
    if rc != 0:
        raise RuntimeError(f"spec_sample_ref failed with status {rc}")
    return out, trace


def softmax(logits, T: float):
    """The oracle's temperature softmax of one row (fp64)."""
    lib = _load()
    l = np.ascontiguousarray(logits, dtype=np.float64)
    p = np.empty_like(l)
    if lib.spec_ref_softmax(_ptr(l), l.size, float(T), _ptr(p)) != 0:
        raise ValueError("softmax needs T > 0")
    return p


def residual(p, q):
    """The oracle's residual weights max(0, p-q) and their total."""
    lib = _load()
    p = np.ascontiguousarray(p, dtype=np.float64)
    q = np.ascontiguousarray(q, dtype=np.float64)
    w = np.empty_like(p)
    R = lib.spec_ref_residual(_ptr(p), _ptr(q), p.size, _ptr(w))
    return w, R


def inverse_cdf(w, u: float):
    """The oracle's inverse-CDF draw: (token, [lo, hi, R])."""
    lib = _load()
    w = np.ascontiguousarray(w, dtype=np.float64)
    cell = np.empty(3, np.float64)
    x = lib.spec_ref_inverse_cdf(_ptr(w), w.size, float(u), _ptr(cell))
    return int(x), cell


# ------------------------------------------------ LM-head-fused verification

def _bf16_to_f64(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) to float64, exactly: a bf16 pattern is the
    upper half of the float32 of the same value."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def lmhead_logits(hidden, lm_head) -> np.ndarray:
    """Target logits of the LM head, t[..., x] = sum_j h[..., j] * W[x, j].

    The verify step scores the k+1 positions with one target forward pass
    ("Speculative Decoding and the Art of Fast LLM Inference", "The Algorithm,
    Step by Step", the verify step), whose last layer is this product.
    hidden: uint16 bf16 bits [..., d]; lm_head: uint16 bf16 bits [V, d].
    Products of two bf16 values are exact in fp64; the sums are fp64 (numpy
    matmul as the one library step)."""
    h = _bf16_to_f64(hidden)
    w = _bf16_to_f64(lm_head)
    lead = h.shape[:-1]
    t = h.reshape(-1, h.shape[-1]) @ w.T
    return t.reshape(*lead, w.shape[0])


def verify_lmhead(hidden, lm_head, draft, tokens, u_accept, u_resample, temperature,
                  nthreads: int = 1, want_trace: bool = True):
    """verify() with the target logits formed from the LM head:
    target = lmhead_logits(hidden, lm_head) rounded once to fp32 (the GPU
    accumulates in fp32; on inputs whose partial sums are all exact in fp32
    the rounding changes nothing).  A bf16 draft is widened to fp32, exactly.
    hidden [B, k+1, d], lm_head [V, d] (uint16 bf16 bits), draft [B, k, V]."""
    t = lmhead_logits(hidden, lm_head).astype(np.float32)
    d, dd = _logits_and_dtype(draft)
    if dd == BF16:
        d = (d.astype(np.uint32) << 16).view(np.float32)
    return verify(t, d, tokens, u_accept, u_resample, temperature, nthreads=nthreads,
                  want_trace=want_trace)


# ------------------------------------------------------- tree verification

def verify_tree(target, draft, parent, tokens, n_nodes, u_accept, u_resample, temperature,
                nthreads: int = 1, want_trace: bool = True):
    """Tree verification (spec_verify_tree_ref_mt in spec_ref.c).  Logits
    [B, N, V] float32 or uint16 (bf16 bits); parent, tokens [B, N] int32;
    n_nodes [B]; u_accept [B, N]; u_resample, temperature [B].  Returns
    (out_tokens [B, N], out_nodes [B, N], num_accepted [B], trace [B, N+3] or
    None)."""
    lib = _load()
    if not hasattr(lib, "_tree_ready"):
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        lib.spec_verify_tree_ref_mt.argtypes = [vp, vp, i32, vp, vp, vp, vp, vp, vp,
                                                i64, i64, i64, vp, vp, vp, vp, i32]
        lib.spec_verify_tree_ref_mt.restype = i32
        lib._tree_ready = True
    target, dt = _logits_and_dtype(target)
    draft, dd = _logits_and_dtype(draft)
    if dt != dd:
        raise TypeError("target and draft must share a dtype")
    B, N, V = target.shape
    if draft.shape != (B, N, V):
        raise ValueError(f"draft shape {draft.shape} != {(B, N, V)}")
    par = np.ascontiguousarray(parent, dtype=np.int32).reshape(B, N)
    tok = np.ascontiguousarray(tokens, dtype=np.int32).reshape(B, N)
    nn = np.ascontiguousarray(n_nodes, dtype=np.int32).reshape(B)
    ua = np.ascontiguousarray(u_accept, dtype=np.float64).reshape(B, N)
    ur = np.ascontiguousarray(u_resample, dtype=np.float64).reshape(B)
    tt = np.ascontiguousarray(temperature, dtype=np.float64).reshape(B)
    out_tokens = np.empty((B, N), np.int32)
    out_nodes = np.empty((B, N), np.int32)
    out_n = np.empty((B,), np.int32)
    trace = np.empty((B, N + 3), np.float64) if want_trace else None
    rc = lib.spec_verify_tree_ref_mt(_ptr(target), _ptr(draft), dt, _ptr(par), _ptr(tok),
                                     _ptr(nn), _ptr(ua), _ptr(ur), _ptr(tt), B, N, V,
                                     _ptr(out_tokens), _ptr(out_nodes), _ptr(out_n),
                                     _ptr(trace) if trace is not None else None,
                                     int(nthreads))
    if rc != 0:
        raise RuntimeError(f"spec_verify_tree_ref failed with status {rc}")
    return out_tokens, out_nodes, out_n, trace
