"""The C ABI library loads, exports every symbol include/*.h declares, and its
host-side checks behave as documented.  No GPU needed: every call here
returns before any CUDA runtime call."""
import ctypes
import glob
import os
import re

import pytest

from tests.conftest import ROOT

import speculative_decoding_verification_65_gb300 as sv
from speculative_decoding_verification_65_gb300 import build as sv_build


@pytest.fixture(scope="module")
def lib():
    sv_build.build()
    return sv.library()


def declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^[A-Za-z_][\w \t\*]*?\b(spec_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for must in ("spec_verify", "spec_verify_workspace_size", "spec_verify_host",
                 "spec_verify_probs", "spec_verify_read_status", "spec_verify_workspace_reset"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    raw = ctypes.CDLL(sv.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(raw, n)]
    assert not missing, missing


def test_abi_version_and_strerror(lib):
    assert sv.spec_verify_abi_version() == 2
    for code in (0, 1, 2, 3):
        assert lib.spec_verify_strerror(code)
    assert b"unknown" in lib.spec_verify_strerror(99)


@pytest.mark.parametrize("B,k,V,dt,ok", [
    (4, 4, 1024, 0, True), (1024, 4, 128256, 1, True), (0, 1, 2, 0, True),
    (1, 32, 2, 1, True), (1, 0, 10, 0, False), (1, 33, 10, 0, False), (1, 1, 1, 0, False),
    (1, 1, (1 << 20) + 1, 0, False), (-1, 1, 10, 0, False), (1, 1, 10, 2, False),
])
def test_workspace_size(lib, B, k, V, dt, ok):
    n = sv.spec_verify_workspace_size(B, k, V, dt)
    if not ok:
        assert n == 0
        assert sv.spec_verify_filtered_workspace_size(B, k, V, dt) == 0
        return
    tile = 32768 // (4 if dt == 0 else 2)
    ns = -(-V // tile)          # tiles per row
    nss = -(-ns // 4)           # super-tiles per row (one partial each)
    ds = -(-V // (tile // 2))   # draw tiles per row
    up = lambda x, a: -(-x // a) * a
    nch = -(-(V * (4 if dt == 0 else 2)) // 4096)  # 4 KB chunks per row
    jobs = up(256 + B * (2 * k + 1) * nss * 16, 256)
    chunks = up(jobs + 80 * B, 256)
    rec = up(chunks + B * up(ds * 4 * 8, 32) * 4, 256)
    filt = up(rec + B * nch * 8, 256)
    # the exact draw: per sequence a 96-byte draw record, a group count, 64
    # groups of 32 bytes, and a 32-byte record per 2048 elements
    rnc = -(-V // 2048)
    resolve = up(filt + B * (2 * k + 1) * 16, 256)
    assert n == resolve + up(96 * B, 256) + up(4 * B, 256) + up(32 * 64 * B, 256) + \
        up(32 * rnc * B, 256)
    # filtered calls with room for the group maxima: one 4-byte key per 8
    # vectors (256 per 32 KB tile) of every row, then per row up to 256 kept
    # tokens of 8 bytes and their 4-byte count
    rows = B * (2 * k + 1)
    kept = up(up(n, 256) + rows * ns * 256 * 4, 256)
    assert sv.spec_verify_filtered_workspace_size(B, k, V, dt) == \
        up(kept + rows * 256 * 8, 256) + rows * 4


def _call(lib, ptrs, B=1, k=1, V=8, dt=0, wsb=1 << 20):
    args = [ctypes.c_void_p(p) for p in ptrs[:8]]
    return lib.spec_verify(*args, B, k, V, dt, ctypes.c_void_p(ptrs[8]), wsb, None)


GOOD = [0x10000 * (i + 1) for i in range(9)]


def test_zero_batch_is_noop(lib):
    assert _call(lib, [0] * 9, B=0) == sv.SPEC_OK


@pytest.mark.parametrize("which", range(9))
def test_null_pointer_rejected(lib, which):
    p = list(GOOD)
    p[which] = 0
    assert _call(lib, p) == sv.SPEC_EINVAL


@pytest.mark.parametrize("which,off", [(0, 8), (1, 4), (2, 2), (8, 8)])
def test_misaligned_pointer_rejected(lib, which, off):
    p = list(GOOD)
    p[which] += off
    assert _call(lib, p) == sv.SPEC_EINVAL


def test_bad_sizes_rejected(lib):
    assert _call(lib, GOOD, k=0) == sv.SPEC_EINVAL
    assert _call(lib, GOOD, V=1) == sv.SPEC_EINVAL
    assert _call(lib, GOOD, dt=5) == sv.SPEC_EINVAL


def test_small_workspace_rejected(lib):
    need = sv.spec_verify_workspace_size(1, 1, 8, 0)
    assert _call(lib, GOOD, wsb=need - 1) == sv.SPEC_ENOSPACE


def test_probs_needs_output(lib):
    args = [ctypes.c_void_p(p) for p in GOOD[:8]] + [None]
    assert lib.spec_verify_probs(*args, 1, 1, 8, 0, ctypes.c_void_p(GOOD[8]), 1 << 20,
                                 None) == sv.SPEC_EINVAL


def test_host_entry_checks(lib):
    n = sv.spec_verify_host_arena_size(2, 3, 100, 1)
    assert n > sv.spec_verify_workspace_size(2, 3, 100, 1)
    args = [ctypes.c_void_p(p) for p in GOOD[:8]]
    # arena not 256-byte aligned
    assert lib.spec_verify_host(*args, 2, 3, 100, 1, ctypes.c_void_p(GOOD[8] + 16), n,
                                None) == sv.SPEC_EINVAL
    assert lib.spec_verify_host(*args, 2, 3, 100, 1, ctypes.c_void_p(GOOD[8]), n - 1,
                                None) == sv.SPEC_ENOSPACE


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    import importlib
    monkeypatch.setattr(sv, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(sv, "_lib", None)
    with pytest.raises(sv.SpecVerifyError):
        sv.library()


# ------------------------------------------------------------ spec_sample

@pytest.mark.parametrize("R,V,dt,ok", [
    (4096, 128256, 1, True), (1, 2, 0, True), (0, 2, 0, True), (3, (1 << 20), 0, True),
    (1, 1, 0, False), (-1, 8, 0, False), (1, (1 << 20) + 1, 1, False), (1, 8, 3, False),
])
def test_sample_workspace_size(lib, R, V, dt, ok):
    n = sv.spec_sample_workspace_size(R, V, dt)
    if not ok:
        assert n == 0
        return
    es = 4 if dt == 0 else 2
    up = lambda x: -(-x // 256) * 256
    chunks = -(-(V * es) // 4096)  # one 8-byte record per 4 KB chunk of a row
    # the exact draw of every row: a 96-byte draw record, a 4-byte count and a
    # 32-byte record per 2048 elements
    rnc = -(-V // 2048)
    assert n == up(256 + R * chunks * 8) + up(96 * R) + up(4 * R) + up(32 * rnc * R)


def _scall(lib, ptrs, R=2, V=100, dt=0, wsb=1 << 20):
    args = [ctypes.c_void_p(p) for p in ptrs[:4]]
    return lib.spec_sample(*args, R, V, dt, ctypes.c_void_p(ptrs[4]), wsb, None)


def test_sample_zero_rows_is_noop(lib):
    assert _scall(lib, [0] * 5, R=0) == sv.SPEC_OK


@pytest.mark.parametrize("which", range(5))
def test_sample_null_pointer_rejected(lib, which):
    p = list(GOOD[:5])
    p[which] = 0
    assert _scall(lib, p) == sv.SPEC_EINVAL


@pytest.mark.parametrize("which,off", [(0, 8), (1, 2), (2, 2), (3, 2), (4, 8)])
def test_sample_misaligned_pointer_rejected(lib, which, off):
    p = list(GOOD[:5])
    p[which] += off
    assert _scall(lib, p) == sv.SPEC_EINVAL


def test_sample_bad_sizes_and_small_workspace(lib):
    assert _scall(lib, GOOD, V=1) == sv.SPEC_EINVAL
    assert _scall(lib, GOOD, dt=7) == sv.SPEC_EINVAL
    assert _scall(lib, GOOD, R=-3) == sv.SPEC_EINVAL
    need = sv.spec_sample_workspace_size(2, 100, 0)
    assert _scall(lib, GOOD, wsb=need - 1) == sv.SPEC_ENOSPACE


def test_wait_selftest_argument_checks(lib):
    assert lib.spec_selftest_wait_timeout(None, 1000, None) == sv.SPEC_EINVAL
    assert lib.spec_selftest_wait_timeout(ctypes.c_void_p(GOOD[0] + 4), 1000, None) == sv.SPEC_EINVAL
    assert lib.spec_selftest_wait_timeout(ctypes.c_void_p(GOOD[0]), 0, None) == sv.SPEC_EINVAL
    assert lib.spec_selftest_wait_timeout(ctypes.c_void_p(GOOD[0]), 10**9, None) == sv.SPEC_EINVAL


# ------------------------------------------------ LM-head-fused verification

def _up(x, a=256):
    return -(-x // a) * a


@pytest.mark.parametrize("B,k,V,d,dt,ok", [
    (1024, 4, 128256, 4096, 1, True), (1, 1, 2, 64, 0, True), (3, 31, 1000, 16384, 0, True),
    (0, 4, 100, 64, 0, False), (1, 0, 100, 64, 0, False), (1, 32, 100, 64, 0, False),
    (1, 4, 1, 64, 0, False), (1, 4, 100, 96, 0, False), (1, 4, 100, 16448, 0, False),
    (1, 4, 100, 64, 2, False), (1, 4, (1 << 20) + 1, 64, 0, False),
    # the GEMMs' tile count (128-row x 256-column tiles) must stay within 2^30
    ((1 << 22), 3, 1 << 20, 64, 0, True), ((1 << 24), 3, 1 << 20, 64, 0, False),
])
def test_lmhead_workspace_size(lib, B, k, V, d, dt, ok):
    n = sv.spec_verify_lmhead_workspace_size(B, k, V, d, dt)
    if not ok:
        assert n == 0
        return
    M = B * (k + 1)
    nt, ng = -(-V // 256), -(-V // 32)
    nc = -(-(V * (4 if dt == 0 else 2)) // 4096)
    part = 256
    tg = _up(part + M * nt * 16)
    rec = _up(tg + M * 4)
    jobs = _up(rec + B * k * nc * 8)
    hdraw = _up(jobs + B * 36)
    grp = _up(hdraw + B * d * 2)
    grp_p = _up(grp + B * ng * 4)
    assert n == _up(grp_p + B * ng * 4)


def _lcall(lib, ptrs, B=2, k=3, V=300, d=64, dt=0, wsb=1 << 26):
    args = [ctypes.c_void_p(p) for p in ptrs[:9]]
    return lib.spec_verify_lmhead(*args, B, k, V, d, dt, ctypes.c_void_p(ptrs[9]), wsb, None)


LGOOD = [0x10000 * (i + 1) for i in range(10)]


@pytest.mark.parametrize("which", range(10))
def test_lmhead_null_pointer_rejected(lib, which):
    p = list(LGOOD)
    p[which] = 0
    assert _lcall(lib, p) == sv.SPEC_EINVAL


@pytest.mark.parametrize("which,off", [(0, 8), (1, 8), (2, 8), (3, 2), (4, 2), (5, 2), (6, 2),
                                       (7, 2), (8, 2), (9, 8)])
def test_lmhead_misaligned_pointer_rejected(lib, which, off):
    p = list(LGOOD)
    p[which] += off
    assert _lcall(lib, p) == sv.SPEC_EINVAL


def test_lmhead_bad_sizes_and_small_workspace(lib):
    assert _lcall(lib, LGOOD, d=100) == sv.SPEC_EINVAL
    assert _lcall(lib, LGOOD, k=32) == sv.SPEC_EINVAL
    assert _lcall(lib, LGOOD, V=1) == sv.SPEC_EINVAL
    assert _lcall(lib, LGOOD, dt=4) == sv.SPEC_EINVAL
    need = sv.spec_verify_lmhead_workspace_size(2, 3, 300, 64, 0)
    assert _lcall(lib, LGOOD, wsb=need - 1) == sv.SPEC_ENOSPACE
    vp = ctypes.c_void_p
    assert lib.spec_lmhead_logits(vp(LGOOD[0]), vp(LGOOD[1]), vp(LGOOD[2]), 4, 300, 96,
                                  vp(LGOOD[3]), None) == sv.SPEC_EINVAL
    assert lib.spec_lmhead_logits(None, vp(LGOOD[1]), vp(LGOOD[2]), 4, 300, 64,
                                  vp(LGOOD[3]), None) == sv.SPEC_EINVAL
    # 2^26 rows x 2^20 columns: 2^31 tiles, more than the GEMM counts
    assert lib.spec_lmhead_logits(vp(LGOOD[0]), vp(LGOOD[1]), vp(LGOOD[2]), 1 << 26, 1 << 20, 64,
                                  vp(LGOOD[3]), None) == sv.SPEC_EINVAL



def test_tree_host_checks(lib):
    """spec_verify_tree rejects bad sizes, null pointers and misaligned
    arrays before any CUDA call; B = 0 is a no-op."""
    buf = (ctypes.c_uint8 * 4096)()
    base = ctypes.addressof(buf)
    a16 = (base + 15) // 16 * 16
    good = [a16] * 11

    def call(ptrs, B=1, N=4, V=16, dt=0):
        return lib.spec_verify_tree(*[ctypes.c_void_p(p) if p else None for p in ptrs],
                                    B, N, V, dt, None)
    assert call([0] * 11, B=0) == 0
    for B, N, V, dt in ((-1, 4, 16, 0), (1, 0, 16, 0), (1, 1025, 16, 0), (1, 4, 1, 0),
                        (1, 4, (1 << 20) + 1, 0), (1, 4, 16, 2)):
        assert call(good, B, N, V, dt) == 1, (B, N, V, dt)
    for i in range(11):
        ptrs = list(good)
        ptrs[i] = 0
        assert call(ptrs) == 1, i
    for i in range(2):  # logits must be 16-byte aligned
        ptrs = list(good)
        ptrs[i] = a16 + 4
        assert call(ptrs) == 1, i
    for i in range(2, 11):  # the rest 4-byte aligned
        ptrs = list(good)
        ptrs[i] = a16 + 2
        assert call(ptrs) == 1, i
