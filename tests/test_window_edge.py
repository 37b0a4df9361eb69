"""The window filter's one-compare test (spec_verify.cu, wfilter_kernel).

A token's window bin is wbin(x) = floor(2 (m - x) c), computed in fp32 as
(m - x) * c and capped at 64 past 32 bits.  Every rounding step is monotone,
so wbin is non-increasing in x and the tokens with wbin(x) <= lim are exactly
those with x >= edge for one float edge.  The kernel finds the edge by
bisection on the order keys between a value two bins outside the window and
the row maximum.  Here that arithmetic is emulated in numpy float32 (IEEE
round-to-nearest subtraction, multiplication and division, as the kernel's
default fp32 operations) and the claim is checked: the bisected edge is in
the window and the float below it is not, and x >= edge agrees with
wbin(x) <= lim on every bf16 value and on fp32 values packed around the edge.
"""
import numpy as np
import pytest

F = np.float32
LOG2E = F(1.4426950408889634)


def wbin(x, m, c):
    with np.errstate(over="ignore"):  # very negative x: the distance overflows to inf (bin 64)
        dd = (F(m) - np.asarray(x, np.float32)).astype(np.float32) * F(c)
        dd = dd.astype(np.float32)
        b = np.where(dd < F(32.0), np.floor(dd * F(2.0)), 64)
    return b.astype(np.int64)


def okey(x):
    b = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    return np.where(b & 0x80000000, (~b) & 0xFFFFFFFF, b | 0x80000000).astype(np.uint64)


def kval(k):
    k = np.uint64(k)
    bits = (k & np.uint64(0x7FFFFFFF)) if (k & np.uint64(0x80000000)) else (~k) & np.uint64(0xFFFFFFFF)
    return np.array([bits], np.uint64).astype(np.uint32).view(np.float32)[0]


def edge_of(lim, m, c):
    lo_v = F(m) - F(F(F(lim) * F(0.5) + F(2.0)) / F(c))
    lo, hi = int(okey(lo_v)), int(okey(F(m)))
    assert wbin(kval(lo), m, c) > lim and wbin(kval(hi), m, c) <= lim
    while hi - lo > 1:
        mid = lo + (hi - lo) // 2
        if wbin(kval(mid), m, c) <= lim:
            hi = mid
        else:
            lo = mid
    return kval(hi)


@pytest.mark.parametrize("seed", range(6))
def test_bisected_edge_is_exact(seed):
    rng = np.random.default_rng(seed)
    all_bf16 = (np.arange(0, 1 << 16, dtype=np.uint32) << 16).view(np.float32)
    all_bf16 = all_bf16[np.isfinite(all_bf16)]
    for _ in range(20):
        m = F(rng.uniform(-30, 30))
        T = F(rng.choice([0.05, 0.3, 0.7, 1.0, 1.5, 4.0]))
        c = F(LOG2E / T)
        lim = int(rng.integers(0, 64))
        e = edge_of(lim, m, c)
        assert wbin(e, m, c) <= lim
        below = np.nextafter(e, F(-np.inf), dtype=np.float32)
        assert wbin(below, m, c) > lim
        # fp32 values packed around the edge, and the bf16 grid below the maximum
        near = (np.asarray(e, np.float32).view(np.uint32).astype(np.int64)
                + np.arange(-4096, 4097)).astype(np.uint32).view(np.float32)
        near = near[np.isfinite(near) & (near <= m)]
        grid = all_bf16[all_bf16 <= m]
        for xs in (near, grid):
            assert np.array_equal(xs >= e, wbin(xs, m, c) <= lim)


def test_bins_are_monotone_in_x():
    rng = np.random.default_rng(9)
    for _ in range(50):
        m = F(rng.uniform(-10, 10))
        c = F(LOG2E / F(rng.choice([0.2, 1.0, 2.5])))
        xs = np.sort(rng.uniform(float(m) - 40, float(m), 20000).astype(np.float32))
        b = wbin(xs, m, c)
        assert np.all(np.diff(b) <= 0)
