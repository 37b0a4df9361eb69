"""The seeded input generators against the recipes they state (CPU).

Every parity test and the benchmark draw their inputs from synth.py, so its
recipes are pinned here:
- the bf16 rounding (nearest, ties to even) and its exact widening;
- the shapes, dtypes and value ranges of the five workloads;
- determinism that does not depend on the thread count;
- the greedy and Gumbel-max draft-token samplers;
- workload 5's three classes;
- the peaks and Zipf constructions;
- the sampling rows taken from a workload's draft rows.
"""
import numpy as np
import pytest
from scipy import special, stats

from speculative_decoding_verification_65_gb300 import synth


# ------------------------------------------------------------------ bf16 bits

def _nearest_even_reference(x32):
    """bf16 bits of float32 values by comparing the two neighbours exactly
    (float64 holds every float32 and bf16 value and their differences)."""
    b = x32.view(np.uint32).astype(np.uint64)
    lo = (b >> np.uint64(16)).astype(np.uint64)           # truncation toward zero
    hi = lo + np.uint64(1)                                  # next bf16 away from zero
    to_f = lambda h: (h.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    x = x32.astype(np.float64)
    dlo, dhi = np.abs(x - to_f(lo)), np.abs(to_f(hi) - x)
    pick_hi = (dhi < dlo) | ((dhi == dlo) & ((lo & np.uint64(1)) == 1))
    return np.where(pick_hi, hi, lo).astype(np.uint16)


def test_bf16_rounding_is_nearest_even():
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 1 << 32, size=200000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[np.isfinite(x) & (np.abs(x) < np.float32(3.0e38))]
    # exact ties: a bf16 value plus half of its last place, both signs
    grid = (np.arange(0, 0x7F7F, 97, dtype=np.uint32) << np.uint32(16)) | np.uint32(0x8000)
    ties = np.concatenate([grid, grid | np.uint32(0x80000000)]).view(np.float32)
    for xs in (x, ties):
        assert np.array_equal(synth.f32_to_bf16_bits(xs), _nearest_even_reference(xs))


def test_bf16_widening_is_exact_on_every_finite_pattern():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    f = synth.bf16_bits_to_f32(bits)
    fin = np.isfinite(f)
    assert np.array_equal(f.view(np.uint32)[fin] >> np.uint32(16), bits[fin].astype(np.uint32))
    assert np.array_equal(synth.f32_to_bf16_bits(f[fin]), bits[fin])


# ------------------------------------------------------------ the workloads

SETS = {1: {1.0}, 2: {1.0}, 3: {0.7}, 4: {0.0, 0.5, 1.0, 1.3}, 5: {1.0}}


@pytest.mark.parametrize("cfg,B,V", [(1, None, None), (2, 6, None), (3, 2, None), (4, 24, 4096),
                                     (5, 6, 8192)])
def test_shapes_dtypes_and_ranges(cfg, B, V):
    c = synth.make_config(cfg, B=B, V=V)
    p = synth.CONFIGS[cfg]
    assert c.B == (B or p["B"]) and c.k == p["k"] and c.V == (V or p["V"])
    B, k, V = c.B, c.k, c.V
    st = np.float32 if p["dtype"] == synth.F32 else np.uint16
    assert c.target.dtype == st and c.target.shape == (B, k + 1, V)
    assert c.draft.dtype == st and c.draft.shape == (B, k, V)
    assert c.tokens.dtype == np.int32 and c.tokens.shape == (B, k)
    assert np.all((c.tokens >= 0) & (c.tokens < V))
    for u in (c.u_accept, c.u_resample):
        assert u.dtype == np.float32 and np.all((u >= 0) & (u < 1))
    allowed = {float(np.float32(x)) for x in SETS[cfg]}
    assert c.temperature.dtype == np.float32 and set(c.temperature.tolist()) <= allowed
    assert np.all(np.isfinite(synth.decode(c.target))) and np.all(np.isfinite(synth.decode(c.draft)))


def test_deterministic_whatever_the_thread_count():
    a = synth.make_config(2, B=6, threads=1)
    b = synth.make_config(2, B=6, threads=4)
    for x, y in ((a.target, b.target), (a.draft, b.draft), (a.tokens, b.tokens),
                 (a.u_accept, b.u_accept), (a.u_resample, b.u_resample)):
        assert np.array_equal(x, y)
    c = synth.make_config(2, B=6, seed_offset=1)
    assert not np.array_equal(a.draft, c.draft)


def test_greedy_tokens_are_the_first_draft_argmax():
    c = synth.make_config(4, B=32, V=4096)
    d = synth.decode(c.draft)
    greedy = c.temperature == 0
    assert greedy.any() and (~greedy).any()
    assert np.array_equal(c.tokens[greedy], np.argmax(d[greedy], axis=2))


def test_gumbel_max_tokens_follow_the_softmax():
    rng = np.random.default_rng(5)
    row = np.array([0.0, 1.0, -0.5, 2.0, 0.3], np.float32)
    for T in (0.5, 1.0, 2.0):
        g = synth._sample_tokens(rng, np.tile(row, (20000, 1)), T)
        obs = np.bincount(g, minlength=row.size)
        exp = special.softmax(row.astype(np.float64) / T) * g.size
        assert stats.chisquare(obs, exp).pvalue > 1e-3, (T, obs, exp)


def test_workload_5_classes():
    c = synth.make_config(5, B=6, V=8192)
    t, d = synth.decode(c.target), synth.decode(c.draft)
    k = c.k
    for b in range(c.B):
        cls = b % 3
        if cls == 0:  # target rows bit-identical to the draft rows; the bonus row fresh
            assert np.array_equal(c.target[b, :k], c.draft[b])
            assert not np.array_equal(c.target[b, k], c.draft[b, k - 1])
        elif cls == 1:  # peaks on ids disjoint from the draft's
            for i in range(k):
                top_t = np.argsort(t[b, i])[-40:]
                top_d = np.argsort(d[b, i])[-40:]
                assert np.intersect1d(top_t, top_d).size == 0
        else:  # t = d + N(0, 0.5^2)
            diff = (t[b, :k] - d[b]).ravel()
            assert 0.45 < diff.std() < 0.55 and abs(diff.mean()) < 0.02


def test_peaks_rows():
    V = 5000
    row, ids = synth._peaks_row(np.random.default_rng(3), V, 2.0, 50, 6.0)
    base = synth._normal(np.random.default_rng(3), V, 2.0)
    assert ids.size == 50 and np.unique(ids).size == 50
    mask = np.zeros(V, bool)
    mask[ids] = True
    assert np.array_equal(row[mask], base[mask] + np.float32(6.0))
    assert np.array_equal(row[~mask], base[~mask])
    _, ids2 = synth._peaks_row(np.random.default_rng(4), V, 2.0, 50, 6.0, exclude=ids)
    assert np.intersect1d(ids, ids2).size == 0


def test_zipf_target_keeps_51_of_the_draft_top_64():
    V = 128256
    rng = np.random.default_rng(8)
    for _ in range(3):
        perm_d = rng.permutation(V)
        perm_t = synth._zipf_target_perm(rng, V, perm_d, 64, 0.8)
        assert np.array_equal(np.sort(perm_t), np.arange(V))
        assert np.intersect1d(perm_t[:64], perm_d[:64]).size == 51
    base = synth._zipf_base(V, 1.1)
    assert base[0] == 0.0 and np.all(np.diff(base) < 0)
    assert np.isclose(base[9], -1.1 * np.log(10.0), rtol=1e-6)


def test_sampling_rows_are_the_draft_rows():
    c = synth.make_config(4, B=8, V=2048)
    sc = synth.make_sample_config(4, B=8, V=2048)
    assert sc.R == c.B * c.k and sc.V == c.V
    assert np.array_equal(sc.logits, c.draft.reshape(sc.R, sc.V))
    assert np.array_equal(sc.temperature, np.repeat(c.temperature, c.k))
    assert sc.u.dtype == np.float32 and np.all((sc.u >= 0) & (sc.u < 1))
