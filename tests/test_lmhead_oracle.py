"""Pins of the LM-head-fused oracle (oracle.lmhead_logits, oracle.verify_lmhead).

The verify step's target pass ends in the LM head, t = h W^T ("Speculative
Decoding and the Art of Fast LLM Inference", "The Algorithm, Step by Step",
the verify step).  Each pin catches a different plausible mistake: a
transposed product (W h, or h W without the transpose), rows of hidden mapped
to the wrong (sequence, position), a bf16 pattern decoded wrongly, the fused
oracle diverging from the pinned unfiltered oracle.
"""
import numpy as np
import pytest

import oracle
from speculative_decoding_verification_65_gb300 import synth


def _bits(x):
    return synth.f32_to_bf16_bits(np.asarray(x, np.float32))


def test_logits_by_hand():
    # B=1, k+1=2 positions, d=3, V=2, written out term by term
    h = np.array([[[1.0, 2.0, -1.0], [0.5, 0.0, 4.0]]], np.float32)
    w = np.array([[3.0, -1.0, 2.0], [0.25, 1.0, 1.0]], np.float32)
    t = oracle.lmhead_logits(_bits(h), _bits(w))
    want = np.array([[[1 * 3 + 2 * -1 + -1 * 2, 1 * 0.25 + 2 * 1 + -1 * 1],
                      [0.5 * 3 + 0 + 4 * 2, 0.5 * 0.25 + 0 + 4 * 1]]])
    np.testing.assert_array_equal(t, want)


def test_logits_equal_a_triple_loop():
    rng = np.random.default_rng(2)
    B, k1, d, V = 2, 3, 5, 4
    h = rng.integers(-3, 4, (B, k1, d)).astype(np.float32) / 2
    w = rng.integers(-3, 4, (V, d)).astype(np.float32) / 4
    t = oracle.lmhead_logits(_bits(h), _bits(w))
    for b in range(B):
        for i in range(k1):
            for x in range(V):
                s = 0.0
                for j in range(d):
                    s += float(h[b, i, j]) * float(w[x, j])
                assert t[b, i, x] == s


def test_bf16_patterns_decode_to_their_values():
    vals = np.array([1.0, -2.5, 0.0078125, 3.0e38, -0.0], np.float32)
    bits = np.array([0x3F80, 0xC020, 0x3C00, 0x7F62, 0x8000], np.uint16)
    h = bits.reshape(1, 1, 5)
    w = np.zeros((5, 5), np.uint16)
    for i in range(5):
        w[i, i] = 0x3F80  # 1.0
    t = oracle.lmhead_logits(h, w)
    np.testing.assert_allclose(t[0, 0], vals.astype(np.float64), rtol=0.004)
    assert t[0, 0, 0] == 1.0 and t[0, 0, 1] == -2.5 and t[0, 0, 2] == 0.0078125


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_identity_head_reduces_to_the_unfiltered_oracle(dtype):
    # W = I (d = V): the logits are the hidden states themselves, so the fused
    # oracle must give exactly what verify() gives on those logits
    B, k, V = 6, 3, 96
    c = synth.gauss_case(B=B, k=k, V=V, dtype="bf16", seed=4, T=(0.0, 0.8, 1.0))
    hidden = c.target  # bf16 bits [B, k+1, V]
    eye = np.zeros((V, V), np.uint16)
    eye[np.arange(V), np.arange(V)] = 0x3F80
    draft = c.draft if dtype == "bf16" else synth.bf16_bits_to_f32(c.draft)
    ft, fn, ftr = oracle.verify_lmhead(hidden, eye, draft, c.tokens, c.u_accept, c.u_resample,
                                       c.temperature)
    rt, rn, rtr = oracle.verify(synth.bf16_bits_to_f32(c.target),
                                synth.bf16_bits_to_f32(c.draft), c.tokens, c.u_accept,
                                c.u_resample, c.temperature)
    assert np.array_equal(ft, rt) and np.array_equal(fn, rn)
    np.testing.assert_array_equal(ftr, rtr)


def test_grid_recipe_logits_are_exact_in_fp32():
    c = synth.make_lmhead_case(B=3, k=2, V=500, d=1024, recipe="grid", seed=5)
    t = oracle.lmhead_logits(c.hidden, c.lm_head)
    assert np.array_equal(t, t.astype(np.float32).astype(np.float64))
    # every partial sum is a multiple of 2^-7 below 2^17: exact in any order
    assert np.all(np.abs(t) * 128 < 2 ** 17)
    assert np.array_equal(t * 128, np.round(t * 128))
    assert 1.0 < t.std() < 10.0


def test_draft_tokens_follow_the_draft_rows():
    c = synth.make_lmhead_case(B=8, k=3, V=300, d=64, recipe="grid", seed=6, T=(0.0,))
    rows = synth.decode(c.draft)
    assert np.array_equal(c.tokens, np.argmax(rows, axis=2))
