"""Pins of the oracle's fixed-point gradient codec (the backward pass's Q_Naive, CPU).

"TAH-Quant" §3.5 / Algorithm 1: the second stage sends a fixed-point quantisation of the
gradient with respect to the activations back to the first (6-8 bits; 10 after the NaN
event of Appendix H); Appendix H eq. (24): g_hat = Q(c g) / c.  The reading (the §3.3
asymmetric uniform quantizer at one width on the activation codec's tiles, c a power of
two) is in ``oracle/tahq_naive_oracle.c``.  These tests pin it to closed forms (ramps and
constants reconstruct exactly), a hand-packed stream, the half-step error bound, the
exact invariance under power-of-two scaling, and the activation codec (independently
pinned) at one width without the outlier transform.
"""
import numpy as np
import pytest

import oracle


def _codes(stream, n, b):
    """Codes of n fields of b bits, least significant bit first (for reading streams)."""
    bits = np.unpackbits(stream, bitorder="little")[: n * b].reshape(n, b)
    return (bits.astype(np.int64) << np.arange(b)).sum(axis=1)


@pytest.mark.parametrize("b", [3, 6, 8, 10, 12])
def test_ramp_reconstructs_exactly(b):
    # a tile holding mn + k s for k = 0 .. 2^b - 1 (s a power of two): D = Q s exactly,
    # inv = 1 / s exactly, so code k is k and the decode is exact
    G = 1 << b
    s = np.float32(2.0 ** -6)
    g = (np.float32(-3.0) + np.arange(G, dtype=np.float32) * s).reshape(1, G)
    perm = np.random.default_rng(b).permutation(G)
    g = g[:, perm]
    codes, scales, zeros = oracle.naive_encode(g, G, b)
    assert scales[0] == s and zeros[0] == np.float32(-3.0)
    assert np.array_equal(_codes(codes, G, b), perm)
    assert np.array_equal(oracle.naive_decode(codes, scales, zeros, 1, G, G, b), g)


def test_hand_packed_ten_bit_stream():
    # codes 1, 2, 1023, 0 at 10 bits: bits 0, 11, 20-29 set -> 01 08 F0 3F 00
    s = np.float32(2.0 ** -4)
    g = np.array([[s, 2 * s, 1023 * s, 0.0]], np.float32)
    codes, scales, zeros = oracle.naive_encode(g, 4, 10)
    assert codes.tolist() == [0x01, 0x08, 0xF0, 0x3F, 0x00]
    assert scales[0] == s and zeros[0] == 0.0


def test_constant_tile():
    g = np.full((2, 16), np.float32(-0.375))
    codes, scales, zeros = oracle.naive_encode(g, 8, 8)
    assert not codes.any() and not scales.any() and np.all(zeros == np.float32(-0.375))
    assert np.array_equal(oracle.naive_decode(codes, scales, zeros, 2, 16, 8, 8), g)


@pytest.mark.parametrize("b", [4, 6, 8, 10, 16])
def test_half_step_error_bound(b):
    # |g_hat - g| <= D / (2 Q) up to a few float roundings, per tile
    rng = np.random.default_rng(40 + b)
    G, T, Cc = 64, 32, 512
    g = (rng.standard_normal((T, Cc)) * 1e-5).astype(np.float32)
    g.reshape(-1, G)[::7, 3] *= 50.0
    codes, scales, zeros = oracle.naive_encode(g, G, b)
    y = oracle.naive_decode(codes, scales, zeros, T, Cc, G, b)
    t = g.reshape(-1, G).astype(np.float64)
    D = t.max(axis=1) - t.min(axis=1)
    Q = (1 << b) - 1
    err = np.abs(y.reshape(-1, G).astype(np.float64) - t).max(axis=1)
    mag = np.abs(t).max(axis=1)
    assert np.all(err <= 0.5 * D / Q * (1 + 2.0 ** -20) + 4 * mag * 2.0 ** -24)
    # and a floor-instead-of-round quantiser would not meet it: the bound is tight
    assert err.max() > 0.4 * (D / Q).min()


@pytest.mark.parametrize("k", [-8, 3, 16])
def test_power_of_two_scaling_is_exact(k):
    # eq. (24) with c = 2^k: the quantiser sees c g, every step scales exactly, so the
    # codes equal those of c = 1 and Q(c g) / c equals Q(g) bit for bit
    rng = np.random.default_rng(7)
    g = (rng.standard_normal((16, 256)) * 3e-3).astype(np.float32)
    c = float(2.0 ** k)
    c1, s1, z1 = oracle.naive_encode(g, 64, 8)
    cc, sc, zc = oracle.naive_encode(g, 64, 8, c)
    assert np.array_equal(cc, c1)
    assert np.array_equal(sc, (s1 * np.float32(c)).astype(np.float32))
    assert np.array_equal(zc, (z1 * np.float32(c)).astype(np.float32))
    assert np.array_equal(oracle.naive_decode(cc, sc, zc, 16, 256, 64, 8, c),
                          oracle.naive_decode(c1, s1, z1, 16, 256, 64, 8))


def test_scaling_rescues_underflow():
    # gradients around 1e-38 sit at the bottom of the normal range: without scaling the
    # tiles' ranges fall below 2^-120 and quantise to their minimum; scaled by 2^40 they
    # keep their shape (the reason for eq. (24))
    rng = np.random.default_rng(3)
    g = (rng.standard_normal((4, 128)) * 1e-37).astype(np.float32)
    c0, s0, z0 = oracle.naive_encode(g, 64, 8)
    assert not s0.any()
    c = float(2.0 ** 40)
    cc, sc, zc = oracle.naive_encode(g, 64, 8, c)
    assert sc.all()
    y = oracle.naive_decode(cc, sc, zc, 4, 128, 64, 8, c)
    rel = np.linalg.norm(y.astype(np.float64) - g) / np.linalg.norm(g.astype(np.float64))
    assert rel < 1e-2


@pytest.mark.parametrize("b", [3, 5, 7])
def test_matches_activation_codec_at_one_width(b):
    # the activation codec with widths {b, b + 1}, budget b (no tile gets b + 1) and
    # tau = infinity (no transform) quantises every tile the same way
    rng = np.random.default_rng(50 + b)
    x = rng.standard_normal((24, 512)).astype(np.float32)
    G = 64
    codes, scales, zeros = oracle.naive_encode(x, G, b)
    enc = oracle.encode(x, G, G, b, b + 1, float(b), 8, tau=float("inf"))
    assert np.all(enc["bits"] == b) and np.all(enc["pivots"] == 0xFF)
    assert np.array_equal(enc["codes"][: codes.size], codes)
    assert np.array_equal(enc["scales"], scales) and np.array_equal(enc["zeros"], zeros)


@pytest.mark.parametrize("G,b,c", [(64, 17, 1.0), (64, 0, 1.0), (6, 5, 1.0),
                                   (64, 8, 3.0), (64, 8, 0.0), (64, 8, float("inf"))])
def test_rejects_invalid_arguments(G, b, c):
    with pytest.raises(ValueError):
        oracle.naive_encode(np.zeros((2, 384), np.float32), G, b, c)


@pytest.mark.parametrize("b", [10, 16])
def test_cutoff_keeps_inverse_finite_and_scale_normal(b):
    # the range cutoff D_min(b) = 2^(b - 126) at widths above 6: a tile {0, D} just below
    # it quantises to its minimum (scale 0, codes 0, decodes to 0); just above it the scale
    # D / Q is a normal float, Q / D finite, and the error stays within half a step
    cut = np.float32(2.0 ** (b - 126))
    for D, live in ((np.nextafter(cut, np.float32(0)), False), (cut, True),
                    (np.float32(cut * np.float32(1.5)), True)):
        g = np.zeros((1, 32), np.float32)
        g[0, 1::2] = D
        codes, scales, zeros = oracle.naive_encode(g, 32, b)
        y = oracle.naive_decode(codes, scales, zeros, 1, 32, 32, b)
        if not live:
            assert scales[0] == 0 and not codes.any() and not y.any()
        else:
            Q = (1 << b) - 1
            assert scales[0] >= np.float32(2.0 ** -126)  # normal
            assert np.isfinite(np.float32(Q) / D)
            step = float(scales[0])
            assert np.abs(y.astype(np.float64) - g).max() <= 0.5 * step * (1 + 1e-3)
            assert y[0, 1] == D and y[0, 0] == 0  # the extremes are exact
