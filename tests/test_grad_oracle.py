"""Oracle of TAH-Quant on gradients with the scaling of Appendix H eq. (24) (CPU).

TAH-Quant Appendix H, Table 10 applies the activation codec itself to backward gradients
(4 bits), and eq. (24) scales a gradient by a constant before quantising it and divides
after: g_hat = Q(c g) / c.  With c a power of two the scaling is exact, the quantiser
(min / max affine, §3.3) commutes with it exactly, and only the entropy keys can differ
in their last bits (the canonical key is scale invariant up to rounding), so the two
encodings agree tile for tile wherever a tile keeps its width.
"""
import numpy as np
import pytest

import oracle
import synth


def _tensor(kind, seed, T=64, C=512):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, C)).astype(np.float32)
    x[:, rng.choice(C, 4, replace=False)] *= 30.0
    if kind == "grad":  # gradient magnitudes: 1e-5 times a per-token RMS
        x *= (1e-5 * np.exp(rng.normal(0.0, 0.5, (T, 1)))).astype(np.float32)
    return x


@pytest.mark.parametrize("kind,k", [("act", 8), ("act", -12), ("grad", 16), ("grad", 24)])
def test_power_of_two_scaling_keeps_codes(kind, k):
    x = _tensor(kind, 100 + k)
    T, C = x.shape
    G, S = 64, 16
    c = float(2.0 ** k)
    r1 = oracle.encode(x, G, G, 3, 4, 3.5, S, want_keys=True)
    rc = oracle.encode_scaled(x, G, G, 3, 4, 3.5, S, c=c, want_keys=True)
    same = r1["bits"] == rc["bits"]
    # only near-ties of the key may change width (keys agree to a few ulp)
    assert (~same).sum() <= 2
    assert np.abs(r1["keys"].astype(np.float64) - rc["keys"]).max() < 1e-5
    assert np.array_equal(r1["pivots"], rc["pivots"])
    assert np.array_equal(rc["scales"][same], (r1["scales"] * np.float32(c))[same])
    assert np.array_equal(rc["zeros"][same], (r1["zeros"] * np.float32(c))[same])
    if same.all():
        assert np.array_equal(r1["codes"], rc["codes"])
        y1 = oracle.decode(r1["codes"], r1["scales"], r1["zeros"], r1["bits"], r1["pivots"],
                           T, C, G, G)
        yc = oracle.decode_scaled(rc["codes"], rc["scales"], rc["zeros"], rc["bits"],
                                  rc["pivots"], T, C, G, G, c=c)
        assert np.array_equal(y1, yc)


def test_bf16_scaling_is_exact():
    x = synth.f32_to_bf16_bits(_tensor("act", 3))
    xs = oracle.scale_input(x, 2.0 ** -20)
    back = synth.bf16_bits_to_f32(xs) * np.float32(2.0 ** 20)
    assert np.array_equal(back, synth.bf16_bits_to_f32(x))


def test_scaling_rescues_tiny_gradients():
    # around 1e-39 the tiles' ranges fall below the 2^-120 cutoff and unscaled they decode
    # to their minimum; scaled by 2^120 (eq. (24)) into an ordinary magnitude they keep
    # their shape.  (At magnitudes near the outlier test's 1e-12 guard the ratio test of
    # eq. (3) also stops transforming tiles; the scaling restores that too.)
    x = _tensor("act", 4) * np.float32(1e-39)
    T, C = x.shape
    r0 = oracle.encode(x, 64, 64, 3, 4, 3.5, 16)
    assert not r0["scales"].any()
    c = float(2.0 ** 120)
    rc = oracle.encode_scaled(x, 64, 64, 3, 4, 3.5, 16, c=c)
    assert rc["scales"].all() and (rc["pivots"] != 0xFF).any()
    y = oracle.decode_scaled(rc["codes"], rc["scales"], rc["zeros"], rc["bits"], rc["pivots"],
                             T, C, 64, 64, c=c)
    y0 = oracle.decode(r0["codes"], r0["scales"], r0["zeros"], r0["bits"], r0["pivots"],
                       T, C, 64, 64)

    def rel(a):
        return np.linalg.norm(a.astype(np.float64) - x) / np.linalg.norm(x.astype(np.float64))
    assert rel(y0) > 0.9 and rel(y) < 0.25


def test_four_bit_gradient_round_trip_bound():
    # Table 10's setting, 4 bits everywhere (budget 4 with widths {3, 4}): every element of
    # a 1e-5-scale gradient comes back within half a quantisation step of its tile
    x = _tensor("grad", 7)
    T, C = x.shape
    c = float(2.0 ** 16)
    r = oracle.encode_scaled(x, 64, 64, 3, 4, 4.0, 16, c=c, tau=float("inf"))
    assert np.all(r["bits"] == 4)
    y = oracle.decode_scaled(r["codes"], r["scales"], r["zeros"], r["bits"], r["pivots"],
                             T, C, 64, 64, c=c)
    step = (r["scales"] / np.float32(c)).astype(np.float64).repeat(64).reshape(T, C)
    assert np.all(np.abs(y.astype(np.float64) - x) <= 0.5 * step * (1 + 1e-3) + 1e-30)


@pytest.mark.parametrize("c", [0.0, 3.0, -2.0, float("inf")])
def test_rejects_scales_that_are_not_powers_of_two(c):
    with pytest.raises(ValueError):
        oracle.encode_scaled(np.zeros((2, 64), np.float32), 64, 64, 3, 4, 3.5, 0, c=c)
