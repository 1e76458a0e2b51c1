"""Pins of the oracle's wire format (CPU only).

"TAH-Quant" §3.2 / §3.4: the 1-bit width map and the per-tile metadata travel with the
payload in one contiguous byte buffer of fixed size; the pages' figure of about 4.41 bits
per element for 80% INT4 + 20% INT3 at a tile of 64 (0.61 bits of metadata) fixes 39
metadata bits per tile.  The fp16 helpers are checked against numpy's float16 and exact
rational arithmetic, the layout against its closed form and an independent parse, and
the quantiser against its defining properties.
"""
import struct
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth

F32 = np.float32


def _f16(bits: int) -> np.float16:
    return np.array([bits], np.uint16).view(np.float16)[0]


def test_f16_value_all_patterns():
    pats = np.arange(65536, dtype=np.uint16)
    ref = pats.view(np.float16).astype(np.float64)
    for p in range(0, 65536, 7):
        v = oracle.f16_value(p)
        if np.isnan(ref[p]):
            assert np.isnan(v)
        else:
            assert v == ref[p]


def test_f16_round_down_is_the_largest_fp16_not_above():
    rng = np.random.default_rng(5)
    xs = np.concatenate([rng.standard_normal(3000) * s for s in (1e-6, 1e-3, 1.0, 300.0, 6e4)])
    xs = np.concatenate([xs, [0.0, -0.0, 65504.0, -65504.0, 6e-8, -6e-8, 1.0 + 2 ** -11]])
    for x in xs.astype(F32):
        h = oracle.f16_round_down(float(x))
        v = _f16(h)
        assert float(v) <= float(x)
        if float(v) < 65504.0:
            up = np.nextafter(v, np.float16(np.inf))
            assert float(up) > float(x)


def test_f16_scale_up_is_the_smallest_covering_scale():
    rng = np.random.default_rng(6)
    for _ in range(3000):
        mn = F32(rng.standard_normal() * 10 ** rng.uniform(-4, 3))
        mx = F32(mn + abs(rng.standard_normal()) * 10 ** rng.uniform(-6, 3))
        Q = int(rng.choice([1, 3, 7, 15, 255]))
        z = float(_f16(oracle.f16_round_down(float(mn))))
        s16 = oracle.f16_scale_up(z, float(mx), Q)
        s = _f16(s16)
        cover = lambda sv: Fraction(z) + Q * Fraction(float(sv)) >= Fraction(float(mx))
        assert cover(s)
        if s16 > 0:
            assert not cover(np.nextafter(s, np.float16(0)))


@pytest.mark.parametrize("b", [2, 3, 4, 8])
def test_wire_quantiser_properties(b):
    tiles = synth.random_tiles(17, 300, 64, "mixed")
    Q = (1 << b) - 1
    for a in tiles:
        q, s16, z16, _ = oracle.quantize_tile_f16(a, b)
        s, z = float(_f16(s16)), float(_f16(z16))
        assert z <= a.min() and s >= 0 and (s16 >> 15) == 0
        assert q.max() <= Q
        y = np.array([np.float32(np.fma(float(qi), s, z)) if hasattr(np, "fma") else
                      F32(Fraction(int(qi)) * Fraction(s) + Fraction(z)) for qi in q], F32)
        assert np.all(np.abs(y.astype(np.float64) - a) <= s / 2 * (1 + 1e-3) + 1e-6 * np.abs(a).max())
        order = np.argsort(a, kind="stable")
        assert np.all(np.diff(q[order].astype(int)) >= 0)        # monotone codes


def test_wire_quantiser_constant_fp16_tile_is_exact():
    a = np.full(64, 0.375, F32)
    q, s16, z16, _ = oracle.quantize_tile_f16(a, 3)
    assert s16 == 0 and float(_f16(z16)) == 0.375 and not q.any()


def test_wire_layout_closed_form_and_4_41_bits():
    T, C, G = 320, 1024, 64                     # n_g = 5120 tiles: K = 80% exactly
    total, off, pay = oracle.wire_layout(T, C, G, 3, 4, 3.8, 0)
    n = T * C // G
    up = lambda v: (v + 15) // 16 * 16
    assert off == [128, 128 + up(n // 8), 128 + up(n // 8) + up(4 * n),
                   128 + up(n // 8) + up(4 * n) + up(n * 6 // 8)]
    assert pay == oracle.payload_size(T, C, G, 3, 4, 3.8, 0)
    assert total == off[3] + up(pay)
    # 39 metadata bits a tile; the payload holds K hi tiles (budget 3.8f is just below 3.8,
    # so K = 4095 of 5120, one short of 80%)
    K = oracle.hi_count(n, 3, 4, 3.8)
    assert K == 4095 and pay == (3 * n + K) * G // 8
    bits_per_elem = (n * (1 + 16 + 16 + 6) + 8 * pay) / (T * C)
    assert bits_per_elem == (39 * n + (3 * n + K) * G) / (T * C)
    assert abs(bits_per_elem - (3.8 + 39 / 64)) < 1e-3 and round(bits_per_elem, 2) == 4.41


def _parse(wire):
    magic, ver, hb, T, C, S = struct.unpack_from("<IHHqqq", wire, 0)
    G, h, lo, hi, pb, _ = struct.unpack_from("<HHBBBB", wire, 32)
    budget, tau = struct.unpack_from("<ff", wire, 40)
    n, om, ome, op, opay, pay, total = struct.unpack_from("<7Q", wire, 48)
    return dict(magic=magic, ver=ver, hb=hb, T=T, C=C, S=S, G=G, h=h, lo=lo, hi=hi, pb=pb,
                budget=budget, tau=tau, n=n, om=om, ome=ome, op=op, opay=opay, pay=pay,
                total=total)


@pytest.mark.parametrize("G,h,S,dt", [(64, 64, 16, "f32"), (128, 32, 0, "f32"),
                                      (32, 32, 8, "bf16"), (16, 16, 24, "f32")])
def test_wire_encode_against_plain_codec(G, h, S, dt):
    rng = np.random.default_rng(G + S)
    x = rng.standard_normal((48, 512)).astype(F32)
    x[:, 7] *= 30
    x[5, 300] = 200.0
    if dt == "bf16":
        x = synth.f32_to_bf16_bits(x)
    lo, hi, beta = 3, 4, 3.5
    wire = oracle.encode_wire(x, G, h, lo, hi, beta, S)
    hd = _parse(wire.tobytes())
    T, C = x.shape
    n = T * C // G
    total, off, pay = oracle.wire_layout(T, C, G, lo, hi, beta, S)
    assert (hd["magic"], hd["ver"], hd["hb"]) == (0x51484154, 1, 128)
    assert wire[:4].tobytes() == b"TAHQ"
    assert (hd["T"], hd["C"], hd["S"], hd["G"], hd["h"], hd["lo"], hd["hi"]) == (T, C, S or T, G, h, lo, hi)
    assert hd["pb"] == int(np.log2(G)) and hd["n"] == n and hd["budget"] == F32(beta)
    assert [hd["om"], hd["ome"], hd["op"], hd["opay"]] == off and hd["pay"] == pay
    assert hd["total"] == total == wire.size
    # widths and transform decisions are the plain codec's
    ref = oracle.encode(x, G, h, lo, hi, beta, S)
    wmap = np.unpackbits(wire[off[0]:off[0] + (n + 7) // 8], bitorder="little")[:n]
    assert np.array_equal(np.where(wmap == 1, hi, lo), ref["bits"])
    meta = wire[off[1]:off[1] + 4 * n].view(np.uint16).reshape(n, 2)
    flag = meta[:, 0] >> 15
    assert np.array_equal(flag == 1, ref["pivots"] != 255)
    pb = hd["pb"]
    pbits = np.unpackbits(wire[off[2]:off[2] + (n * pb + 7) // 8], bitorder="little")[:n * pb]
    piv = (pbits.reshape(n, pb).astype(np.int64) << np.arange(pb)).sum(axis=1)
    assert np.array_equal(np.where(flag == 1, piv, 255), ref["pivots"])
    assert np.all(piv[flag == 0] == 0)
    # each tile decodes within half its fp16 step of the (transformed) values
    y = oracle.decode_wire(wire)
    xf = synth.bf16_bits_to_f32(x) if dt == "bf16" else x
    s = meta[:, 0].copy()
    s &= 0x7FFF
    step = s.view(np.float16).astype(np.float64)
    err = np.linalg.norm((y - xf).reshape(-1, G).astype(np.float64), axis=1)
    tol = np.sqrt(G) * 0.5 * step * (1 + 1e-3) + 1e-5 * np.abs(xf).reshape(-1, G).max(axis=1)
    assert np.all(err <= tol + 1e-30)


def test_wire_decode_rejects_bad_headers():
    x = np.random.default_rng(1).standard_normal((8, 128)).astype(F32)
    wire = oracle.encode_wire(x, 64, 64, 3, 4, 3.5, 0)
    bad = wire.copy(); bad[0] ^= 1
    with pytest.raises(ValueError):
        oracle.decode_wire(bad)
    with pytest.raises((ValueError, RuntimeError)):
        oracle.decode_wire(wire[:200])
