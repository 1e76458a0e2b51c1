"""Pins of the CPU oracle against what the pages and the mathematics fix (no GPU).

Page citations: "TAH-Quant: Effective Activation Quantization in Pipeline Parallelism
over Slow Network" (arXiv 2506.01352v2), and the prior-art page "Training Transformers
with 4-bit Integers" (a summary of arXiv 2306.11987).
"""
import itertools
import math
import os

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
F32 = np.float32


def _ulp(x):
    return np.spacing(np.abs(np.float32(x))).astype(np.float64)


# ------------------------------------------------------------------ canonical log2

def test_lg_exact_at_powers_of_two():
    e = np.arange(-149, 128)
    x = np.ldexp(np.ones(e.size), e).astype(F32)
    assert np.array_equal(oracle.lg(x), e.astype(F32))


def test_lg_exhaustive_mantissas_at_exponent_zero():
    # every float in [1, 2): 2^23 values against a double-precision log2
    x = (np.arange(1 << 23, dtype=np.uint32) | np.uint32(0x3F800000)).view(F32)
    err = np.abs(oracle.lg(x).astype(np.float64) - np.log2(x.astype(np.float64)))
    assert err.max() <= 2.0 ** -23


def test_lg_error_bound_all_exponents_and_subnormals():
    rng = np.random.default_rng(5)
    bits = rng.integers(1, 0x7F800000, 1 << 20, dtype=np.uint32)   # positive finite, incl. subnormal
    x = bits.view(F32)
    got = oracle.lg(x).astype(np.float64)
    ref = np.log2(x.astype(np.float64))
    assert np.all(np.abs(got - ref) <= 2.0 ** -23 + 0.5 * _ulp(got))


def test_lg_tables_are_nearest_floats():
    T, R, k = oracle.log2_tables()
    i = np.arange(128, dtype=np.float64)
    assert np.array_equal(R, (1 / (1 + i / 128)).astype(F32))
    # T_i = -log2 of the stored R_i, so log2(m) = T_i + log2(m R_i) holds exactly
    assert np.array_equal(T, (-np.log2(R.astype(np.float64))).astype(F32))
    assert T[0] == 0 and np.all(np.diff(T) > 0) and T[-1] < 1
    j = np.arange(1, 4)
    assert np.array_equal(k, (((-1.0) ** (j + 1)) / (j * math.log(2))).astype(F32))


# ------------------------------------------------------------------ pairwise sum

def test_pairwise_sum_order():
    e = F32(2.0 ** -24)
    # pairwise: (1 + e) + (e + e) = 1 + 2^-23 ; left-to-right would give exactly 1
    assert oracle.pairwise_sum([1.0, e, e, e]) == F32(1.0 + 2.0 ** -23)
    # exact for sums of equal powers of two
    for n in (8, 16, 32, 64, 128):
        assert oracle.pairwise_sum(np.full(n, 0.375, F32)) == 0.375 * n


# ------------------------------------------------------------------ entropy (eq. 1-2)

@pytest.mark.parametrize("G", [8, 16, 32, 64, 128])
def test_entropy_closed_forms(G):
    rng = np.random.default_rng(G)
    for j in (-20, -3, 0, 5, 30):
        c = F32(2.0 ** j)
        sign = np.where(rng.random(G) < 0.5, -1, 1).astype(F32)
        assert oracle.entropy_key(c * sign) == np.log2(G)          # flat tile -> log2 G
        for spikes in (1, 2, 4):                                   # k equal spikes -> log2 k
            a = np.zeros(G, F32)
            a[rng.choice(G, spikes, replace=False)] = c * sign[:spikes]
            assert oracle.entropy_key(a) == math.log2(spikes)
    assert oracle.entropy_key(np.zeros(G, F32)) == 0.0
    # non-dyadic flat magnitude: log2 G within rounding
    assert abs(oracle.entropy_key(np.full(G, 3.0, F32)) - math.log2(G)) < 1e-6


@pytest.mark.parametrize("kind", ["gauss", "spiky", "positive", "mixed"])
def test_entropy_matches_eq2_literal(kind):
    # canonical fp32 key (bits) vs eq. (1)-(2) evaluated literally in double (nats),
    # with the minus sign of eq. (2) restored; eps = varsigma = 1e-12
    x = synth.random_tiles(11, 300, 64, kind)
    for a in x:
        if np.abs(a).sum() == 0:
            continue
        lit = oracle.entropy_literal(a)
        assert lit >= -1e-9
        assert abs(oracle.entropy_key(a) * math.log(2) - lit) < 1e-5


def test_entropy_ranks_spread_above_spiky():
    # §3.2: H is high when energy is spread evenly, low for a sharp outlier
    rng = np.random.default_rng(0)
    flat = rng.standard_normal(64).astype(F32)
    spiky = flat.copy()
    spiky[17] = 200.0
    assert oracle.entropy_key(flat) > oracle.entropy_key(spiky) + 1.0


def test_entropy_invariances():
    x = synth.random_tiles(3, 200, 64, "gauss")
    rng = np.random.default_rng(1)
    for a in x:
        h = oracle.entropy_key(a)
        assert abs(oracle.entropy_key(a[rng.permutation(64)]) - h) < 1e-5
        assert abs(oracle.entropy_key(a * F32(2.0 ** 7)) - h) < 1e-5
        assert abs(oracle.entropy_key(-a) - h) == 0.0


# ------------------------------------------------------------------ outlier heuristic (eq. 3)

def test_outlier_threshold_cases():
    a = np.zeros(64, F32)
    a[0], a[1] = 1.0, 0.5                       # r = 1/(0.5+1e-12) rounds to 2.0: not > tau
    assert oracle.outlier(a)[:2] == (0, 0)
    a[0] = F32(1.0 + 2.0 ** -23)                # r just above 2: transform
    assert oracle.outlier(a)[:2] == (0, 1)
    assert oracle.outlier(np.zeros(64, F32))[:2] == (0, 0)       # all zero: no transform
    b = np.zeros(64, F32)
    b[9], b[40] = -3.0, 3.0                      # equal maxima: lowest index, r = 1
    assert oracle.outlier(b)[:2] == (9, 0)
    c = np.zeros(64, F32)
    c[33] = -7.0                                 # single spike, rest 0: r = 7/1e-12
    assert oracle.outlier(c)[:2] == (33, 1)


@pytest.mark.parametrize("kind", ["gauss", "spiky", "mixed"])
def test_outlier_against_numpy(kind):
    x = synth.random_tiles(4, 500, 32, kind)
    for a in x:
        d, flag, m1, m2 = oracle.outlier(a)
        mags = np.abs(a)
        assert d == int(np.argmax(mags))                       # first maximum
        assert m1 == mags.max()
        assert m2 == np.sort(np.delete(mags, d))[-1]
        r = F32(m1) / (F32(m2) + F32(1e-12))
        assert flag == int(r > F32(2.0))


# ------------------------------------------------------------------ Hadamard (eq. 4)

def _sylvester(h):
    H = np.array([[1]], dtype=np.int64)
    while H.shape[0] < h:
        H = np.block([[H, H], [H, -H]])
    return H


def _read_golden_matrices():
    mats, cur, name = {}, None, None
    with open(os.path.join(GOLDEN, "sylvester_h4.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("H"):
                name, cur = line, []
                mats[name] = cur
            else:
                cur.append([int(v) for v in line.split()])
    return {k: np.array(v) for k, v in mats.items()}


def test_sylvester_golden_and_orthogonality():
    g = _read_golden_matrices()
    assert np.array_equal(g["H2"], _sylvester(2))
    assert np.array_equal(g["H4"], _sylvester(4))
    for h in (2, 4, 8, 16, 32, 64, 128):
        H = _sylvester(h)
        assert np.array_equal(H @ H.T, h * np.eye(h, dtype=np.int64))


@pytest.mark.parametrize("h", [2, 4, 8, 16, 32, 64, 128])
def test_fwht_is_sylvester_matrix(h):
    H = _sylvester(h)
    for j in range(h):
        e = np.zeros(h, F32)
        e[j] = 1.0
        assert np.array_equal(oracle.fwht(e), H[j].astype(F32))   # row j (H symmetric)
    x = np.random.default_rng(h).integers(-50, 50, h).astype(F32)
    assert np.array_equal(oracle.fwht(x), (x.astype(np.int64) @ H).astype(F32))
    assert np.array_equal(oracle.fwht(oracle.fwht(x)), h * x)     # H H = h I


@pytest.mark.parametrize("G,h", [(64, 64), (32, 32), (128, 128), (64, 16), (128, 32), (8, 8)])
def test_transform_matches_dense(G, h):
    x = synth.random_tiles(7, 50, G, "spiky")
    for a in x:
        d = int(np.argmax(np.abs(a)))
        got = oracle.transform(a, h, d).astype(np.float64)
        p = a.astype(np.float64).copy()
        p[0], p[d] = p[d], p[0]
        ref = np.concatenate([oracle.hadamard_dense(p[b:b + h]) for b in range(0, G, h)])
        bound = math.log2(h) * 2.0 ** -23 * np.abs(a).max() * math.sqrt(h) + 1e-30
        assert np.abs(got - ref).max() <= bound


def test_transform_inverse_and_one_hot():
    # h = 64: 1/sqrt(64) = 1/8 is exact, so a spike c e_d maps to c/8 everywhere
    for d in (0, 5, 63):
        a = np.zeros(64, F32)
        a[d] = -24.0
        t = oracle.transform(a, 64, d)
        assert np.array_equal(t, np.full(64, -3.0, F32))
        assert np.array_equal(oracle.inverse_transform(t, 64, d), a)
    # h = 4, 16: exact scale, integer inputs -> the round trip is exact (P_d P_d = I)
    x = np.random.default_rng(2).integers(-9, 9, 64).astype(F32)
    for h in (4, 16):
        for d in (0, 1, 37):
            assert np.array_equal(oracle.inverse_transform(oracle.transform(x, h, d), h, d), x)


# ------------------------------------------------------------------ quantizer + packing

@pytest.mark.parametrize("b", [1, 2, 3, 4, 5, 8])
def test_quantizer_bounds(b):
    Q = (1 << b) - 1
    x = synth.random_tiles(21, 200, 64, "mixed")
    for v in x:
        q, s, z, _ = oracle.quantize_tile(v, b)
        assert z == v.min()
        if v.max() - v.min() < 2.0 ** -120:
            assert s == 0 and not q.any()
            continue
        assert q[np.argmin(v)] == 0 and q[np.argmax(v)] == Q
        assert q.max() <= Q
        vh = np.array([np.float32(np.float64(qq) * s + z) for qq in q])   # fma: single rounding
        err = np.abs(vh.astype(np.float64) - v)
        assert np.all(err <= s / 2 * (1 + 1e-3) + 4 * _ulp(v) + 4 * _ulp(z))


@pytest.mark.parametrize("b", [2, 3, 4, 8])
def test_quantizer_codes_are_nearest_integers_of_the_exact_product(b):
    # code_k = the integer nearest (v_k - mn) * inv computed exactly, ties to even; the
    # inputs include products that fall within one fp32 rounding of a .5 boundary
    from fractions import Fraction
    Q = (1 << b) - 1
    rng = np.random.default_rng(40 + b)
    tiles = list(synth.random_tiles(41, 60, 64, "mixed"))
    for _ in range(60):    # values on (k + 1/2) / inv, nudged by one ulp either way
        base = rng.standard_normal(64).astype(F32)
        mn, mx = F32(base.min()), F32(base.max())
        inv = F32(F32(Q) / F32(mx - mn))
        k = rng.integers(0, Q, 64)
        tgt = ((k + 0.5) / np.float64(inv) + np.float64(mn)).astype(F32)
        tgt = np.nextafter(tgt, rng.choice([-np.inf, np.inf], 64).astype(F32)).astype(F32)
        v = np.clip(tgt, mn, mx).astype(F32)
        v[0], v[1] = mn, mx
        tiles.append(v)
    for v in tiles:
        q, s, z, _ = oracle.quantize_tile(v, b)
        mn, mx = F32(v.min()), F32(v.max())
        if float(mx) - float(mn) < 2.0 ** -120:
            continue
        inv = F32(F32(Q) / F32(mx - mn))
        for vk, qk in zip(v, q):
            u = Fraction(float(F32(vk - mn))) * Fraction(float(inv))
            n = int(u)                      # u >= 0
            frac = u - n
            want = n + 1 if frac > Fraction(1, 2) or (frac == Fraction(1, 2) and n % 2) else n
            assert int(qk) == min(want, Q), (float(u), int(qk))


def test_quantizer_error_falls_with_bits():
    x = synth.random_tiles(8, 400, 64, "gauss")
    mse = []
    for b in range(2, 9):
        e = 0.0
        for v in x:
            q, s, z, _ = oracle.quantize_tile(v, b)
            e += float(np.sum((q.astype(np.float64) * s + z - v) ** 2))
        mse.append(e)
    ratios = [mse[i] / mse[i + 1] for i in range(len(mse) - 1)]
    assert all(r > 3.0 for r in ratios), ratios          # about 4x per extra bit


def test_pack_golden_order():
    with open(os.path.join(GOLDEN, "pack_order.txt")) as f:
        rows = [ln for ln in f if ln.strip() and not ln.startswith("#")]
    assert rows
    for ln in rows:
        b, codes, packed = (p.strip() for p in ln.split("|"))
        b = int(b)
        codes = np.array([int(c) for c in codes.split()], np.uint8)
        want = np.array([int(h, 16) for h in packed.split()], np.uint8)
        assert np.array_equal(oracle.pack_tile(codes, b), want)
        assert np.array_equal(oracle.unpack_tile(want, codes.size, b), codes)


@pytest.mark.parametrize("b", range(1, 9))
def test_pack_roundtrip(b):
    rng = np.random.default_rng(b)
    for G in (8, 32, 64, 128):
        q = rng.integers(0, 1 << b, G).astype(np.uint8)
        slot = oracle.pack_tile(q, b)
        assert slot.size == G * b // 8
        assert np.array_equal(oracle.unpack_tile(slot, G, b), q)


# ------------------------------------------------------------------ allocation (§3.2)

def _brute_force(H, K):
    """Best K-subset by sum of H; among equal sums the lexicographically smallest."""
    best, best_set = None, None
    for comb in itertools.combinations(range(len(H)), K):
        s = sum(H[i] for i in comb)          # H are small integers / 4: sums are exact
        if best is None or s > best:
            best, best_set = s, comb
    return best_set


def test_allocation_brute_force():
    rng = np.random.default_rng(9)
    for trial in range(60):
        n = int(rng.integers(1, 11))
        H = (rng.integers(0, 6, n) / 4.0).astype(F32)       # many exact ties
        K = int(rng.integers(0, n + 1))
        bits = oracle.allocate(H, K, 3, 4)
        chosen = tuple(np.flatnonzero(bits == 4))
        assert chosen == _brute_force(list(H.astype(np.float64)), K)
        assert np.all((bits == 3) | (bits == 4))


def test_hi_count_and_budget():
    for n_g in (1, 7, 64, 4096, 131072):
        for lo, hi in ((3, 4), (2, 3), (2, 4), (7, 8)):
            assert oracle.hi_count(n_g, lo, hi, lo) == 0
            assert oracle.hi_count(n_g, lo, hi, hi) == n_g
            for beta in np.linspace(lo, hi, 9):
                K = oracle.hi_count(n_g, lo, hi, float(beta))
                assert K == math.floor((float(F32(beta)) - lo) * n_g / (hi - lo))
                assert (K * hi + (n_g - K) * lo) <= float(F32(beta)) * n_g + 1e-9


def test_bits_accounting_golden():
    vals = {}
    with open(os.path.join(GOLDEN, "bits_accounting.txt")) as f:
        for ln in f:
            if ln.strip() and not ln.startswith("#"):
                k, v = ln.split()
                vals[k] = float(v)
    n_g = 4096
    K = oracle.hi_count(n_g, int(vals["bits_lo"]), int(vals["bits_hi"]), vals["budget"])
    # fp32 3.8 lies just below 3.8, and K is a floor (the budget is never exceeded)
    assert abs(K - vals["hi_fraction"] * n_g) <= 1
    G = int(vals["tile"])
    payload = oracle.payload_size(64, n_g, G, 3, 4, vals["budget"], 0)
    # payload bits per element from the stream size, against 0.8*4 + 0.2*3 = 3.8
    assert abs(payload * 8 / (64 * n_g) - vals["payload_bits_per_element"]) < 2e-3
    assert abs(vals["total_bits_per_element"] - vals["metadata_bits_per_element"]
               - vals["payload_bits_per_element"]) < 1e-9


# ------------------------------------------------------------------ whole tensor

def _small(T=48, C=256, seed=0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, C)).astype(F32)
    x[:, 5] *= 40
    x[3, 100] = 900.0
    x[7, 64:128] = 0.0
    x[8, 128:192] = 2.5
    return x


@pytest.mark.parametrize("G,h,lo,hi,beta,S", [
    (64, 64, 3, 4, 3.5, 16), (32, 32, 3, 4, 3.25, 0), (128, 128, 3, 4, 3.9, 24),
    (64, 16, 2, 4, 3.0, 8), (8, 8, 3, 4, 3.5, 12), (16, 8, 3, 5, 4.0, 48)])
def test_encode_structure(G, h, lo, hi, beta, S):
    x = _small()
    T, Cc = x.shape
    r = oracle.encode(x, G, h, lo, hi, beta, S, want_keys=True, want_near=True)
    W = Cc // G
    n_g = (S or T) * W
    K = oracle.hi_count(n_g, lo, hi, beta)
    tiles = x.reshape(-1, G)
    for g in range((T // (S or T))):
        sl = slice(g * n_g, (g + 1) * n_g)
        assert np.count_nonzero(r["bits"][sl] == hi) == K
        assert np.array_equal(r["bits"][sl], oracle.allocate(r["keys"][sl], K, lo, hi))
    slot_total = int(np.sum(r["bits"].astype(np.int64) * G // 8))
    assert slot_total == r["codes"].size == oracle.payload_size(T, Cc, G, lo, hi, beta, S)
    for t in range(tiles.shape[0]):
        assert r["keys"][t] == oracle.entropy_key(tiles[t])
        d, flag, _, _ = oracle.outlier(tiles[t])
        assert r["pivots"][t] == (d if flag else 255)
    # decode stays within the quantisation step (the transform is orthogonal)
    y = oracle.decode(r["codes"], r["scales"], r["zeros"], r["bits"], r["pivots"], T, Cc, G, h)
    err = (y - x).reshape(-1, G).astype(np.float64)
    s = r["scales"].astype(np.float64)
    tol = np.linalg.norm(np.full(G, 0.5), 2) * s * (1 + 1e-3) + 1e-5 * np.abs(tiles).max(axis=1)
    assert np.all(np.linalg.norm(err, axis=1) <= tol + 1e-30)


def test_spike_tile_decodes_exactly():
    x = np.zeros((2, 128), F32)
    x[0, 37] = -96.0
    x[1, 64 + 3] = 0.25
    r = oracle.encode(x, 64, 64, 3, 4, 3.5, 0)
    assert list(r["pivots"]) == [37, 255, 255, 3]
    assert r["scales"][0] == 0 and r["scales"][3] == 0
    y = oracle.decode(r["codes"], r["scales"], r["zeros"], r["bits"], r["pivots"], 2, 128, 64, 64)
    assert np.array_equal(y, x)


def test_eight_bit_roundtrip():
    x = synth.generate(synth.WORKLOADS["c1"])
    r = oracle.encode(x, 64, 64, 7, 8, 8.0, 0)
    assert np.all(r["bits"] == 8)
    y = oracle.decode(r["codes"], r["scales"], r["zeros"], r["bits"], r["pivots"], 256, 1024, 64, 64)
    assert np.linalg.norm(y - x) / np.linalg.norm(x) < 2.0 ** -8


def test_error_falls_with_budget():
    w = synth.WORKLOADS["c4"].with_params(tokens=256, channels=1024, tokens_per_group=64)
    x = synth.bf16_bits_to_f32(synth.generate(w))
    prev = None
    for beta in (3.0, 3.5, 4.0):
        r = oracle.encode(x, 64, 64, 3, 4, beta, 64)
        y = oracle.decode(r["codes"], r["scales"], r["zeros"], r["bits"], r["pivots"], 256, 1024, 64, 64)
        e = np.linalg.norm(y - x) / np.linalg.norm(x)
        assert prev is None or e < prev
        prev = e


def test_group_scope_and_threads():
    x = _small(T=64)
    one = oracle.encode(x, 64, 64, 3, 4, 3.5, 0, want_keys=True)
    grp = oracle.encode(x, 64, 64, 3, 4, 3.5, 16, threads=1, want_keys=True)
    thr = oracle.encode(x, 64, 64, 3, 4, 3.5, 16, threads=4, want_keys=True)
    for k in grp:
        assert np.array_equal(grp[k], thr[k])
    assert np.array_equal(one["keys"], grp["keys"])
    assert not np.array_equal(one["bits"], grp["bits"])       # ranking scope matters
    yd = oracle.decode(grp["codes"], grp["scales"], grp["zeros"], grp["bits"], grp["pivots"],
                       64, 256, 64, 64, threads=3)
    y1 = oracle.decode(grp["codes"], grp["scales"], grp["zeros"], grp["bits"], grp["pivots"],
                       64, 256, 64, 64)
    assert np.array_equal(yd, y1)


def test_bf16_input_is_widened_exactly():
    w = synth.WORKLOADS["c2"].with_params(tokens=64, channels=256, tokens_per_group=32)
    xb = synth.generate(w)
    a = oracle.encode(xb, 64, 64, 3, 4, 3.5, 32)
    b = oracle.encode(synth.bf16_bits_to_f32(xb), 64, 64, 3, 4, 3.5, 32)
    for k in a:
        assert np.array_equal(a[k], b[k])


def test_invalid_arguments_rejected():
    x = np.zeros((4, 128), F32)
    with pytest.raises(ValueError):
        oracle.encode(x, 48, 16, 3, 4, 3.5, 0)      # tile not a power of two
    with pytest.raises(ValueError):
        oracle.encode(x, 64, 64, 3, 4, 4.5, 0)      # budget above hi
    with pytest.raises(ValueError):
        oracle.encode(x, 64, 64, 3, 4, 3.5, 3)      # group does not divide tokens


# ------------------------------------------------------------------ the threshold tau
# (Appendix F: tau = 0 transforms every tile, tau = inf none, tau = 4 fewer than 2)

def test_outlier_tau_cases():
    a = np.zeros(64, F32)
    a[5], a[20] = 3.0, 1.0                       # r = 3 / (1 + 1e-12) rounds to 3.0
    assert oracle.outlier(a, 2.9)[:2] == (5, 1)
    assert oracle.outlier(a, 3.0)[:2] == (5, 0)  # strict: r == tau is no outlier
    assert oracle.outlier(a, 4.0)[:2] == (5, 0)
    assert oracle.outlier(a, 0.0)[:2] == (5, 1)
    assert oracle.outlier(a, np.inf)[:2] == (5, 0)
    assert oracle.outlier(np.zeros(64, F32), 0.0)[:2] == (0, 0)   # r = 0: not > 0
    c = np.zeros(64, F32)
    c[63] = 1e30                                 # r = 1e42 overflows to inf: inf > inf is false
    assert oracle.outlier(c, np.inf)[:2] == (63, 0)
    assert oracle.outlier(c, 3.4e38)[:2] == (63, 1)


@pytest.mark.parametrize("G,h,S", [(64, 64, 16), (32, 16, 0), (8, 8, 12)])
def test_encode_tau(G, h, S):
    x = _small()
    T, Cc = x.shape
    tiles = x.reshape(-1, G)
    base = oracle.encode(x, G, h, 3, 4, 3.5, S)
    same = oracle.encode(x, G, h, 3, 4, 3.5, S, tau=2.0)
    for k in base:
        assert np.array_equal(base[k], same[k]), k
    mags = np.abs(tiles)
    first = np.argmax(mags, axis=1)
    flagged = {}
    for tau in (0.0, 1.5, 2.0, 4.0, np.inf):
        r = oracle.encode(x, G, h, 3, 4, 3.5, S, tau=tau)
        assert np.array_equal(r["bits"], base["bits"])      # the statistics use the raw tile
        f = r["pivots"] != 255
        assert np.array_equal(r["pivots"][f], first[f])
        flagged[tau] = f
        y = oracle.decode(r["codes"], r["scales"], r["zeros"], r["bits"], r["pivots"], T, Cc, G, h)
        err = np.linalg.norm((y - x).reshape(-1, G).astype(np.float64), axis=1)
        tol = np.sqrt(G) * 0.5 * r["scales"].astype(np.float64) * (1 + 1e-3) + 1e-5 * mags.max(axis=1)
        assert np.all(err <= tol + 1e-30)
    assert np.array_equal(flagged[0.0], mags.max(axis=1) > 0)   # every nonzero tile
    assert not flagged[np.inf].any()
    assert np.all(flagged[4.0] <= flagged[2.0]) and np.all(flagged[2.0] <= flagged[1.5])
    assert np.all(flagged[1.5] <= flagged[0.0])
    assert flagged[2.0].any() and (flagged[0.0] & ~flagged[2.0]).any()


def test_encode_tau_untransformed_tiles_match_the_plain_quantizer():
    # tau = inf: every tile is quantised as it is; the codes of tile t are those of the
    # tile-level quantizer and packer applied to the raw tile
    x = _small()[:, :256]
    G = 64
    r = oracle.encode(x, G, G, 3, 4, 3.5, 0, tau=np.inf)
    off = 0
    for t, a in enumerate(x.reshape(-1, G)):
        b = int(r["bits"][t])
        q, s, z, _ = oracle.quantize_tile(a, b)
        assert s == r["scales"][t] and z == r["zeros"][t]
        assert np.array_equal(oracle.pack_tile(q, b), r["codes"][off:off + G * b // 8])
        off += G * b // 8


def test_invalid_tau_rejected():
    x = _small()
    for tau in (-1.0, np.nan):
        with pytest.raises(RuntimeError):
            oracle.encode(x, 64, 64, 3, 4, 3.5, 0, tau=tau)


# ------------------------------------------------------------------ width mixes
# (Appendix G: 100% INT4, 50% INT4 + 50% INT3, 100% INT3; 80% INT2 + 20% INT3)

@pytest.mark.parametrize("lo,hi,beta,frac_hi", [(3, 4, 4.0, 1.0), (3, 4, 3.5, 0.5),
                                                 (3, 4, 3.0, 0.0), (2, 3, 2.2, 0.2)])
def test_appendix_g_width_mixes(lo, hi, beta, frac_hi):
    x = _small()
    T, Cc = x.shape
    G = 64
    r = oracle.encode(x, G, G, lo, hi, beta, 16)
    n_g = 16 * Cc // G
    K = int(np.floor(frac_hi * n_g + 1e-9))
    for g in range(T // 16):
        assert np.count_nonzero(r["bits"][g * n_g:(g + 1) * n_g] == hi) == K
    n = T * Cc // G
    n_hi = np.count_nonzero(r["bits"] == hi)
    assert r["codes"].size == (n * lo + n_hi * (hi - lo)) * G // 8
    assert r["codes"].size * 8 <= beta * T * Cc


# ------------------------------------------------------------------ allocation tiles A != G
# (§3.2 "Tile decomposition": one key per allocation tile of A channels, A a multiple of G
# aligned with the quantisation tiles; A = C is the token-level allocation)

@pytest.mark.parametrize("n", [256, 1024, 8192])
def test_entropy_key_n_closed_forms(n):
    assert oracle.entropy_key_n(np.full(n, 0.5, F32)) == np.log2(n)           # flat
    for k in (1, 2, 4, 64):
        a = np.zeros(n, F32)
        a[np.arange(k) * (n // k)] = -4.0 if k % 2 else 0.5         # powers of two: exact
        assert oracle.entropy_key_n(a) == np.log2(k)                          # k equal spikes
    assert oracle.entropy_key_n(np.zeros(n, F32)) == 0.0


def test_entropy_key_n_matches_the_literal_entropy():
    rng = np.random.default_rng(31)
    for n in (256, 2048):
        for _ in range(20):
            a = (rng.standard_normal(n) * rng.choice([1, 50], n, p=[0.99, 0.01])).astype(F32)
            p = np.abs(a.astype(np.float64)) / np.abs(a.astype(np.float64)).sum()
            lit = -np.sum(np.where(p > 0, p * np.log2(np.where(p > 0, p, 1)), 0.0))
            assert abs(oracle.entropy_key_n(a) - lit) < 2e-5


@pytest.mark.parametrize("A,S", [(128, 16), (256, 8), (512, 48), (64, 16)])
def test_encode_alloc_tiles(A, S):
    x = _small(C=512)
    T, C = x.shape
    G = 64
    m = A // G
    r = oracle.encode(x, G, G, 3, 4, 3.5, S, want_keys=True, alloc_tile=A)
    n = T * C // G
    assert r["keys"].size == n // m
    bits = r["bits"].reshape(-1, m)
    assert np.all(bits == bits[:, :1])                        # one width per allocation tile
    n_ga = S * C // A
    K = oracle.hi_count(n_ga, 3, 4, 3.5)
    for g in range(T // S):
        sl = slice(g * n_ga, (g + 1) * n_ga)
        assert np.count_nonzero(bits[sl, 0] == 4) == K
        assert np.array_equal(bits[sl, 0], oracle.allocate(r["keys"][sl], K, 3, 4))
    rows = x.reshape(-1, A)
    for i in range(0, rows.shape[0], 7):
        assert r["keys"][i] == oracle.entropy_key_n(rows[i])
    assert r["codes"].size == oracle.payload_size(T, C, G, 3, 4, 3.5, S, A) == \
        T // S * (S * C // G * G * 3 // 8 + K * A // 8)
    # the per-tile steps do not depend on A
    base = oracle.encode(x, G, G, 3, 4, 3.5, S)
    assert np.array_equal(r["pivots"], base["pivots"])
    if A == G:
        for k in base:
            assert np.array_equal(base[k], r[k]), k


def test_token_level_allocation_is_a_special_case():
    x = _small(C=512)
    T, C = x.shape
    r = oracle.encode(x, 64, 64, 3, 4, 3.5, 0, want_keys=True, alloc_tile=C)
    tok_bits = r["bits"].reshape(T, -1)
    assert np.all(tok_bits == tok_bits[:, :1])
    hi = tok_bits[:, 0] == 4
    assert hi.sum() == oracle.hi_count(T, 3, 4, 3.5)
    assert r["keys"][hi].min() >= r["keys"][~hi].max()


def test_invalid_alloc_tile_rejected():
    x = _small(C=512)
    for A in (32, 96, 192, 1024):     # below G, not a multiple, not a power-of-two multiple, above C
        with pytest.raises((RuntimeError, ValueError)):
            oracle.encode(x, 64, 64, 3, 4, 3.5, 0, alloc_tile=A)
