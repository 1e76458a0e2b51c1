"""GPU-vs-oracle parity of the sm_103a codec, through the C ABI (``-m gpu``).

Acceptance rule (bits/pivots/scales/zeros bit-exact, codes bit-exact except boundary
elements, decode within 1e-5 relative L2) is in ``_parity.assert_parity``.  Inputs are
seeded synthetic tensors from ``synth`` shaped like the pipeline boundaries of
"TAH-Quant" §5.1; the small cases span several kernel chunks and a ragged tail.
"""
import numpy as np
import pytest

import oracle
import pipeline_activation_quantization_gb300 as tq
import synth
from _parity import assert_parity, gpu_roundtrip, oracle_roundtrip, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_cuda():
    import torch
    assert torch.cuda.is_available(), "the -m gpu tests need a CUDA device"
    tq.lib()


def _check(x, G, h, lo, hi, beta, S, tau=None, alloc_tile=None):
    gpu = gpu_roundtrip(x, G, h, lo, hi, beta, S, tau, alloc_tile)
    ora = oracle_roundtrip(x, G, h, lo, hi, beta, S, tau, alloc_tile)
    return assert_parity(gpu, ora, G)


# ------------------------------------------------------------------ small grid

SMALL = [
    # dtype, dist, G, h, lo, hi, beta, T, C, S
    ("bf16", "gauss_rms_spikes", 64, 64, 3, 4, 3.5, 96, 1088, 32),
    ("f32", "laplace", 64, 64, 3, 4, 3.5, 96, 1088, 32),
    ("bf16", "student_t", 32, 32, 3, 4, 3.25, 80, 2080, 16),
    ("f32", "gauss_fixed_channels", 128, 128, 3, 4, 3.9, 40, 2176, 20),
    ("bf16", "gauss_rms_spikes", 128, 32, 2, 4, 3.0, 48, 1152, 0),
    ("f32", "student_t", 8, 8, 3, 4, 3.5, 30, 264, 10),
    ("bf16", "laplace", 8, 4, 1, 8, 4.4, 24, 200, 12),
    ("f32", "gauss_rms_spikes", 16, 2, 3, 5, 4.0, 33, 400, 11),
    ("bf16", "student_t", 64, 16, 7, 8, 7.5, 64, 1024, 8),
    ("f32", "laplace", 32, 32, 3, 4, 3.0, 64, 512, 0),      # K = 0: all tiles get lo
    ("bf16", "laplace", 64, 64, 3, 4, 4.0, 64, 512, 16),    # K = n_g: all tiles get hi
    ("bf16", "gauss_rms_spikes", 16, 16, 3, 4, 3.5, 512, 2048, 0),   # one group, 64 chunks
    ("f32", "laplace", 128, 64, 3, 4, 3.7, 257, 1024, 257),
]


@pytest.mark.parametrize("dtype,dist,G,h,lo,hi,beta,T,C,S", SMALL)
def test_small_grid(dtype, dist, G, h, lo, hi, beta, T, C, S):
    w = synth.Workload("small", T, C, dtype, G, h, lo, hi, beta, S, 100 + T + G, dist)
    _check(synth.generate(w), G, h, lo, hi, beta, S)


# ------------------------------------------------------------------ the threshold tau
# ("TAH-Quant" Appendix F: tau = 0 always transforms, tau = inf never, tau = 4); every
# layout of the encoder, the one-width kernels included

TAU = [
    # dtype, dist, G, h, lo, hi, beta, T, C, S
    ("f32", "laplace", 128, 128, 3, 4, 3.5, 40, 2176, 20),
    ("f32", "gauss_rms_spikes", 64, 32, 3, 4, 3.5, 96, 1088, 32),
    ("bf16", "gauss_rms_spikes", 64, 64, 3, 4, 3.5, 96, 1088, 32),
    ("f32", "student_t", 16, 16, 3, 4, 3.5, 33, 400, 11),
    ("bf16", "laplace", 32, 8, 3, 4, 3.25, 80, 2080, 16),
    ("f32", "laplace", 64, 64, 3, 4, 3.0, 64, 512, 0),      # one width (K = 0)
    ("bf16", "gauss_rms_spikes", 128, 128, 3, 4, 4.0, 48, 1152, 16),   # one width (K = n_g)
]


@pytest.mark.parametrize("tau", [0.0, 1.5, 4.0, float("inf")])
@pytest.mark.parametrize("dtype,dist,G,h,lo,hi,beta,T,C,S", TAU)
def test_tau(dtype, dist, G, h, lo, hi, beta, T, C, S, tau):
    w = synth.Workload("tau", T, C, dtype, G, h, lo, hi, beta, S, 300 + T + G, dist)
    rep = _check(synth.generate(w), G, h, lo, hi, beta, S, tau)
    print("tau", tau, rep)


def test_tau_rejects_negative_and_nan():
    import torch
    x = torch.zeros(8, 64, device="cuda")
    for tau in (-1.0, float("nan")):
        with pytest.raises(tq.TahqError):
            tq.encode(x, 64, 64, 3, 4, 3.5, 0, tau=tau)


# ------------------------------------------------------------------ allocation tiles
# ("TAH-Quant" §3.2 "Tile decomposition": one key per A channels; A = C is token-level)

ALLOC = [
    # dtype, dist, G, A, lo, hi, beta, T, C, S
    ("f32", "laplace", 128, 256, 3, 4, 3.5, 64, 2048, 16),
    ("f32", "gauss_rms_spikes", 128, 8192, 3, 4, 3.5, 64, 8192, 32),     # token-level, 32 KB
    ("f32", "student_t", 64, 512, 3, 4, 3.25, 96, 1024, 32),
    ("bf16", "gauss_rms_spikes", 64, 4096, 3, 4, 3.5, 80, 4096, 40),     # token-level
    ("bf16", "laplace", 64, 128, 2, 3, 2.2, 96, 1152, 32),
    ("bf16", "student_t", 32, 256, 3, 4, 3.5, 80, 2048, 16),             # narrow layout
    ("f32", "gauss_rms_spikes", 16, 64, 3, 4, 3.5, 33, 448, 11),         # narrow layout
    ("f32", "laplace", 64, 1024, 3, 4, 3.0, 64, 1024, 0),                # K = 0 (one width)
]


@pytest.mark.parametrize("dtype,dist,G,A,lo,hi,beta,T,C,S", ALLOC)
def test_alloc_tiles(dtype, dist, G, A, lo, hi, beta, T, C, S):
    w = synth.Workload("alloc", T, C, dtype, G, G, lo, hi, beta, S, 1100 + T + A, dist)
    print("alloc", A, _check(synth.generate(w), G, G, lo, hi, beta, S, None, A))


# ------------------------------------------------------------------ width mixes
# (Appendix G: 80% INT2 + 20% INT3, 50% INT4 + 50% INT3)

@pytest.mark.parametrize("dtype,G,lo,hi,beta", [("f32", 128, 2, 3, 2.2), ("bf16", 64, 2, 3, 2.2),
                                                ("f32", 32, 2, 3, 2.2), ("bf16", 16, 2, 3, 2.2),
                                                ("f32", 64, 3, 4, 3.5)])
def test_appendix_g_mixes(dtype, G, lo, hi, beta):
    w = synth.Workload("mix", 64, 2048, dtype, G, G, lo, hi, beta, 16, 500 + G, "laplace")
    print("mix", lo, hi, beta, _check(synth.generate(w), G, G, lo, hi, beta, 16))


# ------------------------------------------------------------------ full-size workloads

@pytest.mark.parametrize("name", ["c1", "c2", "c3"])
def test_full_workload(name):
    w = synth.WORKLOADS[name]
    rep = _check(synth.generate(w), w.tile, w.hblock, w.bits_lo, w.bits_hi, w.budget,
                 w.tokens_per_group)
    print(name, rep)


@pytest.fixture(scope="module")
def c4_tensor():
    return synth.generate(synth.WORKLOADS["c4"])


@pytest.mark.parametrize("G,beta", synth.C4_SWEEP)
def test_c4_sweep(c4_tensor, G, beta):
    w = synth.WORKLOADS["c4"]
    rep = _check(c4_tensor, G, G, w.bits_lo, w.bits_hi, beta, w.tokens_per_group)
    print("c4", G, beta, rep)


@pytest.mark.parametrize("index", [0, 1])
def test_c5_fresh_tensors(index):
    w = synth.WORKLOADS["c5"]
    rep = _check(synth.generate(w, index=index), w.tile, w.hblock, w.bits_lo, w.bits_hi,
                 w.budget, w.tokens_per_group)
    print("c5", index, rep)


# ------------------------------------------------------------------ edge cases

def _edge_tensors():
    rng = np.random.default_rng(7)
    out = {}
    out["zeros"] = np.zeros((16, 512), np.float32)                      # all keys tie at 0
    out["constant"] = np.full((16, 512), -2.75, np.float32)
    flat = np.where(rng.random((16, 512)) < 0.5, -1.0, 1.0).astype(np.float32)
    out["flat_signs"] = flat * np.float32(0.5)                           # all keys = log2 G
    sp = np.zeros((16, 512), np.float32)
    for t in range(16 * 8):
        sp.reshape(-1, 64)[t, rng.integers(0, 64)] = np.float32(2.0 ** rng.integers(-10, 10))
    out["spikes"] = sp
    sub = (rng.standard_normal((16, 512)) * 1e-39).astype(np.float32)   # subnormal fp32
    out["subnormal"] = sub
    big = (rng.standard_normal((16, 512)) * 1e30).astype(np.float32)
    out["large"] = big
    edge = np.zeros((16, 512), np.float32)
    edge.reshape(-1, 64)[:, 0] = 1.0
    edge.reshape(-1, 64)[:, 1] = 0.5                                     # r == tau exactly
    edge.reshape(-1, 64)[::2, 0] = np.float32(1.0 + 2.0 ** -23)          # r just above tau
    out["ratio_edge"] = edge
    mixed = rng.standard_normal((16, 512)).astype(np.float32)
    mixed.reshape(-1, 64)[::3] *= np.float32(2.0 ** -20)
    mixed.reshape(-1, 64)[1::5] = 0.0
    out["mixed_scale"] = mixed
    return out


EDGE = _edge_tensors()


@pytest.mark.parametrize("name", sorted(EDGE))
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_edge_cases(name, dtype):
    x = EDGE[name]
    if dtype == "bf16":
        x = synth.f32_to_bf16_bits(x)
    _check(x, 64, 64, 3, 4, 3.5, 4)


# The same value patterns with token groups of whole 32 KB input chunks and tiles of 32 to
# 128 values, the shapes the streaming encoder takes (ranked at 3.5 bits, one width at 3):
# ties of every key in the group (zeros, constant, flat signs), subnormal and huge values,
# ratios at tau and just above.
@pytest.mark.parametrize("name", sorted(EDGE))
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("beta", [3.5, 3.0])
def test_edge_cases_whole_chunk_groups(name, dtype, beta):
    x = np.tile(EDGE[name], (4, 4))  # 64 x 2048; tiles of 64 keep their values
    if dtype == "bf16":
        x = synth.f32_to_bf16_bits(x)
    _check(x, 64, 64, 3, 4, beta, 16)


SMALL_STREAM = [
    # dtype, dist, G, h, beta, T, C, S: groups of whole input chunks
    ("f32", "laplace", 64, 64, 3.5, 64, 2048, 16),
    ("bf16", "gauss_rms_spikes", 64, 32, 3.5, 64, 2048, 16),
    ("f32", "student_t", 32, 32, 3.25, 32, 4096, 8),
    ("bf16", "laplace", 32, 16, 3.75, 64, 2048, 32),
    ("f32", "gauss_fixed_channels", 128, 128, 3.5, 64, 2048, 32),
    ("bf16", "student_t", 128, 64, 3.1, 64, 4096, 16),
]


@pytest.mark.parametrize("dtype,dist,G,h,beta,T,C,S", SMALL_STREAM)
def test_small_whole_chunk_groups(dtype, dist, G, h, beta, T, C, S):
    w = synth.Workload("small", T, C, dtype, G, h, 3, 4, beta, S, 200 + T + G, dist)
    _check(synth.generate(w), G, h, 3, 4, beta, S)


@pytest.mark.parametrize("tau", [0.0, 1.5, 4.0, float("inf")])
@pytest.mark.parametrize("dtype,dist,G,h,beta,T,C,S", [SMALL_STREAM[4], SMALL_STREAM[1],
                                                       ("bf16", "gauss_rms_spikes", 64, 64, 3.0, 64, 2048, 16)])
def test_tau_whole_chunk_groups(dtype, dist, G, h, beta, T, C, S, tau):
    """Outlier thresholds of Appendix F on the streaming encoder's shapes (ranked and one
    width): the pretest's threshold m1 / tau rounded up, the exact test by a division."""
    w = synth.Workload("small", T, C, dtype, G, h, 3, 4, beta, S, 300 + T + G, dist)
    _check(synth.generate(w), G, h, 3, 4, beta, S, tau)


@pytest.mark.parametrize("T,C,S", [(16, 8192, 16), (64, 8192, 64)])
def test_all_keys_tie_in_a_large_group(T, C, S):
    """Every tile's key equal: the whole group is the select's window (2048 candidates:
    the histogram rank; 8192: the radix select over the candidates in memory)."""
    rng = np.random.default_rng(11)
    x = (np.where(rng.random((T, C)) < 0.5, -1.0, 1.0) * 0.75).astype(np.float32)
    _check(x, 64, 64, 3, 4, 3.5, S)


def test_bf16_subnormal_and_single_tile():
    x = (np.arange(64, dtype=np.uint16) + np.uint16(1)).reshape(1, 64)   # bf16 subnormals
    x[0, 5] |= np.uint16(0x8000)
    _check(x, 64, 64, 3, 4, 3.5, 0)
    _check(synth.f32_to_bf16_bits(np.linspace(-3, 5, 8, dtype=np.float32).reshape(1, 8)),
           8, 8, 3, 4, 3.5, 0)


def test_empty_tensor():
    import torch
    x = torch.zeros((0, 128), dtype=torch.float32, device="cuda")
    enc = tq.encode(x, 64, 64, 3, 4, 3.5, 0)
    assert enc["payload_bytes"] == 0
    y = tq.decode(enc, 0, 128, 64, 64)
    torch.cuda.synchronize()
    assert y.shape == (0, 128)
    assert tq.tahq_get_device_status(enc["workspace"])[0] == 0


def test_exact_chunk_multiple():
    # n_g a multiple of the bf16 G=64 chunk (256 tiles), several groups
    w = synth.Workload("chunks", 256, 2048, "bf16", 64, 64, 3, 4, 3.5, 64, 5, "gauss_rms_spikes")
    _check(synth.generate(w), 64, 64, 3, 4, 3.5, 64)


# ------------------------------------------------------------------ device status, bounds

def test_nonfinite_input_sets_status():
    import torch
    x = np.random.default_rng(1).standard_normal((8, 256)).astype(np.float32)
    x[3, 17] = np.nan
    x[5, 200] = np.inf
    enc = tq.encode(to_device(x), 64, 64, 3, 4, 3.5, 0)
    torch.cuda.synchronize()
    rc, word = tq.tahq_get_device_status(enc["workspace"])
    assert rc == 5 and (word & tq.DEV_NONFINITE)
    # a clean call on the same workspace clears the word
    enc = tq.encode(to_device(np.nan_to_num(x, posinf=1.0)), 64, 64, 3, 4, 3.5, 0,
                    workspace=enc["workspace"])
    assert tq.tahq_get_device_status(enc["workspace"]) == (0, 0)


def _encoded_small():
    import torch
    x = synth.generate(synth.Workload("d", 32, 512, "f32", 64, 64, 3, 4, 3.5, 0, 9, "laplace"))
    enc = tq.encode(to_device(x), 64, 64, 3, 4, 3.5, 0)
    torch.cuda.synchronize()
    return x, enc


def test_decode_rejects_bad_bits_and_pivots():
    import torch
    x, enc = _encoded_small()
    good = tq.decode(enc, 32, 512, 64, 64).cpu().numpy()
    bad = dict(enc)
    bad["bits"] = enc["bits"].clone()
    bad["bits"][10] = 0
    bad["bits"][11] = 9
    ws = torch.empty(tq.tahq_decode_workspace_size(32, 512, 64), dtype=torch.uint8, device="cuda")
    y = tq.decode(bad, 32, 512, 64, 64, workspace=ws).cpu().numpy()
    rc, word = tq.tahq_get_device_status(ws)
    assert rc == 5 and (word & tq.DEV_BAD_BITS)
    assert np.all(y.reshape(-1, 64)[10:12] == 0)
    bad = dict(enc)
    bad["pivots"] = enc["pivots"].clone()
    bad["pivots"][3] = 200
    y = tq.decode(bad, 32, 512, 64, 64, workspace=ws).cpu().numpy()
    rc, word = tq.tahq_get_device_status(ws)
    assert rc == 5 and (word & tq.DEV_BAD_BITS)
    assert np.all(y.reshape(-1, 64)[3] == 0)
    assert np.array_equal(y.reshape(-1, 64)[:3], good.reshape(-1, 64)[:3])


def test_decode_truncated_stream_is_bounded():
    import torch
    x, enc = _encoded_small()
    full = enc["codes"]
    cut = full.numel() // 2
    ws = torch.empty(tq.tahq_decode_workspace_size(32, 512, 64), dtype=torch.uint8, device="cuda")
    out = torch.empty((32, 512), dtype=torch.float32, device="cuda")
    rc = tq.tahq_decode(full, cut, enc["scales"], enc["zeros"], enc["bits"], enc["pivots"],
                        32, 512, 64, 64, out, ws, ws.numel())
    assert rc == 0
    rc, word = tq.tahq_get_device_status(ws)
    assert rc == 5 and (word & tq.DEV_STREAM_OVERRUN)
    good = tq.decode(enc, 32, 512, 64, 64).cpu().numpy().reshape(-1, 64)
    y = out.cpu().numpy().reshape(-1, 64)
    slot = enc["bits"].cpu().numpy().astype(np.int64) * 8
    end = np.cumsum(slot)
    inside = end <= cut
    assert np.array_equal(y[inside], good[inside])
    assert np.all(y[~inside] == 0)


# ------------------------------------------------------------------ memory hygiene

def test_outputs_do_not_write_past_their_ends():
    import torch
    T, C, G = 40, 1088, 64
    x = synth.generate(synth.Workload("g", T, C, "bf16", G, G, 3, 4, 3.5, 20, 3, "student_t"))
    n = T * C // G
    pay = tq.tahq_payload_size(T, C, G, 3, 4, 3.5, 20)
    guard = 4096
    dev = "cuda"

    def buf(nbytes):
        b = torch.full((nbytes + 2 * guard,), 0xA5, dtype=torch.uint8, device=dev)
        return b, b[guard:guard + nbytes]

    codes_b, codes = buf(pay)
    sc_b, sc = buf(4 * n)
    ze_b, ze = buf(4 * n)
    bi_b, bi = buf(n)
    pv_b, pv = buf(n)
    ws = torch.empty(tq.tahq_workspace_size(T, C, G, G, 3, 4, 3.5, 20), dtype=torch.uint8, device=dev)
    xt = to_device(x)
    rc = tq.tahq_encode(xt, tq.TAHQ_BF16, T, C, G, G, 3, 4, 3.5, 20, codes, sc, ze, bi, pv,
                        ws, ws.numel())
    assert rc == 0
    out_b, out = buf(4 * T * C)
    dws = torch.empty(tq.tahq_decode_workspace_size(T, C, G), dtype=torch.uint8, device=dev)
    rc = tq.tahq_decode(codes, pay, sc, ze, bi, pv, T, C, G, G, out, dws, dws.numel())
    assert rc == 0
    torch.cuda.synchronize()
    for b in (codes_b, sc_b, ze_b, bi_b, pv_b, out_b):
        h = b.cpu().numpy()
        assert np.all(h[:guard] == 0xA5) and np.all(h[-guard:] == 0xA5)
    ora = oracle.encode(x, G, G, 3, 4, 3.5, 20)
    assert np.array_equal(codes.cpu().numpy(), ora["codes"])


def test_repeat_calls_are_deterministic_and_stream_ordered():
    import torch
    w = synth.WORKLOADS["c2"]
    x = to_device(synth.generate(w))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        a = tq.encode(x, 64, 64, 3, 4, 3.5, 1024)
        ca = a["codes"].clone()
        b = tq.encode(x, 64, 64, 3, 4, 3.5, 1024, workspace=a["workspace"])
    s.synchronize()
    assert torch.equal(ca, b["codes"])
    for k in ("scales", "zeros", "bits", "pivots"):
        assert torch.equal(a[k], b[k])
