"""GPU-vs-oracle parity on the shapes the library encodes with its three-stage encoder
(``-m gpu``, through the C ABI).

The method's defaults — widths {3, 4}, tau = 2 ("TAH-Quant" §3.3 eq. (3)), allocation per
tile (§3.2) — on tiles of 128-byte lines or more (fp32 tiles of 32, 64, 128 values, bf16
of 64, 128) and groups of whole 32 KB input chunks take the streaming encoder (keys and
histograms; select; widths and chunk offsets; quantiser with the exact path); slots that
are not 16-byte multiples (tiles of 32 and 64) are stored a word at a time.  These cases
cover its special inputs: ties of every key, every tile flagged (all through the exact
path), ratio exactly tau, zero and subnormal tiles, several chunks and groups.  The
acceptance rule is ``_parity.assert_parity``.
"""
import numpy as np
import pytest

import pipeline_activation_quantization_gb300 as tq
import synth
from _parity import assert_parity, gpu_roundtrip, oracle_roundtrip

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_cuda():
    import torch
    assert torch.cuda.is_available(), "the -m gpu tests need a CUDA device"
    tq.lib()


def _check(x, beta, S, G=128, tau=None):
    gpu = gpu_roundtrip(x, G, G, 3, 4, beta, S, tau)
    ora = oracle_roundtrip(x, G, G, 3, 4, beta, S, tau)
    return assert_parity(gpu, ora, G)


def _edge(T, C, seed, G=128):
    rng = np.random.default_rng(seed)
    tiles = lambda a: a.reshape(-1, G)  # noqa: E731
    out = {"zeros": np.zeros((T, C), np.float32),
           "constant": np.full((T, C), 1.5, np.float32)}
    out["flat_signs"] = (np.where(rng.random((T, C)) < 0.5, -1.0, 1.0) * 0.25).astype(np.float32)
    # one spike in every tile over small noise: every tile deferred and transformed
    sp = (rng.standard_normal((T, C)) * 1e-3).astype(np.float32)
    n = T * C // G
    tiles(sp)[np.arange(n), rng.integers(0, G, n)] = np.float32(8.0)
    out["spike_every_tile"] = sp
    out["subnormal"] = (rng.standard_normal((T, C)) * 1e-39).astype(np.float32)
    edge = np.zeros((T, C), np.float32)
    tiles(edge)[:, 3] = 1.0
    tiles(edge)[:, G - 9] = 0.5                               # r == tau exactly
    tiles(edge)[::2, 3] = np.float32(1.0 + 2.0 ** -23)        # r just above tau
    out["ratio_edge"] = edge
    mixed = rng.standard_normal((T, C)).astype(np.float32)
    tiles(mixed)[::3] *= np.float32(2.0 ** -20)
    tiles(mixed)[1::5] = 0.0
    tiles(mixed)[2::7, 5] = np.float32(300.0)                 # a flagged tile now and then
    out["mixed_scale"] = mixed
    return out


F32_EDGE = _edge(64, 512, 11)    # 4 tiles a token, groups of 16 tokens = one chunk
BF16_EDGE = _edge(64, 1024, 12)  # 8 tiles a token, groups of 16 tokens = one bf16 chunk


@pytest.mark.parametrize("name", sorted(F32_EDGE))
def test_edge_f32(name):
    print(name, _check(F32_EDGE[name], 3.5, 16))


@pytest.mark.parametrize("name", sorted(BF16_EDGE))
def test_edge_bf16(name):
    print(name, _check(synth.f32_to_bf16_bits(BF16_EDGE[name]), 3.5, 16))


@pytest.mark.parametrize("dtype,dist,beta,T,C,S", [
    ("f32", "laplace", 3.5, 128, 4096, 32),             # 16 chunks a group, 4 groups
    ("f32", "gauss_rms_spikes", 3.25, 96, 2048, 16),    # 4 chunks a group, 6 groups
    ("bf16", "gauss_fixed_channels", 3.75, 64, 4096, 32),
    ("bf16", "student_t", 3.5, 48, 2048, 48),           # one group
])
def test_distributions(dtype, dist, beta, T, C, S):
    w = synth.Workload("three", T, C, dtype, 128, 128, 3, 4, beta, S, 900 + T, dist)
    print(dist, _check(synth.generate(w), beta, S))


# tiles of 32 and 64 values: slots of 12 / 16 and 24 / 32 bytes, stored a word at a time;
# groups of 16 tokens = 2, 4 and 2 chunks
@pytest.mark.parametrize("dtype,G,C", [("f32", 32, 1024), ("f32", 64, 2048), ("bf16", 64, 2048)])
@pytest.mark.parametrize("name", ["spike_every_tile", "ratio_edge", "mixed_scale", "zeros"])
def test_word_slots_edge(dtype, G, C, name):
    x = _edge(64, C, 13 + G, G)[name]
    if dtype == "bf16":
        x = synth.f32_to_bf16_bits(x)
    print(dtype, G, name, _check(x, 3.5, 16, G))


@pytest.mark.parametrize("dtype,G,dist,beta,T,C,S", [
    ("f32", 32, "laplace", 3.5, 96, 2048, 32),
    ("f32", 64, "gauss_rms_spikes", 3.25, 64, 4096, 16),
    ("bf16", 64, "gauss_rms_spikes", 3.5, 128, 4096, 64),   # the bf16 pipeline-boundary shape
    ("bf16", 64, "student_t", 3.75, 64, 2048, 32),
])
def test_word_slots_distributions(dtype, G, dist, beta, T, C, S):
    w = synth.Workload("three", T, C, dtype, G, G, 3, 4, beta, S, 950 + T + G, dist)
    print(dtype, G, dist, _check(synth.generate(w), beta, S, G))


# the outlier threshold as a parameter (Appendix F: 0, 2, 4, infinity; 0.5 and 1.5 also
# take the pretest's rounded-up threshold and, below 1, no shortcut for tiny tiles)
@pytest.mark.parametrize("tau", [0.0, 0.5, 1.5, 4.0, float("inf")])
@pytest.mark.parametrize("dtype,G,C,name", [("f32", 128, 512, "mixed_scale"),
                                            ("f32", 128, 512, "ratio_edge"),
                                            ("bf16", 64, 2048, "spike_every_tile"),
                                            ("f32", 32, 1024, "subnormal")])
def test_tau_edge(dtype, G, C, name, tau):
    x = _edge(64, C, 17 + G, G)[name]
    if dtype == "bf16":
        x = synth.f32_to_bf16_bits(x)
    print(dtype, G, name, tau, _check(x, 3.5, 16, G, tau))


@pytest.mark.parametrize("tau", [0.0, 1.5, 4.0, float("inf")])
def test_tau_distribution(tau):
    w = synth.Workload("three", 96, 2048, "f32", 128, 128, 3, 4, 3.5, 16, 990, "gauss_rms_spikes")
    print(tau, _check(synth.generate(w), 3.5, 16, 128, tau))
