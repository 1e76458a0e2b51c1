"""GPU-vs-oracle parity of the wire format (``-m gpu``), through the C ABI.

"TAH-Quant" §3.2 / §3.4: one fixed-size buffer holding the width map, the per-tile
metadata and the payload.  The acceptance rule is the plain codec's: every byte outside
the payload (header, width map, fp16 scale and zero with the flag, pivot fields, zero
padding) bit-exact; payload codes bit-exact except elements on a rounding boundary (the
oracle flags them); decoded fp32 within 1e-5 relative L2 of the oracle's decode of its
own buffer, and the GPU decoder on the oracle's buffer equally close.
"""
import numpy as np
import pytest

import oracle
import pipeline_activation_quantization_gb300 as tq
import synth
from _parity import code_mismatches, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_cuda():
    import torch
    assert torch.cuda.is_available(), "the -m gpu tests need a CUDA device"
    tq.lib()


def _rel(a, b):
    b64 = b.astype(np.float64)
    den = np.linalg.norm(b64)
    return np.linalg.norm(a.astype(np.float64) - b64) / (den if den > 0 else 1.0)


def _check_wire(x, G, h, lo, hi, beta, S, tau=2.0):
    import torch
    T, C = x.shape
    xt = to_device(x)
    wire_g, ws = tq.encode_wire(xt, G, h, lo, hi, beta, S, tau=tau)
    torch.cuda.synchronize()
    rc, st = tq.tahq_get_device_status(ws)
    assert st == 0, f"encode status {st:#x}"
    gw = wire_g.cpu().numpy()
    ow, near = oracle.encode_wire(x, G, h, lo, hi, beta, S, tau=tau, want_near=True)
    assert gw.size == ow.size == tq.tahq_wire_size(T, C, G, lo, hi, beta, S)
    hd = oracle.wire_header(ow)
    a, b = hd["off_payload"], hd["off_payload"] + hd["payload_bytes"]
    # everything but the payload: bit-exact
    bad = np.flatnonzero(np.concatenate([gw[:a] != ow[:a], gw[b:] != ow[b:]]))
    assert bad.size == 0, f"{bad.size} metadata bytes differ, first at {bad[:8]}"
    # payload: the codes, boundary elements aside
    n = hd["tiles"]
    wmap = np.unpackbits(ow[hd["off_map"]:hd["off_map"] + (n + 7) // 8], bitorder="little")[:n]
    bits = np.where(wmap == 1, hi, lo).astype(np.uint8)
    mism = code_mismatches(gw[a:b], ow[a:b], bits, G)
    if mism.size:
        assert np.all(near.reshape(-1)[mism] == 1), f"code mismatch off a boundary at {mism[:8]}"
        assert mism.size <= 1e-6 * x.size
    # decode: GPU of its own buffer and of the oracle's, against the oracle
    y_ref = oracle.decode_wire(ow)
    y_g, dws = tq.decode_wire(wire_g, T, C, G, h, lo, hi, beta, S)
    y_x, dws2 = tq.decode_wire(torch.from_numpy(ow).cuda(), T, C, G, h, lo, hi, beta, S)
    torch.cuda.synchronize()
    for w in (dws, dws2):
        rc, st = tq.tahq_get_device_status(w)
        assert st == 0, f"decode status {st:#x}"
    assert _rel(y_g.cpu().numpy(), y_ref) <= 1e-5
    assert _rel(y_x.cpu().numpy(), y_ref) <= 1e-5
    return {"code_mismatches": int(mism.size), "wire_bytes": int(gw.size)}


WIRE = [
    # dtype, dist, G, h, lo, hi, beta, T, C, S
    ("f32", "laplace", 128, 128, 3, 4, 3.5, 40, 2176, 20),
    ("f32", "gauss_rms_spikes", 64, 64, 3, 4, 3.8, 96, 1088, 32),
    ("bf16", "gauss_rms_spikes", 64, 64, 3, 4, 3.5, 96, 1088, 32),
    ("bf16", "student_t", 32, 16, 2, 3, 2.2, 80, 2080, 16),
    ("f32", "student_t", 16, 16, 3, 4, 3.5, 33, 400, 11),
    ("f32", "gauss_rms_spikes", 8, 8, 3, 5, 4.0, 30, 264, 10),
    ("f32", "laplace", 64, 64, 3, 4, 3.0, 64, 512, 0),       # one width (K = 0)
    ("bf16", "laplace", 128, 64, 3, 4, 4.0, 48, 1152, 16),   # one width (K = n_g)
    # groups of whole 32 KB chunks: the three-stage encoder with the wire quantiser
    ("f32", "laplace", 128, 128, 3, 4, 3.5, 64, 512, 16),
    ("bf16", "gauss_rms_spikes", 64, 64, 3, 4, 3.5, 64, 2048, 16),
    ("f32", "student_t", 32, 32, 3, 4, 3.25, 64, 1024, 16),
    ("bf16", "laplace", 128, 64, 3, 4, 3.75, 32, 1024, 16),
]


@pytest.mark.parametrize("dtype,dist,G,h,lo,hi,beta,T,C,S", WIRE)
def test_wire_parity(dtype, dist, G, h, lo, hi, beta, T, C, S):
    w = synth.Workload("wire", T, C, dtype, G, h, lo, hi, beta, S, 700 + T + G, dist)
    print("wire", _check_wire(synth.generate(w), G, h, lo, hi, beta, S))


@pytest.mark.parametrize("tau", [0.0, float("inf")])
def test_wire_tau(tau):
    w = synth.Workload("wire", 64, 1024, "f32", 64, 64, 3, 4, 3.5, 16, 901, "gauss_rms_spikes")
    print("wire tau", tau, _check_wire(synth.generate(w), 64, 64, 3, 4, 3.5, 16, tau))


def test_wire_every_tile_flagged():
    # one spike in every tile of 128: the three-stage encoder's exact path on all tiles
    rng = np.random.default_rng(31)
    x = (rng.standard_normal((64, 512)) * 1e-3).astype(np.float32)
    t = x.reshape(-1, 128)
    t[np.arange(t.shape[0]), rng.integers(0, 128, t.shape[0])] = np.float32(-6.0)
    print("wire spikes", _check_wire(x, 128, 128, 3, 4, 3.5, 16))


def test_wire_full_c3():
    w = synth.WORKLOADS["c3"]
    print("wire c3", _check_wire(synth.generate(w), w.tile, w.hblock, w.bits_lo, w.bits_hi,
                                 w.budget, w.tokens_per_group))


def test_wire_empty_tensor_has_a_header():
    import torch
    x = torch.zeros((0, 256), device="cuda")
    wire, _ = tq.encode_wire(x, 64, 64, 3, 4, 3.5, 0)
    torch.cuda.synchronize()
    ow = oracle.encode_wire(np.zeros((0, 256), np.float32), 64, 64, 3, 4, 3.5, 0)
    assert np.array_equal(wire.cpu().numpy(), ow)


def test_wire_header_mismatch_sets_status():
    import torch
    w = synth.Workload("wire", 32, 512, "f32", 64, 64, 3, 4, 3.5, 0, 77, "laplace")
    xt = to_device(synth.generate(w))
    wire, _ = tq.encode_wire(xt, 64, 64, 3, 4, 3.5, 0)
    # the same layout, another hblock: decoded with the caller's, flagged in the status
    y, dws = tq.decode_wire(wire, 32, 512, 64, 32, 3, 4, 3.5, 0)
    torch.cuda.synchronize()
    rc, st = tq.tahq_get_device_status(dws)
    assert st & tq.DEV_BAD_WIRE
