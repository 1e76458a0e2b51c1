"""Helpers of the GPU-vs-oracle parity tests (imported by the ``-m gpu`` test files).

The CUDA path is called through the C ABI (``pipeline_activation_quantization_gb300``);
the oracle through its ctypes wrapper.  The two never share code: only the seeded
inputs from ``synth`` are common.
"""
from __future__ import annotations

import os

import numpy as np

import oracle
import pipeline_activation_quantization_gb300 as tq

HOST_THREADS = min(16, os.cpu_count() or 1)


def to_device(x: np.ndarray):
    import torch
    if x.dtype == np.uint16:
        return torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda()


def gpu_roundtrip(x: np.ndarray, G, h, lo, hi, beta, S, tau=None, alloc_tile=None) -> dict:
    """Encode and decode on the GPU; return host copies plus both status words."""
    import torch
    T, C = x.shape
    xt = to_device(x)
    enc = tq.encode(xt, G, h, lo, hi, beta, S, tau=tau, alloc_tile=alloc_tile)
    y = tq.decode(enc, T, C, G, h)
    torch.cuda.synchronize()
    rc_e, st_e = tq.tahq_get_device_status(enc["workspace"])
    out = {k: enc[k].cpu().numpy() for k in ("codes", "scales", "zeros", "bits", "pivots")}
    out["y"] = y.cpu().numpy()
    out["status_encode"] = st_e
    return out


def oracle_roundtrip(x: np.ndarray, G, h, lo, hi, beta, S, tau=None, alloc_tile=None) -> dict:
    T, C = x.shape
    r = oracle.encode(x, G, h, lo, hi, beta, S, threads=HOST_THREADS, want_near=True, tau=tau,
                      alloc_tile=alloc_tile)
    r["y"] = oracle.decode(r["codes"], r["scales"], r["zeros"], r["bits"], r["pivots"], T, C, G, h,
                           threads=HOST_THREADS)
    return r


def code_mismatches(a: np.ndarray, b: np.ndarray, bits: np.ndarray, G: int) -> np.ndarray:
    """Element indices (tile * G + k) whose unpacked codes differ between two streams."""
    diff = np.flatnonzero(a != b)
    if diff.size == 0:
        return diff
    slot = bits.astype(np.int64) * G // 8
    start = np.concatenate([[0], np.cumsum(slot)])
    tiles = np.unique(np.searchsorted(start, diff, side="right") - 1)
    out = []
    for t in tiles:
        o, n = int(start[t]), int(slot[t])
        qa = oracle.unpack_tile(a[o:o + n], G, int(bits[t]))
        qb = oracle.unpack_tile(b[o:o + n], G, int(bits[t]))
        out.extend(int(t) * G + np.flatnonzero(qa != qb))
    return np.array(out, dtype=np.int64)


def assert_parity(gpu: dict, ora: dict, G: int, max_rel_l2: float = 1e-5) -> dict:
    """The acceptance rule: bits and pivots bit-exact; codes bit-exact except elements
    whose oracle pre-rounding value is within 1e-5 relative of a .5 boundary (at most
    1e-6 of all elements); scales and zeros bit-exact; decoded fp32 within max_rel_l2
    relative L2 of the oracle's decode.  Returns a small report."""
    n_el = ora["y"].size
    assert gpu["status_encode"] == 0, f"device status {gpu['status_encode']:#x}"
    assert np.array_equal(gpu["bits"], ora["bits"]), \
        f"bits differ at {np.flatnonzero(gpu['bits'] != ora['bits'])[:10]}"
    assert np.array_equal(gpu["pivots"], ora["pivots"]), \
        f"pivots differ at {np.flatnonzero(gpu['pivots'] != ora['pivots'])[:10]}"
    assert gpu["codes"].size == ora["codes"].size
    mism = code_mismatches(gpu["codes"], ora["codes"], ora["bits"], G)
    if mism.size:
        near = ora["near"].reshape(-1)
        assert np.all(near[mism] == 1), f"code mismatch off a rounding boundary at {mism[:10]}"
        assert mism.size <= 1e-6 * n_el, f"{mism.size} boundary mismatches"
    assert np.array_equal(gpu["scales"].view(np.uint32), ora["scales"].view(np.uint32)), \
        f"scales differ at {np.flatnonzero(gpu['scales'].view(np.uint32) != ora['scales'].view(np.uint32))[:10]}"
    assert np.array_equal(gpu["zeros"].view(np.uint32), ora["zeros"].view(np.uint32))
    ref = ora["y"].astype(np.float64)
    den = np.linalg.norm(ref)
    rel = np.linalg.norm(gpu["y"].astype(np.float64) - ref) / (den if den > 0 else 1.0)
    assert rel <= max_rel_l2, rel
    return {"code_mismatches": int(mism.size), "near_boundary": int(ora["near"].sum()),
            "rel_l2": float(rel), "decode_bit_exact": bool(np.array_equal(gpu["y"], ora["y"]))}
