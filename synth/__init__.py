"""Seeded synthetic activation tensors shaped like pipeline-stage boundaries.

This module only draws random numbers. It holds none of the codec's arithmetic,
so both the CPU oracle's tests and the CUDA path can take their inputs from it.

Every tensor is row-major ``[tokens, channels]``. ``bf16`` tensors are returned as
``uint16`` bit patterns (rounded from fp32 to nearest-even); ``f32`` tensors as
``float32``. Draws come from ``numpy.random.Generator(PCG64(seed))`` in a fixed
order: base values, per-token RMS, outlier channels, per-channel factors,
element positions, signs. Tensor ``index`` of a workload uses the seed sequence
``SeedSequence([seed, index])``; its first child draws everything but the base
values, and child ``1 + i`` draws the base values of rows ``[1024 i, 1024 (i+1))``
(so blocks can be drawn on several host threads with the same result). Normal
draws are float32; the others are drawn in float64 and rounded to float32.
Counts use Python ``round``.

The workloads stand in for the activations that "TAH-Quant: Effective Activation
Quantization in Pipeline Parallelism over Slow Network" sends between stages
(§5.1: GPT2-XL / Qwen2.5-3B / LLaMA boundaries). No dataset or model weight is used.
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

__all__ = ["Workload", "WORKLOADS", "generate", "f32_to_bf16_bits", "bf16_bits_to_f32",
           "random_tiles"]

_ROW_BLOCK = 1024


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic activation workload and the codec parameters it is run with."""
    name: str
    tokens: int
    channels: int
    dtype: str            # "f32" or "bf16"
    tile: int
    hblock: int
    bits_lo: int
    bits_hi: int
    budget: float
    tokens_per_group: int  # 0 = one group over all tokens
    seed: int
    dist: str             # which value recipe (see ``generate``)

    def with_params(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    @property
    def elements(self) -> int:
        return self.tokens * self.channels

    @property
    def in_bytes(self) -> int:
        return self.elements * (4 if self.dtype == "f32" else 2)


WORKLOADS = {
    # 256 x 1024 fp32, N(0,1), channels {7,300,611,1000} x50; G=h=64, {3,4}, 3.5 bits, seed 0.
    "c1": Workload("c1_256x1024_f32", 256, 1024, "f32", 64, 64, 3, 4, 3.5, 0, 0, "gauss_fixed_channels"),
    # 4 x 1024 x 2048 bf16, 0.5*t(nu=3), 0.5% channels x exp(U[ln20, ln100]); G=64, 3.5 bits, seed 1.
    "c2": Workload("c2_4x1024x2048_bf16", 4096, 2048, "bf16", 64, 64, 3, 4, 3.5, 1024, 1, "student_t"),
    # 8 x 2048 x 4096 bf16, N(0,1)*rms_token (lognormal(0,0.5)), 0.2% channels x100, 1e-4 elements = +-500.
    "c3": Workload("c3_8x2048x4096_bf16", 16384, 4096, "bf16", 64, 64, 3, 4, 3.0, 2048, 2, "gauss_rms_spikes"),
    # same distribution at seed 3; tile/hblock and budget are swept by the caller.
    "c4": Workload("c4_8x2048x4096_bf16", 16384, 4096, "bf16", 64, 64, 3, 4, 3.5, 2048, 3, "gauss_rms_spikes"),
    # 16 x 2048 x 8192 fp32, Laplace(0,1), 0.1% channels x50; G=h=128, 3.5 bits, seed 4.
    "c5": Workload("c5_16x2048x8192_f32", 32768, 8192, "f32", 128, 128, 3, 4, 3.5, 2048, 4, "laplace"),
    # Backward gradients at the 70B-width boundary: 16 x 2048 x 8192 fp32, N(0,1) times a
    # per-token RMS LogNormal(0, 0.5) times 1e-5, 0.1% channels x30; the gradient codecs
    # (tile 64, 8 bits for the fixed-point one, 4 bits for TAH-Quant on gradients).
    "g5": Workload("g5_16x2048x8192_f32", 32768, 8192, "f32", 64, 64, 3, 4, 4.0, 2048, 5, "gradient"),
}

C4_SWEEP = [(g, b) for g in (32, 64, 128) for b in (3.0, 3.5, 4.0)]


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); return the uint16 bit patterns."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rnd = ((b >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((b + rnd) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bit patterns to float32 (exact)."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _draw_rows(blocks, tokens: int, channels: int, draw, threads: int) -> np.ndarray:
    out = np.empty((tokens, channels), dtype=np.float32)

    def one(i):
        r0 = i * _ROW_BLOCK
        r1 = min(tokens, r0 + _ROW_BLOCK)
        out[r0:r1] = draw(np.random.Generator(np.random.PCG64(blocks[i])), (r1 - r0, channels))

    n = (tokens + _ROW_BLOCK - 1) // _ROW_BLOCK
    if threads > 1 and n > 1:
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(one, range(n)))
    else:
        for i in range(n):
            one(i)
    return out


def _values(w: Workload, rng: np.random.Generator, blocks, threads: int) -> np.ndarray:
    T, C = w.tokens, w.channels
    if w.dist == "gauss_fixed_channels":
        x = _draw_rows(blocks, T, C, lambda g, s: g.standard_normal(s, dtype=np.float32), threads)
        chans = [c for c in (7, 300, 611, 1000) if c < C]
        x[:, chans] *= np.float32(50.0)
        return x
    if w.dist == "student_t":
        x = _draw_rows(blocks, T, C, lambda g, s: 0.5 * g.standard_t(3.0, s), threads)
        k = round(0.005 * C)
        chans = rng.choice(C, k, replace=False)
        fac = np.exp(rng.uniform(np.log(20.0), np.log(100.0), k)).astype(np.float32)
        x[:, chans] *= fac[None, :]
        return x
    if w.dist == "gauss_rms_spikes":
        x = _draw_rows(blocks, T, C, lambda g, s: g.standard_normal(s, dtype=np.float32), threads)
        rms = rng.lognormal(0.0, 0.5, T).astype(np.float32)
        x *= rms[:, None]
        k = round(0.002 * C)
        chans = rng.choice(C, k, replace=False)
        x[:, chans] *= np.float32(100.0)
        m = round(1e-4 * T * C)
        pos = rng.choice(T * C, m, replace=False)
        sign = rng.integers(0, 2, m).astype(np.float32) * 2.0 - 1.0
        x.reshape(-1)[pos] = np.float32(500.0) * sign
        return x
    if w.dist == "gradient":
        x = _draw_rows(blocks, T, C, lambda g, s: g.standard_normal(s, dtype=np.float32), threads)
        rms = rng.lognormal(0.0, 0.5, T).astype(np.float32)
        x *= (rms * np.float32(1e-5))[:, None]
        k = round(0.001 * C)
        chans = rng.choice(C, k, replace=False)
        x[:, chans] *= np.float32(30.0)
        return x
    if w.dist == "laplace":
        x = _draw_rows(blocks, T, C, lambda g, s: g.laplace(0.0, 1.0, s), threads)
        k = round(0.001 * C)
        chans = rng.choice(C, k, replace=False)
        x[:, chans] *= np.float32(50.0)
        return x
    raise ValueError(f"unknown distribution {w.dist!r}")


def generate(w: Workload, index: int = 0, threads: int | None = None) -> np.ndarray:
    """Draw tensor number ``index`` ([tokens, channels]) of workload ``w``.

    The steady-state run of the 8192-channel workload uses fresh tensors
    ``index = 0, 1, 2, ...`` of the same seed.
    """
    n_blocks = (w.tokens + _ROW_BLOCK - 1) // _ROW_BLOCK
    kids = np.random.SeedSequence([w.seed, index]).spawn(1 + n_blocks)
    rng = np.random.Generator(np.random.PCG64(kids[0]))
    if threads is None:
        threads = min(16, os.cpu_count() or 1)
    x = _values(w, rng, kids[1:], threads)
    if w.dtype == "bf16":
        return f32_to_bf16_bits(x)
    return x


def random_tiles(seed: int, n_tiles: int, tile: int, kind: str = "gauss") -> np.ndarray:
    """Small float32 test tensors ``[n_tiles, tile]`` with assorted structure.

    kind: "gauss" (N(0,1)), "spiky" (N(0,1) plus one x30 element in a third of
    the tiles), "mixed" (per-tile scale 2^U[-8,8], some constant and all-zero
    tiles, a few exact ties), "positive" (|N(0,1)|+1).
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    x = rng.standard_normal((n_tiles, tile))
    if kind == "gauss":
        pass
    elif kind == "spiky":
        rows = np.arange(0, n_tiles, 3)
        cols = rng.integers(0, tile, rows.size)
        x[rows, cols] *= 30.0
    elif kind == "mixed":
        x *= np.exp2(rng.uniform(-8, 8, (n_tiles, 1)))
        if n_tiles >= 8:
            x[1] = 0.0
            x[2] = 1.25
            x[3, :] = 0.0
            x[3, 5 % tile] = -4.0
            x[4] = np.where(np.arange(tile) % 2 == 0, 2.0, -2.0)
            x[5, 0] = x[5, tile - 1] = np.abs(x[5]).max() * 3.0
    elif kind == "positive":
        x = np.abs(x) + 1.0
    else:
        raise ValueError(kind)
    return x.astype(np.float32)
