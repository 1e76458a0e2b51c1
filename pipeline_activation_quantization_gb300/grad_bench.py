"""Timing of the backward pass's gradient codec (``tahq_naive_encode`` / ``_decode``).

``python -m pipeline_activation_quantization_gb300.grad_bench`` encodes and decodes a
seeded Gaussian fp32 gradient of 32768 tokens x 8192 channels (1e-5 scale, tile 64,
c = 2^16) at 8 and 10 bits on cuda:0: 20 timed calls each after 5 untimed ones, the
L2 flushed (a 256 MiB write) before every call, CUDA events around each call on the
current stream.  Prints the median time and the throughput of the bytes each call moves
(the fp32 gradient, the packed codes, an fp32 scale and zero a tile).
"""
from __future__ import annotations

import argparse

import numpy as np


def main(argv=None) -> int:
    import torch
    from . import naive_decode, naive_encode

    ap = argparse.ArgumentParser()
    ap.add_argument("--tokens", type=int, default=32768)
    ap.add_argument("--channels", type=int, default=8192)
    ap.add_argument("--tile", type=int, default=64)
    ap.add_argument("--bits", type=int, nargs="+", default=[8, 10])
    args = ap.parse_args(argv)
    T, C, G, c = args.tokens, args.channels, args.tile, 2.0 ** 16
    gen = torch.Generator(device="cuda").manual_seed(0)
    g = (torch.randn(T, C, device="cuda", generator=gen) * 1e-5).contiguous()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    y = torch.empty_like(g)
    for b in args.bits:
        codes, scales, zeros = naive_encode(g, G, b, c)
        te, td = [], []
        for i in range(25):
            flush.fill_(1)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            naive_encode(g, G, b, c)
            e1.record()
            flush.fill_(1)
            d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            d0.record()
            naive_decode(codes, scales, zeros, T, C, G, b, c, out=y)
            d1.record()
            torch.cuda.synchronize()
            if i >= 5:
                te.append(e0.elapsed_time(e1))
                td.append(d0.elapsed_time(d1))
        nb = T * C * 4 + T * C * b // 8 + 8 * T * C // G
        me, md = float(np.median(te)), float(np.median(td))
        print(f"bits {b}: encode {me * 1e3:.1f} us ({nb / me / 1e6:.0f} GB/s), "
              f"decode {md * 1e3:.1f} us ({nb / md / 1e6:.0f} GB/s), {nb} bytes a call")
    return 0


if __name__ == "__main__":
    raise SystemExit(main())
