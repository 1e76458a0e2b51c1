"""GPU-vs-oracle parity of the backward pass's fixed-point gradient codec (``-m gpu``).

"TAH-Quant" §3.5 / Algorithm 1 and Appendix H eq. (24): the §3.3 quantizer at one width on
the activation tiles, g_hat = Q(c g) / c.  Codes, scales and zeros bit-exact (codes may
differ only on elements the oracle flags as sitting on a rounding boundary); the decode
of the GPU's own codes bit-exact where the codes agree.
"""
import numpy as np
import pytest

import oracle
import pipeline_activation_quantization_gb300 as tq

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_cuda():
    import torch
    assert torch.cuda.is_available(), "the -m gpu tests need a CUDA device"
    tq.lib()


def _grad(T, C, seed, scale=1e-5):
    rng = np.random.default_rng(seed)
    g = (rng.standard_normal((T, C)) * scale).astype(np.float32)
    g[:, 7::97] *= 40.0                     # a few large channels
    g[3::11] = 0.0                          # all-zero tokens (constant tiles)
    return g


def _unpack(stream, n, b):
    bits = np.unpackbits(stream, bitorder="little")[: n * b].reshape(n, b)
    return (bits.astype(np.int64) << np.arange(b)).sum(axis=1)


@pytest.mark.parametrize("G", [32, 64, 128])
@pytest.mark.parametrize("b", [4, 6, 8, 10, 16])
@pytest.mark.parametrize("c", [1.0, 2.0 ** 12])
def test_naive_parity(G, b, c):
    import torch
    T, C = 40, 1536
    g = _grad(T, C, 100 + G + b)
    codes, scales, zeros = tq.naive_encode(torch.from_numpy(g).cuda(), G, b, c)
    y = tq.naive_decode(codes, scales, zeros, T, C, G, b, c)
    torch.cuda.synchronize()
    oc, os_, oz, near = oracle.naive_encode(g, G, b, c, want_near=True)
    assert np.array_equal(scales.cpu().numpy(), os_)
    assert np.array_equal(zeros.cpu().numpy(), oz)
    gq = _unpack(codes.cpu().numpy(), T * C, b)
    oq = _unpack(oc, T * C, b)
    bad = np.flatnonzero(gq != oq)
    assert np.all(near.reshape(-1)[bad] == 1), f"code mismatch off a boundary at {bad[:8]}"
    yo = oracle.naive_decode(codes.cpu().numpy(), os_, oz, T, C, G, b, c)
    assert np.array_equal(y.cpu().numpy(), yo)


def test_naive_full_size_sampled():
    # a pipeline-boundary gradient, 8 x 2048 x 4096 fp32 at 8 bits, tile 64, c = 2^16
    import torch
    T, C, G, b, c = 16384, 4096, 64, 8, 2.0 ** 16
    rng = np.random.default_rng(5)
    g = (rng.standard_normal((T, C)) * 1e-5).astype(np.float32)
    codes, scales, zeros = tq.naive_encode(torch.from_numpy(g).cuda(), G, b, c)
    y = tq.naive_decode(codes, scales, zeros, T, C, G, b, c).cpu().numpy()
    rows = rng.choice(T, 64, replace=False)
    for r in rows:
        oc, os_, oz = oracle.naive_encode(g[r:r + 1], G, b, c)
        n = C // G
        assert np.array_equal(scales[r * n:(r + 1) * n].cpu().numpy(), os_)
        assert np.array_equal(zeros[r * n:(r + 1) * n].cpu().numpy(), oz)
        nb = C * b // 8
        assert np.array_equal(codes[r * nb:(r + 1) * nb].cpu().numpy(), oc)
        assert np.array_equal(y[r], oracle.naive_decode(oc, os_, oz, 1, C, G, b, c)[0])


def test_naive_empty_and_rejects():
    import torch
    codes, scales, zeros = tq.naive_encode(torch.zeros((0, 128), device="cuda"), 64, 8)
    assert codes.numel() == 0 and scales.numel() == 0
    with pytest.raises(tq.TahqError):
        tq.naive_encode(torch.zeros((4, 128), device="cuda"), 64, 8, 3.0)
    with pytest.raises(tq.TahqError):
        tq.naive_encode(torch.zeros((4, 128), device="cuda"), 16, 8)


@pytest.mark.parametrize("b", [10, 16])
@pytest.mark.parametrize("G", [32, 128])
def test_naive_range_cutoff(G, b):
    # tiles {0, D} with D just below, at and above the width's cutoff 2^(b - 126): below it
    # the tile quantises to its minimum; at and above it the scale is a normal float
    import torch
    cut = np.float32(2.0 ** (b - 126))
    Ds = [np.nextafter(cut, np.float32(0)), cut, np.float32(cut * np.float32(1.5)),
          np.float32(cut * np.float32(3.0))]
    g = np.zeros((len(Ds), G), np.float32)
    for i, D in enumerate(Ds):
        g[i, 1::2] = D
    codes, scales, zeros = tq.naive_encode(torch.from_numpy(g).cuda(), G, b)
    y = tq.naive_decode(codes, scales, zeros, len(Ds), G, G, b)
    torch.cuda.synchronize()
    oc, os_, oz = oracle.naive_encode(g, G, b)
    assert np.array_equal(scales.cpu().numpy(), os_) and os_[0] == 0 and (os_[1:] > 0).all()
    assert np.array_equal(zeros.cpu().numpy(), oz)
    assert np.array_equal(codes.cpu().numpy(), oc)
    assert np.array_equal(y.cpu().numpy(), oracle.naive_decode(oc, os_, oz, len(Ds), G, G, b))


def test_naive_decode_checks_its_buffers():
    import torch
    g = torch.zeros((4, 128), device="cuda")
    codes, scales, zeros = tq.naive_encode(g, 64, 8)
    with pytest.raises(ValueError):
        tq.naive_decode(codes[:-1], scales, zeros, 4, 128, 64, 8)
    with pytest.raises(ValueError):
        tq.naive_decode(codes, scales[:-1], zeros, 4, 128, 64, 8)
    with pytest.raises(ValueError):
        tq.naive_decode(codes, scales, zeros, 4, 128, 64, 8,
                        out=torch.empty((4, 128), dtype=torch.float16, device="cuda"))
