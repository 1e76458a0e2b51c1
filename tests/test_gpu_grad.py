"""TAH-Quant on gradients with eq. (24)'s scaling on the GPU (``-m gpu``): the C entry
points tahq_encode_scaled / tahq_decode_scaled against the CPU oracle (TAH-Quant
Appendix H, Table 10 and eq. (24): g_hat = Q(c g) / c, c a power of two)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
import pipeline_activation_quantization_gb300 as tq  # noqa: E402
import synth  # noqa: E402

pytestmark = pytest.mark.gpu


def _dev(x):
    if x.dtype == np.uint16:
        return torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(x).cuda()


def _check(x, G, lo, hi, beta, S, c, tau=2.0):
    T, C = x.shape
    enc = tq.encode_scaled(_dev(x), G, G, lo, hi, beta, S, tau=tau, scale_c=c)
    y = tq.decode_scaled(enc, T, C, G, G, scale_c=c)
    torch.cuda.synchronize()
    rc, word = tq.tahq_get_device_status(enc["workspace"])
    assert rc == 0, hex(word)
    ref = oracle.encode_scaled(x, G, G, lo, hi, beta, S, c=c, tau=tau, threads=8)
    for k in ("codes", "bits", "pivots", "scales", "zeros"):
        got = enc[k].cpu().numpy()
        assert np.array_equal(got.view(np.uint8), ref[k].view(np.uint8)), k
    yr = oracle.decode_scaled(ref["codes"], ref["scales"], ref["zeros"], ref["bits"],
                              ref["pivots"], T, C, G, G, c=c, threads=8)
    yg = y.cpu().numpy()
    rel = np.linalg.norm(yg.astype(np.float64) - yr) / max(np.linalg.norm(yr.astype(np.float64)), 1e-300)
    assert rel <= 1e-5, rel


@pytest.mark.parametrize("G,beta,c", [(64, 4.0, 2.0 ** 16), (64, 3.5, 2.0 ** 16),
                                      (128, 3.5, 2.0 ** 20), (32, 3.5, 2.0 ** 12)])
def test_scaled_gradient_matches_oracle(G, beta, c):
    w = synth.WORKLOADS["g5"].with_params(tokens=512, channels=1024, tokens_per_group=128)
    _check(synth.generate(w), G, 3, 4, beta, 128, c)


def test_scaled_bf16_gradient_matches_oracle():
    w = synth.WORKLOADS["g5"].with_params(tokens=512, channels=2048, tokens_per_group=256)
    x = synth.f32_to_bf16_bits(synth.generate(w))
    _check(x, 64, 3, 4, 3.5, 256, 2.0 ** 16)


def test_tiny_gradients_and_downscaling():
    rng = np.random.default_rng(9)
    x = (rng.standard_normal((256, 512)) * 1e-39).astype(np.float32)
    _check(x, 64, 3, 4, 3.5, 64, 2.0 ** 120)
    _check(rng.standard_normal((256, 512)).astype(np.float32) * 1e6, 64, 3, 4, 3.5, 64, 2.0 ** -20)


def test_full_size_gradient_sampled():
    # 16 x 2048 x 8192 fp32 gradient at 4 bits (Table 10) scaled by 2^16: the GPU encodes
    # the whole tensor; the oracle checks two of its sixteen 2048-token groups
    w = synth.WORKLOADS["g5"]
    x = synth.generate(w)
    T, C, G, S = w.tokens, w.channels, w.tile, w.tokens_per_group
    c = 2.0 ** 16
    enc = tq.encode_scaled(_dev(x), G, G, 3, 4, 3.5, S, scale_c=c)
    torch.cuda.synchronize()
    assert tq.tahq_get_device_status(enc["workspace"])[0] == 0
    n_g = S * C // G
    gb = enc["payload_bytes"] // (T // S)
    for g in (0, 11):
        ref = oracle.encode_scaled(x[g * S:(g + 1) * S], G, G, 3, 4, 3.5, S, c=c, threads=8)
        sl = slice(g * n_g, (g + 1) * n_g)
        for k in ("bits", "pivots", "scales", "zeros"):
            assert np.array_equal(enc[k][sl].cpu().numpy().view(np.uint8), ref[k].view(np.uint8)), k
        assert np.array_equal(enc["codes"][g * gb:(g + 1) * gb].cpu().numpy(), ref["codes"])


def test_rejects_scale_that_is_not_a_power_of_two():
    x = torch.zeros((64, 256), dtype=torch.float32, device="cuda")
    with pytest.raises(tq.TahqError):
        tq.encode_scaled(x, 64, 64, 3, 4, 3.5, 0, scale_c=3.0)
