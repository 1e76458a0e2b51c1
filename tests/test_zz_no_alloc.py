"""tahq_decode_noalloc: decode for callers that cannot allocate device memory (``-m gpu``).

Some receivers of the activation stream cannot hand the codec a workspace: a stage whose
runtime plans all device memory in advance and passes only inputs and outputs, or a C
caller with no device allocator (where a cudaMalloc in the receive loop would also stall
the device).  This entry point takes its scratch from a fixed array inside the library.
Its output must match tahq_decode's, and the CPU oracle's decode of the same stream,
within the tolerance the other parity tests use, on two calls in a row (the second call
reuses the shared array left by the first).

The file is named so that pytest collects it last.  It passes on its own in a fresh
process (the first call sets up the array's device address) and after the other tests.
"""
import numpy as np
import pytest

import oracle
import pipeline_activation_quantization_gb300 as tq
import synth

pytestmark = pytest.mark.gpu


def _rel_l2(a, b):
    a = a.astype(np.float64)
    b = b.astype(np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


@pytest.mark.parametrize("name", ["c2", "c1"])
def test_noalloc_decode_matches_decode_twice(name):
    import torch
    w = synth.WORKLOADS[name]
    T, C, G, h = w.tokens, w.channels, w.tile, w.hblock
    x_np = synth.generate(w)
    if w.dtype == "bf16":
        x = torch.from_numpy(x_np.view(np.int16)).cuda().view(torch.bfloat16)
    else:
        x = torch.from_numpy(x_np).cuda()
    enc = tq.encode(x, G, h, w.bits_lo, w.bits_hi, w.budget, w.tokens_per_group)
    ref = tq.decode(enc, T, C, G, h)
    torch.cuda.synchronize()
    ref_np = ref.cpu().numpy()
    # the oracle's decode of the stream the GPU wrote
    orc = oracle.decode(enc["codes"].cpu().numpy(), enc["scales"].cpu().numpy(),
                        enc["zeros"].cpu().numpy(), enc["bits"].cpu().numpy(),
                        enc["pivots"].cpu().numpy(), T, C, G, h)
    status = torch.full((1,), 0xFFFFFFFF, dtype=torch.int64, device="cuda")
    for call in range(2):
        out = torch.full((T, C), float("nan"), dtype=torch.float32, device="cuda")
        rc = tq.tahq_decode_noalloc(enc["codes"], enc["codes"].numel(), enc["scales"],
                                    enc["zeros"], enc["bits"], enc["pivots"], T, C, G, h, out,
                                    status)
        assert rc == 0, tq.tahq_status_string(rc)
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        assert np.isfinite(got).all(), f"call {call}: output not fully written"
        assert _rel_l2(got, ref_np) <= 1e-5, f"call {call}: against tahq_decode"
        assert _rel_l2(got, orc) <= 1e-5, f"call {call}: against the oracle's decode"
        assert int(status.cpu().item()) & 0xFFFFFFFF == 0, f"call {call}: device status"


def test_noalloc_rejects_shapes_beyond_its_scratch():
    import torch
    # width-8 tiles: 2048 tiles per decode chunk, so 52289 chunks need more than 256 KiB
    T, C, G = 52289 * 2048 * 8 // 1024, 1024, 8
    assert tq.tahq_decode_workspace_size(T, C, G) > 256 * 1024
    dummy = torch.zeros(16, dtype=torch.uint8, device="cuda")
    f = torch.zeros(4, dtype=torch.float32, device="cuda")
    rc = tq.tahq_decode_noalloc(dummy, 16, f, f, dummy, dummy, T, C, G, G, f)
    assert rc == 3        # TAHQ_ERR_WORKSPACE, before anything is launched
    # the largest accepted shape for this width is still accepted by the size check
    assert tq.tahq_decode_workspace_size(52288 * 2048 * 8 // 1024, C, G) <= 256 * 1024
