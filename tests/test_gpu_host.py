"""The pinned-host round trip (``-m gpu``): chunks of whole token groups copied in,
encoded, decoded and copied out on three streams must give bit for bit the decode of a
whole-tensor encode on the device (the ranking of "TAH-Quant" §3.2 is per group)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import pipeline_activation_quantization_gb300 as tq  # noqa: E402
import synth  # noqa: E402
from pipeline_activation_quantization_gb300.host import HostRoundTrip  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype,G,beta,groups_per_chunk", [("f32", 128, 3.5, 1), ("bf16", 64, 3.5, 2),
                                                           ("bf16", 64, 3.0, 1), ("f32", 32, 3.25, 3)])
def test_host_round_trip_matches_device_codec(dtype, G, beta, groups_per_chunk):
    w = synth.Workload("host", 256, 2048, dtype, G, G, 3, 4, beta, 32, 11 + G, "gauss_rms_spikes")
    x = synth.generate(w)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    x_host = (torch.from_numpy(x.view(np.int16)).view(torch.bfloat16) if dtype == "bf16"
              else torch.from_numpy(x)).pin_memory()
    y_host = torch.empty((w.tokens, w.channels), dtype=torch.float32).pin_memory()
    rt = HostRoundTrip(w.tokens, w.channels, tdt, tile=G, hblock=G, bits_lo=3, bits_hi=4,
                       budget=beta, tokens_per_group=w.tokens_per_group,
                       groups_per_chunk=groups_per_chunk)
    for _ in range(2):  # buffers reused on the second call
        y_host.fill_(float("nan"))
        rt.run(x_host, y_host)
        torch.cuda.synchronize()
        xd = x_host.cuda()
        enc = tq.encode(xd, G, G, 3, 4, beta, w.tokens_per_group)
        y_ref = tq.decode(enc, w.tokens, w.channels, G, G).cpu()
        torch.cuda.synchronize()
        assert torch.equal(y_host.view(torch.int32), y_ref.view(torch.int32))
