"""Bounded waits: a wait that nothing completes gives up after its time limit, flags the
device status word, makes the waits after it return at once, and leaves the workspace
usable.  No GPU fault, trap or hang is involved: the kernel's waits are bounded by the
device's global timer and the kernel returns normally."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
import pipeline_activation_quantization_gb300 as tq  # noqa: E402
import synth  # noqa: E402


def test_wait_gives_up_flags_status_and_fails_fast():
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    elapsed = torch.zeros(2, dtype=torch.int64, device="cuda")
    limit = 2_000_000  # 2 ms
    assert tq.tahq_test_wait_timeout(ws, ws.numel(), limit, elapsed) == 0
    torch.cuda.synchronize()
    rc, word = tq.tahq_get_device_status(ws)
    assert rc == 5 and word & tq.DEV_WAIT_TIMEOUT, (rc, word)
    t_ns, gave_up = (int(v) for v in elapsed.cpu())
    assert gave_up == 8
    # the first wait runs out its limit; the seven after it see the status bit at once
    assert limit <= t_ns < 4 * limit, t_ns


def test_bad_arguments_are_rejected():
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    assert tq.tahq_test_wait_timeout(ws, 512, 1000) == 3
    assert tq.tahq_test_wait_timeout(ws, ws.numel(), 0) == 1


def test_workspace_is_clean_for_the_next_call():
    w = synth.WORKLOADS["c2"].with_params(tokens=512, tokens_per_group=256)
    x = synth.generate(w)
    xt = torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    enc = tq.encode(xt, w.tile, w.hblock, w.bits_lo, w.bits_hi, w.budget, w.tokens_per_group)
    ws = enc["workspace"]
    assert tq.tahq_test_wait_timeout(ws, ws.numel(), 1_000_000) == 0
    torch.cuda.synchronize()
    assert tq.tahq_get_device_status(ws)[0] == 5
    outs = {k: enc[k] for k in ("codes", "scales", "zeros", "bits", "pivots")}
    enc2 = tq.encode(xt, w.tile, w.hblock, w.bits_lo, w.bits_hi, w.budget, w.tokens_per_group,
                     out=outs, workspace=ws)
    torch.cuda.synchronize()
    rc, word = tq.tahq_get_device_status(ws)
    assert rc == 0 and word == 0
    ref = oracle.encode(x, w.tile, w.hblock, w.bits_lo, w.bits_hi, w.budget, w.tokens_per_group)
    for k in ("codes", "bits", "pivots", "scales", "zeros"):
        assert np.array_equal(enc2[k].cpu().numpy().view(np.uint8), ref[k].view(np.uint8)), k
