"""Two pipeline stages in two processes (``-m gpu``): stage a encodes an activation into
TAH-Quant wire buffers chunk by chunk and sends them over gloo (host tensors); stage b,
a second process on the same GPU, receives and decodes them.  Its tensor must equal bit
for bit the decode of a whole-tensor encode in one process (TAH-Quant Algorithm 1, §3.5;
§5.1's TCP transport between stages).  No NCCL, no peer access, no kernel of one process
waits on the other's."""
import json
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _stage(rank, port, name, kw, groups_per_chunk, out_path):
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import synth
    import pipeline_activation_quantization_gb300 as tq
    from pipeline_activation_quantization_gb300 import p2p
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=2)
    torch.cuda.set_device(0)
    w = synth.WORKLOADS[name].with_params(**kw) if kw else synth.WORKLOADS[name]
    args = p2p.CodecArgs(w.tile, w.hblock, w.bits_lo, w.bits_hi, w.budget, w.tokens_per_group)
    x_np = synth.generate(w)
    if w.dtype == "bf16":
        x = torch.from_numpy(x_np.view(np.int16)).cuda().view(torch.bfloat16)
    else:
        x = torch.from_numpy(x_np).cuda()
    if rank == 0:
        info = p2p.send_activation(x, 1, args, groups_per_chunk)
    else:
        y, info = p2p.recv_activation(w.tokens, w.channels, 0, args, torch.device("cuda", 0),
                                      groups_per_chunk)
        # the whole tensor in one process
        wbuf, _ = tq.encode_wire(x, w.tile, w.hblock, w.bits_lo, w.bits_hi, w.budget,
                                 w.tokens_per_group)
        ref, _ = tq.decode_wire(wbuf, w.tokens, w.channels, w.tile, w.hblock, w.bits_lo,
                                w.bits_hi, w.budget, w.tokens_per_group)
        torch.cuda.synchronize()
        same = bool(torch.equal(y.view(torch.int32), ref.view(torch.int32)))
        with open(out_path, "w") as f:
            json.dump({"same": same, "status": info["status"], "chunks": info["chunks"],
                       "bytes": info["bytes"]}, f)
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("name,kw,gpc", [
    ("c2", {}, 1),                                           # 4 chunks of one group
    ("c4", dict(tokens=8192, tile=128, hblock=128), 2),      # 2 chunks of two groups
    ("c1", {}, 1),                                           # one chunk, fp32
])
def test_two_process_stream_equals_one_process_decode(tmp_path, name, kw, gpc):
    import torch.multiprocessing as mp
    out = str(tmp_path / "result.json")
    mp.spawn(_stage, args=(_free_port(), name, kw, gpc, out), nprocs=2, join=True)
    with open(out) as f:
        r = json.load(f)
    assert r["same"], r
    assert all(s == 0 for s in r["status"]), r
