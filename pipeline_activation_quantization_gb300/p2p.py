"""Two pipeline stages in two processes: the activation crosses as TAH-Quant wire buffers.

"TAH-Quant" Algorithm 1 (§3.5): stage a sends Q(a) of the activation it computed, stage b
de-quantises it and goes on; §5.1 runs the stages on separate machines and ships the bytes
over TCP.  Here each stage is a process; the transport is ``torch.distributed`` point to
point over gloo (host tensors, so it works over TCP between machines as well as between two
processes on one host), and the codec runs on each process's GPU through the C ABI:

* the sender splits the activation [tokens, channels] into chunks of whole token groups
  (the ranking is per group, so a chunk's wire buffer holds exactly what a whole-tensor
  encode would hold for those tokens), encodes chunk i + 1 on the GPU while chunk i is on
  the wire (``tahq_encode_wire`` into a device buffer, an asynchronous copy to pinned host
  memory, then ``isend``);
* the receiver posts the receive of chunk i + 1 before it decodes chunk i (a copy to the
  device and ``tahq_decode_wire`` into the chunk's rows of the output).

The decoded tensor is bit for bit the decode of a whole-tensor encode (tested).  Both
processes may share one GPU: neither waits on a kernel of the other, and no device memory
is shared (no NCCL, no peer access).

    python -m pipeline_activation_quantization_gb300.p2p    # a demo on cuda:0
"""
from __future__ import annotations

import dataclasses
import os
import time

from . import (TAHQ_BF16, TAHQ_F32, TahqError, tahq_decode_wire, tahq_encode_wire,
               tahq_wire_decode_workspace_size, tahq_wire_size, tahq_wire_workspace_size)


@dataclasses.dataclass(frozen=True)
class CodecArgs:
    """The codec parameters both stages agree on (the wire header repeats them)."""
    tile: int = 64
    hblock: int = 64
    bits_lo: int = 3
    bits_hi: int = 4
    budget: float = 3.5
    tokens_per_group: int = 0
    tau: float = 2.0


def _chunks(tokens: int, args: CodecArgs, groups_per_chunk: int):
    S = args.tokens_per_group or tokens
    step = S * max(1, groups_per_chunk)
    return [(t, min(tokens, t + step)) for t in range(0, tokens, step)]


def send_activation(x, dst: int, args: CodecArgs, groups_per_chunk: int = 1, group=None) -> dict:
    """Encode the CUDA tensor ``x`` [tokens, channels] chunk by chunk and send the wire
    buffers to rank ``dst``.  Returns the bytes sent and the time taken."""
    import torch
    import torch.distributed as dist
    if x.dtype == torch.float32:
        dt = TAHQ_F32
    elif x.dtype == torch.bfloat16:
        dt = TAHQ_BF16
    else:
        raise ValueError(f"unsupported dtype {x.dtype}")
    x = x.contiguous()
    T, C = x.shape
    a = args
    chunks = _chunks(T, a, groups_per_chunk)
    S = a.tokens_per_group or T
    st = torch.cuda.Stream(device=x.device)
    sizes = [tahq_wire_size(t1 - t0, C, a.tile, a.bits_lo, a.bits_hi, a.budget, min(S, t1 - t0))
             for t0, t1 in chunks]
    wsz = max(tahq_wire_workspace_size(t1 - t0, C, a.tile, a.hblock, a.bits_lo, a.bits_hi,
                                       a.budget, min(S, t1 - t0)) for t0, t1 in chunks)
    if min(sizes) == 0 or wsz == 0:
        raise TahqError(1, "tahq_wire_size")
    big = max(sizes)
    dev_buf = [torch.empty(big, dtype=torch.uint8, device=x.device) for _ in range(2)]
    host_buf = [torch.empty(big, dtype=torch.uint8).pin_memory() for _ in range(2)]
    ws = torch.empty(wsz, dtype=torch.uint8, device=x.device)
    done = [torch.cuda.Event() for _ in range(2)]
    reqs = [None, None]
    t_start = time.perf_counter()
    for i, (t0, t1) in enumerate(chunks):
        s = i % 2
        if reqs[s] is not None:  # the host buffer of chunk i - 2 is free again
            reqs[s].wait()
            reqs[s] = None
        n = sizes[i]
        with torch.cuda.stream(st):
            rc = tahq_encode_wire(x[t0:t1], dt, t1 - t0, C, a.tile, a.hblock, a.bits_lo,
                                  a.bits_hi, a.budget, min(S, t1 - t0), a.tau, dev_buf[s], n,
                                  ws, wsz, st)
            if rc != 0:
                raise TahqError(rc, "tahq_encode_wire")
            host_buf[s][:n].copy_(dev_buf[s][:n], non_blocking=True)
            done[s].record(st)
        if i > 0:  # chunk i - 1 is on the host by now or soon: send it while i encodes
            p = (i - 1) % 2
            done[p].synchronize()
            reqs[p] = dist.isend(host_buf[p][:sizes[i - 1]], dst, group=group)
    last = (len(chunks) - 1) % 2
    done[last].synchronize()
    reqs[last] = dist.isend(host_buf[last][:sizes[-1]], dst, group=group)
    for r in reqs:
        if r is not None:
            r.wait()
    return {"bytes": sum(sizes), "chunks": len(chunks), "seconds": time.perf_counter() - t_start}


def recv_activation(tokens: int, channels: int, src: int, args: CodecArgs, device,
                    groups_per_chunk: int = 1, group=None, out=None) -> tuple:
    """Receive the wire buffers of a [tokens, channels] activation from rank ``src`` and
    decode them into a float32 CUDA tensor (``out`` if given).  Returns (out, info); the
    info holds the device status word of every chunk's decode (0 = clean)."""
    import torch
    import torch.distributed as dist
    a = args
    chunks = _chunks(tokens, a, groups_per_chunk)
    S = a.tokens_per_group or tokens
    sizes = [tahq_wire_size(t1 - t0, channels, a.tile, a.bits_lo, a.bits_hi, a.budget,
                            min(S, t1 - t0)) for t0, t1 in chunks]
    wsz = max(tahq_wire_decode_workspace_size(t1 - t0, channels, a.tile) for t0, t1 in chunks)
    if min(sizes) == 0 or wsz == 0:
        raise TahqError(1, "tahq_wire_size")
    big = max(sizes)
    if out is None:
        out = torch.empty((tokens, channels), dtype=torch.float32, device=device)
    host_buf = [torch.empty(big, dtype=torch.uint8).pin_memory() for _ in range(2)]
    dev_buf = [torch.empty(big, dtype=torch.uint8, device=device) for _ in range(2)]
    ws = [torch.empty(wsz, dtype=torch.uint8, device=device) for _ in range(2)]
    st = torch.cuda.Stream(device=device)
    free = [torch.cuda.Event() for _ in range(2)]
    statuses = []
    t_start = time.perf_counter()
    req = dist.irecv(host_buf[0][:sizes[0]], src, group=group)
    for i, (t0, t1) in enumerate(chunks):
        s = i % 2
        req.wait()
        if i + 1 < len(chunks):  # post the next receive before decoding this chunk
            n = (i + 1) % 2
            free[n].synchronize()  # its host buffer's copy to the device is done
            req = dist.irecv(host_buf[n][:sizes[i + 1]], src, group=group)
        with torch.cuda.stream(st):
            dev_buf[s][:sizes[i]].copy_(host_buf[s][:sizes[i]], non_blocking=True)
            free[s].record(st)
            rc = tahq_decode_wire(dev_buf[s], sizes[i], t1 - t0, channels, a.tile, a.hblock,
                                  a.bits_lo, a.bits_hi, a.budget, min(S, t1 - t0), out[t0:t1],
                                  ws[s], wsz, st)
            if rc != 0:
                raise TahqError(rc, "tahq_decode_wire")
            statuses.append(ws[s][:4].clone())
    st.synchronize()
    words = [int(w.view(torch.int32).item()) & 0xFFFFFFFF for w in statuses]
    return out, {"bytes": sum(sizes), "chunks": len(chunks), "status": words,
                 "seconds": time.perf_counter() - t_start}


def _demo(rank: int, world: int, port: int):
    import numpy as np
    import torch
    import torch.distributed as dist
    import synth
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    torch.cuda.set_device(0)
    w = synth.WORKLOADS["c2"]
    args = CodecArgs(w.tile, w.hblock, w.bits_lo, w.bits_hi, w.budget, w.tokens_per_group)
    if rank == 0:
        x = torch.from_numpy(synth.generate(w).view(np.int16)).cuda().view(torch.bfloat16)
        info = send_activation(x, 1, args)
        print(f"stage a: sent {info['chunks']} chunks, {info['bytes']} bytes in "
              f"{info['seconds'] * 1e3:.1f} ms")
    else:
        y, info = recv_activation(w.tokens, w.channels, 0, args, torch.device("cuda", 0))
        print(f"stage b: received and decoded {info['chunks']} chunks ({info['bytes']} bytes, "
              f"{info['bytes'] * 8 / y.numel():.3f} bits an element) in "
              f"{info['seconds'] * 1e3:.1f} ms, device status {info['status']}")
    dist.destroy_process_group()


if __name__ == "__main__":
    import sys
    import torch.multiprocessing as mp
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    mp.spawn(_demo, args=(2, 29517), nprocs=2, join=True)
