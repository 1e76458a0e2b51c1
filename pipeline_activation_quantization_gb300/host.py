"""Encode and decode an activation that lives in pinned host memory, with the copies
overlapping the codec.

The ranking of "TAH-Quant" §3.2 is per group of tokens, so a chunk of whole token groups
encodes to exactly the bytes a whole-tensor encode gives those tokens.  ``HostRoundTrip``
splits the tensor into such chunks and runs three CUDA streams: chunk i + 1 is copied in
while chunk i is encoded and decoded on the device and chunk i - 1 is copied out (two
device buffers each way).  Every step of the codec runs in the library's kernels through
``encode`` / ``decode``; torch only provides the device buffers, streams and copies.

    rt = HostRoundTrip(tokens, channels, torch.float32, tile=128, hblock=128, budget=3.5,
                       tokens_per_group=2048)
    rt.run(x_host, y_host)   # x_host [tokens, channels] pinned; y_host float32 pinned
"""
from __future__ import annotations

from . import decode, encode, tahq_decode_workspace_size


class HostRoundTrip:
    """Pinned host tensor -> encode -> decode -> pinned host tensor, chunk by chunk of
    ``groups_per_chunk`` token groups, copies in and out overlapping the codec."""

    def __init__(self, tokens: int, channels: int, dtype, tile: int = 64, hblock: int | None = None,
                 bits_lo: int = 3, bits_hi: int = 4, budget: float = 3.5,
                 tokens_per_group: int = 0, groups_per_chunk: int = 1, device=None):
        import torch
        self.T, self.C, self.dtype = tokens, channels, dtype
        self.args = dict(tile=tile, hblock=hblock or tile, bits_lo=bits_lo, bits_hi=bits_hi,
                         budget=budget, tokens_per_group=tokens_per_group)
        S = tokens_per_group or tokens
        step = S * max(1, groups_per_chunk)
        self.chunks = [(t, min(tokens, t + step)) for t in range(0, tokens, step)]
        n = max(t1 - t0 for t0, t1 in self.chunks) if self.chunks else 0
        dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        self.x_dev = [torch.empty((n, channels), dtype=dtype, device=dev) for _ in range(2)]
        self.y_dev = [torch.empty((n, channels), dtype=torch.float32, device=dev) for _ in range(2)]
        self.s_in = torch.cuda.Stream(device=dev)
        self.s_cc = torch.cuda.Stream(device=dev)
        self.s_out = torch.cuda.Stream(device=dev)
        self.ev_in = [torch.cuda.Event() for _ in range(2)]
        self.ev_cc = [torch.cuda.Event() for _ in range(2)]
        self.ev_out = [torch.cuda.Event() for _ in range(2)]
        self._enc = {}  # encode outputs and workspaces by chunk size
        self._dec_ws = {}

    def run(self, x_host, y_host, stream=None):
        """Round-trip ``x_host`` into ``y_host``; work is ordered after ``stream`` (the
        current stream by default) and ``stream`` waits for the last copy out."""
        import torch
        cur = stream or torch.cuda.current_stream()
        a = self.args
        start = torch.cuda.Event()
        start.record(cur)
        for s in (self.s_in, self.s_cc, self.s_out):
            s.wait_event(start)
        for i, (t0, t1) in enumerate(self.chunks):
            k, n = i % 2, t1 - t0
            xd, yd = self.x_dev[k][:n], self.y_dev[k][:n]
            with torch.cuda.stream(self.s_in):
                if i >= 2:
                    self.s_in.wait_event(self.ev_cc[k])  # chunk i - 2 has read the buffer
                if self.dtype == torch.bfloat16:
                    xd.view(torch.int16).copy_(x_host[t0:t1].view(torch.int16), non_blocking=True)
                else:
                    xd.copy_(x_host[t0:t1], non_blocking=True)
                self.ev_in[k].record(self.s_in)
            with torch.cuda.stream(self.s_cc):
                self.s_cc.wait_event(self.ev_in[k])
                if i >= 2:
                    self.s_cc.wait_event(self.ev_out[k])  # chunk i - 2 has left the buffer
                S = min(a["tokens_per_group"] or n, n)
                prev = self._enc.get(n)
                enc = encode(xd, a["tile"], a["hblock"], a["bits_lo"], a["bits_hi"], a["budget"], S,
                             out=prev, workspace=prev["workspace"] if prev else None,
                             stream=self.s_cc)
                self._enc[n] = enc
                ws = self._dec_ws.get(n)
                if ws is None:
                    ws = torch.empty(tahq_decode_workspace_size(n, self.C, a["tile"]),
                                     dtype=torch.uint8, device=xd.device)
                    self._dec_ws[n] = ws
                decode(enc, n, self.C, a["tile"], a["hblock"], out=yd, workspace=ws, stream=self.s_cc)
                self.ev_cc[k].record(self.s_cc)
            with torch.cuda.stream(self.s_out):
                self.s_out.wait_event(self.ev_cc[k])
                y_host[t0:t1].copy_(yd, non_blocking=True)
                self.ev_out[k].record(self.s_out)
        cur.wait_stream(self.s_out)
        return y_host
