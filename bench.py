#!/usr/bin/env python3
"""Throughput of the sm_103a TAH-Quant activation codec (encode + decode round trip).

One step = tahq_encode + tahq_decode of one synthetic activation tensor that is already
resident in HBM (the whole hot path).  Default workload: the 70B-width pipeline
boundary, 16 x 2048 x 8192 fp32 (32768 tokens), tile = Hadamard block = 128, bits
{3, 4}, budget 3.5, ranking per 2048-token sample; steps cycle through several fresh
seeded tensors of that distribution.  Prints one JSON line (rank 0).

  python bench.py [--gpus N --steps K --warmup W --workload c3|c2|c4|c5 ...]
  python bench.py --impl reference     # the CPU oracle on the host cores (reference arm)

value = input-activation GB/s of the round trip, all ranks together (replicas: each GPU
encodes and decodes its own tensor, no collective on the data path).  Every step is timed
with CUDA events on the launching stream; L2 is flushed (a 256 MiB write) between steps,
outside the events.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "encode+decode GB/s of activations (tokens/s) and % of GB300 HBM roofline"
FLUSH_BYTES = 256 << 20


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def _workload(args) -> synth.Workload:
    w = synth.WORKLOADS[args.workload]
    kw = {}
    if args.tile:
        kw["tile"] = args.tile
        kw["hblock"] = args.tile
    if args.hblock:
        kw["hblock"] = args.hblock
    if args.budget is not None:
        kw["budget"] = args.budget
    if args.tokens:
        T, S = args.tokens, w.tokens_per_group
        shape = f"{T // S}x{S}x{w.channels}" if S else f"{T}x{w.channels}"
        kw["tokens"] = T
        kw["name"] = f"{w.name.split('_')[0]}_{shape}_{w.dtype}"
    return w.with_params(**kw) if kw else w


def _config(w: synth.Workload, extra=None, tau=None) -> dict:
    c = {"workload": w.name, "tokens": w.tokens, "channels": w.channels, "input_dtype": w.dtype,
         "tile": w.tile, "hblock": w.hblock, "bits": [w.bits_lo, w.bits_hi], "budget": w.budget,
         "tokens_per_group": w.tokens_per_group, "seed": w.seed,
         "l2": "flushed between steps (256 MiB write, outside the events)"}
    if tau is not None:
        c["tau"] = tau
    if extra:
        c.update(extra)
    return c


def _alg_bytes(w: synth.Workload, payload: int):
    n = w.tokens * w.channels // w.tile
    in_b = w.in_bytes
    enc = in_b + payload + 10 * n
    dec = payload + 10 * n + 4 * w.elements
    return in_b, enc, dec


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed loop runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.rows = []
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        for line in out.splitlines():
            f = [s.strip() for s in line.split(",")]
            if len(f) >= 9:
                self.rows.append(f)

    def summary(self):
        rows = getattr(self, "rows", [])
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


def _traffic_for(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, or None when the
    kernel sources changed since those counters were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except Exception:
        return None
    e = rec.get(f"{kernel}|{workload}")
    if not e or e.get("src_sha") != _src_sha(e.get("src_files")):
        return None
    return e.get("dram_bytes_per_launch")


def _src_sha(files=None) -> str:
    """Hash of the kernel's sources (the listed files of csrc/, else all of them)."""
    h = hashlib.sha256()
    d = os.path.join(ROOT, "pipeline_activation_quantization_gb300", "csrc")
    for name in sorted(files or os.listdir(d)):
        with open(os.path.join(d, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


# ------------------------------------------------------------------ the oracle (CPU)

def _oracle_step(x, w, tokens, tau=None, alloc_tile=None):
    import oracle
    xs = x[:tokens]
    S = min(w.tokens_per_group or w.tokens, tokens)
    r = oracle.encode(xs, w.tile, w.hblock, w.bits_lo, w.bits_hi, w.budget, S, tau=tau,
                      alloc_tile=alloc_tile)
    oracle.decode(r["codes"], r["scales"], r["zeros"], r["bits"], r["pivots"], tokens, w.channels,
                  w.tile, w.hblock)


def cpu_baseline(w: synth.Workload, x, target_s: float = 12.0, tau=None, alloc_tile=None) -> dict:
    """The oracle, single thread, on whole token groups of the same tensor."""
    S = w.tokens_per_group or w.tokens
    t0 = time.perf_counter()
    _oracle_step(x, w, S, tau, alloc_tile)
    one = time.perf_counter() - t0
    groups = max(1, min(w.tokens // S, int(target_s / max(one, 1e-3))))
    t0 = time.perf_counter()
    for g in range(groups):
        _oracle_step(x[g * S:], w, S, tau, alloc_tile)
    dt = time.perf_counter() - t0
    toks = groups * S
    gbs = toks * w.channels * (4 if w.dtype == "f32" else 2) / dt / 1e9
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "tokens_per_s": round(toks / dt, 1),
            "sample": f"{groups} of {w.tokens // S} token groups ({toks} tokens) encoded+decoded, "
                      f"single-threaded scalar C (-O2 -ffp-contract=off), {dt:.1f} s"}


def cpu_baseline_all_cores(w: synth.Workload, x, target_s: float = 6.0, tau=None,
                           alloc_tile=None) -> dict:
    """The same oracle with its token groups (encode) and token ranges (decode) on all host
    cores, whole tensor per step."""
    import oracle
    cores = os.cpu_count() or 1
    S = w.tokens_per_group or w.tokens
    used = max(1, min(cores, w.tokens // S))

    def step():
        r = oracle.encode(x, w.tile, w.hblock, w.bits_lo, w.bits_hi, w.budget, S, threads=cores,
                          tau=tau, alloc_tile=alloc_tile)
        oracle.decode(r["codes"], r["scales"], r["zeros"], r["bits"], r["pivots"], w.tokens,
                      w.channels, w.tile, w.hblock, threads=cores)

    t0 = time.perf_counter()
    step()
    one = time.perf_counter() - t0
    reps = max(1, int(target_s / max(one, 1e-3)))
    t0 = time.perf_counter()
    for _ in range(reps):
        step()
    dt = time.perf_counter() - t0
    toks = reps * w.tokens
    gbs = toks * w.channels * (4 if w.dtype == "f32" else 2) / dt / 1e9
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": used, "kind": "oracle",
            "tokens_per_s": round(toks / dt, 1),
            "sample": f"{reps} x the whole tensor ({w.tokens} tokens) encoded+decoded, "
                      f"{used} token groups on {used} of {cores} host threads "
                      f"(scalar C, -O2 -ffp-contract=off), {dt:.1f} s"}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    w = _workload(args)
    x = synth.generate(w)
    S = w.tokens_per_group or w.tokens
    # size each step's sample so that warm-up + timed steps take about 90 s of host time
    t0 = time.perf_counter()
    _oracle_step(x, w, 16, args.tau, args.alloc_tile or None)
    per_token = (time.perf_counter() - t0) / 16
    tok = int(max(1, min(S, 90.0 / max(1, args.steps + args.warmup) / max(per_token, 1e-9))))
    for _ in range(args.warmup):
        _oracle_step(x, w, tok, args.tau, args.alloc_tile or None)
    t0 = time.perf_counter()
    for k in range(args.steps):
        g = k % max(1, w.tokens // tok)
        _oracle_step(x[g * tok:], w, tok, args.tau, args.alloc_tile or None)
    dt = time.perf_counter() - t0
    in_b = tok * w.channels * (4 if w.dtype == "f32" else 2)
    gbs = in_b * args.steps / dt / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": _config(w, {"sample_tokens_per_step": tok,
                              "alloc_tile": args.alloc_tile or w.tile}, tau=args.tau),
        "tokens_per_s": round(tok * args.steps / dt, 1),
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"each step encodes+decodes {tok} consecutive tokens of the "
                                   f"workload (ranked as one group of {tok} tokens) on one host "
                                   f"core (scalar C oracle)"},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ replicas (N > 1)

def replica_tensor_index(rank: int, n_tensors: int, i: int) -> int:
    """Rank r encodes its own tensors: indices r * n_tensors .. r * n_tensors + n - 1 of the
    workload's generator (replicas, no shared input and no exchange)."""
    return rank * n_tensors + i


def max_over_ranks(ms: float, dist, device) -> float:
    """The job's time: the slowest rank's (all-reduce MAX; the identity on one process)."""
    if dist is None:
        return ms
    import torch
    t = torch.tensor([ms], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(world: int, in_bytes_per_step: int, steps: int, tot_ms: float) -> float:
    """Whole-job throughput in GB/s: the input bytes all ranks processed over the job time."""
    return world * in_bytes_per_step * steps / (tot_ms * 1e-3) / 1e9


# ------------------------------------------------------------------ the other configs

def per_config_workloads():
    """The parity configs besides the headline one, as (key, workload): the 2048-channel
    boundary, the 4096-channel boundary, and the 4096-channel sweep of tile = Hadamard block
    over {32, 64, 128} and budget over {3.0, 3.5, 4.0} (8 x 2048 x 4096 bf16, seed 3)."""
    out = [("c2", synth.WORKLOADS["c2"]), ("c3", synth.WORKLOADS["c3"])]
    base = synth.WORKLOADS["c4"]
    for g, b in synth.C4_SWEEP:
        out.append((f"c4_g{g}_b{b}", base.with_params(tile=g, hblock=g, budget=b)))
    return out


def time_config(tq, w: synth.Workload, x, steps: int, warmup: int, flush, peak: float) -> dict:
    """Encode on one stream and decode on another, each timed alone with CUDA events on its
    own stream, L2 flushed before each; medians (and means) over `steps` calls."""
    import torch
    T, C, G, h = w.tokens, w.channels, w.tile, w.hblock
    sa, sb = torch.cuda.Stream(device=x.device), torch.cuda.Stream(device=x.device)
    with torch.cuda.stream(sa):
        enc = tq.encode(x, G, h, w.bits_lo, w.bits_hi, w.budget, w.tokens_per_group)
    sa.synchronize()
    with torch.cuda.stream(sb):
        y = tq.decode(enc, T, C, G, h)
        dws = torch.empty(tq.tahq_decode_workspace_size(T, C, G), dtype=torch.uint8,
                          device=x.device)
    sb.synchronize()
    outs = {k: enc[k] for k in ("codes", "scales", "zeros", "bits", "pivots")}
    ws = enc["workspace"]
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps + warmup)]
    for k in range(steps + warmup):
        e = ev[k]
        with torch.cuda.stream(sa):
            flush.fill_(k & 255)
            e[0].record(sa)
            tq.encode(x, G, h, w.bits_lo, w.bits_hi, w.budget, w.tokens_per_group, out=outs,
                      workspace=ws, stream=sa)
            e[1].record(sa)
            flush.fill_((k + 7) & 255)
        sb.wait_stream(sa)
        with torch.cuda.stream(sb):
            e[2].record(sb)
            tq.decode(enc, T, C, G, h, out=y, workspace=dws, stream=sb)
            e[3].record(sb)
        sa.wait_stream(sb)
    torch.cuda.synchronize()
    rc, word = tq.tahq_get_device_status(ws, sa)
    if rc != 0:
        raise RuntimeError(f"{w.name}: device status {word:#x}")
    enc_ms = [e[0].elapsed_time(e[1]) for e in ev[warmup:]]
    dec_ms = [e[2].elapsed_time(e[3]) for e in ev[warmup:]]
    in_b, enc_b, dec_b = _alg_bytes(w, enc["payload_bytes"])

    def side(ms, alg):
        med = statistics.median(ms)
        return {"ms_median": round(med, 5), "ms_mean": round(statistics.mean(ms), 5),
                "alg_bytes": alg, "GB_s": round(alg / (med * 1e-3) / 1e9, 2),
                "frac": round(alg / (med * 1e-3) / 1e9 / peak, 4),
                "input_GB_s": round(in_b / (med * 1e-3) / 1e9, 2),
                "tokens_per_s": round(T / (med * 1e-3), 1)}
    return {"workload": w.name, "tile": G, "hblock": h, "budget": w.budget,
            "tokens_per_group": w.tokens_per_group, "steps": steps,
            "encode": side(enc_ms, enc_b), "decode": side(dec_ms, dec_b)}


def run_per_config(tq, dev, steps: int, warmup: int, flush, peak: float) -> dict:
    import torch
    res, cache = {}, {}
    for key, w in per_config_workloads():
        src = (w.tokens, w.channels, w.dtype, w.seed, w.dist)
        if src not in cache:
            cache.clear()
            xi = synth.generate(w)
            cache[src] = torch.from_numpy(xi.view(np.int16)).to(dev).view(torch.bfloat16) \
                if w.dtype == "bf16" else torch.from_numpy(xi).to(dev)
        res[key] = time_config(tq, w, cache[src], steps, warmup, flush, peak)
    target = [v for k, v in res.items() if k != "c2"]
    res["min_frac_4096_channels"] = {
        "encode": min(v["encode"]["frac"] for v in target),
        "decode": min(v["decode"]["frac"] for v in target)}
    return res


# ------------------------------------------------------------------ the backward pass

def run_grad(args):
    """The backward pass's gradient codecs on a gradient-shaped tensor (16 x 2048 x 8192
    fp32 by default): the fixed-point codec (tahq_naive_encode / _decode, 8 bits, tile 64,
    c = 2^16) and TAH-Quant on gradients with eq. (24)'s scaling (tahq_encode_scaled /
    _decode_scaled, widths {3, 4} at 4 bits, Appendix H Table 10).  Outputs and workspaces
    are allocated once; each call is timed alone with CUDA events, L2 flushed before it."""
    import torch
    import pipeline_activation_quantization_gb300 as tq
    w = synth.WORKLOADS[args.grad_workload]
    T, C, G = w.tokens, w.channels, w.tile
    b, c = args.grad_bits, 2.0 ** 16
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    x = torch.from_numpy(synth.generate(w)).to(dev)
    n = T * (C // G)
    nb = tq.tahq_naive_codes_bytes(T, C, G, b)
    codes = torch.empty(max(nb, 16), dtype=torch.uint8, device=dev)
    scales = torch.empty(n, dtype=torch.float32, device=dev)
    zeros = torch.empty(n, dtype=torch.float32, device=dev)
    y = torch.empty((T, C), dtype=torch.float32, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    st = torch.cuda.Stream(device=dev)
    enc_s = tq.encode_scaled(x, G, G, 3, 4, 4.0, w.tokens_per_group, scale_c=c, stream=st)
    outs = {k: enc_s[k] for k in ("codes", "scales", "zeros", "bits", "pivots")}
    dws = torch.empty(tq.tahq_decode_workspace_size(T, C, G), dtype=torch.uint8, device=dev)
    calls = {
        "naive_encode": lambda: tq.tahq_naive_encode(x, T, C, G, b, c, codes, scales, zeros, st),
        "naive_decode": lambda: tq.tahq_naive_decode(codes, scales, zeros, T, C, G, b, c, y, st),
        "tahq_encode_scaled": lambda: tq.encode_scaled(x, G, G, 3, 4, 4.0, w.tokens_per_group,
                                                       scale_c=c, out=outs,
                                                       workspace=enc_s["workspace"], stream=st),
        "tahq_decode_scaled": lambda: tq.decode_scaled(enc_s, T, C, G, G, scale_c=c, out=y,
                                                       workspace=dws, stream=st),
    }
    pay4 = enc_s["payload_bytes"]
    alg = {"naive_encode": 4 * T * C + nb + 8 * n, "naive_decode": nb + 8 * n + 4 * T * C,
           "tahq_encode_scaled": 4 * T * C + pay4 + 10 * n,
           "tahq_decode_scaled": pay4 + 10 * n + 4 * T * C}
    peak, peak_kind = _peaks()
    res = {}
    with torch.cuda.stream(st):
        for name, fn in calls.items():
            ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)]
                  for _ in range(args.steps + args.warmup)]
            for k, e in enumerate(ev):
                flush.fill_(k & 255)
                e[0].record(st)
                rc = fn()
                if isinstance(rc, int) and rc != 0:
                    raise RuntimeError(f"{name}: {tq.tahq_status_string(rc)}")
                e[1].record(st)
            st.synchronize()
            ms = [e[0].elapsed_time(e[1]) for e in ev[args.warmup:]]
            med = statistics.median(ms)
            gbs = alg[name] / (med * 1e-3) / 1e9
            res[name] = {"ms_median": round(med, 5), "ms_mean": round(statistics.mean(ms), 5),
                         "alg_bytes": alg[name], "GB_s": round(gbs, 2),
                         "frac": round(gbs / peak, 4),
                         "tokens_per_s": round(T / (med * 1e-3), 1)}
    rt = res["naive_encode"]["ms_median"] + res["naive_decode"]["ms_median"]
    dom = max(("naive_encode", "naive_decode"), key=lambda k: res[k]["ms_median"])
    kern = {"naive_encode": f"k_naive_encode<{G}>", "naive_decode": f"k_naive_decode<{G}>"}[dom]
    line = {
        "metric": "gradient codec GB/s of gradients (fixed-point, 8 bits) and % of GB300 HBM "
                  "roofline", "value": round(4 * T * C / (rt * 1e-3) / 1e9, 3), "unit": "GB/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(rt, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": w.name, "tokens": T, "channels": C, "tile": G, "bits": b,
                   "scale_c": c, "l2": "flushed before each call (256 MiB write, outside the events)"},
        "calls": res,
        "roofline": {"bound": "hbm", "kernel": kern, "achieved": res[dom]["GB_s"], "peak": peak,
                     "peak_kind": f"{peak_kind} HBM copy GB/s (burst)", "unit": "GB/s",
                     "frac": res[dom]["frac"], "traffic": None},
        "gpu_launches_per_step": 2,
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ the CUDA path

def run_gpu(args):
    import torch
    import pipeline_activation_quantization_gb300 as tq

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    w = _workload(args)
    T, C, G, h = w.tokens, w.channels, w.tile, w.hblock
    n_tensors = args.tensors or (3 if args.workload == "c5" else 1)
    dev = torch.device("cuda", local)
    xs, x_np = [], None
    for i in range(n_tensors):
        xi = synth.generate(w, index=replica_tensor_index(rank, n_tensors, i))
        if x_np is None:
            x_np = xi
        if w.dtype == "bf16":
            xs.append(torch.from_numpy(xi.view(np.int16)).to(dev).view(torch.bfloat16))
        else:
            xs.append(torch.from_numpy(xi).to(dev))
    x = xs[0]
    stream = torch.cuda.Stream(device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)

    lo, hi, beta, S = w.bits_lo, w.bits_hi, w.budget, w.tokens_per_group
    tau = 2.0 if args.tau is None else args.tau
    with torch.cuda.stream(stream):
        enc = tq.encode(x, G, h, lo, hi, beta, S, tau=args.tau, alloc_tile=args.alloc_tile or None)
        y = tq.decode(enc, T, C, G, h)
        dws = torch.empty(tq.tahq_decode_workspace_size(T, C, G), dtype=torch.uint8, device=dev)
        if args.wire:
            wbuf, wws = tq.encode_wire(x, G, h, lo, hi, beta, S, tau=tau)
            y, wdws = tq.decode_wire(wbuf, T, C, G, h, lo, hi, beta, S)
    payload = enc["payload_bytes"]
    out_bufs = {k: enc[k] for k in ("codes", "scales", "zeros", "bits", "pivots")}
    ws = wws if args.wire else enc["workspace"]

    def do_encode(xk):
        if args.wire:
            tq.encode_wire(xk, G, h, lo, hi, beta, S, tau=tau, out=wbuf, workspace=wws, stream=stream)
        else:
            tq.encode(xk, G, h, lo, hi, beta, S, out=out_bufs, workspace=ws, stream=stream,
                      tau=args.tau, alloc_tile=args.alloc_tile or None)

    def do_decode():
        if args.wire:
            tq.decode_wire(wbuf, T, C, G, h, lo, hi, beta, S, out=y, workspace=wdws, stream=stream)
        else:
            tq.decode(enc, T, C, G, h, out=y, workspace=dws, stream=stream)
    K_hi = tq.tahq_hi_count(T, C, G, w.bits_lo, w.bits_hi, w.budget, w.tokens_per_group)
    n_g = (w.tokens_per_group or T) * (C // G)
    if args.alloc_tile:
        n_g //= args.alloc_tile // G      # allocation tiles a group
        K_hi = int(np.floor((w.budget - w.bits_lo) * n_g / (w.bits_hi - w.bits_lo)))
    ranked = 0 < K_hi < n_g
    dt = "bf16" if w.dtype == "bf16" else "f32"
    esize = 2 if w.dtype == "bf16" else 4
    # the encoder's path, as the library chooses it (the launcher in tahq_encode.cuh):
    # the streaming encoder for the method's defaults (tau = 2, A = G, arrays) on tiles of
    # 32..128 values in 128-byte rows: one kernel for one width of 3 or 4 bits, else four
    # for widths {3, 4} ranked per group of whole 32 KB chunks; the three-stage encoder or
    # the work queue for the variants
    n_tiles = T * (C // G)
    n_g_t = (w.tokens_per_group or T) * (C // G)
    ch = 32768 // (G * esize)
    flat_b = w.bits_lo if K_hi == 0 else w.bits_hi
    streaming = (args.alloc_tile in (0, G) and 32 <= G <= 128
                 and (n_tiles * G * esize) % 128 == 0 and (n_g_t * G) % 128 == 0)
    run_flat = streaming and not ranked and flat_b in (3, 4)
    run_ranked = (streaming and ranked and (w.bits_lo, w.bits_hi) == (3, 4)
                  and n_g_t % ch == 0)
    three = (not run_ranked and ranked and G * esize >= 128 and (w.bits_lo, w.bits_hi) == (3, 4)
             and args.alloc_tile in (0, G) and n_g_t % ch == 0)
    if run_flat:
        enc_launches, enc_kernel = 1, f"k_run_flat<{dt},{G},{flat_b}>"
    elif run_ranked:
        enc_launches = 3
        enc_kernel = f"k_run_tiles<{dt},{G}> (+ k_run_select, k_run_compact)"
    elif three:
        enc_launches = 6
        enc_kernel = f"k_stats<{dt},{G}> + k_quant<{dt},{G}> (+ k_gather, k_rank, k_widths, k_chunk_scan)"
    elif ranked:
        enc_launches, enc_kernel = 2, f"k_encode<{dt},{G}> (+ k_items)"
    else:
        enc_launches, enc_kernel = 1, f"k_encode_flat<{dt},{G}>"
    # decode: totals (with the offsets scan), decode; the wire format adds pack and unpack
    launches = enc_launches + 2 + (2 if args.wire else 0)

    def step(ev, k=0):
        ev[0].record(stream)
        do_encode(xs[k % n_tensors])
        ev[1].record(stream)
        flush.fill_((k + 7) & 255)  # the payload is not left in L2 for the decoder
        ev[2].record(stream)
        do_decode()
        ev[3].record(stream)

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    warm = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush.fill_(1)
            step(warm)
    stream.synchronize()
    barrier()
    sampler = ClockSampler(local)
    with sampler:
        t_wall = time.perf_counter()
        with torch.cuda.stream(stream):
            for k in range(args.steps):
                flush.fill_(k & 255)
                step(evs[k], k)
        stream.synchronize()
        t_wall = time.perf_counter() - t_wall
    barrier()
    enc_ms = [e[0].elapsed_time(e[1]) for e in evs]
    dec_ms = [e[2].elapsed_time(e[3]) for e in evs]
    tot_ms = sum(enc_ms) + sum(dec_ms)
    rc, word = tq.tahq_get_device_status(ws, stream)
    if rc != 0:
        raise RuntimeError(f"device status {word:#x} after the timed loop")
    tot_ms = max_over_ranks(tot_ms, dist, dev)

    in_b, enc_b, dec_b = _alg_bytes(w, payload)
    if args.wire:  # the whole buffer is written, then read
        wire_b = tq.tahq_wire_size(T, C, G, lo, hi, beta, S)
        enc_b, dec_b = in_b + wire_b, wire_b + 4 * w.elements
    peak, peak_kind = _peaks()
    ms_step = tot_ms / args.steps
    value = job_value(world, in_b, args.steps, tot_ms)
    e_ms, d_ms = statistics.mean(enc_ms), statistics.mean(dec_ms)
    enc_gbs, dec_gbs = enc_b / (e_ms * 1e-3) / 1e9, dec_b / (d_ms * 1e-3) / 1e9
    dom = ("decode", dec_b, d_ms) if d_ms >= e_ms else ("encode", enc_b, e_ms)
    dom_name = f"k_decode<{G}> (+ k_dec_totals)" if dom[0] == "decode" else enc_kernel
    if args.wire:
        dom_name += " + k_wire_unpack" if dom[0] == "decode" else " + k_wire_pack"

    # end to end through the public API: pinned host input -> device, encode, decode,
    # decoded tensor -> pinned host
    e2e = None
    if not args.no_e2e:
        x_host = torch.from_numpy(x_np.view(np.int16) if w.dtype == "bf16" else x_np).pin_memory()
        y_host = torch.empty((T, C), dtype=torch.float32).pin_memory()
        x_dev = torch.empty_like(x)
        n_e2e = max(3, min(20, args.steps))
        # the arrays format with token groups: the pipelined host round trip of the package
        # (chunks of whole groups, copies in and out overlapping the codec); else one copy
        # in, encode, decode, one copy out
        rt = None
        if not args.wire and S and S < T and T % S == 0 and args.tau is None and not args.alloc_tile:
            from pipeline_activation_quantization_gb300.host import HostRoundTrip
            rt = HostRoundTrip(T, C, x.dtype, tile=G, hblock=h, bits_lo=lo, bits_hi=hi,
                               budget=beta, tokens_per_group=S)
            if w.dtype == "bf16":
                x_host = x_host.view(torch.bfloat16)
        with torch.cuda.stream(stream):
            def e2e_step():
                if rt is not None:
                    rt.run(x_host, y_host, stream=stream)
                    return
                if w.dtype == "bf16":
                    x_dev.view(torch.int16).copy_(x_host, non_blocking=True)
                else:
                    x_dev.copy_(x_host, non_blocking=True)
                do_encode(x_dev)
                do_decode()
                y_host.copy_(y, non_blocking=True)
            e2e_step()
            stream.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(n_e2e):
                e2e_step()
            e1.record(stream)
        stream.synchronize()
        e2e_ms = e0.elapsed_time(e1) / n_e2e
        e2e = {"value": round(world * in_b / (e2e_ms * 1e-3) / 1e9, 3), "unit": "GB/s",
               "h2d_bytes_per_step": in_b, "d2h_bytes_per_step": 4 * w.elements,
               "ms_per_step": round(e2e_ms, 4), "steps": n_e2e,
               "api": ("HostRoundTrip, chunks of one token group, copies overlapping the codec"
                       if rt is not None else "encode + decode between one copy in and one out")}

    if rank != 0:
        return 0
    per_config = None
    if not args.no_per_config and args.workload == "c5" and not (args.tokens or args.tile or args.budget
                                                                 or args.tau is not None
                                                                 or args.alloc_tile or args.wire):
        xs.clear()
        per_config = run_per_config(tq, dev, max(20, args.steps), max(5, args.warmup), flush,
                                    _peaks()[0])
    A = args.alloc_tile or None
    cpu = (None if args.no_cpu_baseline or world > 1
           else cpu_baseline(w, x_np, tau=args.tau, alloc_tile=A))
    cpu_all = (None if args.no_cpu_baseline or world > 1
               else cpu_baseline_all_cores(w, x_np, tau=args.tau, alloc_tile=A))
    clocks = sampler.summary()
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": _config(w, {"parallelism": f"replicas{world}",
                                                     "fresh_tensors_cycled": n_tensors,
                                                     "format": "wire" if args.wire else "arrays",
                                                     "alloc_tile": args.alloc_tile or G},
                                                  tau=args.tau),
        "tokens_per_s": round(world * T / (ms_step * 1e-3), 1),
        "roofline_frac_round_trip": round((enc_b + dec_b) / (ms_step * 1e-3) / 1e9 / peak, 4),
        "encode": {"ms": round(e_ms, 5), "ms_median": round(statistics.median(enc_ms), 5),
                   "alg_bytes": enc_b, "GB_s": round(enc_gbs, 2),
                   "frac": round(enc_gbs / peak, 4), "input_GB_s": round(in_b / (e_ms * 1e-3) / 1e9, 2),
                   "tokens_per_s": round(T / (e_ms * 1e-3), 1)},
        "decode": {"ms": round(d_ms, 5), "ms_median": round(statistics.median(dec_ms), 5),
                   "alg_bytes": dec_b, "GB_s": round(dec_gbs, 2),
                   "frac": round(dec_gbs / peak, 4), "tokens_per_s": round(T / (d_ms * 1e-3), 1)},
        "roofline": {"bound": "hbm", "kernel": dom_name,
                     "achieved": round(dom[1] / (dom[2] * 1e-3) / 1e9, 2), "peak": peak,
                     "peak_kind": f"{peak_kind} HBM copy GB/s (burst)", "unit": "GB/s",
                     "frac": round(dom[1] / (dom[2] * 1e-3) / 1e9 / peak, 4),
                     "traffic": (_traffic_for(dom_name, w.name)
                                 if args.tau is None and not args.wire and not args.alloc_tile
                                 else None)},
        "payload_bytes": payload, "bits_per_element": round(payload * 8 / w.elements, 4),
        "cpu_baseline": cpu, "cpu_baseline_all_cores": cpu_all, "e2e": e2e, "gpu_launches": launches * args.steps,
        "gpu_launches_per_step": launches, "clocks": clocks, "per_config": per_config,
        "wall_s_timed_loop": round(t_wall, 3),
    }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="tahq", choices=["tahq", "reference"])
    ap.add_argument("--workload", default="c5", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--tensors", type=int, default=0,
                    help="distinct seeded tensors cycled over the steps (default 3 for c5, else 1)")
    ap.add_argument("--tokens", type=int, default=0,
                    help="run the workload on its first N tokens (a multiple of its token group)")
    ap.add_argument("--tile", type=int, default=0)
    ap.add_argument("--hblock", type=int, default=0)
    ap.add_argument("--budget", type=float, default=None)
    ap.add_argument("--tau", type=float, default=None,
                    help="outlier threshold (default: the method's 2.0)")
    ap.add_argument("--alloc-tile", type=int, default=0,
                    help="allocation tile A in channels (default: the tile)")
    ap.add_argument("--wire", action="store_true",
                    help="time the wire format (tahq_encode_wire / tahq_decode_wire)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--grad", action="store_true",
                    help="time the backward pass's gradient codecs instead (one JSON line)")
    ap.add_argument("--grad-workload", default="g5", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--grad-bits", type=int, default=8)
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the 2048/4096-channel configs (timed after the headline one)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    return args


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.grad:
        return run_grad(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
