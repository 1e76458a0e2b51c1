"""GB300 (sm_103a) TAH-Quant activation codec: a thin binding of ``include/tahq.h``.

The ``tahq_*`` functions have the names and arguments of the C ABI; they only marshal
arguments (torch tensors become device pointers, the current torch stream is passed
unless one is given).  Every step of the codec runs in the CUDA kernels of
``libtahq.so``; there is no CPU fallback, and importing fails loudly when the library
has not been built (``python -m pipeline_activation_quantization_gb300.build``).

``encode`` / ``decode`` are conveniences that allocate outputs and workspace with torch
(device memory only) and call the same entry points.
"""
from __future__ import annotations

import ctypes as C
import os

from . import build as _build

__all__ = [
    "TAHQ_F32", "TAHQ_BF16", "TahqError", "lib", "tahq_payload_size", "tahq_hi_count",
    "tahq_workspace_size", "tahq_decode_workspace_size", "tahq_encode", "tahq_encode_ex",
    "tahq_decode", "tahq_get_device_status", "tahq_status_string", "tahq_version", "tahq_log2_tables",
    "tahq_decode_noalloc", "tahq_wire_size", "tahq_wire_workspace_size",
    "tahq_wire_decode_workspace_size", "tahq_encode_wire", "tahq_decode_wire", "encode", "decode",
    "encode_wire", "decode_wire", "tahq_naive_codes_bytes", "tahq_naive_encode",
    "tahq_naive_decode", "naive_encode", "naive_decode", "tahq_test_wait_timeout",
    "tahq_scaled_workspace_size", "tahq_encode_scaled", "tahq_decode_scaled", "encode_scaled",
    "decode_scaled", "EXPORTED_SYMBOLS",
]

TAHQ_F32, TAHQ_BF16 = 0, 1
STATUS_NAMES = {0: "TAHQ_OK", 1: "TAHQ_ERR_ARG", 2: "TAHQ_ERR_UNSUPPORTED", 3: "TAHQ_ERR_WORKSPACE",
                4: "TAHQ_ERR_CUDA", 5: "TAHQ_ERR_DEVICE_STATUS"}
DEV_NONFINITE, DEV_WAIT_TIMEOUT, DEV_SELECT_MISMATCH, DEV_BAD_BITS, DEV_STREAM_OVERRUN = 1, 2, 4, 8, 16
DEV_BAD_WIRE = 32

# Every extern "C" function declared in include/tahq.h.
EXPORTED_SYMBOLS = (
    "tahq_payload_size", "tahq_hi_count", "tahq_workspace_size", "tahq_encode", "tahq_encode_ex",
    "tahq_payload_size_ex", "tahq_decode_workspace_size", "tahq_decode", "tahq_get_device_status",
    "tahq_status_string", "tahq_version", "tahq_log2_tables", "tahq_decode_noalloc",
    "tahq_wire_size", "tahq_wire_workspace_size", "tahq_wire_decode_workspace_size",
    "tahq_encode_wire", "tahq_decode_wire", "tahq_naive_codes_bytes", "tahq_naive_encode",
    "tahq_naive_decode", "tahq_test_wait_timeout", "tahq_scaled_workspace_size",
    "tahq_encode_scaled", "tahq_decode_scaled",
)


class TahqError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)}")


_lib = None


def lib(path: str | None = None):
    """Load ``libtahq.so`` (build it first if it is missing or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or _build.build()
    if not os.path.exists(path):
        raise ImportError(f"libtahq.so not found at {path}")
    L = C.CDLL(path)
    i64, i32, sz, p, f32 = C.c_int64, C.c_int, C.c_size_t, C.c_void_p, C.c_float
    sig = {
        "tahq_payload_size": (sz, [i64, i64, i32, i32, i32, f32, i64]),
        "tahq_hi_count": (i64, [i64, i64, i32, i32, i32, f32, i64]),
        "tahq_workspace_size": (sz, [i64, i64, i32, i32, i32, i32, f32, i64]),
        "tahq_decode_workspace_size": (sz, [i64, i64, i32]),
        "tahq_encode": (i32, [p, i32, i64, i64, i32, i32, i32, i32, f32, i64,
                              p, p, p, p, p, p, sz, p]),
        "tahq_encode_ex": (i32, [p, i32, i64, i64, i32, i32, i32, i32, f32, i64, f32, i32,
                                 p, p, p, p, p, p, sz, p]),
        "tahq_payload_size_ex": (sz, [i64, i64, i32, i32, i32, i32, f32, i64]),
        "tahq_decode": (i32, [p, sz, p, p, p, p, i64, i64, i32, i32, p, p, sz, p]),
        "tahq_get_device_status": (i32, [p, C.POINTER(C.c_uint32), p]),
        "tahq_status_string": (C.c_char_p, [i32]),
        "tahq_version": (i32, []),
        "tahq_log2_tables": (None, [p, p, p]),
        "tahq_decode_noalloc": (i32, [p, sz, p, p, p, p, i64, i64, i32, i32, p, p, p]),
        "tahq_wire_size": (sz, [i64, i64, i32, i32, i32, f32, i64]),
        "tahq_wire_workspace_size": (sz, [i64, i64, i32, i32, i32, i32, f32, i64]),
        "tahq_wire_decode_workspace_size": (sz, [i64, i64, i32]),
        "tahq_encode_wire": (i32, [p, i32, i64, i64, i32, i32, i32, i32, f32, i64, f32, p, sz,
                                   p, sz, p]),
        "tahq_decode_wire": (i32, [p, sz, i64, i64, i32, i32, i32, i32, f32, i64, p, p, sz, p]),
        "tahq_naive_codes_bytes": (sz, [i64, i64, i32, i32]),
        "tahq_naive_encode": (i32, [p, i64, i64, i32, i32, f32, p, p, p, p]),
        "tahq_naive_decode": (i32, [p, p, p, i64, i64, i32, i32, f32, p, p]),
        "tahq_test_wait_timeout": (i32, [p, sz, C.c_uint64, p, p]),
        "tahq_scaled_workspace_size": (sz, [i64, i64, i32, i32, i32, i32, f32, i64, i32]),
        "tahq_encode_scaled": (i32, [p, i32, i64, i64, i32, i32, i32, i32, f32, i64, f32, f32,
                                     p, p, p, p, p, p, sz, p]),
        "tahq_decode_scaled": (i32, [p, sz, p, p, p, p, i64, i64, i32, i32, f32, p, p, sz, p]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return L


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ------------------------------------------------------------------ C-ABI names

def tahq_payload_size(tokens, channels, tile, bits_lo, bits_hi, budget, tokens_per_group) -> int:
    return lib().tahq_payload_size(tokens, channels, tile, bits_lo, bits_hi, budget, tokens_per_group)


def tahq_hi_count(tokens, channels, tile, bits_lo, bits_hi, budget, tokens_per_group) -> int:
    return lib().tahq_hi_count(tokens, channels, tile, bits_lo, bits_hi, budget, tokens_per_group)


def tahq_workspace_size(tokens, channels, tile, hblock, bits_lo, bits_hi, budget, tokens_per_group) -> int:
    return lib().tahq_workspace_size(tokens, channels, tile, hblock, bits_lo, bits_hi, budget,
                                     tokens_per_group)


def tahq_decode_workspace_size(tokens, channels, tile) -> int:
    return lib().tahq_decode_workspace_size(tokens, channels, tile)


def tahq_encode(x, dtype, tokens, channels, tile, hblock, bits_lo, bits_hi, budget,
                tokens_per_group, codes, scales, zeros, bits, pivots, workspace,
                workspace_bytes, stream=None) -> int:
    return lib().tahq_encode(_ptr(x), dtype, tokens, channels, tile, hblock, bits_lo, bits_hi,
                             budget, tokens_per_group, _ptr(codes), _ptr(scales), _ptr(zeros),
                             _ptr(bits), _ptr(pivots), _ptr(workspace), workspace_bytes,
                             _stream(stream))


def tahq_encode_ex(x, dtype, tokens, channels, tile, hblock, bits_lo, bits_hi, budget,
                   tokens_per_group, tau, alloc_tile, codes, scales, zeros, bits, pivots,
                   workspace, workspace_bytes, stream=None) -> int:
    return lib().tahq_encode_ex(_ptr(x), dtype, tokens, channels, tile, hblock, bits_lo,
                                bits_hi, budget, tokens_per_group, tau, alloc_tile, _ptr(codes),
                                _ptr(scales), _ptr(zeros), _ptr(bits), _ptr(pivots),
                                _ptr(workspace), workspace_bytes, _stream(stream))


def tahq_payload_size_ex(tokens, channels, tile, alloc_tile, bits_lo, bits_hi, budget,
                         tokens_per_group) -> int:
    return lib().tahq_payload_size_ex(tokens, channels, tile, alloc_tile, bits_lo, bits_hi,
                                      budget, tokens_per_group)


def tahq_decode(codes, codes_bytes, scales, zeros, bits, pivots, tokens, channels, tile, hblock,
                out, workspace, workspace_bytes, stream=None) -> int:
    return lib().tahq_decode(_ptr(codes), codes_bytes, _ptr(scales), _ptr(zeros), _ptr(bits),
                             _ptr(pivots), tokens, channels, tile, hblock, _ptr(out),
                             _ptr(workspace), workspace_bytes, _stream(stream))


def tahq_decode_noalloc(codes, codes_bytes, scales, zeros, bits, pivots, tokens, channels, tile,
                        hblock, out, device_status=None, stream=None) -> int:
    """tahq_decode without a workspace, for callers that cannot allocate device memory
    (the scratch is a fixed array inside the library; see include/tahq.h)."""
    return lib().tahq_decode_noalloc(_ptr(codes), codes_bytes, _ptr(scales), _ptr(zeros),
                                     _ptr(bits), _ptr(pivots), tokens, channels, tile, hblock,
                                     _ptr(out), _ptr(device_status), _stream(stream))


def tahq_test_wait_timeout(workspace, workspace_bytes, limit_ns, elapsed_ns=None,
                           stream=None) -> int:
    return lib().tahq_test_wait_timeout(_ptr(workspace), workspace_bytes, int(limit_ns),
                                        _ptr(elapsed_ns), _stream(stream))


def tahq_get_device_status(workspace, stream=None) -> tuple[int, int]:
    """-> (tahq_status, raw status word)."""
    word = C.c_uint32(0)
    rc = lib().tahq_get_device_status(_ptr(workspace), C.byref(word), _stream(stream))
    return rc, word.value


def tahq_status_string(status: int) -> str:
    return lib().tahq_status_string(status).decode()


def tahq_version() -> int:
    return lib().tahq_version()


def tahq_log2_tables():
    import numpy as np
    T = np.zeros(128, np.float32); R = np.zeros(128, np.float32); k = np.zeros(3, np.float32)
    lib().tahq_log2_tables(T.ctypes.data, R.ctypes.data, k.ctypes.data)
    return T, R, k


# ------------------------------------------------------------------ conveniences (torch memory)

def _check(rc: int, what: str):
    if rc != 0:
        raise TahqError(rc, what)


def encode(x, tile: int = 64, hblock: int | None = None, bits_lo: int = 3, bits_hi: int = 4,
           budget: float = 3.5, tokens_per_group: int = 0, out: dict | None = None,
           workspace=None, stream=None, tau: float | None = None,
           alloc_tile: int | None = None) -> dict:
    """Encode a CUDA tensor ``x`` ([tokens, channels], float32 or bfloat16).  ``tau`` is the
    outlier threshold and ``alloc_tile`` the allocation tile A (None: the method's 2.0 and
    A = tile, through tahq_encode; else tahq_encode_ex).

    Returns ``{"codes", "scales", "zeros", "bits", "pivots", "workspace"}`` (torch tensors on
    x's device).  Pass ``out`` / ``workspace`` from an earlier call to reuse them.
    """
    import torch
    if not x.is_cuda:
        raise ValueError("tahq.encode needs a CUDA tensor")
    if x.dtype == torch.float32:
        dt = TAHQ_F32
    elif x.dtype == torch.bfloat16:
        dt = TAHQ_BF16
    else:
        raise ValueError(f"unsupported dtype {x.dtype}")
    x = x.contiguous()
    T, Cc = x.shape
    h = hblock or tile
    n = T * (Cc // tile)
    pay = (tahq_payload_size(T, Cc, tile, bits_lo, bits_hi, budget, tokens_per_group)
           if not alloc_tile else
           tahq_payload_size_ex(T, Cc, tile, alloc_tile, bits_lo, bits_hi, budget,
                                tokens_per_group))
    ws = tahq_workspace_size(T, Cc, tile, h, bits_lo, bits_hi, budget, tokens_per_group)
    if ws == 0:
        raise TahqError(1, "tahq_workspace_size")
    dev = x.device
    if out is None:
        out = {
            "codes": torch.empty(max(pay, 16), dtype=torch.uint8, device=dev),
            "scales": torch.empty(n, dtype=torch.float32, device=dev),
            "zeros": torch.empty(n, dtype=torch.float32, device=dev),
            "bits": torch.empty(n, dtype=torch.uint8, device=dev),
            "pivots": torch.empty(n, dtype=torch.uint8, device=dev),
        }
    if workspace is None:
        workspace = torch.empty(ws, dtype=torch.uint8, device=dev)
    if tau is None and not alloc_tile:
        rc = tahq_encode(x, dt, T, Cc, tile, h, bits_lo, bits_hi, budget, tokens_per_group,
                         out["codes"], out["scales"], out["zeros"], out["bits"], out["pivots"],
                         workspace, workspace.numel(), stream)
    else:
        rc = tahq_encode_ex(x, dt, T, Cc, tile, h, bits_lo, bits_hi, budget, tokens_per_group,
                            2.0 if tau is None else float(tau), int(alloc_tile or 0),
                            out["codes"], out["scales"], out["zeros"], out["bits"],
                            out["pivots"], workspace, workspace.numel(), stream)
    _check(rc, "tahq_encode")
    res = dict(out)
    res["codes"] = out["codes"][:pay]
    res["workspace"] = workspace
    res["payload_bytes"] = pay
    return res


def decode(enc: dict, tokens: int, channels: int, tile: int = 64, hblock: int | None = None,
           out=None, workspace=None, stream=None):
    """Decode the dict returned by ``encode`` into a float32 CUDA tensor [tokens, channels]."""
    import torch
    dev = enc["scales"].device
    h = hblock or tile
    ws = tahq_decode_workspace_size(tokens, channels, tile)
    if ws == 0:
        raise TahqError(1, "tahq_decode_workspace_size")
    if out is None:
        out = torch.empty((tokens, channels), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = torch.empty(ws, dtype=torch.uint8, device=dev)
    codes = enc["codes"]
    rc = tahq_decode(codes, codes.numel(), enc["scales"], enc["zeros"], enc["bits"], enc["pivots"],
                     tokens, channels, tile, h, out, workspace, workspace.numel(), stream)
    _check(rc, "tahq_decode")
    return out


# ------------------------------------------------------------------ wire format

def tahq_wire_size(tokens, channels, tile, bits_lo, bits_hi, budget, tokens_per_group) -> int:
    return lib().tahq_wire_size(tokens, channels, tile, bits_lo, bits_hi, budget, tokens_per_group)


def tahq_wire_workspace_size(tokens, channels, tile, hblock, bits_lo, bits_hi, budget,
                             tokens_per_group) -> int:
    return lib().tahq_wire_workspace_size(tokens, channels, tile, hblock, bits_lo, bits_hi,
                                          budget, tokens_per_group)


def tahq_wire_decode_workspace_size(tokens, channels, tile) -> int:
    return lib().tahq_wire_decode_workspace_size(tokens, channels, tile)


def tahq_encode_wire(x, dtype, tokens, channels, tile, hblock, bits_lo, bits_hi, budget,
                     tokens_per_group, tau, wire, wire_bytes, workspace, workspace_bytes,
                     stream=None) -> int:
    return lib().tahq_encode_wire(_ptr(x), dtype, tokens, channels, tile, hblock, bits_lo,
                                  bits_hi, budget, tokens_per_group, tau, _ptr(wire), wire_bytes,
                                  _ptr(workspace), workspace_bytes, _stream(stream))


def tahq_decode_wire(wire, wire_bytes, tokens, channels, tile, hblock, bits_lo, bits_hi, budget,
                     tokens_per_group, out, workspace, workspace_bytes, stream=None) -> int:
    return lib().tahq_decode_wire(_ptr(wire), wire_bytes, tokens, channels, tile, hblock, bits_lo,
                                  bits_hi, budget, tokens_per_group, _ptr(out), _ptr(workspace),
                                  workspace_bytes, _stream(stream))


def encode_wire(x, tile: int = 64, hblock: int | None = None, bits_lo: int = 3, bits_hi: int = 4,
                budget: float = 3.5, tokens_per_group: int = 0, tau: float = 2.0, out=None,
                workspace=None, stream=None):
    """Encode a CUDA tensor into one wire buffer (uint8 CUDA tensor of tahq_wire_size bytes).

    Returns ``(wire, workspace)``; pass them back in to reuse them.
    """
    import torch
    if not x.is_cuda:
        raise ValueError("tahq.encode_wire needs a CUDA tensor")
    if x.dtype == torch.float32:
        dt = TAHQ_F32
    elif x.dtype == torch.bfloat16:
        dt = TAHQ_BF16
    else:
        raise ValueError(f"unsupported dtype {x.dtype}")
    x = x.contiguous()
    T, Cc = x.shape
    h = hblock or tile
    size = tahq_wire_size(T, Cc, tile, bits_lo, bits_hi, budget, tokens_per_group)
    ws = tahq_wire_workspace_size(T, Cc, tile, h, bits_lo, bits_hi, budget, tokens_per_group)
    if size == 0 or ws == 0:
        raise TahqError(1, "tahq_wire_size")
    if out is None:
        out = torch.empty(size, dtype=torch.uint8, device=x.device)
    if workspace is None:
        workspace = torch.empty(ws, dtype=torch.uint8, device=x.device)
    rc = tahq_encode_wire(x, dt, T, Cc, tile, h, bits_lo, bits_hi, budget, tokens_per_group,
                          float(tau), out, out.numel(), workspace, workspace.numel(), stream)
    _check(rc, "tahq_encode_wire")
    return out, workspace


def decode_wire(wire, tokens: int, channels: int, tile: int = 64, hblock: int | None = None,
                bits_lo: int = 3, bits_hi: int = 4, budget: float = 3.5, tokens_per_group: int = 0,
                out=None, workspace=None, stream=None):
    """Decode a wire buffer into a float32 CUDA tensor [tokens, channels].

    Returns ``(out, workspace)``; the workspace's status word reports a header that does
    not match the arguments (DEV_BAD_WIRE).
    """
    import torch
    h = hblock or tile
    ws = tahq_wire_decode_workspace_size(tokens, channels, tile)
    if ws == 0:
        raise TahqError(1, "tahq_wire_decode_workspace_size")
    if out is None:
        out = torch.empty((tokens, channels), dtype=torch.float32, device=wire.device)
    if workspace is None:
        workspace = torch.empty(ws, dtype=torch.uint8, device=wire.device)
    rc = tahq_decode_wire(wire, wire.numel(), tokens, channels, tile, h, bits_lo, bits_hi, budget,
                          tokens_per_group, out, workspace, workspace.numel(), stream)
    _check(rc, "tahq_decode_wire")
    return out, workspace


# ------------------------------------------------------------------ backward gradients

def tahq_naive_codes_bytes(tokens, channels, tile, bits) -> int:
    return lib().tahq_naive_codes_bytes(tokens, channels, tile, bits)


def tahq_naive_encode(grad, tokens, channels, tile, bits, scale_c, codes, scales, zeros,
                      stream=None) -> int:
    return lib().tahq_naive_encode(_ptr(grad), tokens, channels, tile, bits, scale_c, _ptr(codes),
                                   _ptr(scales), _ptr(zeros), _stream(stream))


def tahq_naive_decode(codes, scales, zeros, tokens, channels, tile, bits, scale_c, out,
                      stream=None) -> int:
    return lib().tahq_naive_decode(_ptr(codes), _ptr(scales), _ptr(zeros), tokens, channels, tile,
                                   bits, scale_c, _ptr(out), _stream(stream))


def naive_encode(grad, tile: int = 64, bits: int = 8, scale_c: float = 1.0, stream=None):
    """The backward pass's fixed-point codec of a float32 CUDA tensor [tokens, channels]:
    ``(codes, scales, zeros)`` as CUDA tensors."""
    import torch
    if not grad.is_cuda or grad.dtype != torch.float32:
        raise ValueError("tahq.naive_encode needs a float32 CUDA tensor")
    grad = grad.contiguous()
    T, Cc = grad.shape
    nb = tahq_naive_codes_bytes(T, Cc, tile, bits)
    if nb == 0 and T > 0:
        raise TahqError(1, "tahq_naive_codes_bytes")
    n = T * (Cc // tile)
    codes = torch.empty(max(nb, 16), dtype=torch.uint8, device=grad.device)
    scales = torch.empty(n, dtype=torch.float32, device=grad.device)
    zeros = torch.empty(n, dtype=torch.float32, device=grad.device)
    rc = tahq_naive_encode(grad, T, Cc, tile, bits, scale_c, codes, scales, zeros, stream)
    _check(rc, "tahq_naive_encode")
    return codes[:nb], scales, zeros


def naive_decode(codes, scales, zeros, tokens: int, channels: int, tile: int = 64, bits: int = 8,
                 scale_c: float = 1.0, out=None, stream=None):
    """The float32 CUDA tensor [tokens, channels] back from naive_encode's outputs.  The
    buffers are checked against the shape first (the C entry point trusts them)."""
    import torch
    nb = tahq_naive_codes_bytes(tokens, channels, tile, bits)
    n = tokens * (channels // tile) if tile > 0 else 0
    if nb == 0 and tokens > 0:
        raise TahqError(1, "tahq_naive_codes_bytes")
    if codes.numel() < nb or scales.numel() != n or zeros.numel() != n:
        raise ValueError("naive_decode: codes, scales or zeros do not match the shape")
    if scales.dtype != torch.float32 or zeros.dtype != torch.float32:
        raise ValueError("naive_decode: scales and zeros must be float32")
    if out is None:
        out = torch.empty((tokens, channels), dtype=torch.float32, device=codes.device)
    elif (out.dtype != torch.float32 or not out.is_contiguous()
          or tuple(out.shape) != (tokens, channels)):
        raise ValueError("naive_decode: out must be a contiguous float32 [tokens, channels] tensor")
    rc = tahq_naive_decode(codes, scales, zeros, tokens, channels, tile, bits, scale_c, out, stream)
    _check(rc, "tahq_naive_decode")
    return out


# ------------------------------------------------------------------ gradients (eq. (24))

def tahq_scaled_workspace_size(tokens, channels, tile, hblock, bits_lo, bits_hi, budget,
                               tokens_per_group, dtype) -> int:
    return lib().tahq_scaled_workspace_size(tokens, channels, tile, hblock, bits_lo, bits_hi,
                                            budget, tokens_per_group, dtype)


def tahq_encode_scaled(x, dtype, tokens, channels, tile, hblock, bits_lo, bits_hi, budget,
                       tokens_per_group, tau, scale_c, codes, scales, zeros, bits, pivots,
                       workspace, workspace_bytes, stream=None) -> int:
    return lib().tahq_encode_scaled(_ptr(x), dtype, tokens, channels, tile, hblock, bits_lo,
                                    bits_hi, budget, tokens_per_group, tau, scale_c, _ptr(codes),
                                    _ptr(scales), _ptr(zeros), _ptr(bits), _ptr(pivots),
                                    _ptr(workspace), workspace_bytes, _stream(stream))


def tahq_decode_scaled(codes, codes_bytes, scales, zeros, bits, pivots, tokens, channels, tile,
                       hblock, scale_c, out, workspace, workspace_bytes, stream=None) -> int:
    return lib().tahq_decode_scaled(_ptr(codes), codes_bytes, _ptr(scales), _ptr(zeros),
                                    _ptr(bits), _ptr(pivots), tokens, channels, tile, hblock,
                                    scale_c, _ptr(out), _ptr(workspace), workspace_bytes,
                                    _stream(stream))


def encode_scaled(x, tile: int = 64, hblock: int | None = None, bits_lo: int = 3,
                  bits_hi: int = 4, budget: float = 3.5, tokens_per_group: int = 0,
                  tau: float = 2.0, scale_c: float = 1.0, out: dict | None = None,
                  workspace=None, stream=None) -> dict:
    """TAH-Quant on a gradient (float32 or bfloat16 CUDA tensor) with eq. (24)'s scaling by
    the power of two ``scale_c``; returns the dict of ``encode`` (metadata of the scaled
    values)."""
    import torch
    if not x.is_cuda:
        raise ValueError("tahq.encode_scaled needs a CUDA tensor")
    dt = {torch.float32: TAHQ_F32, torch.bfloat16: TAHQ_BF16}.get(x.dtype)
    if dt is None:
        raise ValueError(f"unsupported dtype {x.dtype}")
    x = x.contiguous()
    T, Cc = x.shape
    h = hblock or tile
    n = T * (Cc // tile)
    pay = tahq_payload_size(T, Cc, tile, bits_lo, bits_hi, budget, tokens_per_group)
    ws = tahq_scaled_workspace_size(T, Cc, tile, h, bits_lo, bits_hi, budget, tokens_per_group, dt)
    if ws == 0:
        raise TahqError(1, "tahq_scaled_workspace_size")
    dev = x.device
    if out is None:
        out = {"codes": torch.empty(max(pay, 16), dtype=torch.uint8, device=dev),
               "scales": torch.empty(n, dtype=torch.float32, device=dev),
               "zeros": torch.empty(n, dtype=torch.float32, device=dev),
               "bits": torch.empty(n, dtype=torch.uint8, device=dev),
               "pivots": torch.empty(n, dtype=torch.uint8, device=dev)}
    if workspace is None:
        workspace = torch.empty(ws, dtype=torch.uint8, device=dev)
    rc = tahq_encode_scaled(x, dt, T, Cc, tile, h, bits_lo, bits_hi, budget, tokens_per_group,
                            float(tau), float(scale_c), out["codes"], out["scales"], out["zeros"],
                            out["bits"], out["pivots"], workspace, workspace.numel(), stream)
    _check(rc, "tahq_encode_scaled")
    res = dict(out)
    res["codes"] = out["codes"][:pay]
    res["workspace"] = workspace
    res["payload_bytes"] = pay
    return res


def decode_scaled(enc: dict, tokens: int, channels: int, tile: int = 64,
                  hblock: int | None = None, scale_c: float = 1.0, out=None, workspace=None,
                  stream=None):
    """The gradient back from ``encode_scaled``'s dict: RN(decode / scale_c), float32."""
    import torch
    dev = enc["scales"].device
    h = hblock or tile
    ws = tahq_decode_workspace_size(tokens, channels, tile)
    if ws == 0:
        raise TahqError(1, "tahq_decode_workspace_size")
    if out is None:
        out = torch.empty((tokens, channels), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = torch.empty(ws, dtype=torch.uint8, device=dev)
    codes = enc["codes"]
    rc = tahq_decode_scaled(codes, codes.numel(), enc["scales"], enc["zeros"], enc["bits"],
                            enc["pivots"], tokens, channels, tile, h, float(scale_c), out,
                            workspace, workspace.numel(), stream)
    _check(rc, "tahq_decode_scaled")
    return out
