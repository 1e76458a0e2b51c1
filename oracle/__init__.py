"""CPU oracle of the TAH-Quant activation codec -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may
import this package.  The product (``pipeline_activation_quantization_gb300``) never
imports it and shares no code with it.

The arithmetic lives in ``tahq_oracle.c``, for the wire format in
``tahq_wire_oracle.c`` and for the fixed-point gradient codec of the backward pass in
``tahq_naive_oracle.c`` (plain scalar C, compiled with gcc
``-O2 -ffp-contract=off``, no fast-math); this module only compiles it, marshals numpy
arrays through ctypes, and can split a tensor into its independent token groups to run
them on several host threads (the per-group results are the same as one sequential call).
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRCS = [os.path.join(_HERE, "tahq_oracle.c"), os.path.join(_HERE, "tahq_wire_oracle.c"),
         os.path.join(_HERE, "tahq_naive_oracle.c")]
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libtahq_oracle.so")
CFLAGS = ["-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-std=c11"]

F32, BF16 = 0, 1
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle shared library (in-tree, under ``oracle/_build``)."""
    os.makedirs(_BUILD, exist_ok=True)
    newest = max(os.path.getmtime(f) for f in _SRCS)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < newest:
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.run(["gcc", *CFLAGS, "-o", tmp, *_SRCS, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = C.CDLL(build())
            p, i64, i32, f32 = C.c_void_p, C.c_int64, C.c_int, C.c_float
            sig = {
                "oracle_log2_tables": (None, [p, p, p]),
                "oracle_lg": (f32, [f32]),
                "oracle_lg_array": (None, [p, p, i64]),
                "oracle_pairwise_sum": (f32, [p, i32]),
                "oracle_entropy_key": (f32, [p, i32]),
                "oracle_entropy_literal": (C.c_double, [p, i32, C.c_double, C.c_double]),
                "oracle_outlier": (None, [p, i32, p, p, p, p]),
                "oracle_outlier_tau": (None, [p, i32, f32, p, p, p, p]),
                "oracle_fwht": (None, [p, i32]),
                "oracle_transform": (None, [p, i32, i32, i32]),
                "oracle_inverse_transform": (None, [p, i32, i32, i32]),
                "oracle_hadamard_dense": (None, [p, p, i32]),
                "oracle_quantize_tile": (None, [p, i32, i32, p, p, p, p]),
                "oracle_pack_tile": (None, [p, i32, i32, p]),
                "oracle_unpack_tile": (None, [p, i32, i32, p]),
                "oracle_hi_count": (i64, [i64, i32, i32, f32]),
                "oracle_allocate": (i32, [p, i64, i64, i32, i32, p]),
                "oracle_payload_size": (i64, [i64, i64, i32, i32, i32, f32, i64]),
                "oracle_encode": (i32, [p, i32, i64, i64, i32, i32, i32, i32, f32, i64,
                                        p, p, p, p, p, p, p]),
                "oracle_encode_tau": (i32, [p, i32, i64, i64, i32, i32, i32, i32, f32, i64, f32,
                                            p, p, p, p, p, p, p]),
                "oracle_encode_alloc": (i32, [p, i32, i64, i64, i32, i32, i32, i32, f32, i64, f32,
                                              i32, p, p, p, p, p, p, p]),
                "oracle_entropy_key_n": (f32, [p, i64]),
                "oracle_payload_size_alloc": (i64, [i64, i64, i32, i32, i32, i32, f32, i64]),
                "oracle_decode": (i32, [p, i64, p, p, p, p, i64, i64, i32, i32, p]),
                "oracle_f16_value": (C.c_double, [C.c_uint16]),
                "oracle_f16_round_down": (C.c_uint16, [f32]),
                "oracle_f16_scale_up": (C.c_uint16, [f32, f32, i32]),
                "oracle_quantize_tile_f16": (None, [p, i32, i32, p, p, p, p]),
                "oracle_wire_layout": (i64, [i64, i64, i32, i32, i32, f32, i64, p]),
                "oracle_encode_wire": (i32, [p, i32, i64, i64, i32, i32, i32, i32, f32, i64, f32,
                                             p, i64, p]),
                "oracle_wire_header": (i32, [p, i64, p]),
                "oracle_decode_wire": (i32, [p, i64, p]),
                "oracle_naive_codes_bytes": (C.c_size_t, [i64, i64, i32, i32]),
                "oracle_naive_encode": (i32, [p, i64, i64, i32, i32, f32, p, p, p, p]),
                "oracle_naive_decode": (i32, [p, p, p, i64, i64, i32, i32, f32, p]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32)


# ----------------------------------------------------------------------------- scalars

def log2_tables():
    T = np.zeros(128, np.float32); R = np.zeros(128, np.float32); k = np.zeros(3, np.float32)
    lib().oracle_log2_tables(_ptr(T), _ptr(R), _ptr(k))
    return T, R, k


def lg(x) -> np.ndarray:
    x = _f32(x)
    out = np.empty_like(x)
    lib().oracle_lg_array(_ptr(x), _ptr(out), x.size)
    return out


def pairwise_sum(x) -> float:
    x = _f32(x)
    return float(lib().oracle_pairwise_sum(_ptr(x), x.size))


def entropy_key(a) -> float:
    a = _f32(a)
    return float(lib().oracle_entropy_key(_ptr(a), a.size))


def entropy_literal(a, eps: float = 1e-12, vsig: float = 1e-12) -> float:
    a = _f32(a)
    return float(lib().oracle_entropy_literal(_ptr(a), a.size, eps, vsig))


def outlier(a, tau: float | None = None):
    """-> (pivot, flag, m1, m2) of one tile; flag = r > tau (the method's 2.0 by default)."""
    a = _f32(a)
    d, f = C.c_int(), C.c_int()
    m1, m2 = C.c_float(), C.c_float()
    if tau is None:
        lib().oracle_outlier(_ptr(a), a.size, C.byref(d), C.byref(f), C.byref(m1), C.byref(m2))
    else:
        lib().oracle_outlier_tau(_ptr(a), a.size, float(tau), C.byref(d), C.byref(f),
                                 C.byref(m1), C.byref(m2))
    return d.value, f.value, m1.value, m2.value


def fwht(v) -> np.ndarray:
    v = _f32(v).copy()
    lib().oracle_fwht(_ptr(v), v.size)
    return v


def transform(v, h: int, d: int) -> np.ndarray:
    v = _f32(v).copy()
    lib().oracle_transform(_ptr(v), v.size, h, d)
    return v


def inverse_transform(v, h: int, d: int) -> np.ndarray:
    v = _f32(v).copy()
    lib().oracle_inverse_transform(_ptr(v), v.size, h, d)
    return v


def hadamard_dense(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty_like(x)
    lib().oracle_hadamard_dense(_ptr(x), _ptr(y), x.size)
    return y


def quantize_tile(v, b: int):
    """-> (codes u8[G], scale, zero, near u8[G])."""
    v = _f32(v)
    q = np.zeros(v.size, np.uint8); near = np.zeros(v.size, np.uint8)
    s, z = C.c_float(), C.c_float()
    lib().oracle_quantize_tile(_ptr(v), v.size, b, _ptr(q), C.byref(s), C.byref(z), _ptr(near))
    return q, s.value, z.value, near


def pack_tile(q, b: int) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.uint8)
    slot = np.zeros(q.size * b // 8, np.uint8)
    lib().oracle_pack_tile(_ptr(q), q.size, b, _ptr(slot))
    return slot


def unpack_tile(slot, G: int, b: int) -> np.ndarray:
    slot = np.ascontiguousarray(slot, dtype=np.uint8)
    q = np.zeros(G, np.uint8)
    lib().oracle_unpack_tile(_ptr(slot), G, b, _ptr(q))
    return q


def hi_count(n_g: int, lo: int, hi: int, budget: float) -> int:
    return int(lib().oracle_hi_count(n_g, lo, hi, budget))


def allocate(H, K: int, lo: int, hi: int) -> np.ndarray:
    H = _f32(H)
    bits = np.zeros(H.size, np.uint8)
    rc = lib().oracle_allocate(_ptr(H), H.size, K, lo, hi, _ptr(bits))
    assert rc == 0
    return bits


def payload_size(T, Cc, G, lo, hi, budget, S, alloc_tile: int | None = None) -> int:
    if alloc_tile is None:
        return int(lib().oracle_payload_size(T, Cc, G, lo, hi, budget, S))
    return int(lib().oracle_payload_size_alloc(T, Cc, G, alloc_tile, lo, hi, budget, S))


def entropy_key_n(a) -> float:
    """Entropy key over any power-of-two number of values (an allocation tile)."""
    a = _f32(a)
    return float(lib().oracle_entropy_key_n(_ptr(a), a.size))


# ------------------------------------------------------------------------ whole tensor

def encode(x: np.ndarray, G: int, h: int, lo: int, hi: int, budget: float, S: int = 0,
           threads: int = 1, want_keys: bool = False, want_near: bool = False,
           tau: float | None = None, alloc_tile: int | None = None) -> dict:
    """Encode ``x`` ([T, C] float32, or uint16 bf16 bit patterns).

    Returns a dict with ``codes, scales, zeros, bits, pivots`` (and ``keys`` [n_tiles]
    float32 entropy keys, ``near`` [T, C] boundary flags when asked).  With
    ``threads > 1`` the independent token groups run on host threads.  ``tau`` is the
    outlier threshold (None: the method's 2.0); ``alloc_tile`` the allocation tile A
    (None: A = G), with one key per allocation tile (``keys`` then has n / (A / G)).
    """
    x = np.ascontiguousarray(x)
    dtype = BF16 if x.dtype == np.uint16 else F32
    if dtype == F32:
        x = _f32(x)
    T, Cc = x.shape
    S = S or T
    n = T * (Cc // G)
    A = alloc_tile or G
    total = payload_size(T, Cc, G, lo, hi, budget, S, None if A == G else A)
    if total < 0:
        raise ValueError("invalid codec arguments")
    out = {
        "codes": np.zeros(total, np.uint8),
        "scales": np.zeros(n, np.float32),
        "zeros": np.zeros(n, np.float32),
        "bits": np.zeros(n, np.uint8),
        "pivots": np.zeros(n, np.uint8),
    }
    if want_keys:
        out["keys"] = np.zeros(n // (A // G), np.float32)
    if want_near:
        out["near"] = np.zeros((T, Cc), np.uint8)
    if T == 0:
        return out
    ng = T // S
    n_g = S * (Cc // G)
    gbytes = total // ng

    na_g = n_g // (A // G)

    def run(g):
        sl = slice(g * n_g, (g + 1) * n_g)
        ka = slice(g * na_g, (g + 1) * na_g)
        args = (_ptr(x[g * S:(g + 1) * S]), dtype, S, Cc, G, h, lo, hi, budget, S)
        if A != G:
            fn, args = lib().oracle_encode_alloc, args + (2.0 if tau is None else float(tau), A)
        elif tau is not None:
            fn, args = lib().oracle_encode_tau, args + (float(tau),)
        else:
            fn = lib().oracle_encode
        rc = fn(
            *args,
            _ptr(out["codes"][g * gbytes:(g + 1) * gbytes]), _ptr(out["scales"][sl]),
            _ptr(out["zeros"][sl]), _ptr(out["bits"][sl]), _ptr(out["pivots"][sl]),
            _ptr(out["keys"][ka]) if want_keys else None,
            _ptr(out["near"][g * S:(g + 1) * S]) if want_near else None)
        if rc != 0:
            raise RuntimeError(f"oracle_encode failed on group {g}")

    _run_all(run, ng, threads)
    return out


def decode(codes, scales, zeros, bits, pivots, T: int, Cc: int, G: int, h: int,
           threads: int = 1) -> np.ndarray:
    """Decode to float32 [T, C].  With ``threads > 1`` token ranges run on host threads."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales, zeros = _f32(scales), _f32(zeros)
    bits = np.ascontiguousarray(bits, dtype=np.uint8)
    pivots = np.ascontiguousarray(pivots, dtype=np.uint8)
    out = np.zeros((T, Cc), np.float32)
    if T == 0:
        return out
    W = Cc // G
    parts = max(1, min(threads, T))
    bounds = [T * i // parts for i in range(parts + 1)]
    slot_bytes = bits.astype(np.int64) * G // 8
    start = np.concatenate([[0], np.cumsum(slot_bytes)])

    def run(i):
        t0, t1 = bounds[i], bounds[i + 1]
        if t1 == t0:
            return
        o0 = int(start[t0 * W])
        rc = lib().oracle_decode(_ptr(codes[o0:]), codes.size - o0, _ptr(scales[t0 * W:]),
                                 _ptr(zeros[t0 * W:]), _ptr(bits[t0 * W:]), _ptr(pivots[t0 * W:]),
                                 t1 - t0, Cc, G, h, _ptr(out[t0:t1]))
        if rc != 0:
            raise RuntimeError("oracle_decode rejected its input")

    _run_all(run, parts, threads)
    return out


def _run_all(fn, count: int, threads: int):
    if threads <= 1 or count <= 1:
        for i in range(count):
            fn(i)
        return
    with ThreadPoolExecutor(max_workers=min(threads, count)) as ex:
        list(ex.map(fn, range(count)))


# ------------------------------------------------------------------------ wire format

def f16_value(h: int) -> float:
    return float(lib().oracle_f16_value(int(h)))


def f16_round_down(x: float) -> int:
    return int(lib().oracle_f16_round_down(float(x)))


def f16_scale_up(zero: float, mx: float, Q: int) -> int:
    return int(lib().oracle_f16_scale_up(float(zero), float(mx), int(Q)))


def quantize_tile_f16(v, b: int):
    """-> (codes u8[G], scale16, zero16, near u8[G]) of the wire format's quantiser."""
    v = _f32(v)
    q = np.zeros(v.size, np.uint8); near = np.zeros(v.size, np.uint8)
    s, z = C.c_uint16(), C.c_uint16()
    lib().oracle_quantize_tile_f16(_ptr(v), v.size, b, _ptr(q), C.byref(s), C.byref(z), _ptr(near))
    return q, s.value, z.value, near


def wire_layout(T, Cc, G, lo, hi, budget, S=0):
    """-> (total bytes, [map, meta, pivots, payload offsets], payload bytes)."""
    off = np.zeros(5, np.int64)
    total = int(lib().oracle_wire_layout(T, Cc, G, lo, hi, budget, S, _ptr(off)))
    return total, [int(v) for v in off[:4]], int(off[4])


def encode_wire(x: np.ndarray, G: int, h: int, lo: int, hi: int, budget: float, S: int = 0,
                tau: float = 2.0, want_near: bool = False):
    """The whole tensor as one wire buffer (uint8); with ``want_near`` also the [T, C]
    rounding-boundary flags of its codes."""
    x = np.ascontiguousarray(x)
    dtype = BF16 if x.dtype == np.uint16 else F32
    if dtype == F32:
        x = _f32(x)
    T, Cc = x.shape
    total, _, _ = wire_layout(T, Cc, G, lo, hi, budget, S)
    if total < 0:
        raise ValueError("invalid codec arguments")
    out = np.zeros(total, np.uint8)
    near = np.zeros((T, Cc), np.uint8) if want_near else None
    rc = lib().oracle_encode_wire(_ptr(x), dtype, T, Cc, G, h, lo, hi, budget, S, float(tau),
                                  _ptr(out), total, _ptr(near))
    if rc != 0:
        raise RuntimeError("oracle_encode_wire failed")
    return (out, near) if want_near else out


def wire_header(wire: np.ndarray) -> dict:
    wire = np.ascontiguousarray(wire, dtype=np.uint8)
    f = np.zeros(15, np.int64)
    if lib().oracle_wire_header(_ptr(wire), wire.size, _ptr(f)) != 0:
        raise ValueError("not a wire buffer")
    keys = ["tokens", "channels", "tokens_per_group", "tile", "hblock", "bits_lo", "bits_hi",
            "pivot_bits", "tiles", "off_map", "off_meta", "off_pivots", "off_payload",
            "payload_bytes", "total_bytes"]
    return {k: int(v) for k, v in zip(keys, f)}


def decode_wire(wire: np.ndarray) -> np.ndarray:
    wire = np.ascontiguousarray(wire, dtype=np.uint8)
    hd = wire_header(wire)
    out = np.zeros((hd["tokens"], hd["channels"]), np.float32)
    if lib().oracle_decode_wire(_ptr(wire), wire.size, _ptr(out)) != 0:
        raise RuntimeError("oracle_decode_wire rejected its input")
    return out


# ------------------------------------------------------------------ backward gradients

def naive_codes_bytes(T: int, Cc: int, G: int, b: int) -> int:
    """Bytes of the packed b-bit codes of a [T, Cc] tensor in tiles of G (0: invalid)."""
    return int(lib().oracle_naive_codes_bytes(T, Cc, G, b))


def naive_encode(g: np.ndarray, G: int, b: int, c: float = 1.0, want_near: bool = False):
    """Q_Naive of an fp32 [T, C] gradient at b bits in tiles of G, after scaling by the
    power of two c: (codes uint8, scales [T * C / G], zeros[, near [T, C]])."""
    g = _f32(np.ascontiguousarray(g))
    T, Cc = g.shape
    nb = naive_codes_bytes(T, Cc, G, b)
    if nb == 0 and T * Cc > 0:
        raise ValueError("invalid codec arguments")
    n = T * (Cc // G)
    codes = np.zeros(nb, np.uint8)
    scales = np.zeros(n, np.float32)
    zeros = np.zeros(n, np.float32)
    near = np.zeros((T, Cc), np.uint8) if want_near else None
    if lib().oracle_naive_encode(_ptr(g), T, Cc, G, b, float(c), _ptr(codes), _ptr(scales),
                                 _ptr(zeros), _ptr(near)) != 0:
        raise ValueError("invalid codec arguments")
    return (codes, scales, zeros, near) if want_near else (codes, scales, zeros)


def naive_decode(codes, scales, zeros, T: int, Cc: int, G: int, b: int,
                 c: float = 1.0) -> np.ndarray:
    """The fp32 [T, C] gradient back from Q_Naive's codes, divided by c."""
    out = np.zeros((T, Cc), np.float32)
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales, zeros = _f32(scales), _f32(zeros)
    if lib().oracle_naive_decode(_ptr(codes), _ptr(scales), _ptr(zeros), T, Cc, G, b,
                                 float(c), _ptr(out)) != 0:
        raise ValueError("invalid codec arguments")
    return out


# ------------------------------------------------------------------ TAH-Quant on gradients

def _power_of_two(c: float) -> bool:
    m, _ = np.frexp(np.float32(c))
    return bool(np.isfinite(c) and c > 0 and m == 0.5)


def scale_input(x: np.ndarray, c: float) -> np.ndarray:
    """RN(c x) for a power of two c (exact unless c x leaves the normal range), in x's own
    type: float32, or uint16 bf16 bit patterns (bf16 x 2^k is again a bf16 value)."""
    if not _power_of_two(c):
        raise ValueError("the gradient scale must be a positive finite power of two")
    x = np.ascontiguousarray(x)
    if x.dtype == np.uint16:
        f = (x.astype(np.uint32) << np.uint32(16)).view(np.float32) * np.float32(c)
        b = f.view(np.uint32)
        return ((b + ((b >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)) >> np.uint32(16)).astype(np.uint16)
    return _f32(x) * np.float32(c)


def encode_scaled(x: np.ndarray, G: int, h: int, lo: int, hi: int, budget: float, S: int = 0,
                  c: float = 1.0, tau: float | None = None, threads: int = 1,
                  want_keys: bool = False) -> dict:
    """TAH-Quant applied to a gradient with the scaling of Appendix H eq. (24): the
    activation codec on RN(c g), c a power of two (scales and zeros describe c g)."""
    return encode(scale_input(x, c), G, h, lo, hi, budget, S, threads=threads, tau=tau,
                  want_keys=want_keys)


def decode_scaled(codes, scales, zeros, bits, pivots, T: int, Cc: int, G: int, h: int,
                  c: float = 1.0, threads: int = 1) -> np.ndarray:
    """The gradient back: RN(decode / c), float32 [T, C] (eq. (24): Q(c g) / c)."""
    if not _power_of_two(c):
        raise ValueError("the gradient scale must be a positive finite power of two")
    return decode(codes, scales, zeros, bits, pivots, T, Cc, G, h, threads=threads) / np.float32(c)
