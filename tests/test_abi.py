"""Host-side checks of the C ABI that need no GPU: the library loads, exports every
function include/tahq.h declares, and its size/validation logic agrees with the oracle.
No call here launches a kernel (each invalid call is rejected before any CUDA call)."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import pipeline_activation_quantization_gb300 as tq

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "tahq.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tahq_\w+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    L = tq.lib()
    names = _declared_functions()
    assert len(names) >= 10
    for name in names:
        assert hasattr(L, name), name
    assert sorted(tq.EXPORTED_SYMBOLS) == names


def test_version_and_status_strings():
    assert tq.tahq_version() >= 10000
    for s in range(6):
        assert tq.tahq_status_string(s).startswith(tq.STATUS_NAMES[s])
    assert "unknown" in tq.tahq_status_string(99)


def test_log2_tables_match_oracle():
    a = tq.tahq_log2_tables()
    b = oracle.log2_tables()
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


SHAPES = [
    (256, 1024, 64, 3, 4, 3.5, 0), (4096, 2048, 64, 3, 4, 3.5, 1024),
    (16384, 4096, 64, 3, 4, 3.0, 2048), (16384, 4096, 32, 3, 4, 3.5, 2048),
    (16384, 4096, 128, 3, 4, 4.0, 2048), (32768, 8192, 128, 3, 4, 3.5, 2048),
    (7, 24, 8, 2, 5, 3.3, 7), (0, 64, 64, 3, 4, 3.5, 0), (12, 256, 16, 1, 8, 4.25, 4),
]


@pytest.mark.parametrize("T,C,G,lo,hi,beta,S", SHAPES)
def test_sizes_agree_with_oracle(T, C, G, lo, hi, beta, S):
    pay = tq.tahq_payload_size(T, C, G, lo, hi, beta, S)
    assert pay == max(0, oracle.payload_size(T, C, G, lo, hi, beta, S))
    n_g = (S or T) * (C // G)
    if T:
        assert tq.tahq_hi_count(T, C, G, lo, hi, beta, S) == oracle.hi_count(n_g, lo, hi, beta)
    ws = tq.tahq_workspace_size(T, C, G, G, lo, hi, beta, S)
    assert ws > 0 and ws % 256 == 0
    assert tq.tahq_decode_workspace_size(T, C, G) > 0


@pytest.mark.parametrize("args", [
    (16, 100, 64, 64, 3, 4, 3.5, 0),    # channels not a multiple of tile
    (16, 128, 4, 4, 3, 4, 3.5, 0),      # tile too small
    (16, 256, 256, 256, 3, 4, 3.5, 0),  # tile too large
    (16, 128, 64, 3, 3, 4, 3.5, 0),     # hblock not a power of two
    (16, 128, 64, 128, 3, 4, 3.5, 0),   # hblock above tile
    (16, 128, 64, 64, 4, 4, 4.0, 0),    # lo == hi
    (16, 128, 64, 64, 3, 9, 4.0, 0),    # hi above 8
    (16, 128, 64, 64, 3, 4, 4.5, 0),    # budget above hi
    (16, 128, 64, 64, 3, 4, float("nan"), 0),
    (16, 128, 64, 64, 3, 4, 3.5, 5),    # group does not divide tokens
    (-1, 128, 64, 64, 3, 4, 3.5, 0),
])
def test_invalid_arguments(args):
    assert tq.tahq_workspace_size(*args) == 0
    T, C, G, h, lo, hi, beta, S = args
    fake = 1 << 20   # aligned non-null stand-ins: rejected before any dereference
    rc = tq.tahq_encode(fake, tq.TAHQ_F32, T, C, G, h, lo, hi, beta, S, fake, fake, fake, fake,
                        fake, fake, 1 << 30, 0)
    assert rc == 1


@pytest.mark.parametrize("tau", [-1.0, -0.0 - 1e-30, float("nan"), float("-inf")])
def test_encode_ex_rejects_bad_tau(tau):
    fake = 1 << 20   # rejected before any dereference or launch
    rc = tq.tahq_encode_ex(fake, tq.TAHQ_F32, 16, 128, 64, 64, 3, 4, 3.5, 0, tau, 0, fake, fake, fake,
                           fake, fake, fake, 1 << 30, 0)
    assert rc == 1


def test_unsupported_tile_and_workspace_errors():
    fake = 1 << 20
    # tile 96 is valid for the method but not built (not a power of two)
    rc = tq.tahq_encode(fake, tq.TAHQ_F32, 4, 192, 96, 32, 3, 4, 3.5, 0, fake, fake, fake, fake,
                        fake, fake, 1 << 30, 0)
    assert rc == 2
    need = tq.tahq_workspace_size(16, 128, 64, 64, 3, 4, 3.5, 0)
    rc = tq.tahq_encode(fake, tq.TAHQ_BF16, 16, 128, 64, 64, 3, 4, 3.5, 0, fake, fake, fake, fake,
                        fake, fake, need - 1, 0)
    assert rc == 3
    rc = tq.tahq_encode(fake, tq.TAHQ_BF16, 16, 128, 64, 64, 3, 4, 3.5, 0, fake, fake, fake, fake,
                        fake, fake + 8, need, 0)            # misaligned workspace
    assert rc == 3
    rc = tq.tahq_encode(fake + 4, tq.TAHQ_BF16, 16, 128, 64, 64, 3, 4, 3.5, 0, fake, fake, fake,
                        fake, fake, fake, need, 0)          # misaligned input
    assert rc == 1
    rc = tq.tahq_encode(fake, 7, 16, 128, 64, 64, 3, 4, 3.5, 0, fake, fake, fake, fake,
                        fake, fake, need, 0)                # unknown dtype
    assert rc == 1
    dneed = tq.tahq_decode_workspace_size(16, 128, 64)
    rc = tq.tahq_decode(fake, 100, fake, fake, fake, fake, 16, 128, 64, 64, fake, fake, dneed - 1, 0)
    assert rc == 3
    rc = tq.tahq_decode(fake, 100, fake, fake, fake, fake, 16, 128, 64, 5, fake, fake, dneed, 0)
    assert rc == 1
    assert tq.lib().tahq_get_device_status(None, None, None) == 3


def test_lib_is_in_tree():
    path = tq._build.LIB
    assert os.path.exists(path)
    assert os.path.dirname(os.path.dirname(path)) == os.path.dirname(tq.__file__)
    assert ctypes.CDLL(path) is not None


@pytest.mark.parametrize("T,C,G,lo,hi,beta,S", [(16, 256, 64, 3, 4, 3.8, 0), (48, 512, 128, 3, 4, 3.5, 16),
                                                (33, 400, 16, 3, 5, 4.0, 11), (0, 256, 64, 3, 4, 3.5, 0),
                                                (7, 64, 8, 1, 8, 4.4, 7)])
def test_wire_size_agrees_with_oracle(T, C, G, lo, hi, beta, S):
    assert tq.tahq_wire_size(T, C, G, lo, hi, beta, S) == oracle.wire_layout(T, C, G, lo, hi, beta, S)[0]
    assert tq.tahq_wire_workspace_size(T, C, G, G, lo, hi, beta, S) >= tq.tahq_workspace_size(
        T, C, G, G, lo, hi, beta, S)
    assert tq.tahq_wire_decode_workspace_size(T, C, G) >= tq.tahq_decode_workspace_size(T, C, G)


def test_wire_entry_points_reject_bad_buffers():
    fake = 1 << 20
    size = tq.tahq_wire_size(16, 128, 64, 3, 4, 3.5, 0)
    # short, misaligned or missing buffers, bad tau: rejected before any launch
    assert tq.tahq_encode_wire(fake, tq.TAHQ_F32, 16, 128, 64, 64, 3, 4, 3.5, 0, 2.0, fake,
                               size - 1, fake, 1 << 30, 0) == 1
    assert tq.tahq_encode_wire(fake, tq.TAHQ_F32, 16, 128, 64, 64, 3, 4, 3.5, 0, 2.0, fake + 8,
                               size, fake, 1 << 30, 0) == 1
    assert tq.tahq_encode_wire(fake, tq.TAHQ_F32, 16, 128, 64, 64, 3, 4, 3.5, 0, -1.0, fake,
                               size, fake, 1 << 30, 0) == 1
    assert tq.tahq_decode_wire(0, size, 16, 128, 64, 64, 3, 4, 3.5, 0, fake, fake, 1 << 30, 0) == 1
    assert tq.tahq_decode_wire(fake, size - 16, 16, 128, 64, 64, 3, 4, 3.5, 0, fake, fake,
                               1 << 30, 0) == 1
    assert tq.tahq_encode_wire(fake, tq.TAHQ_F32, 16, 128, 64, 64, 3, 4, 3.5, 0, 2.0, fake, size,
                               fake, 16, 0) == 3      # workspace too small


@pytest.mark.parametrize("T,C,G,A,lo,hi,beta,S", [(16, 512, 64, 128, 3, 4, 3.5, 8),
                                                  (48, 512, 64, 512, 3, 4, 3.5, 0),
                                                  (32, 8192, 128, 8192, 3, 4, 3.5, 16),
                                                  (20, 256, 16, 64, 2, 3, 2.2, 10)])
def test_payload_size_ex_agrees_with_oracle(T, C, G, A, lo, hi, beta, S):
    assert tq.tahq_payload_size_ex(T, C, G, A, lo, hi, beta, S) == \
        oracle.payload_size(T, C, G, lo, hi, beta, S, A)
    assert tq.tahq_payload_size_ex(T, C, G, 0, lo, hi, beta, S) == \
        tq.tahq_payload_size(T, C, G, lo, hi, beta, S)


def test_alloc_tile_argument_errors():
    fake = 1 << 20
    for A in (32, 96, 192, 1024, -64):     # below tile, not a multiple, not 2^k tiles, above C
        assert tq.tahq_payload_size_ex(16, 512, 64, A, 3, 4, 3.5, 0) == 0
        rc = tq.tahq_encode_ex(fake, tq.TAHQ_F32, 16, 512, 64, 64, 3, 4, 3.5, 0, 2.0, A, fake,
                               fake, fake, fake, fake, fake, 1 << 30, 0)
        assert rc == 1
    # an fp32 allocation tile above 32 KB is valid for the method but not built
    rc = tq.tahq_encode_ex(fake, tq.TAHQ_F32, 4, 16384, 64, 64, 3, 4, 3.5, 0, 2.0, 16384, fake,
                           fake, fake, fake, fake, fake, 1 << 30, 0)
    assert rc == 2


def test_naive_codec_sizes_and_argument_errors():
    # the backward pass's gradient codec: sizes, and every host-side rejection before any
    # device call
    assert tq.tahq_naive_codes_bytes(8, 256, 64, 8) == 8 * 256
    assert tq.tahq_naive_codes_bytes(8, 256, 32, 10) == 8 * 256 * 10 // 8
    assert tq.tahq_naive_codes_bytes(8, 256, 16, 8) == 0      # tile not built
    assert tq.tahq_naive_codes_bytes(8, 250, 64, 8) == 0      # channels not whole tiles
    assert tq.tahq_naive_codes_bytes(8, 256, 64, 17) == 0     # width beyond 16
    L = tq.lib()
    assert L.tahq_naive_encode(None, 4, 256, 64, 8, 3.0, None, None, None, None) == 1
    assert L.tahq_naive_encode(None, 4, 256, 64, 0, 1.0, None, None, None, None) == 1
    assert L.tahq_naive_encode(None, 4, 256, 16, 8, 1.0, None, None, None, None) == 2
    assert L.tahq_naive_encode(None, 4, 256, 64, 8, 1.0, None, None, None, None) == 1
    assert L.tahq_naive_encode(None, 0, 256, 64, 8, 1.0, None, None, None, None) == 0
    assert L.tahq_naive_decode(None, None, None, 4, 256, 64, 8, 0.0, None, None) == 1
    assert L.tahq_naive_decode(None, None, None, 0, 256, 64, 8, 1.0, None, None) == 0
