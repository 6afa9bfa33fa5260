"""The C ABI library: it builds for sm_103a, loads, exports every function
include/s4.h declares, and rejects bad arguments on the host before touching
the GPU (these calls never reach CUDA, so they run without a GPU)."""
import ctypes
import os
import re

import pytest

import structured_state_space_gb300 as s4
from structured_state_space_gb300 import build as s4build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "s4.h")


@pytest.fixture(scope="module")
def lib():
    s4build.build()
    return s4.load()


def declared_functions():
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(s4_[a-z0-9_]+)\s*\(", txt)))


def test_header_declares_the_binding_names():
    assert declared_functions() == sorted(s4.ABI_FUNCTIONS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_workspace_bytes(lib):
    # [256 status | H x 1988 far-field constants | H M root values | H 2M spectra
    # | long rows only: 2 x 2M per pair of batch rows], each 256-aligned
    r256 = lambda b: (b + 255) // 256 * 256
    far = lambda H: r256(8 * 1988 * H)
    H, L = 256, 1024
    M = 1024
    assert s4.s4_workspace_bytes(H, 64, 1, L, 16) == 256 + far(H) + 8 * H * M + 16 * H * M
    assert s4.s4_workspace_bytes(3, 4, 1, 100, 1) == 256 + far(3) + 3072 + 6144  # M = 128
    # 2M = 2^15: the four-step scratch, 2 rows of 2M complex per pair (batch 3 -> 2 pairs per channel)
    assert s4.s4_workspace_bytes(2, 4, 1, 16384, 3) == 256 + far(2) + 8 * 2 * 16384 + 16 * 2 * 16384 + 2 * 4 * 32768 * 8
    for bad in [(0, 4, 1, 8, 1), (1, 0, 1, 8, 1), (1, 4, 0, 8, 1), (1, 4, 5, 8, 1), (1, 4, 1, 0, 1),
                (1, 4, 1, 65537, 1), (1, 4, 1, 8, 0), (1, 65537, 1, 8, 1)]:
        assert s4.s4_workspace_bytes(*bad) == 0, bad


def test_status_strings(lib):
    assert s4.s4_status_str(0) == "ok"
    assert s4.s4_status_str(3) == "resonant-diagonal"
    assert s4.s4_status_str(4) == "resonant-correction"
    assert s4.s4_status_str(9) == "timeout"
    assert s4.STATUS[9] == "S4_ERR_TIMEOUT"
    assert s4.s4_status_str(99) == "unknown status"


def _vp(v):
    return ctypes.c_void_p(v)


def test_host_argument_errors(lib):
    A = 0x10000  # aligned stand-in addresses; validation rejects before any use
    ok = [_vp(A)] * 6
    # null output
    assert lib.s4_kernel_gen(*ok, 2, 4, 1, 8, None, _vp(A), 1 << 20, None) == 1
    # null input
    assert lib.s4_kernel_gen(None, *ok[1:], 2, 4, 1, 8, _vp(A), _vp(A), 1 << 20, None) == 1
    # sizes out of range
    assert lib.s4_kernel_gen(*ok, 2, 4, 5, 8, _vp(A), _vp(A), 1 << 20, None) == 1
    assert lib.s4_kernel_gen(*ok, 2, 4, 1, 0, _vp(A), _vp(A), 1 << 20, None) == 1
    assert lib.s4_kernel_gen(*ok, 2, 4, 1, 70000, _vp(A), _vp(A), 1 << 20, None) == 1
    # misaligned kernel output
    assert lib.s4_kernel_gen(*ok, 2, 4, 1, 8, _vp(A + 8), _vp(A), 1 << 20, None) == 1
    # workspace missing / misaligned / too small
    assert lib.s4_kernel_gen(*ok, 2, 4, 1, 8, _vp(A), None, 1 << 20, None) == 2
    assert lib.s4_kernel_gen(*ok, 2, 4, 1, 8, _vp(A), _vp(A + 16), 1 << 20, None) == 2
    assert lib.s4_kernel_gen(*ok, 2, 4, 1, 8, _vp(A), _vp(A), 16, None) == 2
    # convolution
    assert lib.s4_conv_fwd(None, _vp(A), _vp(A), 1, 2, 8, _vp(A), _vp(A), 1 << 20, None) == 1
    assert lib.s4_conv_fwd(_vp(A + 4), _vp(A), _vp(A), 1, 2, 8, _vp(A), _vp(A), 1 << 20, None) == 1
    assert lib.s4_conv_fwd(_vp(A), _vp(A), _vp(A), 0, 2, 8, _vp(A), _vp(A), 1 << 20, None) == 1
    assert lib.s4_conv_fwd(_vp(A), _vp(A), _vp(A), 1, 2, 8, _vp(A), _vp(A), 100, None) == 2
    # layer
    args = [_vp(A)] * 8
    assert lib.s4_layer_fwd(*args, 1, 2, 4, 1, 8, _vp(A), None, _vp(A), 1 << 20, None) == 1
    assert lib.s4_layer_fwd(*args, 1, 2, 4, 1, 8, _vp(A), _vp(A), _vp(A), 10, None) == 2
    # status read without a workspace
    assert lib.s4_get_status(None, None) == 2


def test_host_argument_errors_recurrent_and_ctilde(lib):
    A = 0x10000
    p5 = [_vp(A)] * 5
    assert lib.s4_ctilde(*p5, 2, 4, 1, 8, None, _vp(A), 256, None) == 1           # null output
    assert lib.s4_ctilde(*p5, 2, 300, 1, 8, _vp(A), _vp(A), 256, None) == 1       # N > 256
    assert lib.s4_ctilde(*p5, 2, 4, 1, 8, _vp(A), _vp(A), 64, None) == 2          # ws too small
    p8 = [_vp(A)] * 8
    assert lib.s4_recurrent_fwd(*p8, 1, 2, 4, 1, 8, _vp(A), None, _vp(A), 256, None) == 1
    assert lib.s4_recurrent_fwd(*p8, 1, 2, 4, 5, 8, _vp(A), _vp(A), _vp(A), 256, None) == 1   # r > 4
    assert lib.s4_recurrent_fwd(*p8, 1, 2, 4, 1, 8, _vp(A), _vp(A), None, 256, None) == 2
    assert s4.s4_status_str(8) == "singular-bilinear-matrix"


def test_host_argument_errors_conv_real(lib):
    A = 0x10000
    assert lib.s4_conv_fwd_real(None, _vp(A), _vp(A), 1, 2, 8, _vp(A), _vp(A), 1 << 20, None) == 1
    assert lib.s4_conv_fwd_real(_vp(A), _vp(A), _vp(A), 1, 2, 8, _vp(A + 4), _vp(A), 1 << 20, None) == 1
    assert lib.s4_conv_fwd_real(_vp(A), _vp(A), _vp(A), 1, 2, 8, _vp(A), _vp(A), 100, None) == 2


def test_host_argument_errors_fp32_probe(lib):
    A = 0x10000
    assert lib.s4_fp32_probe(None, 8, 64, None) == 1
    assert lib.s4_fp32_probe(_vp(A), 0, 64, None) == 1
    assert lib.s4_fp32_probe(_vp(A), 8, 0, None) == 1
