"""s4_conv_fwd_noalloc: the convolution entry point for callers that cannot
allocate device memory (for example a host program that owns all device
memory through its own pool, or a loop where cudaMalloc's possible device
synchronisation is not acceptable).  Its scratch is a fixed array inside the
library, so these tests check that two calls in a row -- different sizes,
the second on a smaller problem than the first -- give the same y as
s4_conv_fwd, and that a problem whose scratch would not fit is refused.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import structured_state_space_gb300 as s4  # noqa: E402
from structured_state_space_gb300 import build as s4build  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    s4build.build()
    lib = s4.load()
    f = lib.s4_conv_fwd_noalloc
    f.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 3 + [ctypes.c_void_p] * 2
    f.restype = ctypes.c_int
    return lib


def _inputs(batch, H, L, seed):
    rng = np.random.default_rng(seed)
    u = torch.from_numpy(rng.standard_normal((batch, H, L)).astype(np.float32)).cuda()
    K = torch.from_numpy((rng.standard_normal((H, L)) * 0.05 + 1j * rng.standard_normal((H, L)) * 0.05)
                         .astype(np.complex64)).cuda()
    D = torch.from_numpy(rng.standard_normal(H).astype(np.float32)).cuda()
    return u, K, D


def _noalloc(lib, u, K, D):
    batch, H, L = u.shape
    y = torch.full((batch, H, L), complex(float("nan"), float("nan")), dtype=torch.complex64, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.s4_conv_fwd_noalloc(ctypes.c_void_p(u.data_ptr()), ctypes.c_void_p(K.data_ptr()),
                                 ctypes.c_void_p(D.data_ptr()), batch, H, L,
                                 ctypes.c_void_p(y.data_ptr()), stream)
    torch.cuda.synchronize()
    return rc, y


def _rel(a, b):
    return float(torch.linalg.vector_norm(a - b) / torch.linalg.vector_norm(b))


def test_two_calls_match_the_workspace_entry_point(lib):
    # first call: the benchmark-sized convolution (H = 256, L = 1024, batch 16)
    u1, K1, D1 = _inputs(16, 256, 1024, seed=1)
    rc, y1 = _noalloc(lib, u1, K1, D1)
    assert rc == 0, s4.s4_status_str(rc)
    ref1 = s4.s4_conv_fwd(u1, K1, D1)
    assert _rel(y1, ref1) <= 1e-4
    # second call right after: other sizes, ragged length, fewer channels; the
    # shared scratch still holds the first call's spectrum
    u2, K2, D2 = _inputs(3, 5, 777, seed=2)
    rc, y2 = _noalloc(lib, u2, K2, D2)
    assert rc == 0, s4.s4_status_str(rc)
    ref2 = s4.s4_conv_fwd(u2, K2, D2)
    assert _rel(y2, ref2) <= 1e-4
    assert torch.isfinite(torch.view_as_real(y2)).all()


@pytest.mark.parametrize("batch,H,L", [
    (3, 64, 4096),    # rows of 8192 points: inputs and kernel spectrum staged by bulk copies
    (2, 5, 3001),     # 8192 points, L not a multiple of 4: inputs read directly
    (2, 16, 16384),   # 32768 points: a cluster of CTAs per pair of rows
])
def test_other_row_paths_match_the_workspace_entry_point(lib, batch, H, L):
    # each fits the fixed scratch (256 + 16 H M bytes <= 8 MiB); two calls in a
    # row, the second on the same inputs, must both match s4_conv_fwd
    u, K, D = _inputs(batch, H, L, seed=L + H)
    ref = s4.s4_conv_fwd(u, K, D)
    for _ in range(2):
        rc, y = _noalloc(lib, u, K, D)
        assert rc == 0, s4.s4_status_str(rc)
        assert _rel(y, ref) <= 1e-4


def test_longest_rows_match_the_oracle(lib):
    # L = 40000: M = 65536, rows of 131072 points over 8-CTA clusters (2 MiB of
    # scratch for H = 2); sampled outputs against the direct causal sums
    import oracle.s4_oracle as O
    u, K, D = _inputs(1, 2, 40000, seed=5)
    rc, y = _noalloc(lib, u, K, D)
    assert rc == 0, s4.s4_status_str(rc)
    un, Kn, Dn, yn = u.cpu().numpy(), K.cpu().numpy(), D.cpu().numpy(), y.cpu().numpy()
    ts = [0, 1, 2, 999, 20000, 39998, 39999]
    for h in range(2):
        ref = O.causal_conv_at(Kn[h], un[0, h], Dn[h], ts)
        got = yn[0, h, ts]
        assert np.linalg.norm(got - ref) <= 1e-4 * np.linalg.norm(ref)
    assert _rel(y, s4.s4_conv_fwd(u, K, D)) <= 1e-4


def test_nonfinite_kernel_gives_zeros(lib):
    # a NaN in one channel's kernel makes a non-finite spectrum: with no status
    # block to read, the caller's signal is an all-zero y (and rc 0)
    u, K, D = _inputs(2, 4, 1024, seed=6)
    K[2, 17] = complex(float("nan"), 0.0)
    rc, y = _noalloc(lib, u, K, D)
    assert rc == 0
    assert torch.count_nonzero(y).item() == 0
    # the next call, on a finite kernel, is clean again
    u2, K2, D2 = _inputs(2, 4, 1024, seed=7)
    rc, y2 = _noalloc(lib, u2, K2, D2)
    assert rc == 0 and _rel(y2, s4.s4_conv_fwd(u2, K2, D2)) <= 1e-4


def test_too_large_is_refused(lib):
    # 256 + 16 * H * M bytes must fit 8 MiB: H = 600, L = 1024 needs ~9.4 MiB
    u, K, D = _inputs(1, 600, 1024, seed=3)
    rc, y = _noalloc(lib, u, K, D)
    assert rc == s4.STATUS_CODE["S4_ERR_WORKSPACE"]
    assert torch.isnan(torch.view_as_real(y)).all()   # nothing was written
