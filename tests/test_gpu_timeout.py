"""Failure detection without a GPU fault: the bounded waits of the staged
kernels.

The convolution of rows of 2M = 8192 points stages its input rows and the
kernel spectrum in shared memory by bulk asynchronous copies, and the layer's
kernel-spectrum step stages its twiddle tables the same way for M <= 1024;
each waits on an mbarrier for a bounded number of polls.  With the library's
wait limit set to 0 (s4_set_wait_limit) every such wait gives up at once,
although the copies themselves complete: the kernel must then record
S4_ERR_TIMEOUT, write its output as zeros, issue no further copies, wait for
the copy in flight with the default limit before it exits, and leave the
library usable -- the next call with the default limit is checked against the
oracle.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle.s4_oracle as O  # noqa: E402
import structured_state_space_gb300 as s4  # noqa: E402
from structured_state_space_gb300 import build as s4build  # noqa: E402
from structured_state_space_gb300 import workloads as W  # noqa: E402

pytestmark = pytest.mark.gpu
TIMEOUT = s4.STATUS_CODE["S4_ERR_TIMEOUT"]


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    s4build.build()
    return s4.load()


def rel_l2(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def _with_zero_wait_limit(fn):
    s4.s4_set_wait_limit(0)
    try:
        return fn()
    finally:
        s4.s4_set_wait_limit(-1)


@pytest.mark.parametrize("batch,H,L", [(4, 3, 4096), (3, 2, 2052)])
def test_staged_convolution_wait_runs_out(batch, H, L):
    # L = 2049..4096 and a multiple of 4: rows of 8192 points, inputs and kernel
    # spectrum both staged (an odd batch leaves the last pair with one row)
    rng = np.random.default_rng(L + H)
    u = rng.standard_normal((batch, H, L)).astype(np.float32)
    Kh = ((rng.standard_normal((H, L)) + 1j * rng.standard_normal((H, L))) * 0.05).astype(np.complex64)
    D = rng.standard_normal(H).astype(np.float32)
    ut, Kt, Dt = torch.from_numpy(u).cuda(), torch.from_numpy(Kh).cuda(), torch.from_numpy(D).cuda()
    ws = s4.workspace(H, 1, 1, L, batch)
    y = torch.full((batch, H, L), complex(1.0, 1.0), dtype=torch.complex64, device="cuda")

    def call():
        s4.s4_conv_fwd(ut, Kt, Dt, y=y, ws=ws)
        return s4.s4_get_status(ws)

    assert _with_zero_wait_limit(call) == TIMEOUT
    assert torch.count_nonzero(y).item() == 0
    # default limit again: a clean call that matches the oracle
    assert call() == 0
    yg = y.cpu().numpy()
    rows = [(0, 0), (batch - 1, H - 1), (batch // 2, H // 2)]
    ref = np.stack([O.causal_conv(Kh[h], u[b, h], D[h]) for b, h in rows])
    assert rel_l2(np.stack([yg[b, h] for b, h in rows]), ref) <= 1e-4


def test_staged_twiddle_tables_wait_runs_out():
    # the layer at M = 1024: the kernel-spectrum step stages its twiddle tables
    w = W.custom(16, 1, 5, 1000, 2, seed=31)
    p = W.make_params(w)
    u = W.make_u(w, p)
    d = {k: torch.from_numpy(np.ascontiguousarray(p[k])).cuda() for k in ["Lambda", "P", "Q", "B", "Ctilde", "dt", "D"]}
    ut = torch.from_numpy(u).cuda()
    ws = s4.workspace(w.H, w.N, w.r, w.L, w.batch)
    K = torch.full((w.H, w.L), complex(1.0, 1.0), dtype=torch.complex64, device="cuda")
    y = torch.full((w.batch, w.H, w.L), complex(1.0, 1.0), dtype=torch.complex64, device="cuda")

    def call():
        s4.s4_layer_fwd(d["Lambda"], d["P"], d["Q"], d["B"], d["Ctilde"], d["dt"], d["D"], ut, K=K, y=y, ws=ws)
        return s4.s4_get_status(ws)

    assert _with_zero_wait_limit(call) == TIMEOUT
    assert torch.count_nonzero(K).item() == 0 and torch.count_nonzero(y).item() == 0
    assert call() == 0
    K_ref = O.s4_kernel_channels(p, w.L, [0, 4])
    assert rel_l2(K.cpu().numpy()[[0, 4]], K_ref) <= 1e-4
    y_ref = O.causal_conv(K_ref[1], u[1, 4], p["D"][4])
    assert rel_l2(y.cpu().numpy()[1, 4], y_ref) <= 1e-4


def test_unstaged_kernels_ignore_the_wait_limit():
    # rows of 2048 points take no staged copies: a zero limit changes nothing
    w = W.custom(8, 1, 3, 1024, 2, seed=32)
    p = W.make_params(w)
    u = W.make_u(w, p)
    Kh = O.s4_kernel_channels(p, w.L).astype(np.complex64)
    ws = s4.workspace(w.H, 1, 1, w.L, w.batch)

    def call():
        y = s4.s4_conv_fwd(torch.from_numpy(u).cuda(), torch.from_numpy(Kh).cuda(),
                           torch.from_numpy(p["D"]).cuda(), ws=ws)
        return s4.s4_get_status(ws), y.cpu().numpy()

    st, y = _with_zero_wait_limit(call)
    assert st == 0
    assert rel_l2(y[1, 2], O.causal_conv(Kh[2], u[1, 2], p["D"][2])) <= 1e-4
