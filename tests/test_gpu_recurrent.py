"""Recurrent mode and C~ formation on the GPU vs the float64 oracle, and the
recurrent mode against the convolution path (two GPU paths that must agree)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle.s4_oracle as O  # noqa: E402
import structured_state_space_gb300 as s4  # noqa: E402
from structured_state_space_gb300 import build as s4build  # noqa: E402
from structured_state_space_gb300 import workloads as W  # noqa: E402

pytestmark = pytest.mark.gpu
REL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    s4build.build()
    return s4.load()


def rel_l2(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def _dev(p, keys):
    return {k: torch.from_numpy(np.ascontiguousarray(p[k])).cuda() for k in keys}


def _with_c(w, seed):
    """Workload parameters plus a conventional output vector C (drawn like C~)."""
    p = W.make_params(w)
    rng = np.random.default_rng(seed)
    C = (rng.standard_normal((w.H, w.N)) + 1j * rng.standard_normal((w.H, w.N))) / np.sqrt(2.0)
    p["C"] = C.astype(np.complex64)
    return p


# look-ahead of 16, 8, 4, 2 steps per reduction pass; (16, 4, ...) at rank 4;
# (8, 1, 2, 3) has M = 4, below its look-ahead, and takes single steps
@pytest.mark.parametrize("N,r,H,L", [(4, 1, 3, 64), (64, 1, 8, 1024), (64, 2, 4, 300), (256, 1, 3, 4096),
                                     (33, 3, 2, 100), (16, 4, 2, 200), (8, 1, 2, 3), (128, 2, 2, 64)])
def test_ctilde_matches_oracle(N, r, H, L):
    w = W.custom(N, r, H, L, 1, seed=7 * N + L)
    p = _with_c(w, 11)
    d = _dev(p, ["Lambda", "P", "Q", "dt", "C"])
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    Ct = s4.s4_ctilde(d["Lambda"], d["P"], d["Q"], d["dt"], d["C"], L, ws=ws).cpu().numpy()
    assert s4.s4_get_status(ws) == 0
    M = O.transform_length(L)
    ref = np.array([O.ctilde_from_c(O.bilinear(p["Lambda"][h], p["P"][h], p["Q"][h], p["B"][h], p["dt"][h])[1],
                                    p["C"][h], M) for h in range(H)])
    assert rel_l2(Ct, ref) <= REL, rel_l2(Ct, ref)


def test_kernel_from_c_through_ctilde():
    # C -> C~ (GPU) -> K (GPU filter) equals the definition K_j = C^* Abar^j Bbar.
    w = W.WORKLOADS[1]
    p = _with_c(w, 12)
    d = _dev(p, ["Lambda", "P", "Q", "B", "dt", "C"])
    Ct = s4.s4_ctilde(d["Lambda"], d["P"], d["Q"], d["dt"], d["C"], w.L)
    K = s4.s4_kernel_gen(d["Lambda"], d["P"], d["Q"], d["B"], Ct, d["dt"], w.L).cpu().numpy()
    chans = [0, 5, 100, 255]
    ref = []
    for h in chans:
        _, Ab, Bb = O.bilinear(p["Lambda"][h], p["P"][h], p["Q"][h], p["B"][h], p["dt"][h])
        ref.append(O.kernel_from_c(Ab, Bb, p["C"][h], w.L))
    assert rel_l2(K[chans], np.array(ref)) <= REL


@pytest.mark.parametrize("N,r,H,L,batch", [(4, 1, 2, 64, 1), (64, 1, 6, 1024, 2), (64, 2, 3, 500, 3), (200, 1, 2, 256, 2),
                                           (16, 4, 2, 128, 1), (33, 1, 5, 77, 1)])
def test_recurrent_matches_oracle_and_carries_state(N, r, H, L, batch):
    w = W.custom(N, r, H, L, batch, seed=3 * N + L)
    p = _with_c(w, 13)
    u = W.make_u(w, p)
    d = _dev(p, ["Lambda", "P", "Q", "B", "C", "dt", "D"])
    ut = torch.from_numpy(u).cuda()
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    # two calls: the state of the first continues into the second
    cut = L // 3
    x = torch.zeros((batch, H, N), dtype=torch.complex64, device="cuda")
    y1, x = s4.s4_recurrent_fwd(d["Lambda"], d["P"], d["Q"], d["B"], d["C"], d["dt"], d["D"],
                                ut[:, :, :cut].contiguous(), x=x, ws=ws)
    y2, x = s4.s4_recurrent_fwd(d["Lambda"], d["P"], d["Q"], d["B"], d["C"], d["dt"], d["D"],
                                ut[:, :, cut:].contiguous(), x=x, ws=ws)
    assert s4.s4_get_status(ws) == 0
    y = torch.cat([y1, y2], dim=2).cpu().numpy()
    ref = np.empty((batch, H, L), complex)
    for h in range(H):
        _, Ab, Bb = O.bilinear(p["Lambda"][h], p["P"][h], p["Q"][h], p["B"][h], p["dt"][h])
        for b in range(batch):
            ref[b, h] = O.recurrence(Ab, Bb, p["C"][h], p["D"][h], u[b, h])
    assert rel_l2(y, ref) <= REL, rel_l2(y, ref)


def test_recurrent_equals_convolution_path():
    # The two GPU paths: recurrence with C, and the filter + FFT convolution with C~ = (I - Abar^M)^* C.
    w = W.custom(64, 1, 16, 1024, 2, seed=99)
    p = _with_c(w, 14)
    u = W.make_u(w, p)
    d = _dev(p, ["Lambda", "P", "Q", "B", "C", "dt", "D"])
    ut = torch.from_numpy(u).cuda()
    y_rec, _ = s4.s4_recurrent_fwd(d["Lambda"], d["P"], d["Q"], d["B"], d["C"], d["dt"], d["D"], ut)
    Ct = s4.s4_ctilde(d["Lambda"], d["P"], d["Q"], d["dt"], d["C"], w.L)
    _, y_conv = s4.s4_layer_fwd(d["Lambda"], d["P"], d["Q"], d["B"], Ct, d["dt"], d["D"], ut)
    assert rel_l2(y_conv.cpu().numpy(), y_rec.cpu().numpy()) <= 2 * REL


def test_singular_bilinear_status():
    # lambda_0 = 2/Delta with Delta = 1/4: d_0 = 1 - (Delta/2) lambda_0 = 0 exactly.
    c = lambda v: torch.tensor(v, dtype=torch.complex64, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    lam = c([[8.0, -0.5 + 1j]])
    P = c([[[0.1], [0.2]]])
    dt = torch.tensor([0.25], device="cuda")
    u = torch.ones((1, 1, 4), device="cuda")
    y, x = s4.s4_recurrent_fwd(lam, P, P, c([[1.0, 1.0]]), c([[1.0, 1.0]]), dt, torch.zeros(1, device="cuda"), u, ws=ws)
    assert s4.s4_get_status(ws) == s4.STATUS_CODE["S4_ERR_SINGULAR_BILINEAR"]
    assert torch.count_nonzero(y).item() == 0 and torch.count_nonzero(x).item() == 0
    Ct = s4.s4_ctilde(lam, P, P, dt, c([[1.0, 1.0]]), 4, ws=ws)
    assert s4.s4_get_status(ws) == s4.STATUS_CODE["S4_ERR_SINGULAR_BILINEAR"]
    assert torch.count_nonzero(Ct).item() == 0
