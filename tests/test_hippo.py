"""The library's host routine s4_hippo_dplr against the HiPPO oracle, and the
whole chain HiPPO -> s4_ctilde -> s4_kernel_gen on the GPU against the dense
float64 kernel of the generator.

Eigenvector phases (and within a repeated eigenvalue, the basis) are free, so
the host routine is compared on what the decomposition fixes: the eigenvalues,
the per-eigenvalue Gram matrices P_j P_j^*, and the kernel C^* Abar^j Bbar of
the transformed model, which equals the kernel of (G, B, C).
"""
import numpy as np
import pytest

import oracle.hippo_oracle as HO
import oracle.s4_oracle as O
import structured_state_space_gb300 as s4


@pytest.fixture(scope="module", autouse=True)
def lib():
    from structured_state_space_gb300 import build as s4build
    s4build.build()
    return s4.load()


def _dense_kernel(A, B, C, dt, L):
    N = A.shape[0]
    G = np.eye(N) - dt / 2 * A
    Abar = np.linalg.solve(G, np.eye(N) + dt / 2 * A)
    x = np.linalg.solve(G, dt * np.asarray(B, dtype=np.complex128))
    K = np.empty(L, dtype=np.complex128)
    for j in range(L):
        K[j] = np.vdot(C, x)
        x = Abar @ x
    return K


@pytest.mark.parametrize("kind", HO.KINDS)
@pytest.mark.parametrize("N", [1, 2, 7, 64])
def test_host_routine_matches_oracle(kind, N):
    theta = 2.3
    rng = np.random.default_rng(N)
    B = rng.standard_normal(N) + 1j * rng.standard_normal(N)
    C = rng.standard_normal(N) + 1j * rng.standard_normal(N)
    got = s4.s4_hippo_dplr(kind, N, theta, B=B, C=C)
    ref = HO.hippo_dplr(kind, N, theta, B=B, C=C)
    assert got["rank"] == (2 if kind == "legt" else 1)
    scale = max(1.0, np.abs(ref["Lambda"]).max())
    np.testing.assert_allclose(np.sort(got["Lambda"].imag), np.sort(ref["Lambda"].imag), atol=1e-11 * scale)
    np.testing.assert_allclose(got["Lambda"].real, ref["Lambda"].real, atol=1e-12)
    assert np.all(np.diff(got["Lambda"].imag) >= 0)
    np.testing.assert_array_equal(got["P"], got["Q"])
    # Gram of each row of P (phase-free) where the eigenvalue is simple
    mu_r = ref["Lambda"].imag
    for j in range(N):
        k = int(np.argmin(np.abs(mu_r - got["Lambda"].imag[j])))
        gap = np.min(np.abs(np.delete(mu_r, k) - mu_r[k])) if N > 1 else np.inf
        if gap > 1e-6 * scale:
            g_got = np.outer(got["P"][j], got["P"][j].conj())
            g_ref = np.outer(ref["P"][k], ref["P"][k].conj())
            np.testing.assert_allclose(g_got, g_ref, atol=1e-9 * max(1.0, np.abs(g_ref).max()))
    # kernel of the transformed model == kernel of (G, B, C)
    dt, L = 0.02, 50
    kref = _dense_kernel(HO.generator(kind, N, theta), B, C, dt, L)
    _, Abar, Bbar = O.bilinear(got["Lambda"], got["P"], got["Q"], got["B"], dt)
    k = O.kernel_from_c(Abar, Bbar, got["C"], L)
    assert np.linalg.norm(k - kref) <= 1e-9 * np.linalg.norm(kref)


def test_host_routine_argument_errors():
    for args in [("legt", 4, 0.0), ("legt", 4, float("inf")), ("legs", 0, 1.0), ("legs", 513, 1.0)]:
        with pytest.raises(s4.S4Error) as e:
            s4.s4_hippo_dplr(*args)
        assert e.value.name == "S4_ERR_INVALID_ARG"
    with pytest.raises(ValueError):
        s4.s4_hippo_dplr("legx", 4)


@pytest.mark.gpu
@pytest.mark.parametrize("kind,N,theta", [("legs", 32, 1.0), ("legt", 32, 1.0), ("lagt", 16, 1.0), ("legs", 64, 1.0)])
def test_hippo_chain_on_gpu(kind, N, theta):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    H, L = 4, 256
    rng = np.random.default_rng(11 + N)
    dts = np.exp(rng.uniform(np.log(1e-3), np.log(1e-1), H)).astype(np.float32)
    Lam = np.zeros((H, N), np.complex64)
    Pm = np.zeros((H, N, 2 if kind == "legt" else 1), np.complex64)
    Bm = np.zeros((H, N), np.complex64)
    Cm = np.zeros((H, N), np.complex64)
    refs = []
    for h in range(H):
        B = (rng.standard_normal(N) + 1j * rng.standard_normal(N)) / np.sqrt(2)
        C = (rng.standard_normal(N) + 1j * rng.standard_normal(N)) / np.sqrt(2)
        out = s4.s4_hippo_dplr(kind, N, theta, B=B, C=C)
        Lam[h], Pm[h], Bm[h], Cm[h] = out["Lambda"], out["P"], out["B"], out["C"]
        # the kernel does not depend on the state coordinates: the expected
        # value is the oracle's dense kernel of (G, B, C) at the same Delta
        refs.append(_dense_kernel(HO.generator(kind, N, theta), B, C, float(dts[h]), L))
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    Ct = s4.s4_ctilde(t(Lam), t(Pm), t(Pm), t(dts), t(Cm), L)
    K = s4.s4_kernel_gen(t(Lam), t(Pm), t(Pm), t(Bm), Ct, t(dts), L)
    torch.cuda.synchronize()
    K = K.cpu().numpy()
    for h in range(H):
        e = np.linalg.norm(K[h] - refs[h]) / np.linalg.norm(refs[h])
        assert e <= 1e-4, (h, e)
