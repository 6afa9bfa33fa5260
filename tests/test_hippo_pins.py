"""Pins for the HiPPO -> NPLR -> DPLR oracle (oracle/hippo_oracle.py).

Source: "Recurrent, LSTM, and structured state-space models" (the paragraph
defining the LegS, LegT and LagT generators and their normal-plus-low-rank
structure; the NPLR -> DPLR state change) and the page "lmu.py" (the LMU
cell's continuous state-space matrices, a second printed form of LegT).
"""
import numpy as np
import pytest

import oracle.hippo_oracle as HO
import oracle.s4_oracle as O


def _dplr_dense(out):
    return np.diag(out["Lambda"]) - out["P"] @ out["Q"].conj().T


@pytest.mark.parametrize("N", [1, 2, 5, 8])
@pytest.mark.parametrize("theta", [1.0, 3.5])
def test_legt_matches_lmu_listing(N, theta):
    # lmu.py builds its LegT matrix row-wise: R_i = (2i+1)/theta times -1 above
    # the diagonal and (-1)^(i-j+1) on and below it; B_i = R_i (-1)^i.
    A = np.empty((N, N))
    for i in range(N):
        Ri = (2 * i + 1) / theta
        for j in range(N):
            A[i, j] = Ri * (-1.0 if i < j else (-1.0) ** (i - j + 1))
    np.testing.assert_allclose(HO.generator("legt", N, theta), A, rtol=0, atol=1e-13)
    np.testing.assert_allclose(HO.lmu_legt_b(N, theta), [(2 * i + 1) / theta * (-1.0) ** i for i in range(N)])


@pytest.mark.parametrize("N", [1, 2, 3, 6, 8])
def test_legs_eigenvalues_are_its_diagonal(N):
    # G^S is lower triangular with diagonal -(n+1): the DPLR matrix, similar to
    # it, has eigenvalues -1, ..., -N.
    ev = np.linalg.eigvals(_dplr_dense(HO.hippo_dplr("legs", N)))
    np.testing.assert_allclose(np.sort(ev.real), -np.arange(N, 0, -1.0), atol=1e-6)
    np.testing.assert_allclose(ev.imag, 0.0, atol=1e-6)


@pytest.mark.parametrize("N", [1, 2, 4, 6])
def test_lagt_trace_and_determinant(N):
    # G^L is lower triangular with diagonal -1: trace -N, determinant (-1)^N.
    A = _dplr_dense(HO.hippo_dplr("lagt", N))
    assert abs(np.trace(A) - (-N)) < 1e-12 * N
    assert abs(np.linalg.det(A) - (-1.0) ** N) < 1e-9


@pytest.mark.parametrize("N", [1, 4, 16])
@pytest.mark.parametrize("theta", [1.0, 0.25])
def test_legt_trace(N, theta):
    # trace G^T = -sum (2n+1)/theta = -N^2/theta, invariant under similarity
    A = _dplr_dense(HO.hippo_dplr("legt", N, theta))
    assert abs(np.trace(A) + N * N / theta) < 1e-10 * N * N / theta


@pytest.mark.parametrize("kind,rank", [("legs", 1), ("lagt", 1), ("legt", 2)])
@pytest.mark.parametrize("N", [1, 4, 16, 64])
def test_split_is_normal_plus_low_rank(kind, rank, N):
    Gt, H, U = HO.nplr_split(kind, N, 2.0)
    np.testing.assert_allclose(Gt, H - U @ U.T, atol=1e-12 * max(1.0, np.abs(Gt).max()))
    scale = np.abs(H).max() ** 2 * N
    assert np.abs(H.T @ H - H @ H.T).max() <= 1e-12 * scale
    sv = np.linalg.svd(U @ U.T, compute_uv=False)
    assert int(np.sum(sv > 1e-10 * sv[0])) <= rank
    if N >= 2:
        assert int(np.sum(sv > 1e-10 * sv[0])) == rank


@pytest.mark.parametrize("kind", HO.KINDS)
@pytest.mark.parametrize("N", [1, 3, 16, 64])
def test_similarity_reconstructs_generator(kind, N):
    theta = 1.7
    out = HO.hippo_dplr(kind, N, theta)
    W, s = out["W"], out["s"]
    np.testing.assert_allclose(W.conj().T @ W, np.eye(N), atol=1e-12 * N)
    G = (s[:, None] * (W @ _dplr_dense(out) @ W.conj().T)) / s[None, :]
    ref = HO.generator(kind, N, theta)
    assert np.abs(G - ref).max() <= 1e-12 * N * max(1.0, np.abs(ref).max())
    expect_re = 0.0 if kind == "legt" else -0.5
    np.testing.assert_allclose(out["Lambda"].real, expect_re, atol=1e-12 * N)


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
def test_kernel_invariant_under_state_change(kind):
    rng = np.random.default_rng(7)
    N, theta, dt, L = 8, 1.3, 0.05, 40
    B = rng.standard_normal(N) + 1j * rng.standard_normal(N)
    C = rng.standard_normal(N) + 1j * rng.standard_normal(N)
    out = HO.hippo_dplr(kind, N, theta, B=B, C=C)
    ref = _dense_kernel(HO.generator(kind, N, theta), B, C, dt, L)
    _, Abar, Bbar = O.bilinear(out["Lambda"], out["P"], out["Q"], out["B"], dt)
    K = O.kernel_from_c(Abar, Bbar, out["C"], L)
    assert np.linalg.norm(K - ref) <= 1e-11 * np.linalg.norm(ref)


def test_planted_split_mistake_is_caught(monkeypatch):
    # LegT without the alternating component: H is no longer normal
    real = HO.nplr_split

    def bad(kind, N, theta=1.0):
        Gt, H, U = real(kind, N, theta)
        U = U[:, :1]
        return Gt, Gt + U @ U.T, U

    monkeypatch.setattr(HO, "nplr_split", bad)
    Gt, H, U = HO.nplr_split("legt", 8, 1.0)
    assert np.abs(H.T @ H - H @ H.T).max() > 1e-3
    with pytest.raises(ValueError):
        HO.hippo_dplr("legt", 8, 1.0)


def test_planted_input_transform_mistake_is_caught():
    # B changed with S instead of S^{-1} (LegT, where S is not the identity):
    # the kernel-invariance pin rejects it
    rng = np.random.default_rng(3)
    N, dt, L = 6, 0.05, 20
    B = rng.standard_normal(N) + 0j
    C = rng.standard_normal(N) + 0j
    ref = _dense_kernel(HO.generator("legt", N, 1.0), B, C, dt, L)
    out = HO.hippo_dplr("legt", N, 1.0, B=B, C=C)
    bad_B = out["W"].conj().T @ (B * out["s"])
    _, Abar, Bbar = O.bilinear(out["Lambda"], out["P"], out["Q"], bad_B, dt)
    K = O.kernel_from_c(Abar, Bbar, out["C"], L)
    assert np.linalg.norm(K - ref) > 1e-3 * np.linalg.norm(ref)
