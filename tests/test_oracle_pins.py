"""Pins for the float64 oracle against facts that the pages or the mathematics
fix, so that the oracle is trusted for something other than itself.

Sources: "Recurrent, LSTM, and structured state-space models" ([RSS]) and its
"Examples" page ([EX]).  Each test names the fact it pins.  The last group
plants plausible mistakes in copies of oracle functions and checks that at
least one pin catches each.
"""
import os

import numpy as np
import pytest

import oracle.s4_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            out[key] = np.array([float(v) for v in vals])
    return out


def _rand_dplr(rng, N, r, stable=True, shared=False, dt=None):
    lam = -rng.uniform(0.2, 1.0, N) + 1j * rng.uniform(-5, 5, N)
    if not stable:
        lam = rng.standard_normal(N) + 1j * rng.standard_normal(N)
    P = (rng.standard_normal((N, r)) + 1j * rng.standard_normal((N, r))) / np.sqrt(2 * N)
    Q = P.copy() if shared else (rng.standard_normal((N, r)) + 1j * rng.standard_normal((N, r))) / np.sqrt(2 * N)
    B = rng.standard_normal(N) + 1j * rng.standard_normal(N)
    C = rng.standard_normal(N) + 1j * rng.standard_normal(N)
    if dt is None:
        dt = float(np.exp(rng.uniform(np.log(1e-2), np.log(0.5))))
    return lam, P, Q, B, C, dt


# ----------------------------------------------------------------------------
# [EX] scalar example: A = 0, B = C = 1, D = 0, Delta = 1
# ----------------------------------------------------------------------------

def test_scalar_example_discretisation():
    g = _golden("scalar_example.txt")
    _, Abar, Bbar = O.bilinear([0.0], [[0.0]], [[0.0]], [1.0], 1.0)
    assert Abar.shape == (1, 1)
    assert Abar[0, 0] == g["Abar"][0]
    assert Bbar[0] == g["Bbar"][0]


def test_scalar_example_kernel_conv_recurrence():
    g = _golden("scalar_example.txt")
    L = int(g["L"][0])
    _, Abar, Bbar = O.bilinear([0.0], [[0.0]], [[0.0]], [1.0], 1.0)
    K = O.kernel_from_c(Abar, Bbar, [1.0], L)
    np.testing.assert_array_equal(K, g["K"])
    np.testing.assert_array_equal(O.causal_conv(K, g["u"], 0.0), g["y"])
    np.testing.assert_array_equal(O.recurrence(Abar, Bbar, [1.0], 0.0, g["u"]), g["y"])
    np.testing.assert_array_equal(O.causal_conv_at(K, g["u"], 0.0, range(L)), g["y"])


def test_scalar_example_filter_is_resonant_at_z1():
    # Through the filter path the example has s(1) = 0 = lambda, so the pages'
    # procedure stops with 'resonant-diagonal' at the root z_0 = 1.
    with pytest.raises(O.OracleStatus) as e:
        O.filter_root_values([0.0], [[0.0]], [[0.0]], [1.0], [1.0], 1.0, 8)
    assert e.value.status == "resonant-diagonal"
    assert "k=0" in str(e.value)


# ----------------------------------------------------------------------------
# Closed forms and invariants of the bilinear discretisation
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("N", [1, 3, 7])
def test_diagonal_closed_form(N):
    # With P = Q = 0, A = Lambda is diagonal and the bilinear matrices are the
    # scalar Cayley maps abar = (1 + a lam)/(1 - a lam), bbar = Delta/(1 - a lam).
    rng = np.random.default_rng(N)
    lam, _, _, B, C, dt = _rand_dplr(rng, N, 1)
    Z = np.zeros((N, 1))
    _, Abar, Bbar = O.bilinear(lam, Z, Z, B, dt)
    al = dt / 2
    ab = (1 + al * lam) / (1 - al * lam)
    bb = dt * B / (1 - al * lam)
    np.testing.assert_allclose(Abar, np.diag(ab), atol=1e-14)
    np.testing.assert_allclose(Bbar, bb, rtol=1e-13)
    L = 40
    K = O.kernel_from_c(Abar, Bbar, C, L)
    Kc = np.array([np.sum(np.conj(C) * ab ** j * bb) for j in range(L)])
    np.testing.assert_allclose(K, Kc, rtol=1e-11, atol=1e-14)


def test_bilinear_small_step_matches_exponential():
    # Bilinear discretisation is a second-order accurate approximation of
    # exp(Delta A): the error of Abar shrinks like Delta^3.
    rng = np.random.default_rng(3)
    lam, P, Q, B, _, _ = _rand_dplr(rng, 5, 2)
    A, _, _ = O.bilinear(lam, P, Q, B, 0.1)
    from scipy.linalg import expm
    errs = []
    for dt in [1e-2, 5e-3]:
        _, Abar, _ = O.bilinear(lam, P, Q, B, dt)
        errs.append(np.linalg.norm(Abar - expm(dt * A)))
    ratio = errs[0] / errs[1]
    assert 7.0 < ratio < 9.0, ratio


@pytest.mark.parametrize("seed", range(4))
def test_shared_pq_gives_contraction(seed):
    # With Q = P and Re(lambda) < 0, A + A^* = 2 Re(Lambda) - 2 P P^* is negative
    # definite, so the Cayley transform Abar has spectral norm < 1.
    rng = np.random.default_rng(seed)
    lam, P, _, B, _, dt = _rand_dplr(rng, 6, 2, shared=True)
    P = P * 3.0
    _, Abar, _ = O.bilinear(lam, P, P, B, dt)
    assert np.linalg.norm(Abar, 2) < 1.0


@pytest.mark.parametrize("N,r", [(4, 1), (6, 2), (5, 3)])
def test_dplr_solver_matches_dense(N, r):
    # The recurrent mode's Woodbury solve of G x = b equals the dense solve.
    rng = np.random.default_rng(N * 10 + r)
    lam, P, Q, B, _, dt = _rand_dplr(rng, N, r)
    A, _, _ = O.bilinear(lam, P, Q, B, dt)
    b = rng.standard_normal(N) + 1j * rng.standard_normal(N)
    G = np.eye(N) - dt / 2 * A
    np.testing.assert_allclose(O.recurrent_solve_dplr(lam, P, Q, dt, b), np.linalg.solve(G, b), rtol=1e-11)


@pytest.mark.parametrize("zeros", [1, 2])
def test_dplr_bordered_branch_matches_dense(zeros):
    # d_j = 1 - alpha lambda_j = 0 for some j: the bordered system still solves G x = b.
    rng = np.random.default_rng(40 + zeros)
    N, r = 5, 2
    lam, P, Q, B, _, _ = _rand_dplr(rng, N, r)
    dt = 0.25                      # a power of two: 1 - (dt/2)(2/dt) is exactly 0
    lam = lam.copy()
    lam[:zeros] = 2.0 / dt
    A, _, _ = O.bilinear(lam, P, Q, B, dt)
    b = rng.standard_normal(N) + 1j * rng.standard_normal(N)
    G = np.eye(N) - dt / 2 * A
    np.testing.assert_allclose(O.recurrent_solve_dplr(lam, P, Q, dt, b), np.linalg.solve(G, b), rtol=1e-10)


def test_dplr_bordered_too_many_zeros_is_singular():
    lam = np.array([2.0, 2.0, -1.0 + 1j])
    P = np.ones((3, 1)) * 0.3
    with pytest.raises(O.OracleStatus) as e:
        O.recurrent_solve_dplr(lam, P, P, 1.0, np.ones(3))
    assert e.value.status == "singular-bilinear-matrix"


# ----------------------------------------------------------------------------
# Woodbury, root values and the generating-function identity
# ----------------------------------------------------------------------------

def _dense_root_values(lam, P, Q, B, Ct, dt, M):
    N = len(lam)
    A = np.diag(lam) - np.asarray(P).reshape(N, -1) @ np.asarray(Q).reshape(N, -1).conj().T
    out = []
    for k in range(M):
        z = np.exp(-2j * np.pi * k / M)
        if M > 1 and k == M // 2:
            out.append(dt / 2 * np.vdot(Ct, B))
            continue
        s = 2.0 / dt * (1 - z) / (1 + z)
        out.append(2.0 / (1 + z) * np.vdot(Ct, np.linalg.inv(s * np.eye(N) - A) @ B))
    return np.array(out)


@pytest.mark.parametrize("N,r,M", [(1, 1, 4), (3, 1, 8), (4, 2, 16), (6, 2, 2), (5, 3, 8), (2, 1, 1)])
def test_woodbury_root_values_match_dense_resolvent(N, r, M):
    rng = np.random.default_rng(N * 100 + r * 10 + M)
    lam, P, Q, B, Ct, dt = _rand_dplr(rng, N, r)
    Hw = O.filter_root_values(lam, P, Q, B, Ct, dt, M)
    Hd = _dense_root_values(lam, P, Q, B, Ct, dt, M)
    np.testing.assert_allclose(Hw, Hd, rtol=1e-10, atol=1e-13)


@pytest.mark.parametrize("N,r,L", [(1, 1, 1), (2, 1, 2), (3, 1, 3), (4, 2, 8), (5, 2, 13), (6, 3, 16), (4, 1, 64)])
def test_generating_function_identity(N, r, L):
    # The kernel by its definition (C recovered from C~_M, repeated
    # multiplication) equals the pages' filter: inverse transform of H(z_k).
    rng = np.random.default_rng(N * 1000 + L)
    lam, P, Q, B, Ct, dt = _rand_dplr(rng, N, r)
    K_def = O.s4_kernel(lam, P, Q, B, Ct, dt, L)
    K_filt = O.filter_kernel(lam, P, Q, B, Ct, dt, L)
    assert np.linalg.norm(K_def - K_filt) <= 1e-10 * np.linalg.norm(K_def)


@pytest.mark.parametrize("M", [1, 4, 64])
def test_ctilde_formation_inverts_c_recovery(M):
    # C~ formed from C, then C recovered from C~ (pinned through the
    # generating-function identity), gives C back; and the kernel from C~
    # equals the kernel from C by definition.
    rng = np.random.default_rng(M + 5)
    lam, P, Q, B, C, dt = _rand_dplr(rng, 5, 2)
    _, Abar, Bbar = O.bilinear(lam, P, Q, B, dt)
    Ct = O.ctilde_from_c(Abar, C, M)
    np.testing.assert_allclose(O.c_from_ctilde(Abar, Ct, M), C, rtol=1e-10)
    np.testing.assert_allclose(O.s4_kernel(lam, P, Q, B, Ct, dt, M), O.kernel_from_c(Abar, Bbar, C, M),
                               rtol=1e-10, atol=1e-13)


def test_root_value_at_minus_one_is_finite_formula():
    # z = -1: sum_j K_j (-1)^j over the full length M equals (Delta/2) C~^* B.
    rng = np.random.default_rng(9)
    lam, P, Q, B, Ct, dt = _rand_dplr(rng, 4, 2)
    M = 8
    K = O.s4_kernel(lam, P, Q, B, Ct, dt, M)
    lhs = np.sum(K * (-1.0) ** np.arange(M))
    np.testing.assert_allclose(lhs, dt / 2 * np.vdot(Ct, B), rtol=1e-11)


def test_resonant_correction_status():
    # r = 1, N = 1: W(z) = 1 + conj(q) p / (s - lam) vanishes when
    # conj(q) p = lam - s(z); choose that at the root z = 1 (s = 0).
    # (Here A = lam - p conj(q) = 0, so s(1) = 0 is an eigenvalue of A.)
    # lam = -1/2, p = 1/2, q = -1: conj(q) p = lam, and every product is exact.
    lam = np.array([-0.5 + 0j])
    p = np.array([[0.5 + 0j]])
    q = np.array([[-1.0 + 0j]])
    with pytest.raises(O.OracleStatus) as e:
        O.filter_root_values(lam, p, q, [1.0], [1.0], 0.3, 4)
    assert e.value.status == "resonant-correction"


# ----------------------------------------------------------------------------
# Convolution
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("seed", range(3))
def test_recurrence_equals_convolution(seed):
    rng = np.random.default_rng(seed)
    lam, P, Q, B, C, dt = _rand_dplr(rng, 5, 2)
    _, Abar, Bbar = O.bilinear(lam, P, Q, B, dt)
    L = 50
    u = rng.standard_normal(L)
    D = 0.7
    y_conv = O.causal_conv(O.kernel_from_c(Abar, Bbar, C, L), u, D)
    y_rec = O.recurrence(Abar, Bbar, C, D, u)
    np.testing.assert_allclose(y_conv, y_rec, rtol=1e-11, atol=1e-12)


def test_causal_conv_bruteforce_and_properties():
    rng = np.random.default_rng(5)
    L = 17
    K = rng.standard_normal(L) + 1j * rng.standard_normal(L)
    u = rng.standard_normal(L)
    D = -1.3
    y = O.causal_conv(K, u, D)
    y_bf = np.zeros(L, complex)
    for t in range(L):
        for j in range(t + 1):
            y_bf[t] += K[j] * u[t - j]
        y_bf[t] += D * u[t]
    np.testing.assert_allclose(y, y_bf, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(O.causal_conv_at(K, u, D, [0, 5, L - 1]), y_bf[[0, 5, L - 1]], rtol=1e-13)
    # the skip term alone
    np.testing.assert_array_equal(O.causal_conv(np.zeros(L), u, D), D * u)
    # causality: changing u_t leaves y_{<t} unchanged
    u2 = u.copy()
    u2[9] += 5.0
    y2 = O.causal_conv(K, u2, D)
    np.testing.assert_array_equal(y2[:9], y[:9])
    assert np.all(y2[9:] != y[9:])


# ----------------------------------------------------------------------------
# Transforms and Cauchy products
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("M", [1, 2, 4, 8, 32, 64])
def test_radix2_dft_definition_and_inverse(M):
    rng = np.random.default_rng(M)
    a = rng.standard_normal(M) + 1j * rng.standard_normal(M)
    A = O.radix2_dft(a)
    np.testing.assert_allclose(A, O.dft_direct(a), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(A, np.fft.fft(a), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(O.radix2_dft(A, inverse=True), a, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(O.dft_direct(A, inverse=True), a, rtol=1e-12, atol=1e-12)


def test_dft_matrix_orthogonality():
    # F^* F = M I for the forward DFT matrix.
    M = 16
    F = np.stack([O.radix2_dft(np.eye(M)[j]) for j in range(M)], axis=1)
    np.testing.assert_allclose(F.conj().T @ F, M * np.eye(M), atol=1e-12)
    assert O.radix2_dft(np.array([2.5 - 1j]))[0] == 2.5 - 1j   # M = 1 is the identity


@pytest.mark.parametrize("n,M,s", [(1, 1, 1), (2, 2, 1), (3, 4, 3), (5, 8, 1), (4, 16, 5), (7, 8, 7)])
def test_cauchy_product_tree_matches_direct(n, M, s):
    rng = np.random.default_rng(n * 31 + M)
    mu = (1.0 + rng.uniform(0.05, 0.5, n)) * np.exp(2j * np.pi * rng.uniform(size=n))
    a = rng.standard_normal(n) + 1j * rng.standard_normal(n)
    omega = np.exp(-2j * np.pi * s / M) if M > 1 else 1.0
    y_tree = O.cauchy_product_tree(mu, a, M, s)
    y_dir = O.cauchy_direct(mu, a, M, omega)
    np.testing.assert_allclose(y_tree, y_dir, rtol=1e-9, atol=1e-12)


def test_cauchy_collision_status():
    M = 4
    mu = np.array([1j, 0.3])     # w^3 = e^{-2 pi i 3/4} = i
    with pytest.raises(O.OracleStatus):
        O.cauchy_direct(mu, [1.0, 1.0], M)


def test_root_value_cauchy_form():
    # The pages' Cauchy form of S_uv: (2/(1+z)) u^* R v equals
    # -2 sum conj(u_j) v_j / (a + lam_j) / (z - mu_j) with mu_j = (a - lam_j)/(a + lam_j).
    rng = np.random.default_rng(12)
    N, M = 5, 16
    lam, _, _, B, Ct, dt = _rand_dplr(rng, N, 1)
    a = 2.0 / dt
    mu = (a - lam) / (a + lam)
    wts = -2.0 * np.conj(Ct) * B / (a + lam)
    S = O.cauchy_direct(mu, wts, M)
    for k in range(M):
        if k == M // 2:
            continue
        z = np.exp(-2j * np.pi * k / M)
        s = a * (1 - z) / (1 + z)
        np.testing.assert_allclose(S[k], 2 / (1 + z) * np.sum(np.conj(Ct) * B / (s - lam)), rtol=1e-11)


def test_transform_length():
    assert [O.transform_length(L) for L in [1, 2, 3, 4, 5, 64, 100, 1000, 1024, 65536]] == \
        [1, 2, 4, 4, 8, 64, 128, 1024, 1024, 65536]


# ----------------------------------------------------------------------------
# Planted mistakes: each mutated copy must fail at least one of the checks above
# ----------------------------------------------------------------------------

def _bilinear_mut(kind):
    def f(Lam, P, Q, B, dt):
        Lam, B = np.asarray(Lam, complex), np.asarray(B, complex)
        N = len(Lam)
        P = np.asarray(P, complex).reshape(N, -1)
        Q = np.asarray(Q, complex).reshape(N, -1)
        A = np.diag(Lam) - (P @ Q.T if kind == "no_conj" else P @ Q.conj().T)
        if kind == "plus_pq":
            A = np.diag(Lam) + P @ Q.conj().T
        al = dt / 2
        G = np.eye(N) + al * A if kind == "sign_G" else np.eye(N) - al * A
        return A, np.linalg.solve(G, np.eye(N) + al * A), np.linalg.solve(G, dt * B)
    return f


@pytest.mark.parametrize("kind", ["no_conj", "plus_pq", "sign_G"])
def test_planted_bilinear_mistakes_are_caught(kind, monkeypatch):
    rng = np.random.default_rng(77)
    lam, P, Q, B, Ct, dt = _rand_dplr(rng, 4, 2)
    monkeypatch.setattr(O, "bilinear", _bilinear_mut(kind))
    K_def = O.s4_kernel(lam, P, Q, B, Ct, dt, 16)
    K_filt = O.filter_kernel(lam, P, Q, B, Ct, dt, 16)
    assert np.linalg.norm(K_def - K_filt) > 1e-6 * np.linalg.norm(K_filt)


def test_planted_ctilde_as_c_is_caught():
    rng = np.random.default_rng(78)
    lam, P, Q, B, Ct, dt = _rand_dplr(rng, 4, 1)
    _, Abar, Bbar = O.bilinear(lam, P, Q, B, dt)
    K_wrong = O.kernel_from_c(Abar, Bbar, Ct, 8)     # forgets the (I - Abar^M)^* map
    K_filt = O.filter_kernel(lam, P, Q, B, Ct, dt, 8)
    assert np.linalg.norm(K_wrong - K_filt) > 1e-6 * np.linalg.norm(K_filt)


def test_planted_conv_shift_is_caught():
    g = _golden("scalar_example.txt")
    K = g["K"].astype(complex)
    y_shift = np.convolve(g["u"], K)[1:len(g["u"]) + 1]   # off by one
    assert not np.array_equal(y_shift, g["y"])
    # and the non-mutated oracle matches
    np.testing.assert_array_equal(O.causal_conv(K, g["u"], 0.0), g["y"])
