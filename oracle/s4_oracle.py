"""Plain float64 CPU oracle for the S4 layer forward path.

TEST INFRASTRUCTURE.  This file is the independent reference that the CUDA
path is checked against.  It shares no code with the CUDA path and is only
imported by the tests, by ``__graft_entry__.smoke()`` and by the CPU-baseline
leg of ``bench.py``.  It is deliberately slow and direct: dense matrices,
library LU solves, repeated multiplication, direct O(L^2) convolution.

Sources (page titles and sections):
  [RSS]  "Recurrent, LSTM, and structured state-space models"
         - "Continuous-time linear state-space model" (direct term D u)
         - the complex SISO model, DPLR form, bilinear recurrent matrices,
           truncated output vector C~_M
         - "Radix-two discrete Fourier transform"
         - "Woodbury inverse for a diagonal-plus-low-rank update"
         - "DPLR structured state-space parameterization" (recurrent mode,
           filter mode, root values H(z), statuses)
  [EX]   "Recurrent, LSTM, and structured state-space models -- Examples"
         - scalar state-space example (A = 0, B = C = 1, Delta = 1)
         - "S4 convolution-filter arithmetic and numerical cost"

What the method computes exactly (up to rounding) has a plain definition:
the length-L kernel K_j = C^* Abar^j Bbar of the bilinear-discretised DPLR
model, with C recovered from the supplied C~_M, and the causal convolution
y_t = sum_{j<=t} K_j u_{t-j} + D u_t.  ``s4_kernel`` and ``causal_conv``
compute those definitions directly.  The pages' filter procedure (root values
H(z_k) from resolvents, then an inverse radix-two transform) is written out
separately in ``filter_root_values`` / ``filter_kernel`` so that the tests can
pin one against the other.

Every function here is pinned by a test in tests/test_oracle_pins.py against
facts the pages or the mathematics fix (worked example, closed forms,
invariants, brute force).  No function is parity-unpinned.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "OracleStatus", "bilinear", "c_from_ctilde", "ctilde_from_c", "kernel_from_c", "s4_kernel",
    "s4_kernel_channels", "causal_conv", "causal_conv_at", "recurrence",
    "recurrent_solve_dplr", "transform_length", "radix2_dft", "dft_direct",
    "filter_root_values", "filter_kernel", "s4_layer", "cauchy_direct",
    "cauchy_product_tree",
]


class OracleStatus(Exception):
    """A status the pages define: 'resonant-diagonal', 'resonant-correction',
    'singular-bilinear-matrix' or 'collision'."""

    def __init__(self, status: str, where: str = ""):
        super().__init__(f"{status} {where}".strip())
        self.status = status


def _c(x):
    return np.asarray(x, dtype=np.complex128)


def transform_length(L: int) -> int:
    """M = the least power of two with M >= L ([RSS] filter mode)."""
    if L < 1:
        raise ValueError("L must be >= 1")
    M = 1
    while M < L:
        M *= 2
    return M


# --------------------------------------------------------------------------
# Discretisation and the kernel by its definition
# --------------------------------------------------------------------------

def bilinear(Lam, P, Q, B, dt):
    """Dense bilinear recurrent matrices of one channel.

    [RSS] DPLR parameterization: A = Lambda - P Q^*, alpha = Delta/2,
    G = I - alpha A, Abar = G^{-1}(I + alpha A), Bbar = G^{-1} Delta B.
    G is factored by a library LU solve; a singular G is the status
    'singular-bilinear-matrix'.
    Returns (A, Abar, Bbar).
    """
    Lam, P, Q, B = _c(Lam), _c(P), _c(Q), _c(B)
    N = Lam.shape[0]
    P = P.reshape(N, -1)
    Q = Q.reshape(N, -1)
    dt = float(dt)
    A = np.diag(Lam) - P @ Q.conj().T
    alpha = dt / 2.0
    eye = np.eye(N, dtype=np.complex128)
    G = eye - alpha * A
    try:
        Abar = np.linalg.solve(G, eye + alpha * A)
        Bbar = np.linalg.solve(G, dt * B)
    except np.linalg.LinAlgError as e:
        raise OracleStatus("singular-bilinear-matrix") from e
    return A, Abar, Bbar


def c_from_ctilde(Abar, Ctilde, M: int):
    """Recover C from C~_M = (I - Abar^M)^* C ([RSS] truncated output vector).

    Abar^M by repeated squaring (numpy.linalg.matrix_power), then one solve
    with (I - Abar^M)^*.
    """
    Abar = _c(Abar)
    N = Abar.shape[0]
    AM = np.linalg.matrix_power(Abar, M)
    lhs = (np.eye(N) - AM).conj().T
    return np.linalg.solve(lhs, _c(Ctilde))


def ctilde_from_c(Abar, C, M: int):
    """C~_M = (I - Abar^M)^* C ([RSS] truncated output vector), Abar^M by
    repeated squaring."""
    Abar = _c(Abar)
    N = Abar.shape[0]
    AM = np.linalg.matrix_power(Abar, M)
    return (np.eye(N) - AM).conj().T @ _c(C)


def kernel_from_c(Abar, Bbar, C, L: int):
    """K_j = C^* Abar^j Bbar for 0 <= j < L by repeated multiplication
    ([RSS] length-L impulse kernel; the recurrence x_j = Abar x_{j-1})."""
    Abar, x, C = _c(Abar), _c(Bbar).copy(), _c(C)
    K = np.empty(L, np.complex128)
    for j in range(L):
        K[j] = np.vdot(C, x)          # C^* x  (vdot conjugates its first argument)
        x = Abar @ x
    return K


def s4_kernel(Lam, P, Q, B, Ctilde, dt, L: int):
    """One channel's length-L kernel from the supplied C~ ([EX] filter-cost
    statement: the filter returns K_L = (C^* Abar^j Bbar)_{j<L})."""
    M = transform_length(L)
    _, Abar, Bbar = bilinear(Lam, P, Q, B, dt)
    C = c_from_ctilde(Abar, Ctilde, M)
    return kernel_from_c(Abar, Bbar, C, L)


def s4_kernel_channels(params: dict, L: int, channels=None):
    """K [len(channels)][L] complex128 for the listed channels (all by default)."""
    H = params["Lambda"].shape[0]
    chans = range(H) if channels is None else channels
    out = []
    for h in chans:
        out.append(s4_kernel(params["Lambda"][h], params["P"][h], params["Q"][h],
                             params["B"][h], params["Ctilde"][h], params["dt"][h], L))
    return np.array(out)


# --------------------------------------------------------------------------
# Applying the kernel
# --------------------------------------------------------------------------

def causal_conv(K, u, D=0.0):
    """y_t = sum_{j=0}^{t} K_j u_{t-j} + D u_t for 0 <= t < L.

    [RSS]: the kernel's causal convolution plus the separate direct term;
    [EX] scalar example: sum_{j<=t} K_j u_{t-j}.  numpy.convolve is the direct
    (non-FFT) full linear convolution; its first L entries are the causal sums.
    """
    K, u = _c(K), np.asarray(u, np.float64)
    L = u.shape[-1]
    return np.convolve(u, K)[:L] + float(D) * u


def causal_conv_at(K, u, D, ts):
    """The same sums at selected output positions only (O(t) each)."""
    K, u = _c(K), np.asarray(u, np.float64)
    out = np.empty(len(ts), np.complex128)
    for i, t in enumerate(ts):
        out[i] = np.dot(K[: t + 1], u[t::-1]) + float(D) * u[t]
    return out


def recurrence(Abar, Bbar, C, D, u):
    """x_t = Abar x_{t-1} + Bbar u_t (x_{-1} = 0), y_t = C^* x_t + D u_t
    ([RSS] discrete recurrence with the separate skip term)."""
    Abar, Bbar, C = _c(Abar), _c(Bbar), _c(C)
    x = np.zeros(Abar.shape[0], np.complex128)
    y = np.empty(len(u), np.complex128)
    for t, ut in enumerate(np.asarray(u, np.float64)):
        x = Abar @ x + Bbar * ut
        y[t] = np.vdot(C, x) + float(D) * ut
    return y


def recurrent_solve_dplr(Lam, P, Q, dt, b):
    """Solve G x = b, G = I - alpha(Lambda - P Q^*), the way the recurrent
    mode of [RSS] does: d_j = 1 - alpha lambda_j; if every d_j != 0 use the
    Woodbury inverse with correction I_r + alpha Q^* D^{-1} P, otherwise the
    bordered system over J = {d_j != 0}, Z = {d_j = 0} (|Z| <= r).
    Statuses: 'singular-bilinear-matrix'."""
    Lam, b = _c(Lam), _c(b)
    N = Lam.shape[0]
    P = _c(P).reshape(N, -1)
    Q = _c(Q).reshape(N, -1)
    r = P.shape[1]
    alpha = float(dt) / 2.0
    d = 1.0 - alpha * Lam
    Z = np.flatnonzero(d == 0)
    J = np.flatnonzero(d != 0)
    if Z.size == 0:
        corr = np.eye(r) + alpha * Q.conj().T @ (P / d[:, None])
        if np.linalg.matrix_rank(corr) < r:
            raise OracleStatus("singular-bilinear-matrix")
        # (D + alpha P Q^*)^{-1} b = D^{-1} b - D^{-1} alpha P W^{-1} Q^* D^{-1} b
        Dinv_b = b / d
        z = np.linalg.solve(corr, Q.conj().T @ Dinv_b)
        return Dinv_b - alpha * (P @ z) / d
    s = Z.size
    if s > r:
        raise OracleStatus("singular-bilinear-matrix")
    dJ = d[J]
    PJ, QJ, PZ, QZ = P[J], Q[J], P[Z], Q[Z]
    top_left = np.eye(r) + alpha * QJ.conj().T @ (PJ / dJ[:, None])
    Mb = np.block([[top_left, -QZ.conj().T], [alpha * PZ, np.zeros((s, s))]])
    rhs = np.concatenate([QJ.conj().T @ (b[J] / dJ), b[Z]])
    if np.linalg.matrix_rank(Mb) < r + s:
        raise OracleStatus("singular-bilinear-matrix")
    sol = np.linalg.solve(Mb, rhs)
    z, xZ = sol[:r], sol[r:]
    x = np.empty(N, np.complex128)
    x[J] = (b[J] - alpha * (PJ @ z)) / dJ
    x[Z] = xZ
    return x


# --------------------------------------------------------------------------
# Transforms
# --------------------------------------------------------------------------

def dft_direct(a, inverse=False):
    """O(M^2) definition: ahat_k = sum_j a_j w^{jk}, w = e^{-2 pi i/M};
    the inverse uses conj(w) and divides by M ([RSS] radix-two DFT)."""
    a = _c(a)
    M = a.shape[0]
    j = np.arange(M)
    sign = 1.0 if inverse else -1.0
    F = np.exp(sign * 2j * np.pi * np.outer(j, j) / M)
    out = F @ a
    return out / M if inverse else out


def radix2_dft(a, inverse=False):
    """The radix-two recursion of [RSS]: split into even and odd entries,
    transform each with the root w^2, combine E_k +- w^k O_k.  The inverse
    runs the same recursion with conj(w) and divides by M at the end."""
    a = _c(a)
    M = a.shape[0]
    if M & (M - 1):
        raise ValueError("length must be a power of two")

    def rec(x, w):
        n = x.shape[0]
        if n == 1:
            return x.copy()
        E = rec(x[0::2], w * w)
        O = rec(x[1::2], w * w)
        wk = w ** np.arange(n // 2)
        return np.concatenate([E + wk * O, E - wk * O])

    w = 1.0 + 0j if M == 1 else np.exp((2j if inverse else -2j) * np.pi / M)
    out = rec(a, w)
    return out / M if inverse else out


# --------------------------------------------------------------------------
# The pages' filter procedure (second path, used by the pins)
# --------------------------------------------------------------------------

def filter_root_values(Lam, P, Q, B, Ctilde, dt, M: int):
    """H(z_k) at the M roots z_k = w^k, following [RSS] filter mode.

    z = -1: H = (Delta/2) C~^* B.  Otherwise s(z) = (2/Delta)(1-z)/(1+z);
    an exact zero s(z) - lambda_j is 'resonant-diagonal';
    R(z) = diag(1/(s - lambda_j)), W(z) = I_r + Q^* R P (singular ->
    'resonant-correction'), and
    H(z) = 2/(1+z) (C~^* R B - C~^* R P W^{-1} Q^* R B).
    """
    Lam, B, Ct = _c(Lam), _c(B), _c(Ctilde)
    N = Lam.shape[0]
    P = _c(P).reshape(N, -1)
    Q = _c(Q).reshape(N, -1)
    r = P.shape[1]
    dt = float(dt)
    w = 1.0 + 0j if M == 1 else np.exp(-2j * np.pi / M)
    Hv = np.empty(M, np.complex128)
    for k in range(M):
        # the roots w^k; the real/imag parts at k = 0, M/4, M/2, 3M/4 are exact
        z = _root(M, k) if M > 1 else w
        if z == -1:
            Hv[k] = (dt / 2.0) * np.vdot(Ct, B)
            continue
        s = (2.0 / dt) * (1 - z) / (1 + z)
        den = s - Lam
        if np.any(den == 0):
            raise OracleStatus("resonant-diagonal", f"at k={k}")
        Rd = 1.0 / den
        W = np.eye(r) + Q.conj().T @ (Rd[:, None] * P)
        if abs(np.linalg.det(W)) == 0.0:
            raise OracleStatus("resonant-correction", f"at k={k}")
        CRB = np.vdot(Ct, Rd * B)
        CRP = Ct.conj() @ (Rd[:, None] * P)
        QRB = Q.conj().T @ (Rd * B)
        Hv[k] = 2.0 / (1 + z) * (CRB - CRP @ np.linalg.solve(W, QRB))
    return Hv


def _root(M: int, k: int) -> complex:
    """w^k with w = e^{-2 pi i/M}; exact at the quarter points."""
    k %= M
    if 4 * k % M == 0:
        return [1 + 0j, -1j, -1 + 0j, 1j][4 * k // M]
    return complex(np.exp(-2j * np.pi * k / M))


def filter_kernel(Lam, P, Q, B, Ctilde, dt, L: int):
    """[RSS] filter mode: the first L coefficients of the inverse radix-two
    transform of the root values."""
    M = transform_length(L)
    return radix2_dft(filter_root_values(Lam, P, Q, B, Ctilde, dt, M), inverse=True)[:L]


# --------------------------------------------------------------------------
# Cauchy products on the root grid ([RSS] "Exact Cauchy matrix-vector product
# on a radix-two root grid"): the direct sum and the product-tree procedure.
# --------------------------------------------------------------------------

def cauchy_direct(mu, a, M: int, omega=None):
    """y_k = sum_j a_j / (omega^k - mu_j), 0 <= k < M (the required output)."""
    mu, a = _c(mu), _c(a)
    y = np.zeros(M, np.complex128)
    for k in range(M):
        # default root w = e^{-2 pi i/M}, exact at the quarter points
        zk = (_root(M, k) if M > 1 else 1.0 + 0j) if omega is None else omega ** k
        den = zk - mu
        if np.any(den == 0):
            raise OracleStatus("collision", f"at k={k}")
        y[k] = np.sum(a / den)
    return y


def cauchy_product_tree(mu, a, M: int, s: int = 1):
    """The balanced product-tree procedure: leaves D_j = z - mu_j, P_j = a_j;
    internal nodes D = D1 D2, P = P1 D2 + D1 P2; fold the root polynomials
    modulo z^M - 1; evaluate by the forward DFT at w0^j; reindex for
    omega = w0^s (odd s); divide.  Status 'collision' on a zero D."""
    mu, a = _c(mu), _c(a)
    n = mu.shape[0]
    if n == 0:
        return np.zeros(M, np.complex128)

    def build(lo, hi):
        if hi - lo == 1:
            return np.array([-mu[lo], 1.0 + 0j]), np.array([a[lo]])
        mid = (lo + hi + 1) // 2
        D1, P1 = build(lo, mid)
        D2, P2 = build(mid, hi)
        Dn = np.convolve(D1, D2)
        Pn = np.zeros(len(Dn) - 1, np.complex128)
        t1 = np.convolve(P1, D2)
        t2 = np.convolve(D1, P2)
        Pn[: len(t1)] += t1
        Pn[: len(t2)] += t2
        return Dn, Pn

    Droot, Proot = build(0, n)

    def fold(poly):
        f = np.zeros(M, np.complex128)
        for deg, c in enumerate(poly):
            f[deg % M] += c
        return f

    Dv = radix2_dft(fold(Droot))
    Pv = radix2_dft(fold(Proot))
    idx = [(s * k) % M for k in range(M)] if M > 1 else [0]
    Dk, Pk = Dv[idx], Pv[idx]
    if np.any(Dk == 0):
        raise OracleStatus("collision")
    return Pk / Dk


# --------------------------------------------------------------------------
# The layer
# --------------------------------------------------------------------------

def s4_layer(params: dict, u, channels=None, rows=None):
    """y [batch][len(channels)][L]: kernel per channel, then the causal
    convolution plus D u for each batch row."""
    u = np.asarray(u)
    Bsz, H, L = u.shape
    chans = list(range(H)) if channels is None else list(channels)
    rws = list(range(Bsz)) if rows is None else list(rows)
    K = s4_kernel_channels(params, L, chans)
    y = np.empty((len(rws), len(chans), L), np.complex128)
    for ci, h in enumerate(chans):
        for bi, b in enumerate(rws):
            y[bi, ci] = causal_conv(K[ci], u[b, h], params["D"][h])
    return K, y
