"""Plain float64 CPU oracle for the HiPPO -> NPLR -> DPLR initialisation.

TEST INFRASTRUCTURE.  Independent reference for the library's host routine
``s4_hippo_dplr``; it shares no code with the library.  Only the tests,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import it.

Source: "Recurrent, LSTM, and structured state-space models", the paragraph
that defines the HiPPO state generators (citing Gu, Goel and Re, Theorem 1 /
Appendix C.1, and the HiPPO paper, section 2.3 / Appendices D.1-D.3), and
the same page's DPLR / NPLR definitions (the unitary state change x~ = V^* x
turns B, C into V^* B, V^* C).  Steps, in the pages' order:

1. the real generator G of size N: LegS G^S, LegT G^T (window theta) or the
   original LagT G^L, exactly as the page defines their entries;
2. the similarity S: identity for LegS and LagT, S_0 = diag(sqrt(2n+1))
   diag((-1)^n) for LegT, giving Gt = S^{-1} G S; a state change x = S x~
   maps B, C to S^{-1} B and S^* C;
3. Gt = H - U U^T with H normal and U of rank 1 (LegS, LagT) or 2 (LegT).
   The page states that such a split exists but not the vectors; the plain
   reading taken here is the split whose U follows from the entries by
   inspection (worked out below), and the tests check H normal and the rank;
4. a unitary W with H = W diag(Lambda) W^*: H's Hermitian part is c I (c =
   -1/2 for LegS and LagT, 0 for LegT), so the eigenvectors of the Hermitian
   matrix -i (H - c I) (library eigh) diagonalise H, Lambda = c + i mu;
5. the DPLR form W^* Gt W = Lambda - P Q^* with P = Q = W^* U, and the
   vectors B~ = W^* S^{-1} B, C~ = W^* S^* C.

The splits of step 3 (all derived from the entries of step 1):
  LegS: p_n = sqrt(n + 1/2).  (G^S + p p^T)_nk = -sqrt((2n+1)(2k+1))/2 for
        n > k, +sqrt((2n+1)(2k+1))/2 for n < k and -1/2 on the diagonal:
        -I/2 plus a real skew-symmetric matrix, hence normal.
  LagT: p_n = 1/sqrt(2).  (G^L + p p^T)_nk = -1/2 for n >= k and +1/2 for
        n < k: -I/2 plus a real skew-symmetric matrix.
  LegT: with r_n = sqrt(2n+1) and z_n = (-1)^n, Gt_nk = -r_n r_k/theta for
        n >= k and -r_n r_k (-1)^(k-n)/theta for n < k.  Adding
        (r r^T + (r z)(r z)^T)/(2 theta) leaves -r_n r_k/theta times +1
        (n > k, n + k odd), -1 (n < k, n + k odd) or 0 (n + k even): real
        skew-symmetric.  U = [r, r z] / sqrt(2 theta), rank 2.

Every function is pinned in tests/test_hippo_pins.py (triangular
eigenvalues of G^S, normality and rank of the split, the similarity
reconstruction of G, agreement of G^T with the page "lmu.py" listing's
LegT matrix, and kernel invariance under the state change).
"""
from __future__ import annotations

import numpy as np

__all__ = ["KINDS", "generator", "similarity", "nplr_split", "hippo_dplr", "lmu_legt_b"]

KINDS = ("legs", "legt", "lagt")


def generator(kind: str, N: int, theta: float = 1.0) -> np.ndarray:
    """The real N x N generator G of `kind`, entry by entry from the definitions."""
    G = np.zeros((N, N))
    for n in range(N):
        for k in range(N):
            if kind == "legs":
                if n > k:
                    G[n, k] = -np.sqrt((2 * n + 1) * (2 * k + 1))
                elif n == k:
                    G[n, k] = -(n + 1)
            elif kind == "legt":
                if n >= k:
                    G[n, k] = -(2 * n + 1) * (-1.0) ** (n - k) / theta
                else:
                    G[n, k] = -(2 * n + 1) / theta
            elif kind == "lagt":
                if n >= k:
                    G[n, k] = -1.0
            else:
                raise ValueError(kind)
    return G


def similarity(kind: str, N: int) -> np.ndarray:
    """Diagonal of S (identity, or S_0 = diag(sqrt(2n+1)) diag((-1)^n) for LegT)."""
    if kind == "legt":
        return np.array([np.sqrt(2 * n + 1) * (-1.0) ** n for n in range(N)])
    return np.ones(N)


def nplr_split(kind: str, N: int, theta: float = 1.0):
    """(Gt, H, U): Gt = S^{-1} G S and its split Gt = H - U U^T (step 3)."""
    G = generator(kind, N, theta)
    s = similarity(kind, N)
    Gt = G * s[None, :] / s[:, None]  # (S^{-1} G S)_nk = G_nk s_k / s_n
    n = np.arange(N, dtype=np.float64)
    if kind == "legs":
        U = np.sqrt(n + 0.5)[:, None]
    elif kind == "lagt":
        U = np.full((N, 1), np.sqrt(0.5))
    else:
        r = np.sqrt(2 * n + 1)
        z = (-1.0) ** n
        U = np.stack([r, r * z], axis=1) / np.sqrt(2 * theta)
    H = Gt + U @ U.T
    return Gt, H, U


def hippo_dplr(kind: str, N: int, theta: float = 1.0, B=None, C=None):
    """Steps 1-5.  Returns a dict with Lambda [N], P = Q [N][rank], W (unitary,
    column j = eigenvector of Lambda_j), the similarity diagonal s, and B~, C~
    when B, C are given (complex128)."""
    Gt, H, U = nplr_split(kind, N, theta)
    c = float(np.mean(np.diag(H)))
    herm = (H + H.T) / 2.0
    if not np.allclose(herm, c * np.eye(N), atol=1e-12 * max(1.0, np.abs(H).max())):
        raise ValueError("Hermitian part of H is not a multiple of I")
    mu, W = np.linalg.eigh(-1j * (H - c * np.eye(N)))
    Lam = c + 1j * mu
    P = W.conj().T @ U.astype(np.complex128)
    out = {"Lambda": Lam, "P": P, "Q": P.copy(), "W": W, "s": similarity(kind, N), "rank": U.shape[1]}
    s = out["s"]
    if B is not None:
        out["B"] = W.conj().T @ (np.asarray(B, dtype=np.complex128) / s)
    if C is not None:
        out["C"] = W.conj().T @ (np.asarray(C, dtype=np.complex128) * s)
    return out


def lmu_legt_b(N: int, theta: float = 1.0) -> np.ndarray:
    """The LegT input vector of the page "lmu.py" (the LMU cell's continuous
    state-space matrices): B_n = (2n+1) (-1)^n / theta."""
    n = np.arange(N)
    return (2 * n + 1) * (-1.0) ** n / theta
