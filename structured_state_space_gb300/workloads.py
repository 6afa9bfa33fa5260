"""Seeded synthetic inputs for the S4 layer forward path.

This module only draws random numbers and casts them; it holds none of the
method's arithmetic.  Both the CUDA path (tests, bench) and the CPU oracle take
their inputs from here, so the two sides see byte-identical fp32 arrays.

Parameter shapes (one set of parameters per channel h):
    Lambda [H][N]    complex64  diagonal of Lambda in A = Lambda - P Q^*
    P, Q   [H][N][r] complex64  low-rank factors
    B      [H][N]    complex64  input vector
    Ctilde [H][N]    complex64  truncated output vector C~_M = (I - Abar^M)^* C
    dt     [H]       float32    step size Delta
    D      [H]       float32    direct (skip) term
    u      [batch][H][L] float32 input sequences

The workloads follow the long-sequence setting of "Recurrent, LSTM, and
structured state-space models" (section "DPLR structured state-space
parameterization"): Lambda_n = -0.5 + i*pi*n, n = 0..N-1, identical in every
channel; P, Q, B, C~ drawn per channel; Delta log-uniform per channel.
"Complex N(0,1)" means real and imaginary parts drawn iid N(0,1).
Draw order: Delta[H]; then per channel P, (Q), B, C~; then D[H]; then u.
Everything is drawn in float64 and rounded once to float32.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    N: int
    r: int
    H: int
    L: int
    batch: int
    pq: str            # "shared": Q = P; "independent": Q drawn on its own
    pq_scale: str      # "0.1" (times 0.1) or "1/sqrtN"
    bc_scale: str      # "0.1" or "1/sqrt2"
    dt_lo: float
    dt_hi: float
    seed: int

    @property
    def M(self) -> int:
        return 1 << (self.L - 1).bit_length()

    def describe(self) -> dict:
        return {"workload": self.name, "N": self.N, "r": self.r, "H": self.H,
                "L": self.L, "M": self.M, "batch": self.batch}


# The five workloads, smallest first.  Index 1 is the one the benchmark times.
WORKLOADS = [
    Workload("s4-fwd N4 r1 H2 L64 B1", 4, 1, 2, 64, 1, "shared", "0.1", "0.1", 1e-3, 1e-1, 1000),
    Workload("s4-fwd N64 r1 H256 L1024 B16", 64, 1, 256, 1024, 16, "shared", "1/sqrtN", "1/sqrt2", 1e-3, 1e-1, 1001),
    Workload("s4-fwd N64 r1 H512 L4096 B8", 64, 1, 512, 4096, 8, "shared", "1/sqrtN", "1/sqrt2", 1e-3, 1e-1, 1002),
    Workload("s4-fwd N64 r2 H256 L16384 B4", 64, 2, 256, 16384, 4, "independent", "1/sqrtN", "1/sqrt2", 1e-4, 1e-2, 1003),
    Workload("s4-fwd N256 r1 H1024 L65536 B2", 256, 1, 1024, 65536, 2, "shared", "1/sqrtN", "1/sqrt2", 1e-5, 1e-3, 1004),
]


def custom(N, r, H, L, batch, seed, pq="shared", dt_lo=1e-3, dt_hi=1e-1, name=None) -> Workload:
    """A workload with the second workload's distributions and other sizes."""
    return Workload(name or f"s4-fwd N{N} r{r} H{H} L{L} B{batch}", N, r, H, L, batch,
                    pq, "1/sqrtN", "1/sqrt2", dt_lo, dt_hi, seed)


def _cn(rng, shape):
    return rng.standard_normal(shape) + 1j * rng.standard_normal(shape)


def make_params(w: Workload) -> dict:
    """Per-channel parameters (numpy, fp32/complex64), drawn in the stated order."""
    rng = np.random.default_rng(w.seed)
    H, N, r = w.H, w.N, w.r
    dt = np.exp(rng.uniform(math.log(w.dt_lo), math.log(w.dt_hi), size=H))
    pq_s = 0.1 if w.pq_scale == "0.1" else 1.0 / math.sqrt(N)
    bc_s = 0.1 if w.bc_scale == "0.1" else 1.0 / math.sqrt(2.0)
    P = np.empty((H, N, r), np.complex128)
    Q = np.empty((H, N, r), np.complex128)
    B = np.empty((H, N), np.complex128)
    Ct = np.empty((H, N), np.complex128)
    for h in range(H):
        P[h] = _cn(rng, (N, r)) * pq_s
        Q[h] = P[h] if w.pq == "shared" else _cn(rng, (N, r)) * pq_s
        B[h] = _cn(rng, N) * bc_s
        Ct[h] = _cn(rng, N) * bc_s
    D = rng.standard_normal(H)
    lam_row = -0.5 + 1j * math.pi * np.arange(N)
    Lam = np.broadcast_to(lam_row, (H, N)).copy()
    return {
        "Lambda": Lam.astype(np.complex64), "P": P.astype(np.complex64),
        "Q": Q.astype(np.complex64), "B": B.astype(np.complex64),
        "Ctilde": Ct.astype(np.complex64), "dt": dt.astype(np.float32),
        "D": D.astype(np.float32), "_rng_state": rng.bit_generator.state,
    }


def make_u(w: Workload, params: dict, batch: int | None = None) -> np.ndarray:
    """Input u [batch][H][L] float32, continuing the parameter draw's stream."""
    rng = np.random.default_rng(w.seed)
    rng.bit_generator.state = params["_rng_state"]
    b = w.batch if batch is None else batch
    out = np.empty((b, w.H, w.L), np.float32)
    for i in range(b):  # row by row keeps the float64 temporaries small
        out[i] = rng.standard_normal((w.H, w.L))
    return out


def make_inputs(w: Workload) -> dict:
    p = make_params(w)
    p["u"] = make_u(w, p)
    return p


def scalar_example(L: int, u=None) -> dict:
    """The scalar model A = 0, B = C = 1, D = 0, Delta = 1 (one channel, N = 1, r = 1,
    P = Q = 0).  C~ is not given by that example; callers pass C directly where needed."""
    if u is None:
        u = np.arange(1, L + 1, dtype=np.float32)
    return {
        "Lambda": np.zeros((1, 1), np.complex64), "P": np.zeros((1, 1, 1), np.complex64),
        "Q": np.zeros((1, 1, 1), np.complex64), "B": np.ones((1, 1), np.complex64),
        "C": np.ones((1, 1), np.complex64), "dt": np.ones(1, np.float32),
        "D": np.zeros(1, np.float32), "u": np.asarray(u, np.float32).reshape(1, 1, L),
    }


def sample_channels(w: Workload, extra: int = 4, seed: int = 4242) -> list:
    """Channels checked (and timed on the CPU) for workloads too large to take
    whole: the first two, the two around the middle, the last, and `extra`
    seeded others, sorted.  Small workloads (H <= 8) return every channel."""
    if w.H <= 8:
        return list(range(w.H))
    fixed = {0, 1, w.H // 2 - 1, w.H - 1}
    rest = np.array([h for h in range(w.H) if h not in fixed])
    rng = np.random.default_rng(seed)
    picked = rng.choice(rest, size=min(extra, rest.size), replace=False)
    return sorted(fixed | {int(h) for h in picked})
