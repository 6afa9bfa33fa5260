"""S4 structured state-space layer, forward pass, on one NVIDIA GB300 (sm_103a).

Thin Python binding over the C ABI of ``lib/libs4.so`` (declared in
``include/s4.h``).  The functions here only marshal arguments: they check
shapes and dtypes, take device pointers and the current CUDA stream from
torch tensors, and call the library, whose kernels do all the work.  There is
no fallback: if the library is missing or fails to load, these calls raise.

Entry points (same names as the C ABI):
    s4_kernel_gen(Lambda, P, Q, B, Ctilde, dt, L)      -> K [H][L] complex64
    s4_conv_fwd(u, K, D)                               -> y [batch][H][L] complex64
    s4_conv_fwd_real(u, K, D)                          -> y [batch][H][L] float32 (Re K)
    s4_layer_fwd(Lambda, P, Q, B, Ctilde, dt, D, u)    -> (K, y)
    s4_ctilde(Lambda, P, Q, dt, C, L)                  -> C~ [H][N] complex64
    s4_recurrent_fwd(Lambda, P, Q, B, C, dt, D, u, x)  -> (y, x)   (recurrent mode)
    s4_workspace_bytes(H, N, r, L, batch)
    s4_get_status(ws), s4_status_str(code)
"""
from __future__ import annotations

import ctypes
import os

from .build import LIB as LIB_PATH

__all__ = [
    "S4Error", "load", "s4_kernel_gen", "s4_conv_fwd", "s4_layer_fwd", "s4_workspace_bytes",
    "s4_get_status", "s4_status_str", "workspace", "timing", "STATUS",
]

STATUS = {
    0: "S4_OK", 1: "S4_ERR_INVALID_ARG", 2: "S4_ERR_WORKSPACE", 3: "S4_ERR_RESONANT_DIAGONAL",
    4: "S4_ERR_RESONANT_CORRECTION", 5: "S4_ERR_NONFINITE", 6: "S4_ERR_INVALID_STEP", 7: "S4_ERR_CUDA",
    8: "S4_ERR_SINGULAR_BILINEAR", 9: "S4_ERR_TIMEOUT",
}
STATUS_CODE = {v: k for k, v in STATUS.items()}

# Names of every function the C ABI exports (include/s4.h).
ABI_FUNCTIONS = [
    "s4_workspace_bytes", "s4_kernel_gen", "s4_conv_fwd", "s4_layer_fwd", "s4_get_status",
    "s4_status_str", "s4_timing_enable", "s4_timing_reset", "s4_timing_read",
    "s4_conv_fwd_noalloc", "s4_ctilde", "s4_recurrent_fwd", "s4_conv_fwd_real",
    "s4_hippo_dplr", "s4_fp32_probe", "s4_set_wait_limit", "s4_bounds_violations",
]

HIPPO_KINDS = {"legs": 0, "legt": 1, "lagt": 2}


class S4Error(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = int(code)
        self.name = STATUS.get(self.code, f"status {code}")
        super().__init__(f"{where}: {self.name} ({s4_status_str(self.code)})")


_lib = None


def load(path: str | None = None):
    """Load libs4.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    # S4_LIB: another build of the library (the bounds-checked one, for tests)
    p = path or os.environ.get("S4_LIB") or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"libs4 not built ({p} missing): run structured_state_space_gb300.build.build()")
    lib = ctypes.CDLL(p)
    vp, sz, i32, f64p, i32p = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int)
    lib.s4_workspace_bytes.argtypes = [i32, i32, i32, i32, i32]
    lib.s4_workspace_bytes.restype = sz
    lib.s4_kernel_gen.argtypes = [vp] * 6 + [i32] * 4 + [vp, vp, sz, vp]
    lib.s4_kernel_gen.restype = i32
    lib.s4_conv_fwd.argtypes = [vp, vp, vp, i32, i32, i32, vp, vp, sz, vp]
    lib.s4_conv_fwd.restype = i32
    lib.s4_layer_fwd.argtypes = [vp] * 8 + [i32] * 5 + [vp, vp, vp, sz, vp]
    lib.s4_layer_fwd.restype = i32
    lib.s4_get_status.argtypes = [vp, vp]
    lib.s4_get_status.restype = i32
    lib.s4_status_str.argtypes = [i32]
    lib.s4_status_str.restype = ctypes.c_char_p
    lib.s4_timing_enable.argtypes = [i32]
    lib.s4_timing_enable.restype = None
    lib.s4_timing_reset.argtypes = []
    lib.s4_timing_reset.restype = None
    lib.s4_timing_read.argtypes = [ctypes.c_char_p, i32p, f64p]
    lib.s4_timing_read.restype = i32
    lib.s4_conv_fwd_real.argtypes = [vp, vp, vp, i32, i32, i32, vp, vp, sz, vp]
    lib.s4_conv_fwd_real.restype = i32
    lib.s4_ctilde.argtypes = [vp] * 5 + [i32] * 4 + [vp, vp, sz, vp]
    lib.s4_ctilde.restype = i32
    lib.s4_recurrent_fwd.argtypes = [vp] * 8 + [i32] * 5 + [vp, vp, vp, sz, vp]
    lib.s4_recurrent_fwd.restype = i32
    lib.s4_hippo_dplr.argtypes = [i32, i32, ctypes.c_double] + [vp] * 6 + [i32p]
    lib.s4_hippo_dplr.restype = i32
    lib.s4_fp32_probe.argtypes = [vp, i32, i32, vp]
    lib.s4_fp32_probe.restype = i32
    lib.s4_set_wait_limit.argtypes = [i32]
    lib.s4_set_wait_limit.restype = i32
    lib.s4_bounds_violations.argtypes = []
    lib.s4_bounds_violations.restype = ctypes.c_longlong
    _lib = lib
    return lib


def s4_status_str(code: int) -> str:
    return load().s4_status_str(int(code)).decode()


def s4_workspace_bytes(H: int, N: int, r: int, L: int, batch: int) -> int:
    return int(load().s4_workspace_bytes(H, N, r, L, batch))


# ---------------------------------------------------------------------------
# torch marshalling
# ---------------------------------------------------------------------------

def _torch():
    import torch
    return torch


def _ptr(t, dtype, shape, name):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def workspace(H, N, r, L, batch, device="cuda"):
    """A device workspace of s4_workspace_bytes(...) bytes (a uint8 tensor)."""
    torch = _torch()
    n = s4_workspace_bytes(H, N, r, L, batch)
    if n == 0:
        raise S4Error(1, "s4_workspace_bytes")
    return torch.empty(n, dtype=torch.uint8, device=device)


def _check(code, where):
    if code != 0:
        raise S4Error(code, where)


def s4_kernel_gen(Lambda, P, Q, B, Ctilde, dt, L, K=None, ws=None, stream=None):
    torch = _torch()
    H, N = Lambda.shape
    r = P.shape[-1]
    c64, f32 = torch.complex64, torch.float32
    if K is None:
        K = torch.empty((H, L), dtype=c64, device=Lambda.device)
    if ws is None:
        ws = workspace(H, N, r, L, 1, Lambda.device)
    code = load().s4_kernel_gen(
        _ptr(Lambda, c64, (H, N), "Lambda"), _ptr(P, c64, (H, N, r), "P"), _ptr(Q, c64, (H, N, r), "Q"),
        _ptr(B, c64, (H, N), "B"), _ptr(Ctilde, c64, (H, N), "Ctilde"), _ptr(dt, f32, (H,), "dt"),
        H, N, r, L, _ptr(K, c64, (H, L), "K"), ctypes.c_void_p(ws.data_ptr()), ws.numel(), _stream(stream))
    _check(code, "s4_kernel_gen")
    return K


def s4_conv_fwd(u, K, D, y=None, ws=None, stream=None):
    torch = _torch()
    batch, H, L = u.shape
    c64, f32 = torch.complex64, torch.float32
    if y is None:
        y = torch.empty((batch, H, L), dtype=c64, device=u.device)
    if ws is None:
        ws = workspace(H, 1, 1, L, batch, u.device)
    code = load().s4_conv_fwd(
        _ptr(u, f32, (batch, H, L), "u"), _ptr(K, c64, (H, L), "K"), _ptr(D, f32, (H,), "D"),
        batch, H, L, _ptr(y, c64, (batch, H, L), "y"), ctypes.c_void_p(ws.data_ptr()), ws.numel(),
        _stream(stream))
    _check(code, "s4_conv_fwd")
    return y


def s4_conv_fwd_real(u, K, D, y=None, ws=None, stream=None):
    """y = Re(K) * u + D u, real outputs."""
    torch = _torch()
    batch, H, L = u.shape
    c64, f32 = torch.complex64, torch.float32
    if y is None:
        y = torch.empty((batch, H, L), dtype=f32, device=u.device)
    if ws is None:
        ws = workspace(H, 1, 1, L, batch, u.device)
    code = load().s4_conv_fwd_real(
        _ptr(u, f32, (batch, H, L), "u"), _ptr(K, c64, (H, L), "K"), _ptr(D, f32, (H,), "D"),
        batch, H, L, _ptr(y, f32, (batch, H, L), "y"), ctypes.c_void_p(ws.data_ptr()), ws.numel(),
        _stream(stream))
    _check(code, "s4_conv_fwd_real")
    return y


def s4_layer_fwd(Lambda, P, Q, B, Ctilde, dt, D, u, K=None, y=None, ws=None, stream=None):
    torch = _torch()
    H, N = Lambda.shape
    r = P.shape[-1]
    batch, _, L = u.shape
    c64, f32 = torch.complex64, torch.float32
    if K is None:
        K = torch.empty((H, L), dtype=c64, device=u.device)
    if y is None:
        y = torch.empty((batch, H, L), dtype=c64, device=u.device)
    if ws is None:
        ws = workspace(H, N, r, L, batch, u.device)
    code = load().s4_layer_fwd(
        _ptr(Lambda, c64, (H, N), "Lambda"), _ptr(P, c64, (H, N, r), "P"), _ptr(Q, c64, (H, N, r), "Q"),
        _ptr(B, c64, (H, N), "B"), _ptr(Ctilde, c64, (H, N), "Ctilde"), _ptr(dt, f32, (H,), "dt"),
        _ptr(D, f32, (H,), "D"), _ptr(u, f32, (batch, H, L), "u"), batch, H, N, r, L,
        _ptr(K, c64, (H, L), "K"), _ptr(y, c64, (batch, H, L), "y"), ctypes.c_void_p(ws.data_ptr()),
        ws.numel(), _stream(stream))
    _check(code, "s4_layer_fwd")
    return K, y


def s4_ctilde(Lambda, P, Q, dt, C, L, Ctilde=None, ws=None, stream=None):
    torch = _torch()
    H, N = Lambda.shape
    r = P.shape[-1]
    c64, f32 = torch.complex64, torch.float32
    if Ctilde is None:
        Ctilde = torch.empty((H, N), dtype=c64, device=Lambda.device)
    if ws is None:
        ws = torch.empty(256, dtype=torch.uint8, device=Lambda.device)
    code = load().s4_ctilde(
        _ptr(Lambda, c64, (H, N), "Lambda"), _ptr(P, c64, (H, N, r), "P"), _ptr(Q, c64, (H, N, r), "Q"),
        _ptr(dt, f32, (H,), "dt"), _ptr(C, c64, (H, N), "C"), H, N, r, L,
        _ptr(Ctilde, c64, (H, N), "Ctilde"), ctypes.c_void_p(ws.data_ptr()), ws.numel(), _stream(stream))
    _check(code, "s4_ctilde")
    return Ctilde


def s4_recurrent_fwd(Lambda, P, Q, B, C, dt, D, u, x=None, y=None, ws=None, stream=None):
    """Recurrent mode over u's L steps; x (state, [batch][H][N]) is updated in place."""
    torch = _torch()
    H, N = Lambda.shape
    r = P.shape[-1]
    batch, _, L = u.shape
    c64, f32 = torch.complex64, torch.float32
    if x is None:
        x = torch.zeros((batch, H, N), dtype=c64, device=u.device)
    if y is None:
        y = torch.empty((batch, H, L), dtype=c64, device=u.device)
    if ws is None:
        ws = torch.empty(256, dtype=torch.uint8, device=u.device)
    code = load().s4_recurrent_fwd(
        _ptr(Lambda, c64, (H, N), "Lambda"), _ptr(P, c64, (H, N, r), "P"), _ptr(Q, c64, (H, N, r), "Q"),
        _ptr(B, c64, (H, N), "B"), _ptr(C, c64, (H, N), "C"), _ptr(dt, f32, (H,), "dt"),
        _ptr(D, f32, (H,), "D"), _ptr(u, f32, (batch, H, L), "u"), batch, H, N, r, L,
        _ptr(x, c64, (batch, H, N), "x"), _ptr(y, c64, (batch, H, L), "y"), ctypes.c_void_p(ws.data_ptr()),
        ws.numel(), _stream(stream))
    _check(code, "s4_recurrent_fwd")
    return y, x


def s4_hippo_dplr(kind, N, theta=1.0, B=None, C=None):
    """HiPPO generator `kind` ("legs", "legt", "lagt") of size N in DPLR form
    (host float64 routine of the library).  Returns a dict of complex128
    numpy arrays Lambda [N], P = Q [N][r], and B~, C~ [N] when B, C are given,
    plus the rank r."""
    import numpy as np
    if kind not in HIPPO_KINDS:
        raise ValueError(f"kind must be one of {sorted(HIPPO_KINDS)}")
    lib = load()
    vp = ctypes.c_void_p

    def host_in(v):
        if v is None:
            return None, None
        a = np.ascontiguousarray(np.asarray(v, dtype=np.complex128).reshape(N))
        return a, a.ctypes.data_as(vp)

    Bin, Bp = host_in(B)
    Cin, Cp = host_in(C)
    Lam = np.zeros(N, np.complex128)
    P = np.zeros(2 * N, np.complex128)
    Bt = np.zeros(N, np.complex128) if B is not None else None
    Ct = np.zeros(N, np.complex128) if C is not None else None
    rank = ctypes.c_int(0)
    code = lib.s4_hippo_dplr(HIPPO_KINDS[kind], int(N), float(theta), Bp, Cp, Lam.ctypes.data_as(vp),
                             P.ctypes.data_as(vp), Bt.ctypes.data_as(vp) if Bt is not None else None,
                             Ct.ctypes.data_as(vp) if Ct is not None else None, ctypes.byref(rank))
    _check(code, "s4_hippo_dplr")
    r = rank.value
    out = {"Lambda": Lam, "P": P[: N * r].reshape(N, r).copy(), "rank": r}
    out["Q"] = out["P"].copy()
    if Bt is not None:
        out["B"] = Bt
    if Ct is not None:
        out["C"] = Ct
    return out


def s4_fp32_probe(out, blocks: int, iters: int, stream=None) -> int:
    """Launch the FP32 issue-rate probe (blocks x 256 threads, iters rounded up
    to a multiple of 8, 16 flop per thread and iteration) into the float32
    tensor `out` (at least blocks x 256 elements).  Returns the flop launched."""
    torch = _torch()
    if out.dtype != torch.float32 or not out.is_cuda or out.numel() < blocks * 256:
        raise ValueError("out: a CUDA float32 tensor of blocks x 256 elements")
    _check(load().s4_fp32_probe(ctypes.c_void_p(out.data_ptr()), int(blocks), int(iters), _stream(stream)),
           "s4_fp32_probe")
    return blocks * 256 * ((int(iters) + 7) // 8 * 8) * 16


def s4_set_wait_limit(polls: int) -> None:
    """Polls a kernel's bounded wait on an asynchronous copy makes before it
    reports S4_ERR_TIMEOUT (negative: the default).  A test hook."""
    _check(load().s4_set_wait_limit(int(polls)), "s4_set_wait_limit")


def s4_bounds_violations() -> int:
    """Out-of-extent indices counted by a bounds-checked build (-1: normal build)."""
    return int(load().s4_bounds_violations())


def s4_get_status(ws, stream=None) -> int:
    """Synchronise the stream and return the device-detected status code in ws."""
    return int(load().s4_get_status(ctypes.c_void_p(ws.data_ptr()), _stream(stream)))


class timing:
    """Per-kernel launch timing recorded by the library (CUDA events on the
    launch stream)."""

    @staticmethod
    def enable(on=True):
        load().s4_timing_enable(1 if on else 0)

    @staticmethod
    def reset():
        load().s4_timing_reset()

    @staticmethod
    def read(name):
        n = ctypes.c_int(0)
        ms = ctypes.c_double(0.0)
        rc = load().s4_timing_read(name.encode(), ctypes.byref(n), ctypes.byref(ms))
        if rc != 0:
            raise RuntimeError("s4_timing_read failed")
        return n.value, ms.value
