"""Small calls of every kernel family, for the bounds-checked build.

Run as a child process with S4_LIB pointing at libs4_checked.so (see
tests/test_gpu_bounds.py): it makes the calls, checks that each returns S4_OK
with finite outputs, and prints one JSON line with the number of out-of-extent
indices the instrumented kernels counted (s4_bounds_violations)."""
import ctypes
import json
import os
import sys

import numpy as np
import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import structured_state_space_gb300 as s4  # noqa: E402
from structured_state_space_gb300 import workloads as W  # noqa: E402


def dev(p, keys):
    return {k: torch.from_numpy(np.ascontiguousarray(p[k])).cuda() for k in keys}


def finite(t):
    return bool(torch.isfinite(torch.view_as_real(t) if t.is_complex() else t).all())


def main():
    lib = s4.load()
    assert s4.s4_bounds_violations() >= 0, "not a bounds-checked build"
    calls = 0
    keys = ["Lambda", "P", "Q", "B", "Ctilde", "dt", "D"]
    # the layer: tiny rows, short rows (staged twiddles at M <= 1024), 8192-point
    # rows (staged inputs, and unstaged at a ragged L), the four-step long rows
    for (N, r, H, L, batch) in [(4, 1, 3, 1, 2), (6, 2, 2, 20, 3), (8, 1, 3, 1000, 3), (8, 1, 2, 4000, 3),
                                (8, 1, 2, 3001, 2), (8, 2, 2, 9000, 3), (8, 1, 2, 16384, 3), (8, 1, 2, 40000, 1),
                                (16, 4, 2, 300, 1)]:
        w = W.custom(N, r, H, L, batch, seed=N + L)
        p = W.make_params(w)
        d = dev(p, keys)
        u = torch.from_numpy(W.make_u(w, p)).cuda()
        ws = s4.workspace(H, N, r, L, batch)
        K, y = s4.s4_layer_fwd(d["Lambda"], d["P"], d["Q"], d["B"], d["Ctilde"], d["dt"], d["D"], u, ws=ws)
        assert s4.s4_get_status(ws) == 0 and finite(K) and finite(y), ("layer", N, r, H, L, batch)
        # kernel generation alone (cluster inverse transforms on long rows)
        K1 = s4.s4_kernel_gen(d["Lambda"], d["P"], d["Q"], d["B"], d["Ctilde"], d["dt"], L, ws=ws)
        # the convolutions alone
        y1 = s4.s4_conv_fwd(u, K1, d["D"], ws=ws)
        y2 = s4.s4_conv_fwd_real(u, K1, d["D"], ws=ws)
        assert s4.s4_get_status(ws) == 0 and finite(K1) and finite(y1) and finite(y2), ("parts", L)
        calls += 4
        if 256 + 16 * H * w.M <= (8 << 20):  # the allocation-free convolution, where it fits
            f = lib.s4_conv_fwd_noalloc
            f.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 3 + [ctypes.c_void_p] * 2
            f.restype = ctypes.c_int
            y3 = torch.empty_like(y)
            rc = f(ctypes.c_void_p(u.data_ptr()), ctypes.c_void_p(K1.data_ptr()), ctypes.c_void_p(d["D"].data_ptr()),
                   batch, H, L, ctypes.c_void_p(y3.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
            torch.cuda.synchronize()
            assert rc == 0 and finite(y3), ("noalloc", L)
            calls += 1
    # recurrent mode and C~, both branches of the solver (a zero d_j in channel 0)
    for (N, r, H, L, batch) in [(40, 1, 3, 50, 3), (80, 2, 2, 30, 2)]:
        w = W.custom(N, r, H, L, batch, seed=7 * N)
        p = W.make_params(w)
        p["dt"][0] = np.float32(0.25)  # lambda = 2/Delta = 8 exactly: d_1 = 1 - (Delta/2) lambda = 0
        p["Lambda"][0, 1] = np.complex64(8.0)
        p["P"][0, 1, 0] = 4.0
        p["Q"] = p["P"].copy()
        p["C"] = p["Ctilde"]
        d = dev(p, keys + ["C"])
        u = torch.from_numpy(W.make_u(w, p)).cuda()
        ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
        yr, x = s4.s4_recurrent_fwd(d["Lambda"], d["P"], d["Q"], d["B"], d["C"], d["dt"], d["D"], u, ws=ws)
        st1 = s4.s4_get_status(ws)
        Ct = s4.s4_ctilde(d["Lambda"], d["P"], d["Q"], d["dt"], d["C"], L, ws=ws)
        st2 = s4.s4_get_status(ws)
        assert st1 == 0 and st2 == 0 and finite(yr) and finite(x) and finite(Ct), ("recurrent", N, r, st1, st2)
        calls += 2
    print(json.dumps({"calls": calls, "violations": s4.s4_bounds_violations()}))


if __name__ == "__main__":
    main()
