"""CUDA path vs the float64 oracle, element by element, on the same seeded inputs.

Tolerances (fp32 arithmetic against float64): relative L2 error <= 1e-4 on K
and on y, and max |y_gpu - y_ref| <= 1e-3 * max|y_ref|.  Large workloads are
compared on sampled channels: their whole kernels and every batch row of them,
whole (or sampled output positions where a case says so).
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle.s4_oracle as O  # noqa: E402
import structured_state_space_gb300 as s4  # noqa: E402
from structured_state_space_gb300 import build as s4build  # noqa: E402
from structured_state_space_gb300 import workloads as W  # noqa: E402

pytestmark = pytest.mark.gpu

REL_K = 1e-4
REL_Y = 1e-4
MAXABS_Y = 1e-3


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    s4build.build()
    return s4.load()


def dev(params, keys=("Lambda", "P", "Q", "B", "Ctilde", "dt", "D")):
    return {k: torch.from_numpy(np.ascontiguousarray(params[k])).cuda() for k in keys}


def rel_l2(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def check_y(y_gpu, y_ref, what):
    e = rel_l2(y_gpu, y_ref)
    m = float(np.max(np.abs(y_gpu - y_ref)))
    scale = float(np.max(np.abs(y_ref)))
    assert e <= REL_Y, f"{what}: rel-L2 {e:.3e}"
    assert m <= MAXABS_Y * scale, f"{what}: max abs {m:.3e} vs {scale:.3e}"
    return e


def run_layer(p, u):
    d = dev(p)
    ut = torch.from_numpy(u).cuda()
    K, y = s4.s4_layer_fwd(d["Lambda"], d["P"], d["Q"], d["B"], d["Ctilde"], d["dt"], d["D"], ut)
    torch.cuda.synchronize()
    return K.cpu().numpy(), y.cpu().numpy()


# sampled channels per workload: all of them for the small ones, else the
# first two, the middle two, the last and `count - 4` seeded others
def _channels(w, count):
    if w.H <= count:
        return list(range(w.H))
    return W.sample_channels(w, extra=count - 4)


@pytest.mark.parametrize("wi,nch", [(0, 2), (1, 256), (2, 16), (3, 8), (4, 8)])
def test_layer_matches_oracle(wi, nch):
    w = W.WORKLOADS[wi]
    p = W.make_params(w)
    u = W.make_u(w, p)
    K_gpu, y_gpu = run_layer(p, u)
    chans = _channels(w, nch)
    K_ref = O.s4_kernel_channels(p, w.L, chans)
    assert rel_l2(K_gpu[chans], K_ref) <= REL_K, rel_l2(K_gpu[chans], K_ref)
    # every batch row of the sampled channels, whole
    ys_gpu, ys_ref = [], []
    for ci, h in enumerate(chans):
        for b in range(w.batch):
            ys_ref.append(O.causal_conv(K_ref[ci], u[b, h], p["D"][h]))
            ys_gpu.append(y_gpu[b, h])
    check_y(np.concatenate(ys_gpu), np.concatenate(ys_ref), w.name)
    assert np.all(np.isfinite(y_gpu))


@pytest.mark.parametrize("N,r,H,L,batch", [
    (4, 1, 3, 1, 2), (4, 1, 3, 2, 2), (5, 2, 2, 3, 1), (6, 1, 5, 16, 3), (8, 2, 4, 100, 2),
    (7, 3, 2, 33, 2), (4, 4, 2, 64, 1), (300, 1, 2, 200, 2), (16, 1, 9, 1000, 3),
    (16, 2, 3, 5000, 2), (4, 1, 3, 6000, 3), (4, 1, 3, 3001, 3), (4, 1, 3, 4000, 3), (12, 1, 2, 16384, 1), (8, 1, 2, 20000, 2),
    (8, 2, 2, 40000, 1),
    # L = M on long rows: the spectrum's even bins taken from the root values
    (8, 1, 3, 8192, 3), (6, 2, 2, 32768, 1), (4, 1, 2, 65536, 1),
    # N = 256 at rank 1 on grids of H M >= 2^19.6: far-field series with pole groups,
    # with the half spectrum at radix 16 (L = M = 16384) and the full one (L < M)
    (256, 1, 48, 16384, 2), (256, 1, 16, 40000, 1),
    # the far-field series at ranks 3 and 4 (N >= 48 poles, M >= 8192 roots), long rows
    (64, 3, 2, 8192, 2), (48, 4, 2, 16384, 1),
    # M = 32 and 512 (kspec with staged twiddle tables), M = 2048 (unstaged)
    (6, 1, 3, 20, 3), (8, 1, 3, 300, 2), (8, 2, 2, 2048, 3),
])
def test_edge_sizes(N, r, H, L, batch):
    w = W.custom(N, r, H, L, batch, seed=N * 1000 + L)
    p = W.make_params(w)
    u = W.make_u(w, p)
    K_gpu, y_gpu = run_layer(p, u)
    # the oracle's kernel on a sample of channels where it is costly; whole rows
    chans = [0, H // 2, H - 1] if N * N * L * H > 2e10 else list(range(H))
    K_ref = O.s4_kernel_channels(p, L, chans)
    assert rel_l2(K_gpu[chans], K_ref) <= REL_K, rel_l2(K_gpu[chans], K_ref)
    y_ref = np.stack([[O.causal_conv(K_ref[ci], u[b, h], p["D"][h]) for ci, h in enumerate(chans)]
                      for b in range(batch)])
    check_y(y_gpu[:, chans], y_ref, f"edge N{N} r{r} L{L}")


def test_kernel_gen_and_conv_separately():
    w = W.WORKLOADS[1]
    p = W.make_params(w)
    u = W.make_u(w, p)
    d = dev(p)
    K = s4.s4_kernel_gen(d["Lambda"], d["P"], d["Q"], d["B"], d["Ctilde"], d["dt"], w.L)
    chans = [0, 7, 200]
    K_ref = O.s4_kernel_channels(p, w.L, chans)
    assert rel_l2(K.cpu().numpy()[chans], K_ref) <= REL_K
    # the convolution alone, fed a kernel given in complex64
    Kin = (np.random.default_rng(3).standard_normal((w.H, w.L)) * 0.05 + 1j * 0.02).astype(np.complex64)
    y = s4.s4_conv_fwd(torch.from_numpy(u).cuda(), torch.from_numpy(Kin).cuda(), d["D"]).cpu().numpy()
    rows = [(0, 0), (3, 17), (15, 255)]
    y_ref = np.stack([O.causal_conv(Kin[h], u[b, h], p["D"][h]) for b, h in rows])
    check_y(np.stack([y[b, h] for b, h in rows]), y_ref, "conv only")


@pytest.mark.parametrize("batch,H,L", [(2, 30, 32768), (3, 26, 65536)])
def test_long_row_conv_many_pairs(batch, H, L):
    # the four-step convolution alone on 30 and 52 pairs of rows (2M = 2^16 with
    # radix-16 columns, 2^17 with radix 32; the odd batch leaves each channel's
    # last pair with one row), rows across the whole scratch
    rng = np.random.default_rng(H * L + batch)
    u = rng.standard_normal((batch, H, L)).astype(np.float32)
    Kin = ((rng.standard_normal((H, L)) + 1j * rng.standard_normal((H, L))) * 0.01).astype(np.complex64)
    D = rng.standard_normal(H).astype(np.float32)
    ut, Kt, Dt = torch.from_numpy(u).cuda(), torch.from_numpy(Kin).cuda(), torch.from_numpy(D).cuda()
    y = s4.s4_conv_fwd(ut, Kt, Dt).cpu().numpy()
    assert np.array_equal(y, s4.s4_conv_fwd(ut, Kt, Dt).cpu().numpy())
    pb = (batch + 1) // 2
    # pair p = h pb + b // 2: the first pairs, the middle, the last pair
    rows = [(0, 0), (batch - 1, H - 1), (0, 24 // pb), (batch - 1, 25 // pb), (batch // 2, H // 2), (1, H - 2)]
    y_ref = np.stack([O.causal_conv(Kin[h], u[b, h], D[h]) for b, h in rows])
    check_y(np.stack([y[b, h] for b, h in rows]), y_ref, f"conv L{L} pairs {pb * H}")


def test_scalar_example_conv_gives_prefix_sums():
    # Page example: K = (1, ..., 1), D = 0  =>  y_t = sum_{s<=t} u_s.
    L = 8
    g = W.scalar_example(L, u=[3, -1, 4, 1, -5, 9, 2, -6])
    K = torch.ones((1, L), dtype=torch.complex64, device="cuda")
    y = s4.s4_conv_fwd(torch.from_numpy(g["u"]).cuda(), K, torch.zeros(1, device="cuda")).cpu().numpy()
    np.testing.assert_allclose(y[0, 0].real, [3, 2, 6, 7, 2, 11, 13, 7], atol=1e-5)
    np.testing.assert_allclose(y[0, 0].imag, 0, atol=1e-5)


def test_scalar_example_kernel_gen_is_resonant():
    # Through the filter, A = 0 resonates at z = 1 (s(1) = 0 = lambda).
    g = W.scalar_example(8)
    d = {k: torch.from_numpy(g[k]).cuda() for k in ["Lambda", "P", "Q", "B", "dt"]}
    ws = s4.workspace(1, 1, 1, 8, 1)
    K = s4.s4_kernel_gen(d["Lambda"], d["P"], d["Q"], d["B"], d["B"], d["dt"], 8, ws=ws)
    assert s4.s4_get_status(ws) == s4.STATUS_CODE["S4_ERR_RESONANT_DIAGONAL"]
    assert torch.count_nonzero(K).item() == 0


def test_resonant_correction_status():
    # lambda = -1/2, p = 1/2, q = -1: W(1) = 1 + conj(q) p / (0 - lambda) = 0 exactly.
    c = lambda v: torch.tensor(v, dtype=torch.complex64, device="cuda")
    ws = s4.workspace(1, 1, 1, 4, 1)
    K = s4.s4_kernel_gen(c([[-0.5]]), c([[[0.5]]]), c([[[-1.0]]]), c([[1.0]]), c([[1.0]]),
                         torch.tensor([0.3], device="cuda"), 4, ws=ws)
    assert s4.s4_get_status(ws) == s4.STATUS_CODE["S4_ERR_RESONANT_CORRECTION"]
    assert torch.count_nonzero(K).item() == 0


@pytest.mark.parametrize("bad", [0.0, -1e-3, float("nan"), float("inf")])
def test_invalid_step_status(bad):
    w = W.WORKLOADS[0]
    p = W.make_params(w)
    p["dt"][1] = bad
    d = dev(p)
    ws = s4.workspace(w.H, w.N, w.r, w.L, 1)
    K = s4.s4_kernel_gen(d["Lambda"], d["P"], d["Q"], d["B"], d["Ctilde"], d["dt"], w.L, ws=ws)
    assert s4.s4_get_status(ws) == s4.STATUS_CODE["S4_ERR_INVALID_STEP"]
    assert torch.count_nonzero(K).item() == 0


def test_status_clears_on_next_call():
    w = W.WORKLOADS[0]
    p = W.make_params(w)
    d = dev(p)
    ws = s4.workspace(w.H, w.N, w.r, w.L, 1)
    bad = d["dt"].clone()
    bad[0] = -1.0
    s4.s4_kernel_gen(d["Lambda"], d["P"], d["Q"], d["B"], d["Ctilde"], bad, w.L, ws=ws)
    assert s4.s4_get_status(ws) != 0
    s4.s4_kernel_gen(d["Lambda"], d["P"], d["Q"], d["B"], d["Ctilde"], d["dt"], w.L, ws=ws)
    assert s4.s4_get_status(ws) == 0


def _layer(d, u, ws, K=None, y=None, dt=None):
    return s4.s4_layer_fwd(d["Lambda"], d["P"], d["Q"], d["B"], d["Ctilde"], d["dt"] if dt is None else dt,
                           d["D"], u, K=K, y=y, ws=ws)


def test_layer_status_protocol():
    # a bad step in the last channel zeroes K and y of the whole call, and the
    # next good call on the same workspace clears the status again
    w = W.WORKLOADS[1]
    p = W.make_params(w)
    d = dev(p)
    ut = torch.from_numpy(W.make_u(w, p)).cuda()
    ws = s4.workspace(w.H, w.N, w.r, w.L, w.batch)
    bad = d["dt"].clone()
    bad[w.H - 1] = -1.0
    K, y = _layer(d, ut, ws, dt=bad)
    assert s4.s4_get_status(ws) == s4.STATUS_CODE["S4_ERR_INVALID_STEP"]
    assert torch.count_nonzero(K).item() == 0 and torch.count_nonzero(y).item() == 0
    K, y = _layer(d, ut, ws)
    assert s4.s4_get_status(ws) == 0
    assert torch.count_nonzero(K).item() > 0 and torch.count_nonzero(y).item() > 0
    # a status left by another entry point is cleared by the layer call too
    s4.s4_kernel_gen(d["Lambda"], d["P"], d["Q"], d["B"], d["Ctilde"], bad, w.L, ws=ws)
    assert s4.s4_get_status(ws) != 0
    _layer(d, ut, ws, K=K, y=y)
    assert s4.s4_get_status(ws) == 0


def test_layer_status_on_an_uninitialised_workspace():
    # layer calls do not reset the status block: flags carry the call's
    # generation, so whatever the workspace held before reads as clear
    w = W.WORKLOADS[1]
    p = W.make_params(w)
    d = dev(p)
    ut = torch.from_numpy(W.make_u(w, p)).cuda()
    ws = s4.workspace(w.H, w.N, w.r, w.L, w.batch)
    ws.fill_(0xFF)
    K, y = _layer(d, ut, ws)
    assert s4.s4_get_status(ws) == 0
    K_ref, y_ref = _layer(d, ut, s4.workspace(w.H, w.N, w.r, w.L, w.batch))
    assert torch.equal(K, K_ref) and torch.equal(y, y_ref)


def test_layer_flags_do_not_leak_into_other_entry_points():
    w = W.WORKLOADS[1]
    p = W.make_params(w)
    d = dev(p)
    ut = torch.from_numpy(W.make_u(w, p)).cuda()
    ws = s4.workspace(w.H, w.N, w.r, w.L, w.batch)
    bad = d["dt"].clone()
    bad[3] = float("nan")
    K, _ = _layer(d, ut, ws)
    for clean in (lambda: s4.s4_conv_fwd(ut, K, d["D"], ws=ws),
                  lambda: s4.s4_kernel_gen(d["Lambda"], d["P"], d["Q"], d["B"], d["Ctilde"], d["dt"], w.L, ws=ws),
                  lambda: s4.s4_ctilde(d["Lambda"], d["P"], d["Q"], d["dt"], d["Ctilde"], w.L, ws=ws)):
        _layer(d, ut, ws, dt=bad)
        assert s4.s4_get_status(ws) == s4.STATUS_CODE["S4_ERR_INVALID_STEP"]
        clean()
        assert s4.s4_get_status(ws) == 0


@pytest.mark.parametrize("L", [8, 32])
def test_layer_resonance_zeroes_outputs(L):
    # L = 32 takes the three-kernel layer path, L = 8 the generic one
    g = W.scalar_example(L, u=list(range(1, L + 1)))
    d = {k: torch.from_numpy(g[k]).cuda() for k in ["Lambda", "P", "Q", "B", "dt"]}
    ws = s4.workspace(1, 1, 1, L, 1)
    K, y = s4.s4_layer_fwd(d["Lambda"], d["P"], d["Q"], d["B"], d["B"], d["dt"],
                           torch.zeros(1, device="cuda"), torch.from_numpy(g["u"]).cuda(), ws=ws)
    assert s4.s4_get_status(ws) == s4.STATUS_CODE["S4_ERR_RESONANT_DIAGONAL"]
    assert torch.count_nonzero(K).item() == 0 and torch.count_nonzero(y).item() == 0


def test_layer_calls_in_a_graph_match_eager():
    # consecutive layer calls captured in one graph (each call's kernels chained
    # by programmatic dependent launch) give bitwise the results of eager calls
    w = W.WORKLOADS[1]
    p = W.make_params(w)
    d = dev(p)
    u1 = torch.from_numpy(W.make_u(w, p)).cuda()
    u2 = u1.flip(-1).contiguous()
    ws = s4.workspace(w.H, w.N, w.r, w.L, w.batch)
    K1e, y1e = _layer(d, u1, ws)
    K2e, y2e = _layer(d, u2, ws)
    torch.cuda.synchronize()
    K1, y1 = torch.empty_like(K1e), torch.empty_like(y1e)
    K2, y2 = torch.empty_like(K2e), torch.empty_like(y2e)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        _layer(d, u1, ws, K=K1, y=y1)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        _layer(d, u1, ws, K=K1, y=y1)
        _layer(d, u2, ws, K=K2, y=y2)
    y1.zero_()
    y2.zero_()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        for _ in range(3):
            g.replay()
    s.synchronize()
    assert torch.equal(y1, y1e) and torch.equal(y2, y2e) and torch.equal(K2, K2e)
    assert s4.s4_get_status(ws, s) == 0


def test_graph_replay_after_a_flagged_replay():
    # a replay whose inputs were fixed after a flagged replay must not see the
    # earlier replay's flag: each execution of a captured call is a new call
    w = W.WORKLOADS[1]
    p = W.make_params(w)
    d = dev(p)
    u = torch.from_numpy(W.make_u(w, p)).cuda()
    ws = s4.workspace(w.H, w.N, w.r, w.L, w.batch)
    K_ref, y_ref = _layer(d, u, ws)
    K_ref2 = s4.s4_kernel_gen(d["Lambda"], d["P"], d["Q"], d["B"], d["Ctilde"], d["dt"], w.L, ws=ws)
    y_ref2 = s4.s4_conv_fwd(u, K_ref2, d["D"], ws=ws)
    torch.cuda.synchronize()
    dt = d["dt"].clone()
    K, y = torch.empty_like(K_ref), torch.empty_like(y_ref)
    K2, y2 = torch.empty_like(K_ref2), torch.empty_like(y_ref2)
    s = torch.cuda.Stream()

    def calls():  # the layer call last: s4_get_status reports the last call
        s4.s4_kernel_gen(d["Lambda"], d["P"], d["Q"], d["B"], d["Ctilde"], dt, w.L, K=K2, ws=ws, stream=s)
        s4.s4_conv_fwd(u, K2, d["D"], y=y2, ws=ws, stream=s)
        with torch.cuda.stream(s):
            _layer(d, u, ws, K=K, y=y, dt=dt)

    with torch.cuda.stream(s):
        calls()
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        calls()
    for bad in (True, False, True, False):
        with torch.cuda.stream(s):  # the input update is ordered before the replay
            dt.copy_(d["dt"])
            if bad:
                dt[7] = float("nan")
            g.replay()
        s.synchronize()
        st = s4.s4_get_status(ws, s)
        if bad:
            assert st == s4.STATUS_CODE["S4_ERR_INVALID_STEP"]
            assert torch.count_nonzero(y).item() == 0
        else:
            assert st == 0
            assert torch.equal(K, K_ref) and torch.equal(y, y_ref)
            assert torch.equal(K2, K_ref2) and torch.equal(y2, y_ref2)


def test_entry_points_chained_in_a_graph_match_eager():
    # kernel generation and the two convolutions, alternating in one graph, each
    # call's first kernel a programmatic dependent of the previous call's last:
    # bitwise the eager results, and the status of the last call
    w = W.WORKLOADS[1]
    p = W.make_params(w)
    d = dev(p)
    u = torch.from_numpy(W.make_u(w, p)).cuda()
    ws = s4.workspace(w.H, w.N, w.r, w.L, w.batch)
    Ke = s4.s4_kernel_gen(d["Lambda"], d["P"], d["Q"], d["B"], d["Ctilde"], d["dt"], w.L, ws=ws)
    ye = s4.s4_conv_fwd(u, Ke, d["D"], ws=ws)
    yre = s4.s4_conv_fwd_real(u, Ke, d["D"], ws=ws)
    torch.cuda.synchronize()
    K, y, yr = torch.empty_like(Ke), torch.empty_like(ye), torch.empty_like(yre)
    s = torch.cuda.Stream()

    def calls():
        s4.s4_kernel_gen(d["Lambda"], d["P"], d["Q"], d["B"], d["Ctilde"], d["dt"], w.L, K=K, ws=ws, stream=s)
        s4.s4_conv_fwd(u, K, d["D"], y=y, ws=ws, stream=s)
        s4.s4_conv_fwd_real(u, K, d["D"], y=yr, ws=ws, stream=s)

    with torch.cuda.stream(s):
        calls()
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        calls()
        calls()
    K.zero_()
    y.zero_()
    yr.zero_()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        for _ in range(3):
            g.replay()
    s.synchronize()
    assert torch.equal(K, Ke) and torch.equal(y, ye) and torch.equal(yr, yre)
    assert s4.s4_get_status(ws, s) == 0


def test_host_errors_raise():
    w = W.WORKLOADS[0]
    p = W.make_params(w)
    d = dev(p)
    small = torch.empty(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(s4.S4Error) as e:
        s4.s4_kernel_gen(d["Lambda"], d["P"], d["Q"], d["B"], d["Ctilde"], d["dt"], w.L, ws=small)
    assert e.value.code == 2
    with pytest.raises(TypeError):
        s4.s4_kernel_gen(d["Lambda"].to(torch.complex128), d["P"], d["Q"], d["B"], d["Ctilde"], d["dt"], w.L)


def test_deterministic():
    w = W.WORKLOADS[1]
    p = W.make_params(w)
    u = W.make_u(w, p)
    K1, y1 = run_layer(p, u)
    K2, y2 = run_layer(p, u)
    assert np.array_equal(K1, K2) and np.array_equal(y1, y2)


def test_timing_hooks_count_launches():
    w = W.WORKLOADS[1]
    p = W.make_params(w)
    u = W.make_u(w, p)
    d = dev(p)
    ut = torch.from_numpy(u).cuda()
    s4.timing.reset()
    s4.timing.enable(True)
    try:
        for _ in range(3):
            s4.s4_layer_fwd(d["Lambda"], d["P"], d["Q"], d["B"], d["Ctilde"], d["dt"], d["D"], ut)
        torch.cuda.synchronize()
        # the benchmark workload's layer path: root values, fused inverse
        # transform + kernel spectrum, convolution
        for name in ["cauchy", "kspec", "conv"]:
            n, ms = s4.timing.read(name)
            assert n == 3 and ms > 0.0, (name, n, ms)
        for name in ["ifft", "spectrum"]:
            assert s4.timing.read(name)[0] == 0
    finally:
        s4.timing.enable(False)
        s4.timing.reset()


@pytest.mark.parametrize("H,L,batch", [(3, 1, 3), (2, 3, 1), (5, 16, 3), (4, 100, 2), (6, 1024, 5),
                                       (3, 5000, 3), (2, 16384, 3), (2, 40000, 1)])
def test_conv_real_matches_oracle(H, L, batch):
    # y = Re(K) * u + D u with real outputs
    rng = np.random.default_rng(H * 1000 + L)
    u = rng.standard_normal((batch, H, L)).astype(np.float32)
    K = ((rng.standard_normal((H, L)) + 1j * rng.standard_normal((H, L))) * 0.05).astype(np.complex64)
    D = rng.standard_normal(H).astype(np.float32)
    y = s4.s4_conv_fwd_real(torch.from_numpy(u).cuda(), torch.from_numpy(K).cuda(),
                            torch.from_numpy(D).cuda()).cpu().numpy()
    assert y.dtype == np.float32
    Kr = K.real.astype(np.float64)
    ref = np.stack([[O.causal_conv(Kr[h], u[b, h], D[h]).real for h in range(H)] for b in range(batch)])
    check_y(y, ref, f"real L{L}")


@pytest.mark.gpu
def test_fp32_probe_runs_and_counts_flop():
    # every lane's chain a <- a m + c converges to c / (1 - m); the flop count
    # is blocks x 256 x iters (rounded to 8) x 16
    out = torch.full((2 * 256,), float("nan"), dtype=torch.float32, device="cuda")
    flop = s4.s4_fp32_probe(out, 2, 13)
    torch.cuda.synchronize()
    assert flop == 2 * 256 * 16 * 16
    assert bool(torch.isfinite(out).all())


def test_packed_root_values_equal_scalar_bitwise():
    # The root-value kernel takes packed fp32x2 pairs of roots on large grids and
    # the scalar loop on small ones; both do the same per-lane operations in the
    # same order, so one channel alone (H = 1, scalar) and the same channel
    # repeated 64 times (packed) give identical kernels, bit for bit.  (N = 32
    # poles: the far-root series is not used below 48 poles, so every root takes
    # the direct sum in both.)
    w = W.custom(32, 1, 1, 16384, 1, seed=4242)
    p = W.make_params(w)
    rep = {k: np.repeat(p[k], 64, axis=0) for k in ["Lambda", "P", "Q", "B", "Ctilde", "dt"]}
    d1, d64 = dev(p, keys=("Lambda", "P", "Q", "B", "Ctilde", "dt")), dev(rep, keys=("Lambda", "P", "Q", "B", "Ctilde", "dt"))
    K1 = s4.s4_kernel_gen(d1["Lambda"], d1["P"], d1["Q"], d1["B"], d1["Ctilde"], d1["dt"], w.L).cpu().numpy()
    K64 = s4.s4_kernel_gen(d64["Lambda"], d64["P"], d64["Q"], d64["B"], d64["Ctilde"], d64["dt"], w.L).cpu().numpy()
    assert np.array_equal(K1[0].view(np.uint32), K64[0].view(np.uint32))
    assert np.array_equal(K64[0].view(np.uint32), K64[63].view(np.uint32))
    K_ref = O.s4_kernel_channels(p, w.L, [0])
    assert rel_l2(K1, K_ref) <= REL_K


@pytest.mark.parametrize("r,dt", [(1, 1e-4), (1, 1e-2), (2, 1e-3), (3, 1e-3), (4, 1e-4)])
def test_far_root_series_against_the_definition(r, dt):
    # Channels whose roots are almost all far from the poles (N = 256 poles spread
    # over 800 along the imaginary axis, a = 2/Delta >= 200): nearly every CTA
    # of roots takes the truncated series instead of the direct sum.  The kernel
    # must still match the definition K_j = C^* Abar^j Bbar, here to 1e-5 (ten
    # times tighter than the parity tolerance), in one call that mixes the two
    # forms (the CTAs around z = 1 stay direct).
    w = W.custom(256, r, 4, 32768, 1, seed=77 + r, dt_lo=dt, dt_hi=dt)
    p = W.make_params(w)
    d = dev(p, keys=("Lambda", "P", "Q", "B", "Ctilde", "dt"))
    K = s4.s4_kernel_gen(d["Lambda"], d["P"], d["Q"], d["B"], d["Ctilde"], d["dt"], w.L).cpu().numpy()
    K_ref = O.s4_kernel_channels(p, w.L, [0, 3])
    assert rel_l2(K[[0, 3]], K_ref) <= 1e-5, rel_l2(K[[0, 3]], K_ref)


@pytest.mark.parametrize("dt", [1e-3, 1e-4])
def test_pole_group_series_against_the_definition(dt):
    # Rank 1 on a grid large enough for the packed kernel (H M >= 2^19.6), N = 256
    # poles: the far-field series' second level is on.  With a = 2/Delta = 2e3
    # about 15 % of the roots lie within 1.5 R of the poles' centre; their warps sum
    # directly only over the pole groups they are near and take the group series
    # for the others.  K must match the definition to 1e-5 here too.
    w = W.custom(256, 1, 16, 65536, 1, seed=91, dt_lo=dt, dt_hi=dt)
    p = W.make_params(w)
    d = dev(p, keys=("Lambda", "P", "Q", "B", "Ctilde", "dt"))
    K = s4.s4_kernel_gen(d["Lambda"], d["P"], d["Q"], d["B"], d["Ctilde"], d["dt"], w.L).cpu().numpy()
    K_ref = O.s4_kernel_channels(p, w.L, [0, 11])
    assert rel_l2(K[[0, 11]], K_ref) <= 1e-5, rel_l2(K[[0, 11]], K_ref)
    assert np.all(np.isfinite(K))
