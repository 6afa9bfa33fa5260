"""The seeded input generators: shapes, dtypes, determinism and the
distribution readings stated for each workload."""
import numpy as np
import pytest

from structured_state_space_gb300 import workloads as W
import oracle.s4_oracle as O


@pytest.mark.parametrize("i", range(3))
def test_shapes_dtypes_determinism(i):
    w = W.WORKLOADS[i]
    a = W.make_inputs(w)
    b = W.make_inputs(w)
    H, N, r, L, Bsz = w.H, w.N, w.r, w.L, w.batch
    assert a["Lambda"].shape == (H, N) and a["Lambda"].dtype == np.complex64
    assert a["P"].shape == (H, N, r) and a["Q"].shape == (H, N, r)
    assert a["B"].shape == (H, N) and a["Ctilde"].shape == (H, N)
    assert a["dt"].shape == (H,) and a["dt"].dtype == np.float32
    assert a["D"].shape == (H,) and a["u"].shape == (Bsz, H, L) and a["u"].dtype == np.float32
    for k in ["Lambda", "P", "Q", "B", "Ctilde", "dt", "D", "u"]:
        np.testing.assert_array_equal(a[k], b[k])
    assert np.all(a["dt"] >= np.float32(w.dt_lo)) and np.all(a["dt"] <= np.float32(w.dt_hi))
    np.testing.assert_array_equal(a["Lambda"][0], (-0.5 + 1j * np.pi * np.arange(N)).astype(np.complex64))
    if w.pq == "shared":
        np.testing.assert_array_equal(a["P"], a["Q"])


def test_transform_lengths():
    assert [w.M for w in W.WORKLOADS] == [64, 1024, 4096, 16384, 65536]
    assert [W.custom(4, 1, 1, L, 1, 0).M for L in [1, 2, 3, 100, 1000]] == [1, 2, 4, 128, 1024]


def test_independent_pq_workload_is_stable():
    # With Q drawn independently of P, A = Lambda - P Q^* is not guaranteed
    # stable; check every channel of that workload has Re(eig A) < 0.
    w = W.WORKLOADS[3]
    p = W.make_params(w)
    assert not np.array_equal(p["P"], p["Q"])
    worst = max(np.linalg.eigvals(O.bilinear(p["Lambda"][h], p["P"][h], p["Q"][h],
                                             p["B"][h], p["dt"][h])[0]).real.max() for h in range(w.H))
    assert worst < -0.1
