"""bench.cauchy_work: the root-value kernel's algorithmic flop, replayed from the
parameters as the kernel splits the roots (direct sums near the poles, the
far-field series elsewhere, pole groups for near warps at rank 1).  Host logic,
no GPU."""
import bench
from structured_state_space_gb300 import workloads as W

SMS = 152


def test_direct_sum_below_the_series_thresholds():
    # rows of M < 8192 roots, or N < 48 poles: every (root, pole) term summed directly
    for N, L in [(64, 1024), (32, 16384)]:
        w = W.custom(N, 1, 4, L, 1, seed=3)
        p = W.make_params(w)
        flop, frac = bench.cauchy_work(p, w, SMS)
        assert frac == 1.0
        assert flop == w.H * w.M * N * bench.cauchy_flop(1)


def test_far_split_on_a_grouped_grid():
    # rank 1, N = 256, H M = 2^20 >= 512 x 10 x 152: the packed kernel with pole groups
    w = W.custom(256, 1, 16, 65536, 1, seed=91, dt_lo=1e-3, dt_hi=1e-3)
    p = W.make_params(w)
    flop, frac = bench.cauchy_work(p, w, SMS)
    full = w.H * w.M * w.N * bench.cauchy_flop(1)
    # some terms are summed directly (the roots near z = 1), most are not
    assert 0.0 < frac < 0.25, frac
    assert 0 < flop < 0.5 * full, flop / full
    # at least the series' set-up for every root
    assert flop >= 24 * w.H * w.M


def test_more_near_roots_cost_more():
    # a smaller a = 2/Delta brings more roots within 1.5 R of the poles
    fl = []
    for dt in (1e-4, 1e-2):
        w = W.custom(256, 1, 16, 65536, 1, seed=91, dt_lo=dt, dt_hi=dt)
        fl.append(bench.cauchy_work(W.make_params(w), w, SMS))
    assert fl[1][1] > fl[0][1]
    assert fl[1][0] > fl[0][0]
