"""The library's partition tuner (exact dynamic program) against the
oracle's Algorithm 1 brute force.  No GPU."""
import numpy as np
import pytest

from communication_overlap_gb300 import fo
from oracle import plan as OP
from oracle import tune as OT


def _desc(M, N, W, tn=256, parts=()):
    return fo.make_desc(M=M, N=N, K=64, tile_n=tn, swizzle=8, wave_width=W,
                        group_waves=parts, host_only=True)


@pytest.mark.parametrize("seed", range(8))
def test_dp_finds_the_brute_force_minimum(seed):
    rng = np.random.default_rng(seed)
    W = int(rng.integers(2, 9))
    tm, tn = int(rng.integers(2, 7)), int(rng.integers(2, 6))
    tiles = tm * tn
    T = OP.wave_count(tiles, W)
    if T > 11:
        T = 11
        W = -(-tiles // T)
        T = OP.wave_count(tiles, W)
    tile_bytes = 128 * 256 * 2
    dur = float(rng.uniform(50, 500))
    xs = np.sort(rng.choice(np.arange(1, 4 * tiles + 1), 5, replace=False)) * tile_bytes / 2
    ys = np.sort(rng.uniform(1, 80, 5)) if seed % 2 else rng.uniform(1, 80, 5)
    curve = list(zip(xs.tolist(), ys.tolist()))
    best, t_min = OT.best_partition(T, dur, curve, W, tiles, tile_bytes)
    parts, pred = fo.fo_tune_partition(_desc(tm * 128, tn * 256, W), dur, curve)
    assert sum(parts) == T and min(parts) >= 1
    assert pred == pytest.approx(t_min, rel=1e-12, abs=1e-9)
    # the returned partition really has that prediction
    assert OT.predict(tuple(parts), dur, curve, W, tiles, tile_bytes) == pytest.approx(t_min)
    # and the predictor agrees with the oracle on every candidate
    for cand in OP.design_space(T)[:64]:
        p = fo.fo_predict_partition(_desc(tm * 128, tn * 256, W, parts=cand), dur, curve)
        assert p == pytest.approx(OT.predict(cand, dur, curve, W, tiles, tile_bytes))


def test_large_T_is_fast_and_no_worse_than_one_then_two():
    # the grouped workload has about 98 waves: 2^97 candidates
    W, tiles_m, tiles_n = 148, 259, 56
    d = _desc(tiles_m * 128, tiles_n * 256, W)
    _, T = fo.fo_wave_count(d)
    curve = [(65536 * 16, 4.0), (65536 * 148, 20.0), (65536 * 2960, 300.0)]
    parts, pred = fo.fo_tune_partition(d, 2700.0, curve)
    assert sum(parts) == T
    base = OP.one_then_two(T)
    p_base = fo.fo_predict_partition(_desc(tiles_m * 128, tiles_n * 256, W, parts=base),
                                     2700.0, curve)
    assert pred <= p_base + 1e-9
    assert pred >= 2700.0   # never below the GEMM itself


def test_bad_curves_rejected():
    d = _desc(512, 1024, 4)
    for curve in ([(1, 2.0)], [(1, 2.0), (1, 3.0)], [(1, float("nan")), (2, 1.0)]):
        with pytest.raises(fo.FoError):
            fo.fo_tune_partition(d, 10.0, curve)


@pytest.mark.parametrize("T", [1, 2, 7, 8, 9, 98, 122])
def test_curve_sample_points(T):
    """The group sizes at which the benchmark samples the latency curve:
    strictly increasing, every size up to 8, T itself, and gaps that grow
    no faster than a quarter of the size (so interpolation stays local)."""
    pytest.importorskip("torch")
    from communication_overlap_gb300.tuning import sample_waves
    ks = sample_waves(T)
    assert ks[-1] == T and ks[0] == 1
    assert all(b > a for a, b in zip(ks, ks[1:]))
    assert [k for k in ks if k <= 8] == list(range(1, min(T, 8) + 1))
    assert all(b - a <= max(1, a // 4) for a, b in zip(ks, ks[1:-1]))


@pytest.mark.parametrize("seed", range(8))
def test_interference_dp_finds_the_brute_force_minimum(seed):
    """The exact search with the interference factors against the oracle's
    brute force, and the predictor against the oracle on every candidate."""
    rng = np.random.default_rng(50 + seed)
    W = int(rng.integers(2, 7))
    tm, tn = int(rng.integers(2, 6)), int(rng.integers(2, 5))
    tiles = tm * tn
    T = OP.wave_count(tiles, W)
    tile_bytes = 128 * 256 * 2
    dur = float(rng.uniform(50, 500))
    xs = np.sort(rng.choice(np.arange(1, 4 * tiles + 1), 4, replace=False)) * tile_bytes / 2
    ys = np.sort(rng.uniform(1, 80, 4))
    curve = list(zip(xs.tolist(), ys.tolist()))
    sigma, rho = float(rng.uniform(1.0, 1.4)), float(rng.uniform(0.7, 2.5))
    best, t_min = OT.best_partition(T, dur, curve, W, tiles, tile_bytes, sigma, rho)
    d = _desc(tm * 128, tn * 256, W)
    parts, pred = fo.fo_tune_partition(d, dur, curve, sigma, rho)
    assert sum(parts) == T and pred == pytest.approx(t_min, rel=1e-9, abs=1e-9)
    assert tuple(parts) == tuple(best)          # exhaustive: the first on ties
    assert OT.predict(tuple(parts), dur, curve, W, tiles, tile_bytes, sigma, rho) == \
        pytest.approx(t_min)
    for cand in OP.design_space(T)[:64]:
        p = fo.fo_predict_partition(_desc(tm * 128, tn * 256, W, parts=cand), dur, curve,
                                    sigma, rho)
        assert p == pytest.approx(OT.predict(cand, dur, curve, W, tiles, tile_bytes, sigma, rho))
    # sigma = rho = 1 is the plain call
    assert fo.fo_tune_partition(d, dur, curve, 1.0, 1.0) == fo.fo_tune_partition(d, dur, curve)


def test_interference_factors_must_be_positive():
    d = _desc(512, 1024, 4)
    curve = [(1, 2.0), (2, 3.0)]
    for sigma, rho in ((0.0, 1.0), (1.0, -0.5), (float("inf"), 1.0), (1.0, float("nan"))):
        with pytest.raises(fo.FoError):
            fo.fo_tune_partition(d, 10.0, curve, sigma, rho)


def test_interference_large_T_local_search():
    """Beyond 20 waves the search is local: it is never worse than its
    starting points (the plain optimum, the finest partition, one wave then
    groups of two) under the interference model."""
    W, tiles_m, tiles_n = 148, 259, 56
    d = _desc(tiles_m * 128, tiles_n * 256, W)
    _, T = fo.fo_wave_count(d)
    assert T > 20
    curve = [(65536 * 16, 4.0), (65536 * 148, 20.0), (65536 * 2960, 300.0)]
    sigma, rho = 1.05, 1.3
    parts, pred = fo.fo_tune_partition(d, 2700.0, curve, sigma, rho)
    assert sum(parts) == T
    assert pred == pytest.approx(fo.fo_predict_partition(
        _desc(tiles_m * 128, tiles_n * 256, W, parts=parts), 2700.0, curve, sigma, rho))
    plain, _ = fo.fo_tune_partition(d, 2700.0, curve)
    for start in (plain, [1] * T, OP.one_then_two(T)):
        p0 = fo.fo_predict_partition(_desc(tiles_m * 128, tiles_n * 256, W, parts=start),
                                     2700.0, curve, sigma, rho)
        assert pred <= p0 + 1e-9
