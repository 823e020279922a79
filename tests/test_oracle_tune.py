"""Pins of the oracle's Algorithm 1 (predictive wave-group tuning).

Hand-computed predictions (tests/golden/tuning_hand_cases.txt), an
independent tick-by-tick simulation of one compute stream feeding one
communication channel, closed forms of the curve interpolation, and planted
mistakes that the pins must catch.  No GPU.
"""
import itertools
import os

import numpy as np
import pytest

from oracle import plan as P
from oracle import tune as T

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "tuning_hand_cases.txt")
CURVES = {"latency": [(1, 15.0), (2, 15.0)], "bandwidth": [(1, 5.0), (2, 10.0)]}


def _cases():
    rows = [l.split() for l in open(GOLDEN, encoding="utf-8")
            if l.strip() and not l.startswith("#")]
    preds = [(r[0], tuple(int(x) for x in r[1].split(",")), float(r[2]))
             for r in rows if r[0] != "best"]
    bests = [(r[1], float(r[2]), tuple(int(x) for x in r[3].split(",")))
             for r in rows if r[0] == "best"]
    return preds, bests


def test_hand_computed_predictions():
    preds, bests = _cases()
    for case, part, want in preds:
        assert T.predict(part, 40.0, CURVES[case], 1, 4, 1) == pytest.approx(want), (case, part)
    for case, t_min, part in bests:
        got, t = T.best_partition(4, 40.0, CURVES[case], 1, 4, 1)
        assert t == pytest.approx(t_min) and got == part


def _simulate(partition, duration, curve, W, tiles, tile_bytes, tick=0.01):
    """Tick-by-tick: the GEMM finishes wave after wave; a group becomes ready
    when its last wave is done; one channel sends ready groups in order,
    each for its interpolated latency."""
    T_ = sum(partition)
    sizes = T.group_bytes(partition, W, tiles, tile_bytes)
    ready_at, w = [], 0
    for g in partition:
        w += g
        ready_at.append(duration * w / T_)
    t, busy_until, j, done = 0.0, 0.0, 0, 0.0
    while j < len(partition):
        if t >= ready_at[j] - 1e-9 and t >= busy_until - 1e-9:
            busy_until = t + T.interp_latency(curve, sizes[j])
            done = busy_until
            j += 1
        t = round(t + tick, 6)
    return done


@pytest.mark.parametrize("seed", range(6))
def test_matches_tick_simulation(seed):
    rng = np.random.default_rng(seed)
    W, tiles = 3, 3 * 5 - 1       # last wave partial
    curve = sorted(zip(rng.choice(np.arange(1, 40), 4, replace=False) * 1.0,
                       np.round(rng.uniform(1, 30, 4), 2)))
    for part in P.design_space(5):
        got = T.predict(part, 50.0, curve, W, tiles, 2)
        sim = _simulate(part, 50.0, curve, W, tiles, 2)
        assert got == pytest.approx(sim, abs=0.02), part


def test_interpolation_closed_forms():
    c = [(10, 3.0), (30, 7.0), (20, 4.0)]          # unsorted on purpose
    assert T.interp_latency(c, 10) == 3.0
    assert T.interp_latency(c, 15) == pytest.approx(3.5)
    assert T.interp_latency(c, 25) == pytest.approx(5.5)
    assert T.interp_latency(c, 5) == 3.0            # floor below the samples
    assert T.interp_latency(c, 40) == pytest.approx(10.0)   # last slope 0.3/byte


def test_group_bytes_partial_last_wave():
    assert T.group_bytes((1, 2, 1), 148, 512, 65536) == [148 * 65536, 296 * 65536, 68 * 65536]


def test_planted_missing_max_is_caught(monkeypatch):
    def wrong(partition, duration, curve, W, tiles, tb):
        sizes = T.group_bytes(partition, W, tiles, tb)
        tp = tm = 0.0
        for g, b in zip(partition, sizes):
            tp += duration / sum(partition) * g
            tm = tm + T.interp_latency(curve, b)     # forgot the max
        return tm
    monkeypatch.setattr(T, "predict", wrong)
    with pytest.raises(AssertionError):
        test_hand_computed_predictions()


def test_planted_previous_group_size_is_caught(monkeypatch):
    real = T.group_bytes

    def shifted(partition, W, tiles, tb):   # the garbled G_{i-1} read literally
        b = real(partition, W, tiles, tb)
        return b[-1:] + b[:-1]
    monkeypatch.setattr(T, "group_bytes", shifted)
    with pytest.raises(AssertionError):
        test_hand_computed_predictions()


# ------------------------------------------------------------ interference

GOLDEN_I = os.path.join(os.path.dirname(__file__), "golden", "tuning_interference_cases.txt")


def _interference_cases():
    rows = [l.split() for l in open(GOLDEN_I, encoding="utf-8")
            if l.strip() and not l.startswith("#")]
    preds = [(float(r[0]), float(r[1]), tuple(int(x) for x in r[2].split(",")), float(r[3]))
             for r in rows if r[0] != "best"]
    bests = [(float(r[1]), float(r[2]), float(r[3]), tuple(int(x) for x in r[4].split(",")))
             for r in rows if r[0] == "best"]
    return preds, bests


def test_hand_computed_interference():
    preds, bests = _interference_cases()
    curve = CURVES["bandwidth"]
    for sigma, rho, part, want in preds:
        got = T.predict(part, 40.0, curve, 1, 4, 1, gemm_slowdown=sigma, comm_slowdown=rho)
        assert got == pytest.approx(want), (sigma, rho, part)
    for sigma, rho, t_min, part in bests:
        got, t = T.best_partition(4, 40.0, curve, 1, 4, 1, sigma, rho)
        assert t == pytest.approx(t_min) and got == part


def test_no_interference_is_the_pages_predictor():
    """sigma = rho = 1 gives back every hand-computed case of the pages'
    loop."""
    preds, _ = _cases()
    for case, part, want in preds:
        got = T.predict(part, 40.0, CURVES[case], 1, 4, 1, gemm_slowdown=1.0,
                        comm_slowdown=1.0)
        assert got == pytest.approx(want)


def _simulate_interference(partition, duration, curve, W, tiles, tile_bytes, sigma, rho,
                           tick=0.002):
    """Tick by tick: the GEMM does duration / T of work per wave, at 1/sigma
    of a tick per tick while a communication runs; one channel sends ready
    groups in order, each needing its curve latency of work, done at 1/rho
    per tick while the GEMM runs, 1 per tick after."""
    T_ = sum(partition)
    sizes = T.group_bytes(partition, W, tiles, tile_bytes)
    ready_work, w = [], 0
    for g in partition:
        w += g
        ready_work.append(duration * w / T_)
    t, g_done, j, left, done = 0.0, 0.0, 0, None, 0.0
    while j < len(partition):
        if left is None and g_done >= ready_work[j] - 1e-9:
            left = T.interp_latency(curve, sizes[j])
        gemm_on = g_done < duration - 1e-9
        if gemm_on:
            g_done += tick / sigma if left is not None else tick
        if left is not None:
            left -= tick / rho if gemm_on else tick
            if left <= 1e-9:
                done = t + tick
                left = None
                j += 1
        t = round(t + tick, 6)
    return done


@pytest.mark.parametrize("seed", range(4))
def test_interference_matches_tick_simulation(seed):
    rng = np.random.default_rng(100 + seed)
    W, tiles = 2, 2 * 5 - 1
    # latency grows with the size (a falling curve extrapolates below zero)
    curve = list(zip(np.sort(rng.choice(np.arange(1, 30), 3, replace=False)) * 1.0,
                     np.sort(np.round(rng.uniform(1, 20, 3), 2))))
    sigma, rho = float(rng.uniform(1.0, 1.5)), float(rng.uniform(0.7, 3.0))
    for part in P.design_space(5):
        got = T.predict(part, 40.0, curve, W, tiles, 2, sigma, rho)
        sim = _simulate_interference(part, 40.0, curve, W, tiles, 2, sigma, rho)
        assert got == pytest.approx(sim, abs=0.05), part


def test_planted_slowdown_throughout_is_caught(monkeypatch):
    """A predictor that slows every wave and every communication by the
    factors, whether or not the other side runs, fails the hand-computed
    cases."""
    real = T.predict

    def always(partition, duration, curve, W, tiles, tb, gemm_slowdown=1.0,
               comm_slowdown=1.0):
        slow = [(b, t * comm_slowdown) for b, t in curve]
        return real(partition, duration * gemm_slowdown, slow, W, tiles, tb)
    monkeypatch.setattr(T, "predict", always)
    with pytest.raises(AssertionError):
        test_hand_computed_interference()


def test_planted_swapped_factors_are_caught(monkeypatch):
    """Factors applied to the wrong side fail the hand-computed cases."""
    real = T.predict

    def swapped(partition, duration, curve, W, tiles, tb, gemm_slowdown=1.0,
                comm_slowdown=1.0):
        return real(partition, duration, curve, W, tiles, tb, comm_slowdown, gemm_slowdown)
    monkeypatch.setattr(T, "predict", swapped)
    with pytest.raises(AssertionError):
        test_hand_computed_interference()
