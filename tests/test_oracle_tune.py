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
