"""Offline measurements and the predictive search on the GPU (-m gpu):
the sampled latency curve is positive and grows with the group size, the
tuned partition is valid, and re-planning keeps the path bit-exact."""
import pytest
import torch

from communication_overlap_gb300 import fo
from communication_overlap_gb300 import workloads as W
from communication_overlap_gb300.tuning import Tuner

from gpu_checks import check_run

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("kernels", ["direct", "separate"])
def test_tuner_small_allreduce(kernels):
    w = W.scaled(W.WORKLOADS["allreduce"], M=1024, N=2048, K=256, wave_width=8)
    t = Tuner(w, reps=3, kernels=kernels)
    try:
        gemm = t.gemm_us()
        curve = t.curve()
        assert gemm > 0 and len(curve) == t.pipe.waves
        assert all(us > 0 for _, us in curve)
        assert curve[-1][1] > curve[0][1]          # more bytes take longer
        parts, pred = fo.fo_tune_partition(t.desc(), gemm, curve)
        assert sum(parts) == t.pipe.waves and pred >= gemm
        t.pipe.replan(parts)
        t.pipe.step()
        res = t.pipe.results()
        check_run(t.pipe, t.inp, res)
    finally:
        t.close()


def test_interference_factors_and_tuned_partition():
    """The measured interference factors are finite and at least 1; the
    search with them returns a valid partition whose step is exact."""
    w = W.scaled(W.WORKLOADS["allreduce"], M=1024, N=2048, K=256, wave_width=8)
    t = Tuner(w, reps=3)
    try:
        gemm = t.gemm_us()
        curve = t.curve()
        sigma, rho = t.interference(gemm, reps=3)
        assert 0.9 <= sigma < 10.0 and 0.25 <= rho <= 8.0
        parts, pred = fo.fo_tune_partition(t.desc(), gemm, curve, sigma, rho)
        plain = fo.fo_predict_partition(t.desc(parts), gemm, curve)
        assert sum(parts) == t.pipe.waves and pred > 0
        t.pipe.replan(parts)
        t.pipe.step()
        check_run(t.pipe, t.inp, t.pipe.results())
    finally:
        t.close()


def test_curve_in_one_launch():
    """The latency curve measured inside one persistent consumer launch:
    positive, growing with the group size, and below the curve of one
    launch per group (no launch or ramp-up per group)."""
    w = W.scaled(W.WORKLOADS["allreduce"], M=2048, N=2048, K=256, wave_width=4)
    t = Tuner(w, reps=3)
    try:
        alone = dict(t.curve())
        inl = t.curve_in_launch()
        assert len(inl) >= 2 and all(us > 0 for _, us in inl)
        assert inl[-1][1] > inl[0][1]
        b0, us0 = inl[0]
        assert us0 < alone[b0]
    finally:
        t.close()
