"""Pins of the oracle's element-wise epilogue and the ReduceScatter ->
AllGather row exchange: closed forms, an independent fp64 formulation of
SiLU, and the round trip C -> slices -> gathered rows == C."""
import numpy as np
import pytest

from oracle import bf16 as B
from oracle import comm as cm
from oracle import epilogue as E
from oracle import plan as P


def _bits(v):
    return B.round_to_bf16(np.asarray(v, dtype=np.float64))


def test_relu_and_bias_closed_forms():
    x = _bits([[-1.0, 0.0, -0.0, 2.5, -3.0, 7.0]])
    assert np.array_equal(E.elementwise(x, act=E.ACT_RELU), _bits([[0, 0, 0, 2.5, 0, 7]]))
    b = _bits([1.0, 1.0, 1.0, 1.0, 4.0, -10.0])
    assert np.array_equal(E.elementwise(x, b), _bits([[0, 1, 1, 3.5, 1, -3]]))
    assert np.array_equal(E.elementwise(x, b, E.ACT_RELU), _bits([[0, 1, 1, 3.5, 1, 0]]))
    # the plain path is the identity on bf16 values
    y = _bits(np.random.default_rng(0).standard_normal((7, 9)))
    assert np.array_equal(E.elementwise(y), y)


def test_silu_against_tanh_form():
    """x * sigmoid(x) == x * (1 + tanh(x/2)) / 2, computed in fp64 here;
    the oracle's fp32 result rounded to bf16 may differ by one bf16 ulp at
    most, and only rarely."""
    x = _bits(np.linspace(-12, 12, 4001))
    got = B.bits_to_f64(E.elementwise(x, act=E.ACT_SILU))
    xv = B.bits_to_f64(x)
    ref = B.bits_to_f64(_bits(xv * (1 + np.tanh(xv / 2)) / 2))
    ulp = np.maximum(np.abs(ref), 2.0 ** -126) * 2.0 ** -7
    assert (np.abs(got - ref) <= ulp).all()
    assert np.mean(got != ref) < 0.02
    assert E.elementwise(_bits([0.0]), act=E.ACT_SILU)[0] == 0
    assert B.bits_to_f64(E.elementwise(_bits([20.0]), act=E.ACT_SILU))[0] == 20.0
    # silu(-x) = silu(x) - x
    pos = B.bits_to_f64(E.elementwise(_bits([3.0]), act=E.ACT_SILU))[0]
    neg = B.bits_to_f64(E.elementwise(_bits([-3.0]), act=E.ACT_SILU))[0]
    assert neg == pytest.approx(pos - 3.0, abs=2 ** -8 * 3)


@pytest.mark.parametrize("layout", [P.LAYOUT_RS_SUBTILE, P.LAYOUT_RS_ROWBLOCK])
def test_reducescatter_then_allgather_round_trip(layout):
    """Scattering C's tiles to R slices, reordering inside each slice and
    gathering the slices back with the row exchange returns C."""
    R = 4
    M = 8 * 128
    tiles = (M // 128) * 2
    W = 5
    p = P.build_plan([M], 512, 64, 128, 256, 2, W,
                     P.one_then_two(P.wave_count(tiles, W)), layout, R)
    C = np.random.default_rng(1).integers(0, 0x7F00, (M, 512)).astype(np.uint16)
    slices = cm.reorder_back_rs(p, cm.consume_rs(p, cm.pre_reorder(p, C), []))
    assert np.array_equal(E.allgather_rows(p, slices), C)


def test_planted_row_exchange_mistake_is_caught(monkeypatch):
    real = E.allgather_rows

    def swapped(p, slices):          # slices taken in reverse order
        return real(p, slices[::-1])
    monkeypatch.setattr(E, "allgather_rows", swapped)
    with pytest.raises(AssertionError):
        test_reducescatter_then_allgather_round_trip(P.LAYOUT_RS_SUBTILE)


def test_planted_silu_sign_mistake_is_caught(monkeypatch):
    real_exp = np.exp
    monkeypatch.setattr(E.np, "exp", lambda v: real_exp(-v))   # sigmoid of -x
    with pytest.raises(AssertionError):
        test_silu_against_tanh_form()
