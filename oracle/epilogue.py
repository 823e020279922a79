"""Element-wise epilogue and the ReduceScatter -> AllGather row exchange
(TEST INFRASTRUCTURE ONLY).

Pages (see ``oracle/__init__`` for the titles):
  [P1] 五、CUTLASS 扩展实现 "Epilogue 集成": element-wise operations after a
       matrix product (ReLU, SiLU, bias addition) are usually fused into the
       kernel; FlashOverlap fuses the post-communication reorder with them,
       saving a kernel launch.
  [P1] 二 (2) ReduceScatter + AllGather: after the AllGather the row order is
       fixed by a local row exchange -- a plain block-cyclic permutation that
       needs no mapping table and fuses with element-wise operations.

Definitions taken (the pages name the operations, not their arithmetic):
  y = act(x + bias[col]) with x and bias the exact bf16 values, the addition
  and the activation in fp32, one rounding to bf16 (nearest even);
  relu(v) = v if v > 0 else 0;  silu(v) = v / (1 + exp(-v)).
"""
import numpy as np

from .bf16 import bits_to_f64, f32_round_to_bf16
from . import plan as P

ACT_NONE, ACT_RELU, ACT_SILU = 0, 1, 2


def elementwise(x_bits, bias_bits=None, act=ACT_NONE):
    """act(x + bias) over an array whose last axis is the column; bias_bits
    has one bf16 value per column (or None)."""
    v = bits_to_f64(x_bits).astype(np.float32)
    if bias_bits is not None:
        v = v + bits_to_f64(bias_bits).astype(np.float32)
    if act == ACT_RELU:
        v = np.where(v > np.float32(0), v, np.float32(0)).astype(np.float32)
    elif act == ACT_SILU:
        with np.errstate(over="ignore"):
            v = (v / (np.float32(1) + np.exp(-v))).astype(np.float32)
    elif act != ACT_NONE:
        raise ValueError(act)
    return f32_round_to_bf16(v)


def allgather_rows(p, slices):
    """The AllGather stand-in followed by the local row exchange: the R
    row-major slices ((M / R) x N each, as the post-ReduceScatter reorder
    leaves them) assembled into the M x N output in global row order.

    rs_subtile: slice k row h*tm + i is global row tile_m*tm + h*k + i
      (h = tile_m / R): a block-cyclic permutation of h-row blocks.
    rs_rowblock: slice k holds global rows k M/R .. (k+1) M/R - 1.
    """
    R = p.n_dest
    rows_per = p.M // R
    out = np.zeros((p.M, p.N), dtype=np.uint16)
    h = p.tile_m // R
    for k in range(R):
        for rho in range(rows_per):
            if p.layout == P.LAYOUT_RS_SUBTILE:
                tm, i = divmod(rho, h)
                g = p.tile_m * tm + h * k + i
            elif p.layout == P.LAYOUT_RS_ROWBLOCK:
                g = k * rows_per + rho
            else:
                raise ValueError(p.layout)
            out[g] = slices[k][rho]
    return out
