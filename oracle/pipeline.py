"""One whole pass of the path on the CPU (TEST INFRASTRUCTURE ONLY).

GEMM -> pre-comm reorder -> counting table -> communication stand-in ->
post-comm reorder, in the order of [P2] Figure 5's caption and [P1] 核心设计
(see ``oracle/__init__`` for the page titles).  Every stage is timed so the
benchmark can report the oracle as a CPU baseline.
"""
from dataclasses import dataclass, field
import time

from . import plan as P
from . import comm as cm
from .gemm import grouped_gemm_bf16

CONSUMERS = ("copy", "sum", "rs", "a2a")


@dataclass
class Result:
    plan: object
    C: object = None              # stacked GEMM output, row-major bf16 bits
    C_r: object = None            # reordered buffer [units, tile_n]
    counting: list = None         # final counting table
    fired: list = None            # groups in firing order
    comm_out: object = None       # consumer output (array or list of arrays)
    final: object = None          # post-comm reorder output(s)
    seconds: dict = field(default_factory=dict)


def run(expert_rows, N, K, tile_m, tile_n, swizzle, wave_width, partition,
        layout, consumer, A, B_list, partials=(), n_dest=1, row_token=None,
        row_slot=None, top_k=2, C_given=None, pad_expert_tile_rows=False,
        serpentine=False):
    """Run the path once.  ``C_given`` may be passed to skip the GEMM stage
    (to check the later stages on a given GEMM output)."""
    res = Result(plan=None)
    t = time.perf_counter()
    p = P.build_plan(expert_rows, N, K, tile_m, tile_n, swizzle, wave_width,
                     partition, layout, n_dest, row_token, row_slot,
                     pad_expert_tile_rows=pad_expert_tile_rows, serpentine=serpentine)
    res.plan = p
    res.seconds["plan"] = time.perf_counter() - t

    t = time.perf_counter()
    res.C = grouped_gemm_bf16(A, B_list, expert_rows) if C_given is None else C_given
    res.seconds["gemm"] = time.perf_counter() - t

    t = time.perf_counter()
    res.C_r = cm.pre_reorder(p, res.C)
    snaps, fired = P.simulate_counting(p)
    res.counting = snaps[-1]
    res.fired = [j for wave in fired for j in wave]
    res.seconds["pre_reorder"] = time.perf_counter() - t

    t = time.perf_counter()
    if consumer == "copy":
        res.comm_out = cm.consume_copy(p, res.C_r)
    elif consumer == "sum":
        res.comm_out = cm.consume_sum(p, res.C_r, list(partials))
    elif consumer == "rs":
        res.comm_out = cm.consume_rs(p, res.C_r, list(partials))
    elif consumer == "a2a":
        res.comm_out = cm.consume_a2a(p, res.C_r)
    else:
        raise ValueError(consumer)
    res.seconds["consumer"] = time.perf_counter() - t

    t = time.perf_counter()
    if layout == P.LAYOUT_TILE:
        res.final = cm.reorder_back_tile(p, res.comm_out)
    elif layout in (P.LAYOUT_RS_SUBTILE, P.LAYOUT_RS_ROWBLOCK):
        res.final = cm.reorder_back_rs(p, res.comm_out)
    else:
        res.final = cm.reorder_back_a2a(p, res.comm_out, top_k)
    res.seconds["post_reorder"] = time.perf_counter() - t
    return res
