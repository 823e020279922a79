"""Seeded random shapes through the whole path (-m gpu), against the oracle.

Each case draws a workload kind, tile width, M (ragged where the layout
allows), N, K, wave width, band height and wave-group partition, and for the
All-to-All layer the token count, experts and ranks, and the band order
(forward or serpentine), from one fixed seed;
the cases rotate through the separate kernels, the fused kernel and the
direct consumer+reorder.  Every table, reorder and consumer output must be
bit-exact, the GEMM within the tolerance, as in the hand-picked cases.
"""
import numpy as np
import pytest

from communication_overlap_gb300 import fo
from communication_overlap_gb300 import workloads as W
from communication_overlap_gb300.pipeline import Pipeline

from gpu_checks import check_run, fill_comm_sentinel, step_mode

pytestmark = pytest.mark.gpu

KINDS = ["wave_pattern", "allreduce", "reducescatter", "rowblock", "alltoall"]
MODES = [False, True, "direct"]


def _case(i):
    rng = np.random.default_rng(20261202 + i)
    kind = KINDS[i % len(KINDS)]
    tile_n = int(rng.choice([128, 256]))
    kw = dict(N=tile_n * int(rng.integers(1, 7)), K=64 * int(rng.integers(1, 9)),
              tile_n=tile_n, wave_width=int(rng.integers(1, 25)),
              swizzle=int(rng.integers(1, 10)), serpentine=bool(rng.integers(0, 2)))
    if kind in ("wave_pattern", "allreduce"):
        w = W.scaled(W.WORKLOADS[kind], M=int(rng.integers(1, 1600)), **kw)
    elif kind == "reducescatter":
        w = W.scaled(W.WORKLOADS[kind], M=128 * int(rng.integers(1, 13)), **kw)
    elif kind == "rowblock":
        w = W.scaled(W.WORKLOADS["reducescatter"], M=512 * int(rng.integers(1, 4)),
                     layout=W.LAYOUT_RS_ROWBLOCK, **kw)
    else:
        n_tok = int(rng.integers(40, 700))
        # expert grids padded to even tile-row counts when W is even (CTA
        # pairs), unpadded when it is odd
        w = W.scaled(W.WORKLOADS[kind], M=2 * n_tok, n_tokens=n_tok,
                     n_experts=int(rng.integers(2, 7)), n_dest=int(rng.choice([2, 4, 8])),
                     pad_expert_tile_rows=kw["wave_width"] % 2 == 0, **kw)
    return w, rng, MODES[i % len(MODES)]


def _partition(rng, T):
    cuts = sorted(int(c) for c in rng.choice(np.arange(1, T), size=int(rng.integers(0, T)),
                                             replace=False)) if T > 1 else []
    edges = [0] + cuts + [T]
    return [b - a for a, b in zip(edges, edges[1:])]


@pytest.mark.parametrize("i", range(60))
def test_random_shape(i):
    w, rng, mode = _case(i)
    inp = W.make_inputs(w)
    probe = fo.make_desc(M=w.M, N=w.N, K=w.K, tile_n=w.tile_n, swizzle=w.swizzle,
                         wave_width=w.wave_width, layout=w.layout, n_dest=w.n_dest,
                         expert_rows=inp.expert_rows if w.grouped else None,
                         row_token=inp.row_token, row_slot=inp.row_slot, host_only=True,
                         pad_expert_tile_rows=w.pad_expert_tile_rows,
                         band_order=fo.FO_BAND_SERPENTINE if w.serpentine else fo.FO_BAND_FORWARD)
    _, T = fo.fo_wave_count(probe)
    pipe = Pipeline(w, inp, partition=_partition(rng, T))
    try:
        if mode == "direct":
            fill_comm_sentinel(pipe)
        for _ in range(2):
            pipe.step(**step_mode(mode))
        check_run(pipe, inp, pipe.results(), direct=mode == "direct")
        assert fo.fo_plan_device_status(pipe.plan) == 0
    finally:
        pipe.close()
