"""Degenerate and edge shapes through the whole path, against the oracle
(-m gpu): one tile, one row, more CTAs than tiles, one group per wave, one
k-block, the last-wave split at its smallest K, 128-wide tiles with CTA
pairs and the split, an expert with no rows, and a routing with no tokens."""
import numpy as np
import pytest
import torch

from communication_overlap_gb300 import fo
from communication_overlap_gb300 import workloads as W
from communication_overlap_gb300.pipeline import Pipeline

from gpu_checks import check_run, fill_comm_sentinel, run_workload, step_mode

pytestmark = pytest.mark.gpu


def _run(w, partition=None, fused=False, variant=None, **kw):
    inp = W.make_inputs(w)
    pipe = Pipeline(w, inp, partition=partition, gemm_variant=variant, **kw)
    try:
        if fused == "direct":
            fill_comm_sentinel(pipe)
        for _ in range(2):
            pipe.step(**step_mode(fused))
        res = pipe.results()
        check_run(pipe, inp, res, direct=fused == "direct")
        assert fo.fo_plan_device_status(pipe.plan) == 0
        return pipe.tiles, pipe.waves, pipe.partition
    finally:
        pipe.close()


@pytest.mark.parametrize("fused", [False, True, "direct"])
@pytest.mark.parametrize("case", [
    dict(M=128, N=256, K=64, wave_width=1),           # one tile, one k-block
    dict(M=1, N=256, K=128, wave_width=1),            # one row
    dict(M=200, N=512, K=192, wave_width=148),        # more CTAs than tiles: one wave
    dict(M=384, N=768, K=64, wave_width=2),           # K of one block: no split possible
])
def test_tiny_shapes(case, fused):
    w = W.scaled(W.WORKLOADS["wave_pattern"], swizzle=2, **case)
    _run(w, fused=fused)


def test_one_group_per_wave():
    w = W.scaled(W.WORKLOADS["allreduce"], M=512, N=1024, K=256, wave_width=3)
    tiles, T, _ = _run(w, partition=None)
    _run(w, partition=[1] * T)


@pytest.mark.parametrize("variant", [fo.FO_GEMM_SINGLE, fo.FO_GEMM_PAIRS])
def test_split_with_two_k_blocks(variant):
    """K = 128: each half of a split tile is a single k-block."""
    w = W.scaled(W.WORKLOADS["wave_pattern"], M=512, N=1024, K=128, wave_width=12)
    inp = W.make_inputs(w)
    pipe = Pipeline(w, inp, gemm_variant=variant)
    try:
        assert fo.fo_plan_set_split(pipe.plan, True) == 4
        pipe.step()
        check_run(pipe, inp, pipe.results())
    finally:
        pipe.close()


@pytest.mark.parametrize("fused", [False, True, "direct"])
def test_tile_n_128_pairs_and_split(fused):
    """128 x 128 tiles: 32 tiles on W = 20 (last wave 12, not split) and on
    W = 24 (last wave 8, split), with CTA pairs."""
    for Wd, n_split in ((20, 0), (24, 8)):
        w = W.scaled(W.WORKLOADS["wave_pattern"], M=512, N=1024, K=256, tile_n=128,
                     wave_width=Wd, swizzle=4)
        inp = W.make_inputs(w)
        pipe = Pipeline(w, inp, gemm_variant=fo.FO_GEMM_PAIRS)
        try:
            assert fo.fo_plan_set_split(pipe.plan, True) == n_split
            if fused == "direct":
                fill_comm_sentinel(pipe)
            pipe.step(**step_mode(fused))
            check_run(pipe, inp, pipe.results(), direct=fused == "direct")
        finally:
            pipe.close()


def test_a2a_expert_without_rows():
    """An expert that received no token has no tiles; the others are routed
    as usual."""
    w = W.scaled(W.WORKLOADS["alltoall"], M=2 * 300, N=512, K=128, n_tokens=300,
                 n_experts=4, wave_width=5, pad_expert_tile_rows=False)
    er, tok, sl = W.routing(w)
    # move expert 1's rows to expert 0: expert 1 ends up empty
    inp = W.make_inputs(w)
    e0, e1 = er[0], er[1]
    er2 = [e0 + e1, 0] + list(er[2:])
    inp.expert_rows = er2
    pipe = Pipeline(w, inp)
    try:
        pipe.step(fused=True)
        check_run(pipe, inp, pipe.results())
    finally:
        pipe.close()


def test_routing_with_no_tokens():
    """A routing in which every row is empty: nothing is computed, sent or
    written, every group is still signalled, and a real routing afterwards
    is exact."""
    w = W.scaled(W.WORKLOADS["alltoall_dynamic"], M=4 * 256, N=512, K=128, n_tokens=300,
                 n_experts=4, capacity=256, wave_width=5)
    inp = W.make_inputs(w)
    pipe = Pipeline(w, inp)
    try:
        empty = torch.full((w.M,), -1, dtype=torch.int32, device=pipe.device)
        zeros = torch.zeros((w.M,), dtype=torch.int32, device=pipe.device)
        for f in pipe.buf.final:
            f.zero_()
        pipe.route(empty, zeros)
        pipe.step(fused=True)
        res = pipe.results()
        assert res["status"] == 0
        assert res["count"] == pipe.group_tiles
        assert pipe.dest_units == [0] * w.n_dest
        assert set(fo.fo_plan_table(pipe.plan, fo.FO_TAB_SLOT_LIVE)) == {0}
        assert all(not f.any() for f in res["final"])
        tok = torch.from_numpy(np.asarray(inp.row_token, np.int32)).to(pipe.device)
        sl = torch.from_numpy(np.asarray(inp.row_slot, np.int32)).to(pipe.device)
        pipe.route(tok, sl)
        pipe.step(fused=True)
        check_run(pipe, inp, pipe.results())
    finally:
        pipe.close()
