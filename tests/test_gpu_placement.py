"""Bit-exact placement of the pre-communication reorder (-m gpu).

The GEMM's epilogue stores every tile row (unit) straight to its place in
the reordered buffer C_r ([P1] 二、重排机制 "预通信重排"; 五 "Epilogue 集成").
With exact-entry inputs (entries in {-1, 0, 1}, at most 256 non-zero
columns per row of A) every output value is an exact integer, so the GPU's
raw C_r must equal, unit for unit and bit for bit, the oracle's pre-reorder
of the oracle's own GEMM -- in every layout: whole tiles, ReduceScatter
subtiles, ReduceScatter row blocks, All-to-All sub-tokens on unpadded and on
padded expert grids, a routing rebuilt on the device, and a split last wave.
The consumer and the post-communication reorder are then checked bit for
bit from the oracle's C_r, in each step variant.  At full size the same
comparison covers every unit of every workload.
"""
import numpy as np
import pytest
import torch

from communication_overlap_gb300 import fo
from communication_overlap_gb300 import workloads as W
from communication_overlap_gb300.pipeline import Pipeline

from gpu_checks import check_exact_run, exact_inputs, fill_comm_sentinel, step_mode

pytestmark = pytest.mark.gpu

MODES = [False, True, "direct"]

CASES = {
    # whole tiles, single CTAs (odd W) and CTA pairs (even W)
    "tile_single": ("allreduce", dict(M=640, N=1024, K=256, wave_width=5), {}),
    "tile_pairs": ("wave_pattern", dict(M=512, N=1024, K=192, wave_width=6), {}),
    "tile_ragged": ("wave_pattern", dict(M=300, N=768, K=128, wave_width=4, swizzle=3), {}),
    "tile_128": ("worked_example", dict(M=640, N=384, K=256, wave_width=5, uniform=False), {}),
    # a last wave of 4 tiles on W = 12, split over two CTAs per tile
    "split_single": ("wave_pattern", dict(M=512, N=1024, K=256, wave_width=12),
                     dict(gemm_variant=fo.FO_GEMM_SINGLE)),
    "split_pairs": ("wave_pattern", dict(M=512, N=1024, K=256, wave_width=12),
                    dict(gemm_variant=fo.FO_GEMM_PAIRS)),
    # ReduceScatter: subtile k of every tile to rank k; the row-block reading
    "rs_subtile": ("reducescatter", dict(M=1024, N=512, K=192, wave_width=7), {}),
    "rs_subtile_pairs": ("reducescatter", dict(M=1024, N=512, K=256, wave_width=8), {}),
    # other rank counts: 64-row subtiles (R = 2) and 16-row subtiles (R = 8)
    "rs_subtile_r2": ("reducescatter", dict(M=1024, N=512, K=128, wave_width=5, n_dest=2), {}),
    "rs_subtile_r8": ("reducescatter", dict(M=1024, N=768, K=128, wave_width=6, n_dest=8), {}),
    "rs_rowblock": ("reducescatter", dict(M=1024, N=512, K=192, wave_width=3,
                                          layout=W.LAYOUT_RS_ROWBLOCK), {}),
    # All-to-All sub-tokens: unpadded grids (odd W), padded grids as pairs
    "a2a_unpadded": ("alltoall", dict(M=2 * 700, N=768, K=256, n_tokens=700, n_experts=5,
                                      wave_width=9, pad_expert_tile_rows=False), {}),
    "a2a_unpadded_even_w": ("alltoall", dict(M=2 * 700, N=768, K=256, n_tokens=700,
                                             n_experts=5, wave_width=8,
                                             pad_expert_tile_rows=False), {}),
    "a2a_padded_pairs": ("alltoall", dict(M=2 * 700, N=768, K=256, n_tokens=700, n_experts=5,
                                          wave_width=8, pad_expert_tile_rows=True),
                         dict(gemm_variant=fo.FO_GEMM_PAIRS)),
    # the serpentine band order: odd bands walk their columns right to left
    "serp_tile_pairs": ("allreduce", dict(M=1024, N=1024, K=256, wave_width=6, swizzle=2,
                                          serpentine=True),
                        dict(gemm_variant=fo.FO_GEMM_PAIRS)),
    "serp_tile_single": ("wave_pattern", dict(M=640, N=768, K=128, wave_width=7, swizzle=2,
                                              serpentine=True), {}),
    "serp_rs_subtile": ("reducescatter", dict(M=1024, N=768, K=192, wave_width=6, swizzle=3,
                                              serpentine=True), {}),
    "serp_a2a_padded_pairs": ("alltoall", dict(M=2 * 700, N=768, K=256, n_tokens=700,
                                               n_experts=5, wave_width=8, swizzle=2,
                                               pad_expert_tile_rows=True, serpentine=True),
                              dict(gemm_variant=fo.FO_GEMM_PAIRS)),
}


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("case", list(CASES))
def test_exact_placement(case, mode):
    name, kw, pipe_kw = CASES[case]
    w = W.scaled(W.WORKLOADS[name], **kw)
    inp = exact_inputs(w)
    pipe = Pipeline(w, inp, **pipe_kw)
    try:
        if "split" in case:
            assert fo.fo_plan_set_split(pipe.plan, True) == 4
        if pipe_kw.get("gemm_variant") == fo.FO_GEMM_PAIRS:
            assert pipe.pairable
        if mode == "direct":
            fill_comm_sentinel(pipe)
        for _ in range(2):
            pipe.step(**step_mode(mode))
        check_exact_run(pipe, inp, pipe.results(), direct=mode == "direct")
        assert fo.fo_plan_device_status(pipe.plan) == 0
    finally:
        pipe.close()


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("pad,serp", [(False, False), (True, False), (True, True)])
def test_exact_placement_device_routing(mode, pad, serp):
    """A routing rebuilt on the device (fo_plan_route): the GEMM stores each
    sub-token to the place the device tables give, bit for bit as the oracle
    places it for that routing; with padded and unpadded expert grids."""
    w = W.scaled(W.WORKLOADS["alltoall_dynamic"], M=5 * 384, N=768, K=256, n_tokens=700,
                 n_experts=5, capacity=384, wave_width=8, swizzle=2,
                 pad_expert_tile_rows=pad, serpentine=serp)
    inp = exact_inputs(w)
    pipe = Pipeline(w, inp)
    try:
        for step in (1, 2):
            er, tok, sl = W.routing(w, step)
            # the same token matrix, gathered by the new routing
            X = np.zeros((w.n_tokens, w.K), dtype=np.uint16)
            win = np.zeros(w.n_tokens, dtype=np.int64)
            old = np.asarray(inp.row_token)
            X[old[old >= 0]] = inp.A[old >= 0]
            win[old[old >= 0]] = inp.window[old >= 0]
            inp.row_token, inp.row_slot, inp.expert_rows = tok, sl, er
            inp.A = W.gather_rows(X, tok)
            inp.window = np.where(tok >= 0, win[np.maximum(tok, 0)], 0)
            pipe.set_A(inp.A)
            dev = pipe.device
            pipe.route(torch.from_numpy(tok).to(dev), torch.from_numpy(sl).to(dev))
            if mode == "direct":
                fill_comm_sentinel(pipe)
            for f in pipe.buf.final:
                f.zero_()
            pipe.step(**step_mode(mode))
            check_exact_run(pipe, inp, pipe.results(), direct=mode == "direct")
    finally:
        pipe.close()


FULL = ["wave_pattern", "allreduce", "reducescatter", "alltoall", "alltoall_dynamic"]


@pytest.mark.parametrize("name", FULL)
def test_exact_placement_full_size(name):
    """Each workload at full size, in the benchmark's launch configuration
    (overlapped, the direct consumer+reorder): every unit of C_r bit for bit
    against the oracle, then the final outputs bit for bit."""
    w = W.WORKLOADS[name]
    inp = exact_inputs(w)
    pipe = Pipeline(w, inp)
    try:
        fill_comm_sentinel(pipe)
        for _ in range(2):
            pipe.step(fused=True, direct=True)
        check_exact_run(pipe, inp, pipe.results(), direct=True)
    finally:
        pipe.close()


@pytest.mark.parametrize("per_sm", [0, 1, 4])
def test_exact_placement_direct_bucket_grids(per_sm):
    """The direct All-to-All bucket at its default grid (one CTA per SM, 8
    vectors per thread in flight), at an explicit one per SM and at four per
    SM (4 vectors per thread): the same bytes, bit for bit."""
    w = W.scaled(W.WORKLOADS["alltoall"], M=2 * 700, N=768, K=256, n_tokens=700, n_experts=5,
                 wave_width=8, pad_expert_tile_rows=True)
    sm = torch.cuda.get_device_properties(0).multi_processor_count
    inp = exact_inputs(w)
    pipe = Pipeline(w, inp, consumer_ctas=per_sm * sm)
    try:
        fill_comm_sentinel(pipe)
        for _ in range(2):
            pipe.step(fused=True, direct=True)
        check_exact_run(pipe, inp, pipe.results(), direct=True)
    finally:
        pipe.close()
