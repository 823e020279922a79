"""Routing tables built on the device (fo_plan_route) against the host
planner and the oracle, and the whole path run on routings that never went
through the host (-m gpu).

Expert capacities are fixed, so the GEMM shape, tiles, waves and groups
never change; each step brings a new assignment of tokens to rows, empty
rows included.  The tables the device builds must equal, bit for bit, those
the host planner and the oracle build from the same routing, and every
output of the step must match the oracle's for that routing.
"""
from dataclasses import replace

import numpy as np
import pytest
import torch

from communication_overlap_gb300 import fo
from communication_overlap_gb300 import workloads as W
from communication_overlap_gb300.pipeline import Pipeline

from gpu_checks import check_run, fill_comm_sentinel, oracle_plan, step_mode

pytestmark = pytest.mark.gpu

_TABLES = (fo.FO_TAB_UNIT, fo.FO_TAB_PART_START, fo.FO_TAB_PART_LEN, fo.FO_TAB_PART_DST,
           fo.FO_TAB_DEST_UNITS, fo.FO_TAB_FINAL_ROWS, fo.FO_TAB_DEST_CAPACITY,
           fo.FO_TAB_SLOT_LIVE, fo.FO_TAB_UNIT_PLACE)


def _small(capacity=384, **kw):
    args = dict(M=5 * capacity, N=768, K=256, n_tokens=700, n_experts=5,
                capacity=capacity, wave_width=7, swizzle=3)
    args.update(kw)
    return W.scaled(W.WORKLOADS["alltoall_dynamic"], **args)


def _inputs_for_step(w, base, step):
    """The step's routing and its routed A (the dispatch gather of the token
    matrix), with the same B."""
    er, tok, sl = W.routing(w, step)
    return replace(base, A=W.gather_rows(W.token_matrix(w), tok), expert_rows=er,
                   row_token=tok, row_slot=sl)


def _host_tables(w, inp, partition):
    desc = fo.make_desc(M=w.M, N=w.N, K=w.K, tile_n=w.tile_n, swizzle=w.swizzle,
                        wave_width=w.wave_width, group_waves=partition, layout=w.layout,
                        n_dest=w.n_dest, expert_rows=inp.expert_rows,
                        row_token=inp.row_token, row_slot=inp.row_slot, host_only=True,
                        pad_expert_tile_rows=w.pad_expert_tile_rows,
                        band_order=fo.FO_BAND_SERPENTINE if w.serpentine else fo.FO_BAND_FORWARD)
    plan = fo.fo_plan_groups(desc)
    try:
        return {t: fo.fo_plan_table(plan, t) for t in _TABLES}
    finally:
        fo.fo_plan_destroy(plan)


def _route(pipe, inp):
    dev = pipe.device
    tok = torch.from_numpy(np.asarray(inp.row_token, np.int32)).to(dev)
    sl = torch.from_numpy(np.asarray(inp.row_slot, np.int32)).to(dev)
    pipe.route(tok, sl)


@pytest.mark.parametrize("capacity,wave_width", [(384, 7), (300, 7), (200, 7), (300, 8)])
def test_device_tables_equal_host_tables(capacity, wave_width):
    """(300 rows = 3 tile rows per expert: with W = 8 each expert's grid is
    padded with an empty tile row, which the routing kernels count too.)"""
    w = _small(capacity, wave_width=wave_width)
    base = W.make_inputs(w)
    pipe = Pipeline(w, base)
    try:
        for step in (1, 2):
            inp = _inputs_for_step(w, base, step)
            _route(pipe, inp)
            torch.cuda.synchronize()
            assert int(pipe.buf.status.item()) == 0
            got = {t: fo.fo_plan_table(pipe.plan, t) for t in _TABLES}
            # the final sizes follow the workload's token count, which the
            # host planner reads off the routing: equal when every token is in
            want = _host_tables(w, inp, pipe.partition)
            n_tok = int(np.max(inp.row_token)) + 1
            for t in _TABLES:
                if t in (fo.FO_TAB_FINAL_ROWS, fo.FO_TAB_DEST_CAPACITY) and n_tok != w.n_tokens:
                    continue
                assert got[t] == want[t], t
            op = oracle_plan(w, inp, pipe.partition)
            unit = np.array(got[fo.FO_TAB_UNIT]).reshape(op.tiles, 128)
            assert np.array_equal(unit, op.unit)
            assert got[fo.FO_TAB_PART_LEN] == op.part_len.reshape(-1).tolist()
    finally:
        pipe.close()


@pytest.mark.parametrize("fused,wave_width", [(False, 7), (True, 7), (True, 8), ("direct", 8)])
def test_steps_on_device_routings_match_oracle(fused, wave_width):
    """Three steps, each on a routing handed over in device memory; after
    each, every table, the reorders and the consumer match the oracle for
    that step's routing, bit for bit (W = 8: padded grids, CTA pairs)."""
    w = _small(300 if wave_width == 8 else 384, wave_width=wave_width)
    base = W.make_inputs(w)
    pipe = Pipeline(w, base)
    try:
        for step in (1, 2, 3):
            inp = _inputs_for_step(w, base, step)
            pipe.set_A(inp.A)
            for f in pipe.buf.final:
                f.zero_()
            _route(pipe, inp)
            if fused == "direct":
                fill_comm_sentinel(pipe)
            pipe.step(**step_mode(fused))
            res = pipe.results()
            check_run(pipe, inp, res, direct=fused == "direct")
    finally:
        pipe.close()


def test_dropped_tokens_and_ragged_capacity():
    w = _small(200)   # below the mean load: the router drops rows
    base = W.make_inputs(w)
    pipe = Pipeline(w, base)
    try:
        inp = _inputs_for_step(w, base, 4)
        pipe.set_A(inp.A)
        for f in pipe.buf.final:
            f.zero_()
        _route(pipe, inp)
        pipe.step()
        check_run(pipe, inp, pipe.results())
    finally:
        pipe.close()


@pytest.mark.parametrize("bad", ["token", "slot", "duplicate"])
def test_invalid_routing_routes_nothing(bad):
    """A routing with a token or slot out of range, or a (token, slot) pair
    twice, sets FO_ERR_ARG and leaves a plan that sends no row; a valid
    routing afterwards works again."""
    w = _small(384)
    base = W.make_inputs(w)
    pipe = Pipeline(w, base)
    try:
        inp = _inputs_for_step(w, base, 1)
        tok, sl = np.array(inp.row_token), np.array(inp.row_slot)
        if bad == "token":
            tok[5] = w.n_tokens
        elif bad == "slot":
            sl[7] = w.top_k
        else:   # give every empty row the pair (token 0, slot 0)
            tok[tok < 0] = 0
            sl[tok == 0] = 0
        pipe.buf.status.zero_()
        _route(pipe, replace(inp, row_token=tok, row_slot=sl))
        pipe.step()
        res = pipe.results()
        assert res["status"] == fo.FO_ERR_ARG
        assert pipe.dest_units == [0] * w.n_dest
        assert set(fo.fo_plan_table(pipe.plan, fo.FO_TAB_UNIT)) == {-1}
        assert set(fo.fo_plan_table(pipe.plan, fo.FO_TAB_SLOT_LIVE)) == {0}   # GEMM skips all
        assert res["count"] == pipe.group_tiles      # the GEMM still signals every group
        # recovery
        pipe.buf.status.zero_()
        pipe.set_A(inp.A)
        for f in pipe.buf.final:
            f.zero_()
        _route(pipe, inp)
        pipe.step()
        check_run(pipe, inp, pipe.results())
    finally:
        pipe.close()


def test_full_size_dynamic_alltoall():
    """The 8 x 5120-row capacity layer at full size: two device routings,
    the first with the separate kernels, the second with the direct
    consumer+reorder the benchmark's step runs; every table and data
    movement bit-exact, the GEMM on 2048 sampled rows."""
    w = W.WORKLOADS["alltoall_dynamic"]
    base = W.make_inputs(w)
    pipe = Pipeline(w, base)
    try:
        rng = np.random.default_rng(321)
        for step, mode in ((1, False), (2, "direct")):
            inp = _inputs_for_step(w, base, step)
            pipe.set_A(inp.A)
            for f in pipe.buf.final:
                f.zero_()
            _route(pipe, inp)
            if mode == "direct":
                fill_comm_sentinel(pipe)
            pipe.step(**step_mode(mode))
            res = pipe.results()
            rows = np.sort(rng.choice(w.M, size=2048, replace=False))
            check_run(pipe, inp, res, gemm_rows=rows, full_gemm=False, direct=mode == "direct")
    finally:
        pipe.close()


@pytest.mark.parametrize("variant", [fo.FO_GEMM_SINGLE, fo.FO_GEMM_PAIRS])
def test_empty_tiles_are_skipped_but_counted(variant):
    """Capacity far above the load leaves whole tiles empty: the GEMM skips
    their mainloop (single CTAs: each empty tile; pairs: both tiles of a pair
    empty), still counts them, and every output matches the oracle."""
    w = _small(768, M=5 * 768, wave_width=8, swizzle=4)
    base = W.make_inputs(w)
    pipe = Pipeline(w, base, gemm_variant=variant)
    try:
        live = fo.fo_plan_table(pipe.plan, fo.FO_TAB_SLOT_LIVE)
        assert 0 in live and 1 in live
        if variant == fo.FO_GEMM_PAIRS:
            assert pipe.pairable
        for step in (1, 2):
            inp = _inputs_for_step(w, base, step)
            pipe.set_A(inp.A)
            for f in pipe.buf.final:
                f.zero_()
            _route(pipe, inp)
            pipe.step()
            res = pipe.results()
            assert res["count"] == pipe.group_tiles
            check_run(pipe, inp, res)
    finally:
        pipe.close()


@pytest.mark.parametrize("wave_width", [7, 8])
def test_many_steps_cycling_device_routings(wave_width):
    """As the benchmark runs the dynamic layer: four routings resident in
    device memory, taken in turn for 60 overlapped steps of the direct
    consumer+reorder, each step routed on the device first.  The first time
    a routing comes up its outputs are checked against the oracle; every
    later step on it must give the same final bytes (device digests), with
    the communication buffers never written.  (W = 8: padded grids, CTA
    pairs.)"""
    w = _small(300, wave_width=wave_width)
    base = W.make_inputs(w)
    pipe = Pipeline(w, base)
    try:
        dev = pipe.device
        routes = []
        for k in range(1, 5):
            inp = _inputs_for_step(w, base, k)
            routes.append((inp,
                           torch.from_numpy(np.asarray(inp.row_token, np.int32)).to(dev),
                           torch.from_numpy(np.asarray(inp.row_slot, np.int32)).to(dev),
                           torch.from_numpy(inp.A.view(np.int16)).to(dev)))
        fill_comm_sentinel(pipe)
        first = {}
        for step in range(60):
            k = step % len(routes)
            inp, tok, sl, A = routes[k]
            pipe.buf.A = A
            for f in pipe.buf.final:
                f.zero_()
            pipe.route(tok, sl)
            pipe.step(fused=True, direct=True)
            digest = [(int(f.view(torch.int16).to(torch.int64).sum()),
                       int((f.view(torch.int16).to(torch.int64).reshape(-1) *
                            (torch.arange(f.numel(), device=dev) % 65521 + 1)).sum()))
                      for f in pipe.buf.final]
            if k not in first:
                check_run(pipe, inp, pipe.results(), direct=True)
                first[k] = digest
            else:
                assert digest == first[k], step
                assert int(pipe.buf.status.item()) == 0, step
    finally:
        pipe.close()
