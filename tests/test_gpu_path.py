"""GPU parity of the whole path against the CPU oracle (-m gpu).

Tables, reorders, consumer outputs and the counting table are compared
bit-exact (the reorders and consumers on the GPU's own GEMM output); the
GEMM within relative Frobenius 5e-3 and |d| <= 2e-2 (1 + |ref|) per element
against the fp64 oracle, and bit-exact where the result is exact.
"""
import numpy as np
import pytest
import torch

from communication_overlap_gb300 import fo
from communication_overlap_gb300 import workloads as W
from communication_overlap_gb300.pipeline import Pipeline
from oracle import bf16 as OB
from oracle import gemm as OG

from gpu_checks import (COMM_SENTINEL, check_run, fill_comm_sentinel, gpu_gemm_output,
                        oracle_plan, run_workload, step_mode)

pytestmark = pytest.mark.gpu


def _small(name, **kw):
    return W.scaled(W.WORKLOADS[name], **kw)


def test_worked_example_end_to_end():
    pipe, inp, res = run_workload(W.WORKLOADS["worked_example"])
    try:
        assert res["count"] == [2, 4, 2]   # the page's final counting table
        check_run(pipe, inp, res)
    finally:
        pipe.close()


@pytest.mark.parametrize("overlap", [True, False])
@pytest.mark.parametrize("case", [
    dict(name="wave_pattern", M=512, N=1024, K=512, wave_width=6),          # 16 tiles
    dict(name="wave_pattern", M=300, N=768, K=192, wave_width=4, swizzle=3),  # ragged M
    dict(name="worked_example", M=640, N=384, K=320, wave_width=5),          # BN=128
    dict(name="allreduce", M=512, N=1024, K=448, wave_width=5),
    dict(name="reducescatter", M=1024, N=512, K=384, wave_width=7),
])
def test_small_cases(case, overlap):
    case = dict(case)
    w = _small(case.pop("name"), **case)
    pipe, inp, res = run_workload(w, overlap=overlap)
    try:
        check_run(pipe, inp, res)
    finally:
        pipe.close()


def test_rowblock_layout():
    w = _small("reducescatter", M=1024, N=512, K=192, wave_width=3,
               layout=W.LAYOUT_RS_ROWBLOCK)
    pipe, inp, res = run_workload(w)
    try:
        check_run(pipe, inp, res)
    finally:
        pipe.close()


def test_small_alltoall_ragged_experts():
    w = _small("alltoall", M=2 * 700, N=768, K=256, n_tokens=700, n_experts=5,
               wave_width=9, pad_expert_tile_rows=False)
    pipe, inp, res = run_workload(w)
    try:
        assert any(m % 128 for m in inp.expert_rows)
        check_run(pipe, inp, res)
    finally:
        pipe.close()


@pytest.mark.parametrize("fused", [False, True, "direct"])
def test_alltoall_padded_grids_run_as_pairs(fused):
    """Expert grids padded to even tile-row counts (an explicit plan input)
    let the GEMM run as CTA pairs; everything matches the oracle."""
    w = _small("alltoall", M=2 * 700, N=768, K=256, n_tokens=700, n_experts=5,
               wave_width=8, pad_expert_tile_rows=True)
    inp = W.make_inputs(w)
    assert any(-(-m // 128) % 2 for m in inp.expert_rows)
    pipe = Pipeline(w, inp, gemm_variant=fo.FO_GEMM_PAIRS)
    try:
        assert pipe.pairable
        if fused == "direct":
            fill_comm_sentinel(pipe)
        for _ in range(2):
            pipe.step(**step_mode(fused))
        check_run(pipe, inp, pipe.results(), direct=fused == "direct")
    finally:
        pipe.close()


def test_gemm_exact_unit_entries_and_identity():
    """Entries in {-1, 0, 1} with K <= 256 give exact integer sums: the GPU
    result must equal the oracle bit for bit; an identity A returns B."""
    w = _small("wave_pattern", M=384, N=512, K=256, wave_width=4)
    rng = np.random.default_rng(5)
    inp = W.make_inputs(w)
    inp.A = OB.round_to_bf16(rng.integers(-1, 2, (w.M, w.K)).astype(np.float64))
    inp.B = [OB.round_to_bf16(rng.integers(-1, 2, (w.K, w.N)).astype(np.float64))]
    pipe, inp, res = run_workload(w, inp)
    try:
        op = oracle_plan(w, inp, pipe.partition)
        C = gpu_gemm_output(pipe, res, op)
        assert np.array_equal(C, OG.gemm_bf16(inp.A, inp.B[0]))
    finally:
        pipe.close()
    w2 = _small("wave_pattern", M=256, N=512, K=256, wave_width=4)
    inp2 = W.make_inputs(w2)
    inp2.A = OB.round_to_bf16(np.eye(256))
    pipe, inp2, res = run_workload(w2, inp2)
    try:
        op = oracle_plan(w2, inp2, pipe.partition)
        assert np.array_equal(gpu_gemm_output(pipe, res, op), inp2.B[0])
    finally:
        pipe.close()


def test_signals_off_and_repeat_epochs():
    """With count/flags NULL the GEMM writes the same C_r and signals
    nothing (it leaves the flags alone); with signals, every step's flags
    hold its own epoch."""
    w = _small("wave_pattern", M=512, N=1024, K=256, wave_width=6)
    inp = W.make_inputs(w)
    pipe = Pipeline(w, inp)
    try:
        for _ in range(3):
            pipe.step()
        ref = pipe.results()
        assert ref["flags"] == [3] * pipe.P
        pipe.buf.C_r.zero_()
        torch.cuda.synchronize()
        pipe.gemm(pipe.s0, 99, signal=False)
        torch.cuda.synchronize()
        res = pipe.results()
        assert np.array_equal(res["C_r"], ref["C_r"])
        assert res["flags"] == [3] * pipe.P
    finally:
        pipe.close()


def test_per_group_calls_match_whole_call():
    """Consuming and reordering group by group gives the same bytes as the
    single all-groups call; so does the direct consumer+reorder called group
    by group."""
    w = _small("allreduce", M=512, N=1024, K=256, wave_width=3)
    inp = W.make_inputs(w)
    pipe = Pipeline(w, inp)
    try:
        pipe.step()
        whole = pipe.results()
        for c in pipe.buf.comm + pipe.buf.final:
            c.zero_()
        torch.cuda.synchronize()
        e = pipe.epoch
        for j in range(pipe.P):
            pipe.consume(pipe.s1, e, group=j)
            pipe.reorder(pipe.s1, j, j + 1)
        torch.cuda.synchronize()
        parts = pipe.results()
        for a, b in zip(whole["comm"] + whole["final"], parts["comm"] + parts["final"]):
            assert np.array_equal(a, b)
        # the direct consumer+reorder, group by group (last group first)
        for f in pipe.buf.final:
            f.zero_()
        fill_comm_sentinel(pipe)
        torch.cuda.synchronize()
        for j in reversed(range(pipe.P)):
            pipe.consume_reorder(pipe.s1, e, group=j, direct=True)
        torch.cuda.synchronize()
        direct = pipe.results()
        assert direct["status"] == 0
        for a, b in zip(whole["final"], direct["final"]):
            assert np.array_equal(a, b)
        for c in direct["comm"]:
            assert (c == COMM_SENTINEL).all()
    finally:
        pipe.close()


FULL = ["wave_pattern", "allreduce", "reducescatter", "alltoall"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_workload(name):
    """Each workload at full size, overlapped: every table, reorder and
    consumer output bit-exact; the GEMM on 4096 sampled rows (every row when
    M <= 4096) against the fp64 oracle."""
    w = W.WORKLOADS[name]
    pipe, inp, res = run_workload(w, steps=3)
    try:
        rng = np.random.default_rng(123)
        rows = np.sort(rng.choice(w.M, size=min(w.M, 4096), replace=False))
        check_run(pipe, inp, res, gemm_rows=rows, full_gemm=False)
        # the direct fused variant, as the benchmark also times it: the same
        # final buffers, bit for bit, and the communication buffers untouched
        fill_comm_sentinel(pipe)
        for f in pipe.buf.final:
            f.zero_()
        for _ in range(2):
            pipe.step(fused=True, direct=True)
        got = pipe.results()
        assert got["status"] == 0
        for g, r in zip(got["final"], res["final"]):
            assert np.array_equal(g, r)
        for c in got["comm"]:
            assert (c == COMM_SENTINEL).all()
    finally:
        pipe.close()


@pytest.mark.parametrize("variant", [fo.FO_GEMM_SINGLE, fo.FO_GEMM_PAIRS])
@pytest.mark.parametrize("split", [True, False])
def test_last_wave_split(variant, split):
    """16 tiles on W = 12 CTAs: the last wave holds 4 tiles, so CTAs 0-3 and
    4-7 each compute half of K of those tiles (pairs: CTA pairs), the owners
    add the helpers' partial sums; everything matches the oracle with and
    without the split, and the counting table and flags are the same."""
    w = _small("wave_pattern", M=512, N=1024, K=512, wave_width=12)
    inp = W.make_inputs(w)
    pipe = Pipeline(w, inp, gemm_variant=variant)
    try:
        n = fo.fo_plan_set_split(pipe.plan, split)
        assert n == (4 if split else 0)
        for _ in range(3):
            pipe.step()
        res = pipe.results()
        check_run(pipe, inp, res)
        assert fo.fo_plan_device_status(pipe.plan) == 0
    finally:
        pipe.close()


def test_last_wave_split_exact_entries():
    """Entries in {-1, 0, 1} give exact sums in any order: the split tiles of
    the last wave equal the oracle bit for bit."""
    w = _small("wave_pattern", M=512, N=1024, K=256, wave_width=12)
    rng = np.random.default_rng(7)
    inp = W.make_inputs(w)
    inp.A = OB.round_to_bf16(rng.integers(-1, 2, (w.M, w.K)).astype(np.float64))
    inp.B = [OB.round_to_bf16(rng.integers(-1, 2, (w.K, w.N)).astype(np.float64))]
    pipe, inp, res = run_workload(w, inp)
    try:
        assert fo.fo_plan_set_split(pipe.plan, True) == 4
        op = oracle_plan(w, inp, pipe.partition)
        assert np.array_equal(gpu_gemm_output(pipe, res, op), OG.gemm_bf16(inp.A, inp.B[0]))
    finally:
        pipe.close()


def test_gemm_resets_the_counting_table():
    """Whatever the counting table holds before the launch, the kernel resets
    it before counting: after the step it holds |G_j| again."""
    w = _small("wave_pattern", M=512, N=1024, K=256, wave_width=6)
    inp = W.make_inputs(w)
    pipe = Pipeline(w, inp)
    try:
        for junk in (7, -3, 1 << 20):
            pipe.buf.count.fill_(junk)
            pipe.step()
            res = pipe.results()
            assert res["count"] == pipe.group_tiles
            assert res["status"] == 0
            check_run(pipe, inp, res)
    finally:
        pipe.close()


@pytest.mark.parametrize("mode", [True, "direct"])
@pytest.mark.parametrize("name,kw", [
    ("allreduce", dict(M=1024, N=1024, K=256, wave_width=6)),
    ("reducescatter", dict(M=1024, N=512, K=192, wave_width=7)),
    ("alltoall", dict(M=2 * 700, N=768, K=256, n_tokens=700, n_experts=5, wave_width=8)),
])
def test_paced_consumer(name, kw, mode):
    """fo_plan_set_pacing: with only a few consumer CTAs working while the
    GEMM runs (the rest joining at the last group's flag), every output is
    still the oracle's, bit for bit, over repeated steps."""
    w = _small(name, **kw)
    inp = W.make_inputs(w)
    pipe = Pipeline(w, inp)
    try:
        for pace in (1, 3, 40):
            fo.fo_plan_set_pacing(pipe.plan, pace)
            if mode == "direct":
                fill_comm_sentinel(pipe)
            for f in pipe.buf.final:
                f.zero_()
            for _ in range(3):
                pipe.step(**step_mode(mode))
            check_run(pipe, inp, pipe.results(), direct=mode == "direct")
        with pytest.raises(fo.FoError):
            fo.fo_plan_set_pacing(pipe.plan, -1)
    finally:
        pipe.close()
