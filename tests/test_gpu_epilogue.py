"""GPU parity of the fused post-communication epilogue and of the
ReduceScatter -> AllGather row exchange (-m gpu), against the oracle
applied to the GPU's own consumer output.  Bit-exact for the identity, bias
and ReLU; SiLU within one bf16 ulp (fp32 exp on two machines)."""
import numpy as np
import pytest
import torch

from communication_overlap_gb300 import fo
from communication_overlap_gb300 import workloads as W
from oracle import bf16 as OB
from oracle import comm as OC
from oracle import epilogue as OE

from gpu_checks import (COMM_SENTINEL, check_run, fill_comm_sentinel, gpu_gemm_output,
                        oracle_plan, run_workload)

pytestmark = pytest.mark.gpu

CASES = [
    dict(name="allreduce", M=512, N=1024, K=256, wave_width=4),
    dict(name="reducescatter", M=1024, N=512, K=192, wave_width=8),
    dict(name="reducescatter", M=1024, N=512, K=192, wave_width=3, layout=W.LAYOUT_RS_ROWBLOCK),
    dict(name="alltoall", M=2 * 600, N=768, K=128, n_tokens=600, n_experts=4, wave_width=7,
         pad_expert_tile_rows=False),
    dict(name="worked_example"),
]
ACTS = [(fo.FO_ACT_NONE, False), (fo.FO_ACT_RELU, True), (fo.FO_ACT_SILU, True)]


def _workload(case):
    case = dict(case)
    w = W.WORKLOADS[case.pop("name")]
    return W.scaled(w, **case) if case else w


def _close(got, want, act):
    if act != fo.FO_ACT_SILU:
        return np.array_equal(got, want)
    g, r = OB.bits_to_f64(got), OB.bits_to_f64(want)
    ulp = np.maximum(np.abs(r), 2.0 ** -126) * 2.0 ** -7
    return bool((np.abs(g - r) <= ulp).all() and np.mean(got != want) < 0.02)


def _bias(N, seed=3):
    return OB.round_to_bf16(np.random.default_rng(seed).standard_normal(N))


@pytest.mark.parametrize("case", CASES)
def test_fused_reorder_epilogue(case):
    w = _workload(case)
    pipe, inp, res = run_workload(w)
    try:
        check_run(pipe, inp, res)
        op = oracle_plan(w, inp, pipe.partition)
        bias = _bias(w.N)
        dbias = torch.from_numpy(bias.view(np.int16)).cuda()
        for act, with_bias in ACTS:
            outs = [torch.empty_like(f) for f in pipe.buf.final]
            fo.fo_reorder_back_fused(pipe.plan, 0, pipe.P, [c.data_ptr() for c in pipe.buf.comm],
                                     [o.data_ptr() for o in outs],
                                     dbias.data_ptr() if with_bias else 0, act,
                                     pipe.s0.cuda_stream)
            torch.cuda.synchronize()
            if w.layout == W.LAYOUT_TILE:
                ref = [OC.reorder_back_tile(op, res["comm"][0])]
            elif w.layout == W.LAYOUT_A2A:
                ref = OC.reorder_back_a2a(op, res["comm"], w.top_k)
            else:
                ref = OC.reorder_back_rs(op, res["comm"])
            for o, r in zip(outs, ref):
                want = OE.elementwise(r, bias if with_bias else None, act)
                got = o.cpu().numpy().view(np.uint16)
                assert _close(got, want, act), (w.name, act, with_bias)
    finally:
        pipe.close()


@pytest.mark.parametrize("case", [CASES[1], CASES[2]])
def test_allgather_row_exchange(case):
    w = _workload(case)
    pipe, inp, res = run_workload(w)
    try:
        op = oracle_plan(w, inp, pipe.partition)
        C = gpu_gemm_output(pipe, res, op)
        bias = _bias(w.N, 4)
        dbias = torch.from_numpy(bias.view(np.int16)).cuda()
        out = torch.empty((w.M, w.N), dtype=torch.int16, device="cuda")
        # the identity epilogue gathers back exactly the reduced rows
        fo.fo_allgather_rows(pipe.plan, [f.data_ptr() for f in pipe.buf.final], out.data_ptr(),
                             0, fo.FO_ACT_NONE, pipe.s0.cuda_stream)
        torch.cuda.synchronize()
        gathered = out.cpu().numpy().view(np.uint16)
        assert np.array_equal(gathered, OE.allgather_rows(op, res["final"]))
        summed = OC.consume_rs(op, OC.pre_reorder(op, C), inp.partials)
        assert np.array_equal(gathered, OE.allgather_rows(op, OC.reorder_back_rs(op, summed)))
        for act in (fo.FO_ACT_RELU, fo.FO_ACT_SILU):
            fo.fo_allgather_rows(pipe.plan, [f.data_ptr() for f in pipe.buf.final],
                                 out.data_ptr(), dbias.data_ptr(), act, pipe.s0.cuda_stream)
            torch.cuda.synchronize()
            want = OE.elementwise(OE.allgather_rows(op, res["final"]), bias, act)
            assert _close(out.cpu().numpy().view(np.uint16), want, act)
    finally:
        pipe.close()


@pytest.mark.parametrize("case", CASES)
def test_fused_consume_reorder(case):
    """One kernel for the consumer and the reorder: the same bytes in the
    communication and the final buffers as the two separate calls, with the
    GEMM running alongside; with an epilogue, the oracle's result."""
    w = _workload(case)
    pipe, inp, res = run_workload(w, steps=2)           # separate calls
    try:
        check_run(pipe, inp, res)
        for c in pipe.buf.comm + pipe.buf.final:
            c.zero_()
        torch.cuda.synchronize()
        for _ in range(2):                               # fused, overlapped, twice
            pipe.step(fused=True)
        fused = pipe.results()
        assert fused["status"] == 0
        for a, b in zip(res["comm"] + res["final"], fused["comm"] + fused["final"]):
            assert np.array_equal(a, b)
        op = oracle_plan(w, inp, pipe.partition)
        bias = _bias(w.N, 5)
        dbias = torch.from_numpy(bias.view(np.int16)).cuda()
        pipe.epoch += 1
        pipe.gemm(pipe.s0, pipe.epoch)
        pipe.consume_reorder(pipe.s0, pipe.epoch, bias=dbias.data_ptr(), act=fo.FO_ACT_SILU)
        got = pipe.results()
        assert got["status"] == 0
        for g, r in zip(got["final"], res["final"]):
            assert _close(g, OE.elementwise(r, bias, fo.FO_ACT_SILU), fo.FO_ACT_SILU)
    finally:
        pipe.close()


@pytest.mark.parametrize("case", CASES)
def test_fused_direct(case):
    """The direct variant (no communication buffers): the final buffers equal
    the oracle's reorder of the oracle's consumer output, bit for bit, and
    the communication buffers are never touched; with an epilogue, the
    oracle's element-wise result."""
    w = _workload(case)
    pipe, inp, res = run_workload(w, steps=2, fused="direct")
    try:
        check_run(pipe, inp, res, direct=True)
        bias = _bias(w.N, 6)
        dbias = torch.from_numpy(bias.view(np.int16)).cuda()
        want = [OE.elementwise(r, bias, fo.FO_ACT_RELU) for r in res["final"]]
        for f in pipe.buf.final:
            f.zero_()
        pipe.epoch += 1
        pipe.gemm(pipe.s0, pipe.epoch)
        pipe.consume_reorder(pipe.s0, pipe.epoch, bias=dbias.data_ptr(), act=fo.FO_ACT_RELU,
                             direct=True)
        got = pipe.results()
        assert got["status"] == 0
        for c in got["comm"]:
            assert (c == COMM_SENTINEL).all()
        for g, r in zip(got["final"], want):
            assert np.array_equal(g, r)
    finally:
        pipe.close()
