"""The allocation-free consumer entry point (fo_consume_group_noalloc).

It serves callers that may not allocate device memory while they run the
overlap (graph capture, runtimes whose pool owns all device memory,
latency-critical loops): its chunk counters live in a fixed array inside
the library instead of the plan's scratch.  Its output must equal the
regular entry point's, bit for bit (the consumer's tolerance), on two calls
in a row -- once with the flags already raised and once overlapped with a
fresh GEMM launch -- and a plan with more groups than the array holds is
refused without a launch.

Kept in a file of its own that pytest collects last.
"""
import numpy as np
import pytest
import torch

from communication_overlap_gb300 import fo
from communication_overlap_gb300 import workloads as W
from communication_overlap_gb300.pipeline import Pipeline

pytestmark = pytest.mark.gpu


def _noalloc(pipe, epoch, stream):
    b = pipe.buf
    fo.fo_consume_group_noalloc(pipe.plan, -1, pipe.kind, b.C_r.data_ptr(),
                                [p.data_ptr() for p in b.partials],
                                [c.data_ptr() for c in b.comm], b.flags.data_ptr(), epoch, 0,
                                b.status.data_ptr(), stream.cuda_stream)


def _comm(pipe):
    torch.cuda.synchronize()
    return [c.cpu().numpy().copy() for c in pipe.buf.comm]


@pytest.mark.parametrize("name,kw", [
    ("allreduce", dict(M=512, N=1024, K=256, wave_width=3)),
    ("reducescatter", dict(M=1024, N=512, K=192, wave_width=5)),
])
def test_noalloc_matches_regular_entry_point(name, kw):
    w = W.scaled(W.WORKLOADS[name], **kw)
    pipe = Pipeline(w, W.make_inputs(w))
    try:
        pipe.step()                       # regular path: GEMM + fo_consume_group
        ref = _comm(pipe)
        assert int(pipe.buf.status.item()) == 0
        for call in range(2):
            for c in pipe.buf.comm:
                c.fill_(0x7FC0)           # poison the outputs between calls
            torch.cuda.synchronize()
            if call == 0:                 # flags of this epoch already raised
                _noalloc(pipe, pipe.epoch, pipe.s0)
            else:                         # a fresh epoch, overlapped with the GEMM
                pipe.epoch += 1
                pipe.set_overlap(True)
                pipe.gemm(pipe.s0, pipe.epoch)
                _noalloc(pipe, pipe.epoch, pipe.s0)
            got = _comm(pipe)
            assert int(pipe.buf.status.item()) == 0
            for a, b in zip(ref, got):
                assert np.array_equal(a, b), f"call {call} differs"
    finally:
        pipe.close()


def test_noalloc_refuses_too_many_groups():
    n = fo.FO_NOALLOC_MAX_GROUPS + 1      # one wave per group, one tile per wave
    desc = fo.make_desc(M=128 * n, N=128, K=64, tile_n=128, swizzle=1, wave_width=1,
                        group_waves=[1] * n)
    plan = fo.fo_plan_groups(desc)
    try:
        buf = torch.zeros(16, dtype=torch.int32, device="cuda")
        with pytest.raises(fo.FoError) as e:
            fo.fo_consume_group_noalloc(plan, -1, fo.FO_CONS_COPY, buf.data_ptr(), [],
                                        [buf.data_ptr()], buf.data_ptr(), 1, 0,
                                        buf.data_ptr(), 0)
        assert e.value.status == fo.FO_ERR_ARG
    finally:
        fo.fo_plan_destroy(plan)
