"""Failure handling on the GPU without faulting it (-m gpu).

A consumer whose flags are never raised must give up after its bounded
wait, report FO_ERR_TIMEOUT in the status word and leave the context usable.
No trap, no bad address, no endless loop: the wait is a flag nothing sets.
"""
import numpy as np
import pytest
import torch

from communication_overlap_gb300 import fo
from communication_overlap_gb300 import workloads as W
from communication_overlap_gb300.pipeline import Pipeline

pytestmark = pytest.mark.gpu


def _pipe():
    w = W.scaled(W.WORKLOADS["wave_pattern"], M=256, N=512, K=128, wave_width=2)
    return Pipeline(w, W.make_inputs(w))


def test_consumer_times_out_without_gemm():
    pipe = _pipe()
    try:
        pipe.buf.flags.zero_()
        pipe.buf.status.zero_()
        torch.cuda.synchronize()
        pipe.consume(pipe.s1, epoch=12345, spin_limit_ns=2_000_000)   # 2 ms
        torch.cuda.synchronize()
        assert int(pipe.buf.status.item()) == fo.FO_ERR_TIMEOUT
        # the context still works: a normal iteration afterwards is clean
        pipe.buf.status.zero_()
        torch.cuda.synchronize()
        pipe.step()
        res = pipe.results()
        assert res["status"] == 0
        assert res["count"] == pipe.group_tiles
    finally:
        pipe.close()


def test_stale_epoch_times_out():
    """Flags left at an older epoch do not satisfy a newer wait."""
    pipe = _pipe()
    try:
        pipe.step()
        torch.cuda.synchronize()
        pipe.buf.status.zero_()
        torch.cuda.synchronize()
        pipe.consume(pipe.s1, epoch=pipe.epoch + 1, spin_limit_ns=1_000_000)
        torch.cuda.synchronize()
        assert int(pipe.buf.status.item()) == fo.FO_ERR_TIMEOUT
        assert fo.fo_plan_device_status(pipe.plan) == 0   # the GEMM never timed out
    finally:
        pipe.close()


def test_bad_arguments_launch_nothing():
    pipe = _pipe()
    try:
        with pytest.raises(fo.FoError) as e:
            fo.fo_consume_group(pipe.plan, 7, fo.FO_CONS_COPY, pipe.buf.C_r.data_ptr(), [],
                                [pipe.buf.comm[0].data_ptr()], pipe.buf.flags.data_ptr(), 1,
                                0, pipe.buf.status.data_ptr(), 0)
        assert e.value.status == fo.FO_ERR_ARG
        with pytest.raises(fo.FoError):
            fo.fo_reorder_back(pipe.plan, 1, 0, [pipe.buf.comm[0].data_ptr()],
                               [pipe.buf.final[0].data_ptr()], 0)
        with pytest.raises(fo.FoError):   # misaligned A
            fo.fo_signaled_gemm(pipe.plan, pipe.buf.A.data_ptr() + 2,
                                [pipe.buf.B[0].data_ptr()], pipe.buf.C_r.data_ptr(), 0, 0,
                                1, 0)
    finally:
        pipe.close()


def test_overlapped_reorder_waits_for_its_groups():
    """With overlap on, fo_reorder_back is the consumer's programmatic
    dependent and waits until each group it moves has been consumed.  When
    the consumer gives up (flags never raised for its epoch), the reorder's
    bounded wait runs out, the plan's status word says so, and the next
    iteration is clean."""
    pipe = _pipe()
    try:
        pipe.step()
        torch.cuda.synchronize()
        pipe.buf.status.zero_()
        torch.cuda.synchronize()
        pipe.set_overlap(True)
        pipe.consume(pipe.s1, epoch=pipe.epoch + 7, spin_limit_ns=2_000_000)
        pipe.reorder(pipe.s1)
        torch.cuda.synchronize()
        assert int(pipe.buf.status.item()) == fo.FO_ERR_TIMEOUT
        assert fo.fo_plan_device_status(pipe.plan, clear=True) == fo.FO_ERR_TIMEOUT
        pipe.buf.status.zero_()
        torch.cuda.synchronize()
        pipe.step()
        res = pipe.results()
        assert res["status"] == 0
        assert fo.fo_plan_device_status(pipe.plan) == 0
    finally:
        pipe.close()


def test_misaligned_buffers_are_argument_errors():
    """Buffers that are not 16-byte aligned (data) or 4-byte aligned
    (counters, flags, status) are refused on the host with FO_ERR_ARG,
    before any launch; the plan stays usable."""
    w = W.scaled(W.WORKLOADS["allreduce"], M=256, N=512, K=128, wave_width=2)
    inp = W.make_inputs(w)
    pipe = Pipeline(w, inp)
    try:
        b = pipe.buf
        s = pipe.s0.cuda_stream
        parts = [p.data_ptr() for p in b.partials]
        bad = [
            lambda: fo.fo_consume_group(pipe.plan, -1, fo.FO_CONS_SUM, b.C_r.data_ptr() + 2,
                                        parts, [b.comm[0].data_ptr()], b.flags.data_ptr(), 1,
                                        0, b.status.data_ptr(), s),
            lambda: fo.fo_consume_group(pipe.plan, -1, fo.FO_CONS_SUM, b.C_r.data_ptr(),
                                        parts[:-1] + [parts[-1] + 8], [b.comm[0].data_ptr()],
                                        b.flags.data_ptr(), 1, 0, b.status.data_ptr(), s),
            lambda: fo.fo_consume_group(pipe.plan, -1, fo.FO_CONS_SUM, b.C_r.data_ptr(), parts,
                                        [b.comm[0].data_ptr() + 4], b.flags.data_ptr(), 1, 0,
                                        b.status.data_ptr(), s),
            lambda: fo.fo_consume_group(pipe.plan, -1, fo.FO_CONS_SUM, b.C_r.data_ptr(), parts,
                                        [b.comm[0].data_ptr()], b.flags.data_ptr() + 2, 1, 0,
                                        b.status.data_ptr(), s),
            lambda: fo.fo_consume_reorder(pipe.plan, -1, fo.FO_CONS_SUM, b.C_r.data_ptr(), parts,
                                          None, [b.final[0].data_ptr() + 2], 0, fo.FO_ACT_NONE,
                                          b.flags.data_ptr(), 1, 0, b.status.data_ptr(), s),
            lambda: fo.fo_consume_group_noalloc(pipe.plan, -1, fo.FO_CONS_SUM,
                                                b.C_r.data_ptr() + 8, parts,
                                                [b.comm[0].data_ptr()], b.flags.data_ptr(), 1, 0,
                                                b.status.data_ptr(), s),
            lambda: fo.fo_signaled_gemm(pipe.plan, b.A.data_ptr(), [x.data_ptr() for x in b.B],
                                        b.C_r.data_ptr(), b.count.data_ptr() + 1,
                                        b.flags.data_ptr(), 1, s),
        ]
        for call in bad:
            with pytest.raises(fo.FoError) as e:
                call()
            assert e.value.status == fo.FO_ERR_ARG
        torch.cuda.synchronize()
        pipe.step(fused=True, direct=True)          # still usable
        assert pipe.results()["status"] == 0
    finally:
        pipe.close()
