"""The allocation-free consumer entry point (fo_consume_group_noalloc).

It serves callers that may not allocate device memory while they run the
overlap (graph capture, runtimes whose pool owns all device memory,
latency-critical loops): its chunk counters live in a fixed array inside
the library instead of the plan's scratch.  Its output must equal the
regular entry point's, bit for bit (the consumer's tolerance), on two calls
in a row -- once with the flags already raised and once overlapped with a
fresh GEMM launch.  Further cases: per-group calls feeding an overlapped
post-communication reorder; two plans with different group counts consumed
back to back on one stream (the second call must not start while the first
still takes chunks from the shared array); a call after one whose wait ran
out; and a plan with more groups than the array holds, refused without a
launch.

Kept in a file of its own that pytest collects last.
"""
import numpy as np
import pytest
import torch

from communication_overlap_gb300 import fo
from communication_overlap_gb300 import workloads as W
from communication_overlap_gb300.pipeline import Pipeline

pytestmark = pytest.mark.gpu

POISON = 0x7FC0


def _noalloc(pipe, epoch, stream, group=-1, spin_limit_ns=0):
    b = pipe.buf
    fo.fo_consume_group_noalloc(pipe.plan, group, pipe.kind, b.C_r.data_ptr(),
                                [p.data_ptr() for p in b.partials],
                                [c.data_ptr() for c in b.comm], b.flags.data_ptr(), epoch,
                                spin_limit_ns, b.status.data_ptr(), stream.cuda_stream)


def _outputs(pipe, final=False):
    torch.cuda.synchronize()
    bufs = pipe.buf.comm + (pipe.buf.final if final else [])
    return [c.cpu().numpy().copy() for c in bufs]


def _poison(pipe, final=False):
    for c in pipe.buf.comm + (pipe.buf.final if final else []):
        c.fill_(POISON)
    torch.cuda.synchronize()


def _same(ref, got, what):
    assert len(ref) == len(got)
    for k, (a, b) in enumerate(zip(ref, got)):
        assert np.array_equal(a, b), f"{what}: buffer {k} differs"


CASES = [
    ("allreduce", dict(M=512, N=1024, K=256, wave_width=3)),
    ("reducescatter", dict(M=1024, N=512, K=192, wave_width=5)),
]


@pytest.mark.parametrize("name,kw", CASES)
def test_noalloc_matches_regular_entry_point(name, kw):
    w = W.scaled(W.WORKLOADS[name], **kw)
    pipe = Pipeline(w, W.make_inputs(w))
    try:
        pipe.step()                       # regular path: GEMM + fo_consume_group
        ref = _outputs(pipe)
        assert int(pipe.buf.status.item()) == 0
        for call in range(2):
            _poison(pipe)                 # poison the outputs between calls
            if call == 0:                 # flags of this epoch already raised
                _noalloc(pipe, pipe.epoch, pipe.s0)
            else:                         # a fresh epoch, overlapped with the GEMM
                pipe.epoch += 1
                pipe.set_overlap(True)
                pipe.gemm(pipe.s0, pipe.epoch)
                _noalloc(pipe, pipe.epoch, pipe.s0)
            got = _outputs(pipe)
            assert int(pipe.buf.status.item()) == 0
            _same(ref, got, f"call {call}")
    finally:
        pipe.close()


def test_noalloc_per_group_calls_feed_the_overlapped_reorder():
    """Group by group, each no-alloc consume followed by an overlapped
    fo_reorder_back of that group (which waits on the consumed flags the
    consume publishes through the shared array): the same bytes as the
    regular whole-step path."""
    w = W.scaled(W.WORKLOADS["allreduce"], M=512, N=1024, K=256, wave_width=3)
    pipe = Pipeline(w, W.make_inputs(w))
    try:
        pipe.step()
        ref = _outputs(pipe, final=True)
        _poison(pipe, final=True)
        pipe.epoch += 1
        pipe.set_overlap(True)
        pipe.gemm(pipe.s0, pipe.epoch)
        for j in range(pipe.P):
            _noalloc(pipe, pipe.epoch, pipe.s0, group=j)
            pipe.reorder(pipe.s0, j, j + 1)
        got = _outputs(pipe, final=True)
        assert int(pipe.buf.status.item()) == 0
        assert fo.fo_plan_device_status(pipe.plan) == 0
        _same(ref, got, "per-group calls")
    finally:
        pipe.close()


def test_noalloc_two_plans_back_to_back_on_one_stream():
    """Two plans with different group counts: both GEMMs, then both no-alloc
    consumes issued back to back on one stream with overlap on, then again
    with the flags already raised.  Each plan's output equals its regular
    fo_consume_group output bit for bit."""
    wa = W.scaled(W.WORKLOADS["allreduce"], M=512, N=1024, K=256, wave_width=3)
    wb = W.scaled(W.WORKLOADS["wave_pattern"], M=768, N=1024, K=192, wave_width=2)
    pa = Pipeline(wa, W.make_inputs(wa))
    pb = Pipeline(wb, W.make_inputs(wb))
    try:
        assert pa.P != pb.P
        refs = []
        for p in (pa, pb):
            p.step()
            refs.append(_outputs(p))
        s = pa.s0
        for rnd in range(3):
            for p in (pa, pb):
                _poison(p)
                p.set_overlap(True)
            if rnd < 2:               # fresh epochs: both GEMMs first
                for p in (pa, pb):
                    p.epoch += 1
                    p.gemm(s, p.epoch)
            for p in (pa, pb):
                _noalloc(p, p.epoch, s)
            for p, ref in zip((pa, pb), refs):
                got = _outputs(p)
                assert int(p.buf.status.item()) == 0, (rnd, p.w.name)
                _same(ref, got, f"round {rnd}, {p.w.name}")
    finally:
        pa.close()
        pb.close()


def test_noalloc_after_a_wait_that_ran_out():
    """A no-alloc consume whose flags nothing raises gives up after its
    bounded wait and reports FO_ERR_TIMEOUT; its last CTA still resets the
    shared counters, so the next call's output is right."""
    w = W.scaled(W.WORKLOADS["allreduce"], M=512, N=1024, K=256, wave_width=3)
    pipe = Pipeline(w, W.make_inputs(w))
    try:
        pipe.step()
        ref = _outputs(pipe)
        pipe.buf.status.zero_()
        torch.cuda.synchronize()
        _noalloc(pipe, pipe.epoch + 7, pipe.s0, spin_limit_ns=2_000_000)   # 2 ms
        torch.cuda.synchronize()
        assert int(pipe.buf.status.item()) == fo.FO_ERR_TIMEOUT
        pipe.buf.status.zero_()
        _poison(pipe)
        _noalloc(pipe, pipe.epoch, pipe.s0)
        got = _outputs(pipe)
        assert int(pipe.buf.status.item()) == 0
        _same(ref, got, "after a timeout")
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
