"""The consumer on SMs reserved for it (fo_plan_set_consumer_placement).

[P1] 四、实时调优, offline stage: the communication kernel takes some SMs and
the GEMM's waves are counted over the SMs left to it.  With the reserved
placement the consumer's CTAs may not share an SM with a CTA of the signaled
GEMM; the plan's W leaves the SMs for them.  Checked here: every output is
still the oracle's (bit for bit where the path is exact), and the consumer's
CTAs of an overlapped step ran on no more SMs than the GEMM left free (their
own %smid records).
"""
import pytest
import torch

from communication_overlap_gb300 import fo
from communication_overlap_gb300 import workloads as W
from communication_overlap_gb300.pipeline import Pipeline

from gpu_checks import check_run, fill_comm_sentinel, step_mode

pytestmark = pytest.mark.gpu

FREE_SMS = 8   # the SMs the GEMM leaves to the consumer in these cases


def _sm_count():
    return torch.cuda.get_device_properties(0).multi_processor_count


CASES = [
    ("allreduce", dict(M=2048, N=4096, K=256, n_partials=3)),          # 256 tiles, sums
    ("reducescatter", dict(M=4096, N=2048, K=256)),                      # subtile layout
    ("wave_pattern", dict(M=2048, N=4096, K=256)),                       # copy
    ("alltoall", dict(M=2 * 2048, N=2048, K=256, n_tokens=2048)),        # bucket by rank
]


def _reserved_pipe(name, kw):
    w = W.scaled(W.WORKLOADS[name], wave_width=_sm_count() - FREE_SMS, **kw)
    inp = W.make_inputs(w)
    return w, inp, Pipeline(w, inp, reserved_consumer_sms=True)


@pytest.mark.parametrize("mode", [False, True, "direct"])
@pytest.mark.parametrize("name,kw", CASES, ids=[c[0] for c in CASES])
def test_reserved_consumer_parity(name, kw, mode):
    """Overlapped steps with the consumer on reserved SMs: every output is
    the oracle's (the placement changes no arithmetic and no address)."""
    w, inp, pipe = _reserved_pipe(name, kw)
    try:
        if mode == "direct":
            fill_comm_sentinel(pipe)
        for f in pipe.buf.final:
            f.zero_()
        for _ in range(3):
            pipe.step(**step_mode(mode))
        check_run(pipe, inp, pipe.results(), direct=mode == "direct")
    finally:
        pipe.close()


@pytest.mark.parametrize("mode", [False, "direct"])
@pytest.mark.parametrize("name", ["allreduce", "alltoall"])
def test_reserved_consumer_sms(name, mode):
    """The consumer's CTAs of an overlapped step run on no more SMs than the
    GEMM leaves free.  K = 4096 keeps the GEMM's CTAs resident (one or two
    64-deep main loops each) long after the consumer, launched as its
    programmatic dependent, has placed its CTAs; the default grid is as many
    CTAs as the free SMs hold at once (at most 8 each: 2048 threads)."""
    kw = dict(CASES)[name]
    w, inp, pipe = _reserved_pipe(name, dict(kw, K=4096))
    try:
        assert pipe.tiles > w.wave_width   # every GEMM CTA holds an SM
        ctas = 8 * FREE_SMS
        trace = torch.zeros(2 * pipe.P + 4 * ctas, dtype=torch.int64, device="cuda")
        fo.fo_plan_set_trace(pipe.plan, 0, trace.data_ptr())
        for _ in range(3):
            pipe.step(**step_mode(mode))
        torch.cuda.synchronize()
        fo.fo_plan_set_trace(pipe.plan, 0, 0)
        assert int(pipe.buf.status.item()) == 0
        assert pipe.buf.count.cpu().tolist() == pipe.group_tiles
        rec = trace.cpu().numpy()[2 * pipe.P:].reshape(ctas, 4)
        ran = rec[rec[:, 2] > 0]              # the CTAs of the launch stamp their end
        assert len(ran) >= FREE_SMS
        sms = {int(x) for x in ran[:, 0]}
        assert len(sms) <= FREE_SMS, (len(sms), FREE_SMS)
    finally:
        pipe.close()


def test_reserved_placement_arguments():
    sm = _sm_count()
    w = W.scaled(W.WORKLOADS["wave_pattern"], M=2048, N=8192, K=128, wave_width=sm)
    pipe = Pipeline(w, W.make_inputs(w))
    try:
        assert pipe.tiles >= sm
        # the GEMM holds every SM: nothing to reserve
        with pytest.raises(fo.FoError):
            fo.fo_plan_set_consumer_placement(pipe.plan, fo.FO_CONSUMER_RESERVED)
        with pytest.raises(fo.FoError):
            fo.fo_plan_set_consumer_placement(pipe.plan, 7)
        fo.fo_plan_set_consumer_placement(pipe.plan, fo.FO_CONSUMER_SHARED)
    finally:
        pipe.close()
