"""The signal protocol under repetition (-m gpu).

Before every overlapped step the reordered buffer C_r is filled with a
sentinel (0xFFFF, a NaN no real output carries) and the consumer's buffers
are cleared.  A consumer that ever read a unit before the GEMM had stored it
and raised the group's flag would copy the sentinel.  Over 1000 steps per case
the consumer's and the reorder's outputs must equal, bit for bit, those of
the first step, which is checked against the oracle.  Covers the separate and
the fused kernels (with and without the communication buffers), and all
four consumers.
"""
import numpy as np
import pytest
import torch

from communication_overlap_gb300 import workloads as W
from communication_overlap_gb300.pipeline import Pipeline

from gpu_checks import check_run, fill_comm_sentinel, step_mode

pytestmark = pytest.mark.gpu

CASES = [
    ("wave_pattern", dict(M=512, N=1024, K=256, wave_width=6)),
    ("allreduce", dict(M=512, N=1024, K=256, wave_width=5)),
    ("reducescatter", dict(M=1024, N=512, K=192, wave_width=7)),
    ("alltoall", dict(M=2 * 700, N=768, K=256, n_tokens=700, n_experts=5, wave_width=9,
                      pad_expert_tile_rows=False)),
]


def _digest(tensors):
    """Per-buffer digest computed on the device: the sum and a position-
    weighted sum of the 16-bit patterns (int64), so that a changed or
    displaced element shows."""
    out = []
    for t in tensors:
        v = t.view(torch.int16).to(torch.int64).reshape(-1) & 0xFFFF
        idx = torch.arange(v.numel(), device=v.device, dtype=torch.int64) % 65521 + 1
        out.append((int(v.sum()), int((v * idx).sum())))
    return out


@pytest.mark.parametrize("fused", [False, True, "direct"])
@pytest.mark.parametrize("name,kw", CASES)
def test_repeated_overlapped_steps(name, kw, fused):
    w = W.scaled(W.WORKLOADS[name], **kw)
    inp = W.make_inputs(w)
    pipe = Pipeline(w, inp)
    try:
        reps = 1000
        sentinel = torch.full_like(pipe.buf.C_r, -1)   # 0xFFFF in every element
        first = None
        for rep in range(reps):
            pipe.buf.C_r.copy_(sentinel)
            for c in pipe.buf.comm + pipe.buf.final:
                c.zero_()
            if fused == "direct":
                fill_comm_sentinel(pipe)
            pipe.step(**step_mode(fused))
            if rep == 0:
                res = pipe.results()
                check_run(pipe, inp, res, direct=fused == "direct")
                assert not any((c == 0xFFFF).any() for c in res["comm"] + res["final"])
                first = _digest(pipe.buf.comm + pipe.buf.final)
            else:
                assert _digest(pipe.buf.comm + pipe.buf.final) == first, rep
                assert int(pipe.buf.status.item()) == 0, rep
        assert pipe.buf.count.cpu().tolist() == pipe.group_tiles
    finally:
        pipe.close()
