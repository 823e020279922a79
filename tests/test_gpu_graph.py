"""A whole step captured in a CUDA graph and replayed with one epoch (-m gpu).

The GEMM, the consumer and the reorder are captured once on the step's
stream (the consumer as the GEMM's programmatic dependent, as in a step) and
the graph is replayed with the same kernel parameters, epoch and per-launch
sequence numbers included, on new activations every time.  Every replay
must match the oracle: the flags are cleared by each launch and every
per-launch handshake (the counting table's reset, the split tiles' partial
sums, the overlapped reorder's consumed flags) is withdrawn once used, so a
replay can never pass on its predecessor's signals.
"""
from dataclasses import replace

import numpy as np
import pytest
import torch

from communication_overlap_gb300 import workloads as W
from communication_overlap_gb300.pipeline import Pipeline

from gpu_checks import check_run, fill_comm_sentinel, step_mode

pytestmark = pytest.mark.gpu

CASES = [
    # CTA pairs, 256-wide tiles, a split last wave: partials received early
    ("wave_pattern", dict(M=512, N=1024, K=256, wave_width=12), "direct"),
    # the separate kernels: the overlapped reorder waits on consumed flags
    ("wave_pattern", dict(M=512, N=1024, K=256, wave_width=12), False),
    # single CTAs (odd W), a split last wave received by the epilogue
    ("allreduce", dict(M=512, N=1024, K=256, wave_width=5), "direct"),
    ("allreduce", dict(M=512, N=1024, K=256, wave_width=5), True),
    ("reducescatter", dict(M=1024, N=512, K=192, wave_width=6), False),
    ("alltoall", dict(M=2 * 500, N=768, K=256, n_tokens=500, n_experts=4, wave_width=8),
     "direct"),
]


@pytest.mark.parametrize("name,kw,mode", CASES)
def test_graph_replays_match_the_oracle(name, kw, mode):
    w = W.scaled(W.WORKLOADS[name], **kw)
    inp = W.make_inputs(w)
    pipe = Pipeline(w, inp)
    try:
        if mode == "direct":
            fill_comm_sentinel(pipe)
        pipe.step(**step_mode(mode))      # outside the capture: one-time setup
        torch.cuda.synchronize()
        epoch = pipe.epoch + 1
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=pipe.s0):
            pipe.gemm(pipe.s0, epoch)
            if mode:
                pipe.consume_reorder(pipe.s0, epoch, direct=mode == "direct")
            else:
                pipe.consume(pipe.s0, epoch)
                pipe.reorder(pipe.s0)
        pipe.epoch = epoch
        rng = np.random.default_rng(4242)
        for _ in range(4):
            A = W.to_bf16_bits((rng.standard_normal((w.M, w.K)) / np.sqrt(w.K))
                               .astype(np.float32))
            with torch.cuda.stream(pipe.s0):
                pipe.set_A(A)
                graph.replay()
            torch.cuda.synchronize()
            check_run(pipe, replace(inp, A=A), pipe.results(), direct=mode == "direct")
    finally:
        pipe.close()
