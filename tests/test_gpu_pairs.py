"""The two GEMM variants on the GPU (-m gpu): one CTA per tile, and CTA
pairs sharing a tcgen05.mma.cta_group::2 (M = 256).  Both must pass every
parity check on shapes whose launch order pairs vertically adjacent tiles,
and agree with each other."""
import numpy as np
import pytest

from communication_overlap_gb300 import fo
from communication_overlap_gb300 import workloads as W

from gpu_checks import check_run, run_workload

pytestmark = pytest.mark.gpu

PAIRABLE = [
    dict(name="worked_example"),                                          # W=2, 8 tiles, BN=128
    dict(name="wave_pattern", M=512, N=1024, K=512, wave_width=6),        # 16 tiles, ragged wave
    dict(name="wave_pattern", M=1024, N=768, K=192, wave_width=4, swizzle=4),
    dict(name="worked_example", M=768, N=512, K=320, wave_width=6, swizzle=2),  # BN=128
    dict(name="allreduce", M=512, N=1024, K=448, wave_width=4),
    dict(name="reducescatter", M=1024, N=512, K=384, wave_width=8),
]


@pytest.mark.parametrize("case", PAIRABLE)
def test_pairs_match_single(case):
    case = dict(case)
    w = W.WORKLOADS[case.pop("name")]
    w = W.scaled(w, **case) if case else w
    outs = {}
    for variant in (fo.FO_GEMM_SINGLE, fo.FO_GEMM_PAIRS):
        pipe, inp, res = run_workload(w, gemm_variant=variant)
        try:
            assert pipe.pairable
            check_run(pipe, inp, res)
            outs[variant] = res["C_r"]
        finally:
            pipe.close()
    a, b = outs[fo.FO_GEMM_SINGLE].astype(np.int32), outs[fo.FO_GEMM_PAIRS].astype(np.int32)
    # both are within tolerance of the oracle; report how often they differ
    assert np.mean(a != b) < 0.01


def test_pairs_refused_when_not_pairable():
    w = W.scaled(W.WORKLOADS["wave_pattern"], M=300, N=768, K=192, wave_width=4, swizzle=3)
    with pytest.raises(fo.FoError) as e:
        run_workload(w, gemm_variant=fo.FO_GEMM_PAIRS)
    assert e.value.status == fo.FO_ERR_UNSUPPORTED
