"""The exact-entry inputs of the bit-exact placement tests (no GPU).

Entries of A and B are -1, 0 or 1 and every row of A has its non-zero
entries inside one window of at most 256 columns, so every value of the
product is an integer of magnitude <= 256: exact in fp32 whatever the
order of the additions, and exact in bf16.  The placement tests compute the
oracle's GEMM of such inputs window by window; here that equals the
oracle's dense product, and the values are the integers the argument says.
"""
import numpy as np
import pytest

from communication_overlap_gb300 import workloads as W
from oracle import bf16 as OB
from oracle import gemm as OG

from gpu_checks import exact_gemm_oracle, exact_inputs


@pytest.mark.parametrize("name,kw", [
    ("allreduce", dict(M=640, N=1024, K=768, wave_width=5)),
    ("reducescatter", dict(M=512, N=512, K=192, wave_width=3)),
    ("alltoall", dict(M=2 * 300, N=512, K=1024, n_tokens=300, n_experts=4, wave_width=5)),
])
def test_window_product_is_the_dense_product(name, kw):
    w = W.scaled(W.WORKLOADS[name], **kw)
    inp = exact_inputs(w)
    A = OB.bits_to_f64(inp.A)
    assert set(np.unique(A)) <= {-1.0, 0.0, 1.0}
    assert set(np.unique(OB.bits_to_f64(inp.B[0]))) == {-1.0, 0.0, 1.0}
    assert ((A != 0).sum(axis=1) <= 256).all()
    C = exact_gemm_oracle(w, inp)
    assert np.array_equal(C, OG.grouped_gemm_bf16(inp.A, inp.B, inp.expert_rows))
    v = OB.bits_to_f64(C)
    assert np.array_equal(v, np.rint(v)) and np.abs(v).max() <= 256
    # the values are spread: a unit stored in another unit's place shows
    units = C.reshape(-1, w.tile_n)
    assert len(np.unique(units, axis=0)) == len(units) - int((~units.any(axis=1)).sum()) + \
        int((~units.any(axis=1)).any())
