"""The GEMM of the path, as its plain definition (TEST INFRASTRUCTURE ONLY).

[P1] 核心设计 "计算侧": the GEMM stays one kernel and is not split or changed;
the method only observes when its output tiles finish.  So the value the
path must produce is plain C = A . B.  The oracle takes the exact values of
the bf16 inputs, accumulates the products in fp64 (numpy's matmul is the
library primitive for that step) and rounds each result once to bf16 with
round-to-nearest-even.

For the grouped (All-to-All / MoE) workload, the routed rows are stacked
expert after expert and expert e's rows are multiplied by its own B_e.
"""
import numpy as np

from .bf16 import bits_to_f64, round_to_bf16


def gemm_f64(A_bits, B_bits):
    """C = A . B in fp64 from bf16 bit arrays A [M, K], B [K, N]."""
    A = bits_to_f64(A_bits)
    B = bits_to_f64(B_bits)
    if A.shape[1] != B.shape[0]:
        raise ValueError("inner dimensions differ")
    return A @ B


def gemm_bf16(A_bits, B_bits):
    """C = A . B rounded once to bf16 (uint16 bits)."""
    return round_to_bf16(gemm_f64(A_bits, B_bits))


def grouped_gemm_bf16(A_bits, B_list, expert_rows):
    """Stacked C: rows of expert e are A[rows of e] . B_e, rounded to bf16."""
    out = []
    r0 = 0
    for e, m_e in enumerate(expert_rows):
        out.append(gemm_bf16(A_bits[r0:r0 + m_e], B_list[e]))
        r0 += m_e
    return np.concatenate(out, axis=0)


def gemm_rows_bf16(A_bits, B_list, expert_rows, rows):
    """Only the given rows of the (stacked) product, for sampled checks at
    full size.  ``rows`` index the stacked output; each uses its expert's B."""
    rows = np.asarray(rows, dtype=np.int64)
    bounds = np.cumsum([0] + list(expert_rows))
    expert = np.searchsorted(bounds, rows, side="right") - 1
    out = np.empty((len(rows), B_list[0].shape[1]), dtype=np.uint16)
    for e in np.unique(expert):
        sel = np.nonzero(expert == e)[0]
        out[sel] = gemm_bf16(A_bits[rows[sel]], B_list[e])
    return out
