"""Shared checks of the CUDA path against the oracle (used by -m gpu tests
and by __graft_entry__.smoke)."""
import numpy as np
import torch

from communication_overlap_gb300 import workloads as W
from communication_overlap_gb300.pipeline import Pipeline
from oracle import bf16 as OB
from oracle import comm as OC
from oracle import gemm as OG
from oracle import plan as OP

_LAYOUT = {W.LAYOUT_TILE: OP.LAYOUT_TILE, W.LAYOUT_RS_SUBTILE: OP.LAYOUT_RS_SUBTILE,
           W.LAYOUT_RS_ROWBLOCK: OP.LAYOUT_RS_ROWBLOCK, W.LAYOUT_A2A: OP.LAYOUT_A2A}

# GEMM tolerance against the fp64 oracle (fp32 accumulation, bf16 output)
FROB_TOL = 5e-3
ELEM_TOL = 2e-2


def oracle_plan(w, inp, partition):
    return OP.build_plan(inp.expert_rows, w.N, w.K, w.tile_m, w.tile_n, w.swizzle,
                         w.wave_width, partition, _LAYOUT[w.layout], w.n_dest,
                         inp.row_token, inp.row_slot)


def gemm_close(got_bits, ref_bits):
    """Relative Frobenius <= 5e-3 and |d| <= 2e-2 (1 + |ref|) per element."""
    got, ref = OB.bits_to_f64(got_bits), OB.bits_to_f64(ref_bits)
    frob = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    elem = np.abs(got - ref) <= ELEM_TOL * (1.0 + np.abs(ref))
    return frob, bool(elem.all())


def gpu_gemm_output(pipe, res, op):
    """Row-major C recovered from the GPU's C_r by the oracle's inverse map
    (independent of the GPU's own post-reorder)."""
    C = np.zeros((op.M, op.N), dtype=np.uint16)
    for s in range(op.tiles):
        rows = op.tile_rows(s)
        r0, c0 = op.tile_row0(s), op.tile_col0(s)
        u = op.unit[s, :rows]
        keep = u >= 0          # rows that hold no token are never stored
        C[r0:r0 + rows, c0:c0 + op.tile_n][keep] = res["C_r"][u[keep]]
    return C


def token_rows(w, inp):
    """Rows of the stacked GEMM output that hold a token (all of them but
    the empty capacity rows of an All-to-All routing)."""
    if inp.row_token is None:
        return np.ones(w.M, dtype=bool)
    return np.asarray(inp.row_token) >= 0


# A bf16 NaN pattern no output carries: the communication buffers hold it
# before a step of the direct variant, which must leave them untouched.
COMM_SENTINEL = 0x7FC1


def fill_comm_sentinel(pipe):
    for c in pipe.buf.comm:
        c.view(torch.int16).fill_(COMM_SENTINEL)


def step_mode(mode):
    """Pipeline.step keywords of a test mode: False (separate kernels), True
    (fused) or "direct" (fused, without communication buffers)."""
    return dict(fused=bool(mode), direct=mode == "direct")


def check_run(pipe, inp, res, gemm_rows=None, full_gemm=True, direct=False):
    """Every check of one GPU pass.  Returns a dict of findings; raises
    AssertionError on the first mismatch.  direct: the pass used the direct
    variant, so the communication buffers must still hold COMM_SENTINEL and
    the final buffers are checked against the oracle's reorder of the
    oracle's consumer output."""
    w = pipe.w
    op = oracle_plan(w, inp, pipe.partition)
    out = {}
    # counting table and flags
    assert res["count"] == op.group_tiles.tolist(), (res["count"], op.group_tiles)
    assert res["flags"] == [pipe.epoch] * op.n_groups
    assert res["status"] == 0
    # GEMM (C recovered through the oracle's map of the GPU's C_r)
    C_gpu = gpu_gemm_output(pipe, res, op)
    stored = token_rows(w, inp)
    if full_gemm:
        C_ref = OG.grouped_gemm_bf16(inp.A, inp.B, inp.expert_rows)
        frob, ok = gemm_close(C_gpu[stored], C_ref[stored])
    else:
        rows = np.asarray(gemm_rows)
        rows = rows[stored[rows]]
        C_ref = OG.gemm_rows_bf16(inp.A, inp.B, inp.expert_rows, rows)
        frob, ok = gemm_close(C_gpu[rows], C_ref)
    out["gemm_frob"] = frob
    assert frob <= FROB_TOL and ok, f"GEMM off: frob {frob}"
    # pre-comm reorder of the GPU's own output: bit-exact
    C_r_ref = OC.pre_reorder(op, C_gpu)
    assert np.array_equal(res["C_r"][:op.n_units], C_r_ref)
    # consumer, from the GPU's own C_r: bit-exact
    if w.consumer == W.CONS_COPY:
        comm = [OC.consume_copy(op, C_r_ref)]
    elif w.consumer == W.CONS_SUM:
        comm = [OC.consume_sum(op, C_r_ref, inp.partials)]
    elif w.consumer == W.CONS_RS:
        comm = OC.consume_rs(op, C_r_ref, inp.partials)
    else:
        comm = OC.consume_a2a(op, C_r_ref)
    assert len(comm) == len(res["comm"])
    for k, (g, r) in enumerate(zip(res["comm"], comm)):
        if direct:
            assert (g == COMM_SENTINEL).all(), f"consumer buffer {k} was written"
        else:
            assert np.array_equal(g, r), f"consumer buffer {k} differs"
    # post-comm reorder: bit-exact
    if w.layout == W.LAYOUT_TILE:
        final = [OC.reorder_back_tile(op, comm[0])]
    elif w.layout in (W.LAYOUT_RS_SUBTILE, W.LAYOUT_RS_ROWBLOCK):
        final = OC.reorder_back_rs(op, comm)
    else:
        final = OC.reorder_back_a2a(op, comm, w.top_k, n_tokens=w.n_tokens)
    for k, (g, r) in enumerate(zip(res["final"], final)):
        assert np.array_equal(g, r), f"final buffer {k} differs"
    if w.layout == W.LAYOUT_TILE and w.consumer == W.CONS_COPY:
        assert np.array_equal(res["final"][0], C_gpu)
    return out


def run_workload(w, inp=None, overlap=True, steps=2, fused=False, **kw):
    """fused: a test mode of step_mode."""
    inp = inp or W.make_inputs(w)
    pipe = Pipeline(w, inp, **kw)
    try:
        if fused == "direct":
            fill_comm_sentinel(pipe)
        for _ in range(steps):
            pipe.step(overlap=overlap, **step_mode(fused))
        res = pipe.results()
    except Exception:
        pipe.close()
        raise
    return pipe, inp, res
