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
                         inp.row_token, inp.row_slot,
                         pad_expert_tile_rows=w.pad_expert_tile_rows,
                         serpentine=w.serpentine)


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


def unit_errors(got_bits, ref_bits, tile_n):
    """Relative Frobenius error of every tile-row segment (unit) of the
    compared rows: a unit stored to the wrong place shows as an error near
    1 in its own segment, however large the matrix."""
    got = OB.bits_to_f64(got_bits).reshape(got_bits.shape[0], -1, tile_n)
    ref = OB.bits_to_f64(ref_bits).reshape(ref_bits.shape[0], -1, tile_n)
    num = np.linalg.norm(got - ref, axis=2)
    den = np.maximum(np.linalg.norm(ref, axis=2), 1e-30)
    return np.where(num == 0, 0.0, num / den)


def check_signals(pipe, op, res):
    """The final counting table equals |G_j|, every flag holds the epoch and
    no wait ran out."""
    assert res["count"] == op.group_tiles.tolist(), (res["count"], op.group_tiles)
    assert res["flags"] == [pipe.epoch] * op.n_groups
    assert res["status"] == 0


def check_consumer_and_final(pipe, op, inp, C_r_src, res, direct=False):
    """The consumer's and the post-communication reorder's outputs against
    the oracle's, fed with C_r_src, bit for bit.  direct: the pass used the
    direct variant, so the communication buffers must still hold
    COMM_SENTINEL and the final buffers are checked against the oracle's
    reorder of the oracle's consumer output."""
    w = pipe.w
    if w.consumer == W.CONS_COPY:
        comm = [OC.consume_copy(op, C_r_src)]
    elif w.consumer == W.CONS_SUM:
        comm = [OC.consume_sum(op, C_r_src, inp.partials)]
    elif w.consumer == W.CONS_RS:
        comm = OC.consume_rs(op, C_r_src, inp.partials)
    else:
        comm = OC.consume_a2a(op, C_r_src)
    assert len(comm) == len(res["comm"])
    for k, (g, r) in enumerate(zip(res["comm"], comm)):
        if direct:
            assert (g == COMM_SENTINEL).all(), f"consumer buffer {k} was written"
        else:
            assert np.array_equal(g, r), f"consumer buffer {k} differs"
    if w.layout == W.LAYOUT_TILE:
        final = [OC.reorder_back_tile(op, comm[0])]
    elif w.layout in (W.LAYOUT_RS_SUBTILE, W.LAYOUT_RS_ROWBLOCK):
        final = OC.reorder_back_rs(op, comm)
    else:
        final = OC.reorder_back_a2a(op, comm, w.top_k, n_tokens=w.n_tokens)
    for k, (g, r) in enumerate(zip(res["final"], final)):
        assert np.array_equal(g, r), f"final buffer {k} differs"
    return final


def check_run(pipe, inp, res, gemm_rows=None, full_gemm=True, direct=False):
    """Every check of one GPU pass.  Returns a dict of findings; raises
    AssertionError on the first mismatch.

    The GEMM is checked through the oracle's own unit table: the GPU's C_r is
    read back into row-major C by the oracle's mapping, and C (every row, or
    the sampled gemm_rows) must be within the tolerance of the fp64 oracle,
    over the whole compared block and unit by unit (a unit stored to another
    unit's place fails its own segment).  The consumer and the reorder are
    then fed the GPU's own C_r and compared bit for bit."""
    w = pipe.w
    op = oracle_plan(w, inp, pipe.partition)
    out = {}
    check_signals(pipe, op, res)
    C_gpu = gpu_gemm_output(pipe, res, op)
    stored = token_rows(w, inp)
    if full_gemm:
        rows = np.nonzero(stored)[0]
        C_ref = OG.grouped_gemm_bf16(inp.A, inp.B, inp.expert_rows)[rows]
    else:
        rows = np.asarray(gemm_rows)
        rows = rows[stored[rows]]
        C_ref = OG.gemm_rows_bf16(inp.A, inp.B, inp.expert_rows, rows)
    frob, ok = gemm_close(C_gpu[rows], C_ref)
    out["gemm_frob"] = frob
    assert frob <= FROB_TOL and ok, f"GEMM off: frob {frob}"
    worst = unit_errors(C_gpu[rows], C_ref, w.tile_n)
    out["unit_frob_max"] = float(worst.max()) if worst.size else 0.0
    assert out["unit_frob_max"] <= FROB_TOL, f"a unit is off: {out['unit_frob_max']}"
    # the consumer and the reorder, fed the GPU's own C_r: bit-exact
    check_consumer_and_final(pipe, op, inp, res["C_r"][:op.n_units], res, direct)
    if w.layout == W.LAYOUT_TILE and w.consumer == W.CONS_COPY:
        assert np.array_equal(res["final"][0], C_gpu)
    return out


# ---------------------------------------------------------------------------
# Exact-entry inputs: A and B hold only -1, 0 and 1, and every row of A has
# its non-zero entries inside one window of at most 256 consecutive columns.
# Every product sum is then an integer of magnitude <= 256 -- exact in fp32
# (any order) and in bf16 -- so the GPU's GEMM output must equal the oracle's
# bit for bit, and so must the pre-communication reorder: the GPU's raw C_r
# is compared with the oracle's pre_reorder of the oracle's own GEMM.  The
# oracle computes each row's product from its window alone (the entries
# outside it are zero and add nothing).

EXACT_WINDOW = 256


def exact_inputs(w, seed=11):
    """Inputs of workload w with exact entries (see above); partials and the
    routing stay the workload's own."""
    inp = W.make_inputs(w)
    rng = np.random.default_rng(seed)
    win = min(EXACT_WINDOW, w.K)
    n_win = w.K // win
    # bf16 bit patterns of -1, 0 and 1, indexed by a draw from {0, 1, 2}
    table = OB.round_to_bf16(np.array([-1.0, 0.0, 1.0]))

    def draw(shape):
        return table[rng.integers(0, 3, size=shape, dtype=np.int8)]

    def rows_of(n):
        off = rng.integers(0, n_win, size=n) * win
        X = np.zeros((n, w.K), dtype=np.uint16)
        cols = off[:, None] + np.arange(win)[None, :]
        X[np.arange(n)[:, None], cols] = draw((n, win))
        return X, off

    if w.grouped:
        X, off_x = rows_of(w.n_tokens)
        tok = np.asarray(inp.row_token)
        inp.A = W.gather_rows(X, tok)
        inp.window = np.where(tok >= 0, off_x[np.maximum(tok, 0)], 0)
    else:
        inp.A, inp.window = rows_of(w.M)
    inp.B = [draw((w.K, w.N)) for _ in inp.B]
    return inp


def exact_gemm_oracle(w, inp):
    """The oracle's GEMM of exact-entry inputs, row by row from each row's
    window (rows of one expert and one window in one oracle call)."""
    win = min(EXACT_WINDOW, w.K)
    C = np.zeros((sum(inp.expert_rows), w.N), dtype=np.uint16)
    r0 = 0
    for e, m_e in enumerate(inp.expert_rows):
        rows = np.arange(r0, r0 + m_e)
        for off in np.unique(inp.window[rows]):
            sel = rows[inp.window[rows] == off]
            C[sel] = OG.gemm_bf16(inp.A[sel, off:off + win], inp.B[e][off:off + win])
        r0 += m_e
    return C


def check_exact_run(pipe, inp, res, direct=False):
    """A pass on exact-entry inputs: the counting table and flags, the GPU's
    raw C_r against the oracle's pre-reorder of the oracle's GEMM (every unit,
    bit for bit), then the consumer and the reorder bit for bit."""
    w = pipe.w
    op = oracle_plan(w, inp, pipe.partition)
    check_signals(pipe, op, res)
    C_r_ref = OC.pre_reorder(op, exact_gemm_oracle(w, inp))
    got = res["C_r"][:op.n_units]
    bad = np.nonzero((got != C_r_ref).any(axis=1))[0]
    assert bad.size == 0, f"{bad.size} of {op.n_units} units differ, first {bad[:8].tolist()}"
    check_consumer_and_final(pipe, op, inp, C_r_ref, res, direct)
    return op


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
