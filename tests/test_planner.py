"""The CUDA path's host planner against the oracle, table by table,
bit-exact (no GPU: host-only plans)."""
import numpy as np
import pytest

from communication_overlap_gb300 import fo
from communication_overlap_gb300 import workloads as W
from oracle import comm as OC
from oracle import plan as OP

_LAYOUT_NAME = {fo.FO_LAYOUT_TILE: OP.LAYOUT_TILE, fo.FO_LAYOUT_RS_SUBTILE: OP.LAYOUT_RS_SUBTILE,
                fo.FO_LAYOUT_RS_ROWBLOCK: OP.LAYOUT_RS_ROWBLOCK,
                fo.FO_LAYOUT_A2A_SUBTOKEN: OP.LAYOUT_A2A}


def _oracle_places(op, layout, tok, sl):
    """Each unit's final place as the oracle's consumer and post-communication
    reorder put it: every unit of C_r carries its number + 1 in its first
    three columns (14 bits each: finite bf16 patterns, which a one-source
    fp32 sum keeps), the oracle moves the units, and the outputs are read
    back.  Place = k << 28 | row x N / 8 + first column / 8."""
    n = op.n_units
    ids = np.arange(1, n + 1, dtype=np.int64)
    C_r = np.zeros((n, op.tile_n), dtype=np.uint16)
    for c in range(3):
        C_r[:, c] = (ids >> (14 * c)) & 0x3FFF
    if layout == fo.FO_LAYOUT_TILE:
        outs = [OC.reorder_back_tile(op, OC.consume_copy(op, C_r))]
    elif layout == fo.FO_LAYOUT_A2A_SUBTOKEN:
        top_k = int(sl[tok >= 0].max()) + 1
        outs = OC.reorder_back_a2a(op, OC.consume_a2a(op, C_r), top_k,
                                   n_tokens=int(tok.max()) + 1)
    else:
        outs = OC.reorder_back_rs(op, OC.consume_rs(op, C_r, []))
    place = np.full(n, -1, dtype=np.int64)
    for k, out in enumerate(outs):
        blocks = out.reshape(out.shape[0], -1, op.tile_n).astype(np.int64)
        got = blocks[..., 0] | (blocks[..., 1] << 14) | (blocks[..., 2] << 28)
        r, c = np.nonzero(got)
        place[got[r, c] - 1] = (k << 28) | (r * (op.N // 8) + c * (op.tile_n // 8))
    return place


def _compare(expert_rows, N, K, tile_n, S, Wd, layout, R=1, tok=None, sl=None,
             partition=None, pad=False, serp=False):
    M = int(sum(expert_rows))
    grouped = tok is not None or len(expert_rows) > 1
    args = dict(M=M, N=N, K=K, tile_n=tile_n, swizzle=S, wave_width=Wd, layout=layout,
                n_dest=R, expert_rows=list(expert_rows) if grouped else None,
                row_token=tok, row_slot=sl, host_only=True, pad_expert_tile_rows=pad,
                band_order=fo.FO_BAND_SERPENTINE if serp else fo.FO_BAND_FORWARD)
    tiles, T = fo.fo_wave_count(fo.make_desc(**args))
    if partition is None:
        partition = OP.one_then_two(OP.wave_count(tiles, Wd))
    plan = fo.fo_plan_groups(fo.make_desc(**args, group_waves=partition))
    try:
        op = OP.build_plan(list(expert_rows), N, K, 128, tile_n, S, Wd, partition,
                           _LAYOUT_NAME[layout], R, tok, sl, pad_expert_tile_rows=pad,
                           serpentine=serp)
        assert (tiles, T) == (op.tiles, op.waves)
        t, waves, gt, t2s = fo.fo_plan_info(plan)
        assert (t, waves) == (op.tiles, op.waves)
        assert gt == op.group_tiles.tolist()
        assert t2s == op.tile_to_slot.tolist()
        assert fo.fo_plan_table(plan, fo.FO_TAB_SLOT_TILE) == op.slot_to_tile.tolist()
        assert fo.fo_plan_table(plan, fo.FO_TAB_SLOT_GROUP) == op.slot_group.tolist()
        unit = np.array(fo.fo_plan_table(plan, fo.FO_TAB_UNIT)).reshape(op.tiles, 128)
        assert np.array_equal(unit, op.unit)
        for which, ref in ((fo.FO_TAB_PART_START, op.part_start),
                           (fo.FO_TAB_PART_LEN, op.part_len),
                           (fo.FO_TAB_PART_DST, op.part_dst)):
            assert fo.fo_plan_table(plan, which) == ref.reshape(-1).tolist()
        assert fo.fo_plan_table(plan, fo.FO_TAB_DEST_UNITS) == \
            [OP.dest_rows(op, k) for k in range(op.part_start.shape[1])]
        live = fo.fo_plan_table(plan, fo.FO_TAB_SLOT_LIVE)
        assert live == (op.unit >= 0).any(axis=1).astype(int).tolist()
        if op.n_units * tile_n <= (1 << 26):   # the id payload stays small
            place = fo.fo_plan_table(plan, fo.FO_TAB_UNIT_PLACE)
            assert place == _oracle_places(op, layout, tok, sl).tolist()
        if layout == fo.FO_LAYOUT_A2A_SUBTOKEN:
            # output rows: every slot of every token of the rank
            n_tok, k = int(tok.max()) + 1, int(sl[tok >= 0].max()) + 1
            fr = fo.fo_plan_table(plan, fo.FO_TAB_FINAL_ROWS)
            assert fr == [len(range(d, n_tok, R)) * k for d in range(R)]
            assert fo.fo_plan_table(plan, fo.FO_TAB_DEST_CAPACITY) == \
                [f * (N // tile_n) for f in fr]
    finally:
        fo.fo_plan_destroy(plan)


def test_worked_example_tables():
    _compare([256], 512, 256, 128, 2, 2, fo.FO_LAYOUT_TILE, partition=(1, 2, 1))


@pytest.mark.parametrize("name", ["wave_pattern", "allreduce", "reducescatter"])
def test_workload_tables(name):
    w = W.WORKLOADS[name]
    _compare([w.M], w.N, w.K, w.tile_n, w.swizzle, w.wave_width, w.layout, w.n_dest)


def test_alltoall_workload_tables():
    w = W.WORKLOADS["alltoall"]
    er, tok, sl = W.routing(w)
    assert w.pad_expert_tile_rows
    _compare(er, w.N, w.K, w.tile_n, w.swizzle, w.wave_width, w.layout, w.n_dest, tok, sl,
             pad=True)
    # the same layer unpadded: the grids are exactly the GEMM's output tiles
    _compare(er, w.N, w.K, w.tile_n, w.swizzle, w.wave_width, w.layout, w.n_dest, tok, sl)


def test_rowblock_tables():
    _compare([1024], 1024, 64, 256, 3, 5, fo.FO_LAYOUT_RS_ROWBLOCK, R=4)


@pytest.mark.parametrize("rows", [[300], [128, 5, 0, 260], [1]])
def test_ragged_tile_tables(rows):
    _compare(rows, 768, 64, 256, 2, 3, fo.FO_LAYOUT_TILE)


def test_ragged_a2a_tables():
    rng = np.random.default_rng(0)
    n_tok, E, k, D = 300, 5, 2, 8
    picks = np.argsort(rng.random((n_tok, E)), axis=1)[:, :k]
    tok = np.repeat(np.arange(n_tok), k)
    sl = np.tile(np.arange(k), n_tok)
    ex = picks.reshape(-1)
    order = np.lexsort((sl, tok, ex))
    er = np.bincount(ex, minlength=E).tolist()
    _compare(er, 512, 64, 128, 3, 7, fo.FO_LAYOUT_A2A_SUBTOKEN, D, tok[order], sl[order])


@pytest.mark.parametrize("capacity", [384, 300, 200])
def test_capacity_padded_a2a_tables(capacity):
    """Experts of a fixed capacity: rows the routing leaves empty (token -1)
    get no unit; at 200 rows some routed rows are dropped, at 300 the
    capacity is not a multiple of 128."""
    w = W.scaled(W.WORKLOADS["alltoall_dynamic"], M=5 * capacity, N=768, K=64,
                 n_tokens=700, n_experts=5, capacity=capacity, wave_width=7, swizzle=3)
    er, tok, sl = W.routing(w, step=2)
    routed = (tok >= 0).sum()
    assert (routed < 700 * 2) if capacity == 200 else (routed == 700 * 2 and (tok < 0).any())
    _compare(er, w.N, w.K, w.tile_n, w.swizzle, w.wave_width, w.layout, w.n_dest, tok, sl)


def test_alltoall_dynamic_workload_tables():
    w = W.WORKLOADS["alltoall_dynamic"]
    er, tok, sl = W.routing(w)
    _compare(er, w.N, w.K, w.tile_n, w.swizzle, w.wave_width, w.layout, w.n_dest, tok, sl)


@pytest.mark.parametrize("tm,tn,S,Wd", [(3, 5, 2, 4), (4, 4, 8, 3), (5, 3, 3, 7)])
def test_every_partition_tables(tm, tn, S, Wd):
    T = OP.wave_count(tm * tn, Wd)
    for part in OP.design_space(T):
        _compare([tm * 128], tn * 128, 64, 128, S, Wd, fo.FO_LAYOUT_TILE, partition=part)
        _compare([tm * 128], tn * 128, 64, 128, S, Wd, fo.FO_LAYOUT_RS_SUBTILE, R=4,
                 partition=part)


@pytest.mark.parametrize("Wd,pad", [(6, True), (6, False), (5, True)])
def test_padded_a2a_tables(Wd, pad):
    """All-to-All with pad_expert_tile_rows: odd expert grids get an empty
    tile row (whatever W); without it the grids are the GEMM's output tiles
    (even W included).  The host planner's tables equal the oracle's."""
    rng = np.random.default_rng(3)
    n_tok, E, k, D = 150, 3, 2, 4
    picks = np.argsort(rng.random((n_tok, E)), axis=1)[:, :k]
    tok = np.repeat(np.arange(n_tok), k)
    sl = np.tile(np.arange(k), n_tok)
    ex = picks.reshape(-1)
    order = np.lexsort((sl, tok, ex))
    er = np.bincount(ex, minlength=E).tolist()
    assert any(-(-m // 128) % 2 for m in er)
    _compare(er, 512, 64, 256, 4, Wd, fo.FO_LAYOUT_A2A_SUBTOKEN, D, tok[order], sl[order],
             pad=pad)
    tiles, _ = fo.fo_wave_count(fo.make_desc(
        M=int(sum(er)), N=512, K=64, tile_n=256, swizzle=4, wave_width=Wd,
        layout=fo.FO_LAYOUT_A2A_SUBTOKEN, n_dest=D, expert_rows=er, row_token=tok[order],
        row_slot=sl[order], host_only=True, pad_expert_tile_rows=pad))
    tm = [-(-m // 128) for m in er]
    assert tiles == 2 * sum(t + (t % 2 if pad else 0) for t in tm)


def test_padding_is_an_all_to_all_option():
    """The padding of expert grids is refused for the other layouts."""
    d = fo.make_desc(M=384, N=512, K=64, tile_n=256, swizzle=2, wave_width=4,
                     group_waves=(1, 1), host_only=True, pad_expert_tile_rows=True)
    with pytest.raises(fo.FoError) as e:
        fo.fo_plan_groups(d)
    assert e.value.status == fo.FO_ERR_ARG
    with pytest.raises(ValueError):
        OP.build_plan([384], 512, 64, 128, 256, 2, 4, (1, 1), OP.LAYOUT_TILE,
                      pad_expert_tile_rows=True)


@pytest.mark.parametrize("tm,tn,S,Wd", [(5, 3, 2, 4), (4, 4, 1, 3), (7, 2, 3, 6)])
def test_serpentine_tables(tm, tn, S, Wd):
    """The serpentine band order (odd bands right to left): every table
    equals the oracle's, for every partition of a small grid, in the tile
    and ReduceScatter layouts."""
    T = OP.wave_count(tm * tn, Wd)
    for part in OP.design_space(T):
        _compare([tm * 128], tn * 128, 64, 128, S, Wd, fo.FO_LAYOUT_TILE, partition=part,
                 serp=True)
        _compare([tm * 128], tn * 128, 64, 128, S, Wd, fo.FO_LAYOUT_RS_SUBTILE, R=4,
                 partition=part, serp=True)


@pytest.mark.parametrize("pad", [False, True])
def test_serpentine_a2a_tables(pad):
    rng = np.random.default_rng(4)
    n_tok, E, k, D = 500, 4, 2, 8
    picks = np.argsort(rng.random((n_tok, E)), axis=1)[:, :k]
    tok = np.repeat(np.arange(n_tok), k)
    sl = np.tile(np.arange(k), n_tok)
    ex = picks.reshape(-1)
    order = np.lexsort((sl, tok, ex))
    er = np.bincount(ex, minlength=E).tolist()
    _compare(er, 768, 64, 256, 2, 6, fo.FO_LAYOUT_A2A_SUBTOKEN, D, tok[order], sl[order],
             pad=pad, serp=True)


@pytest.mark.parametrize("name", ["wave_pattern", "allreduce", "reducescatter"])
def test_serpentine_workload_tables(name):
    w = W.WORKLOADS[name]
    _compare([w.M], w.N, w.K, w.tile_n, w.swizzle, w.wave_width, w.layout, w.n_dest,
             serp=True)
