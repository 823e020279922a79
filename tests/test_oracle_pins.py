"""Pins of the CPU oracle against what the pages and mathematics fix.

Every check here is independent of the oracle's own code path: printed
values from the pages (tests/golden, each with its citation), closed forms,
brute force on tiny inputs, and an independent library conversion (torch)
for bf16 rounding.  No GPU.
"""
import itertools
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import bf16 as B
from oracle import plan as P
from oracle import comm as cm
from oracle import gemm as G
from oracle import pipeline

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _lines(name):
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        return [l.split() for l in f if l.strip() and not l.startswith("#")]


# ---------------------------------------------------------------- bf16

def _torch_bf16(x32):
    return (torch.from_numpy(np.asarray(x32, np.float32)).to(torch.bfloat16)
            .view(torch.int16).numpy().view(np.uint16))


def test_bf16_matches_torch_on_random_fp32():
    rng = np.random.default_rng(0)
    mant = rng.uniform(1, 2, 200000)
    expo = rng.integers(-140, 128, 200000)
    x = (mant * np.exp2(expo.astype(np.float64))).astype(np.float32)
    x *= np.where(rng.random(200000) < 0.5, -1, 1).astype(np.float32)
    assert np.array_equal(B.f32_round_to_bf16(x), _torch_bf16(x))


def test_bf16_ties_subnormals_overflow_signed_zero():
    # exact halfway cases between neighbouring bf16 values: ties go to even
    base = np.arange(0x3F80, 0x3F90, dtype=np.uint32) << 16
    ties = (base | 0x8000).view(np.float32)
    special = np.array([0.0, -0.0, np.inf, -np.inf, 1e-45, -1e-45, 3e-39,
                        3.3895314e38, 3.3961775e38, 3.4028235e38,
                        np.float32(2 ** -133), np.float32(1.5 * 2 ** -133)],
                       dtype=np.float32)
    x = np.concatenate([ties, special])
    assert np.array_equal(B.f32_round_to_bf16(x), _torch_bf16(x))
    # signed zero keeps its sign
    assert B.round_to_bf16(np.array([-0.0]))[0] == 0x8000


def test_bf16_fp64_is_nearest_by_brute_force():
    """fp64 values (sums of the GEMM) round to the nearest bf16, ties to even,
    checked against an enumeration of all finite positive bf16 values."""
    allbits = np.arange(0x0000, 0x7F80, dtype=np.uint16)
    vals = B.bits_to_f64(allbits)
    rng = np.random.default_rng(1)
    x = rng.uniform(-4, 4, 5000) * np.exp2(rng.integers(-20, 20, 5000))
    got = B.round_to_bf16(x)
    for xi, gi in zip(x, got):
        a = abs(xi)
        i = np.searchsorted(vals, a)
        cands = [c for c in (i - 1, i) if 0 <= c < len(vals)]
        d = [abs(vals[c] - a) for c in cands]
        best = [c for c, dc in zip(cands, d) if dc == min(d)]
        if len(best) > 1:   # tie: even fraction bit pattern
            best = [c for c in best if allbits[c] % 2 == 0]
        want = allbits[best[0]] | (0x8000 if xi < 0 else 0)
        assert gi == want


# ---------------------------------------------------------------- plan pins

def test_worked_example_counting_table():
    rows = _lines("worked_example_counting.txt")
    want_sizes = [int(v) for v in rows[0][1:]]
    p = P.build_plan([256], 512, 256, 128, 128, 2, 2, (1, 2, 1), P.LAYOUT_TILE)
    assert p.tiles == 8 and p.waves == 4
    assert list(p.group_tiles) == want_sizes
    snaps, fired = P.simulate_counting(p)
    for w, line in enumerate(rows[1:]):
        assert int(line[1]) == w + 1
        table = [int(v) for v in line[3:6]]
        assert snaps[w] == table
        fires = [] if line[7] == "-" else [int(v) - 1 for v in line[7].split(",")]
        assert fired[w] == fires
    assert snaps[-1] == want_sizes


def test_wave_counts_and_design_space_from_pages():
    for line in _lines("wave_counts.txt"):
        if line[0] == "waves":
            M, N, tm, tn, sms, want = map(int, line[1:])
            tiles = (M // tm) * (N // tn)
            assert P.wave_count(tiles, sms) == want
        elif line[0] == "space":
            T, count = int(line[1]), int(line[2])
            space = P.design_space(T)
            assert len(space) == count == 2 ** (T - 1)
            assert len(set(space)) == count
            for member in line[3:]:
                assert tuple(int(v) for v in member.split(",")) in space


def test_mapping_illustration_convention():
    """The mapping table sends a tile to its contiguous reordered index and the
    inverse sends an index back to its tile; each tile moves as one block."""
    rows = {r[0]: r[1:] for r in _lines("mapping_illustration.txt")}
    order = [int(v) for v in rows["order"]]
    want_map = dict(tuple(map(int, kv.split(":"))) for kv in rows["map"])
    want_inv = dict(tuple(map(int, kv.split(":"))) for kv in rows["inverse"])
    # a 1 x 4 grid whose tiles are dispatched in that order, one wave
    p = P.build_plan([128], 4 * 128, 64, 128, 128, 1, 4, (1,), P.LAYOUT_TILE)
    p.slot_tile = [(0, 0, t) for t in order]
    p.slot_to_tile = np.array(order)
    p.tile_to_slot = np.argsort(p.slot_to_tile)
    P._assign_units(p)
    assert {t: int(p.tile_to_slot[t]) for t in range(4)} == want_map
    assert {s: int(p.slot_to_tile[s]) for s in range(4)} == want_inv
    C = np.arange(128 * 512, dtype=np.uint16).reshape(128, 512)
    C_r = cm.pre_reorder(p, C).reshape(4, 128, 128)
    for idx, t in want_inv.items():
        assert np.array_equal(C_r[idx], C[:, t * 128:(t + 1) * 128])


def test_swizzle_reading_worked_grid():
    # the banded order taken for the worked example's 2 x 4 grid, band 2
    assert P.launch_order(2, 4, 2) == [(0, 0), (1, 0), (0, 1), (1, 1),
                                       (0, 2), (1, 2), (0, 3), (1, 3)]
    # band 1 is plain row-major; a band as tall as the grid is column-major
    assert P.launch_order(3, 2, 1) == [(0, 0), (0, 1), (1, 0), (1, 1), (2, 0), (2, 1)]
    assert P.launch_order(3, 2, 8) == [(0, 0), (1, 0), (2, 0), (0, 1), (1, 1), (2, 1)]


def test_serpentine_launch_order():
    """The serpentine band order (a plan input): the second band of a 5 x 3
    grid in bands of 2 walks its columns right to left, the third left to
    right again; every tile is launched once, a band's tiles stay
    consecutive, and vertical neighbours stay in consecutive slots."""
    got = P.launch_order(5, 3, 2, serpentine=True)
    assert got == [(0, 0), (1, 0), (0, 1), (1, 1), (0, 2), (1, 2),
                   (2, 2), (3, 2), (2, 1), (3, 1), (2, 0), (3, 0),
                   (4, 0), (4, 1), (4, 2)]
    fwd = P.launch_order(5, 3, 2)
    assert sorted(got) == sorted(fwd) and len(set(got)) == 15
    for a, b in zip(range(0, 12, 2), range(1, 12, 2)):
        (ra, ca), (rb, cb) = got[a], got[b]
        assert ca == cb and rb == ra + 1
    # one band: the same order as the forward one (the worked example)
    assert P.launch_order(2, 4, 2, serpentine=True) == P.launch_order(2, 4, 2)


@pytest.mark.parametrize("tm,tn,S,W", [(3, 5, 2, 4), (4, 4, 8, 3), (5, 3, 3, 7),
                                       (2, 4, 2, 2), (7, 2, 4, 5)])
def test_every_partition_brute_force(tm, tn, S, W):
    """All 2**(T-1) partitions of tiny grids: groups are consecutive wave
    ranges, sizes sum to the tiles, the table fills every group exactly
    once and in order, and the mapping tables are inverse permutations."""
    tiles = tm * tn
    T = P.wave_count(tiles, W)
    assert T <= 8
    for part in P.design_space(T):
        p = P.build_plan([tm * 128], tn * 128, 64, 128, 128, S, W, part,
                         P.LAYOUT_TILE)
        assert int(p.group_tiles.sum()) == tiles
        assert sorted(p.tile_to_slot.tolist()) == list(range(tiles))
        assert np.array_equal(p.slot_to_tile[p.tile_to_slot], np.arange(tiles))
        waves_before = 0
        for j, g in enumerate(part):
            s0, s1 = p.group_slots[j]
            assert s0 == min(tiles, waves_before * W)
            assert s1 == min(tiles, (waves_before + g) * W)
            waves_before += g
        snaps, fired = P.simulate_counting(p)
        assert snaps[-1] == p.group_tiles.tolist()
        assert [j for w in fired for j in w] == list(range(len(part)))


def test_one_then_two_partition():
    assert P.one_then_two(4) == (1, 2, 1)
    assert P.one_then_two(7) == (1, 2, 2, 2)
    assert P.one_then_two(1) == (1,)
    assert sum(P.one_then_two(98)) == 98 and len(P.one_then_two(98)) == 50


# ---------------------------------------------------------------- layouts

def _tiny_plan(layout, R=4, M=3 * 128, N=4 * 64, tn=64, W=5, S=2, ragged=None,
               tokens=None):
    if layout == P.LAYOUT_A2A:
        er, tok, sl = tokens
        tiles = sum(-(-m // 128) for m in er) * (N // tn)
        return P.build_plan(er, N, 64, 128, tn, S, W,
                            P.one_then_two(P.wave_count(tiles, W)), layout, R, tok, sl)
    rows = [M if ragged is None else ragged]
    tiles = -(-rows[0] // 128) * (N // tn)
    return P.build_plan(rows, N, 64, 128, tn, S, W,
                        P.one_then_two(P.wave_count(tiles, W)), layout, R)


def _tiny_routing(n_tok=40, E=3, k=2, D=4, seed=0):
    rng = np.random.default_rng(seed)
    picks = np.argsort(rng.random((n_tok, E)), axis=1)[:, :k]
    tok = np.repeat(np.arange(n_tok), k)
    sl = np.tile(np.arange(k), n_tok)
    ex = picks.reshape(-1)
    order = np.lexsort((sl, tok, ex))
    return np.bincount(ex, minlength=E).tolist(), tok[order], sl[order]


@pytest.mark.parametrize("ragged", [None, 300])
def test_tile_layout_round_trip_and_contiguity(ragged):
    p = _tiny_plan(P.LAYOUT_TILE, ragged=ragged)
    M = p.M
    C = np.random.default_rng(2).integers(0, 65535, (M, p.N)).astype(np.uint16)
    C_r = cm.pre_reorder(p, C)
    assert p.n_units * p.tile_n == M * p.N     # same element count as C
    # every group is one contiguous range and the ranges tile the buffer
    ends = [cm.group_units(p, j) for j in range(p.n_groups)]
    assert ends[0][0] == 0 and ends[-1][1] == p.n_units
    assert all(a[1] == b[0] for a, b in zip(ends, ends[1:]))
    # a group's range holds exactly its tiles, whole, in slot order
    for j in range(p.n_groups):
        a, b = cm.group_units(p, j)
        s0, s1 = p.group_slots[j]
        blocks = [C[p.tile_row0(s):p.tile_row0(s) + p.tile_rows(s),
                    p.tile_col0(s):p.tile_col0(s) + p.tile_n] for s in range(s0, s1)]
        assert np.array_equal(C_r[a:b], np.concatenate(blocks))
    back = cm.reorder_back_tile(p, cm.consume_copy(p, C_r))
    assert np.array_equal(back, C)


def test_rs_subtile_kth_subtiles_form_whole_rows():
    """[P1] 二 (2): subtile k of every tile goes to rank k, and all k-th
    subtiles together form complete rows."""
    R = 4
    p = _tiny_plan(P.LAYOUT_RS_SUBTILE, R=R, M=4 * 128)
    C = np.random.default_rng(3).integers(0, 65535, (p.M, p.N)).astype(np.uint16)
    C_r = cm.pre_reorder(p, C)
    # the scatter of the ReduceScatter stand-in, on unsummed data
    S = cm.consume_copy(p, C_r)
    slices = [np.zeros((P.dest_rows(p, k), p.tile_n), np.uint16) for k in range(R)]
    for j in range(p.n_groups):
        for k in range(R):
            st, n, o = int(p.part_start[j, k]), int(p.part_len[j, k]), int(p.part_dst[j, k])
            slices[k][o:o + n] = S[st:st + n]
    outs = cm.reorder_back_rs(p, slices)
    h = 128 // R
    for k in range(R):
        assert outs[k].shape == (p.M // R, p.N)
        for tm in range(p.M // 128):
            assert np.array_equal(outs[k][h * tm:h * (tm + 1)],
                                  C[128 * tm + h * k:128 * tm + h * (k + 1)])
    # every group splits evenly across ranks
    assert (p.part_len == p.part_len[:, :1]).all()


def test_rs_rowblock_literal_reading():
    R = 4
    p = _tiny_plan(P.LAYOUT_RS_ROWBLOCK, R=R, M=8 * 128)
    # finite values only: the sum stand-in rounds through fp32 (NaN payloads
    # would not survive it)
    C = np.random.default_rng(4).integers(0, 0x7F00, (p.M, p.N)).astype(np.uint16)
    slices = cm.consume_rs(p, cm.pre_reorder(p, C), [])
    outs = cm.reorder_back_rs(p, slices)
    for k in range(R):
        assert np.array_equal(outs[k], C[k * p.M // R:(k + 1) * p.M // R])


def test_a2a_every_routed_row_lands_once():
    D, k = 4, 2
    er, tok, sl = _tiny_routing(D=D)
    p = _tiny_plan(P.LAYOUT_A2A, R=D, N=3 * 64, tokens=(er, tok, sl))
    C = np.random.default_rng(5).integers(0, 65535, (p.M, p.N)).astype(np.uint16)
    C_r = cm.pre_reorder(p, C)
    # the parts of group j, destination d hold only rows routed to d
    for s in range(p.tiles):
        u = p.unit[s, :p.tile_rows(s)]
        j = p.slot_group[s]
        d = tok[p.tile_row0(s) + np.arange(p.tile_rows(s))] % D
        lo = p.part_start[j, d]
        assert ((u >= lo) & (u < lo + p.part_len[j, d])).all()
    assert sorted(p.unit[p.unit >= 0].tolist()) == list(range(p.n_units))
    recv = cm.consume_a2a(p, C_r)
    outs = cm.reorder_back_a2a(p, recv, k)
    for rho in range(p.M):
        t, q = int(tok[rho]), int(sl[rho])
        assert np.array_equal(outs[t % D][(t // D) * k + q], C[rho])
    assert sum(o.shape[0] for o in outs) == p.M


def test_a2a_expert_grid_padding_is_an_explicit_input():
    """Reading R16: an expert's grid is ceil(m_e / 128) tile rows -- the
    GEMM's output tiles -- whatever W is.  Only with pad_expert_tile_rows
    does an odd count get one empty tile row, so that launch slots 2i, 2i+1
    are vertically adjacent tiles of one expert and column; the empty tiles
    hold no rows, take slots and count in |G_j|; every routed row still
    lands once either way."""
    D, k = 4, 2
    er, tok, sl = _tiny_routing(n_tok=100, E=3, D=D)     # 200 rows over 3 experts
    tm = [-(-m // 128) for m in er]
    assert any(t % 2 for t in tm)
    for W, pad in ((6, True), (6, False), (5, True), (5, False)):
        tiles = sum(t + (t % 2 if pad else 0) for t in tm) * 3
        p = P.build_plan(er, 3 * 64, 64, 128, 64, 4, W,
                         P.one_then_two(P.wave_count(tiles, W)), P.LAYOUT_A2A, D, tok, sl,
                         pad_expert_tile_rows=pad)
        assert p.tiles == tiles
        assert p.expert_tiles_m == [t + (t % 2 if pad else 0) for t in tm]
        assert int(p.group_tiles.sum()) == p.tiles
        empty = [s for s in range(p.tiles) if p.tile_rows(s) == 0]
        assert len(empty) == (sum(t % 2 for t in tm) * 3 if pad else 0)
        if pad:
            for s in range(0, p.tiles, 2):
                e0, tm0, tn0 = p.slot_tile[s]
                e1, tm1, tn1 = p.slot_tile[s + 1]
                assert (e0, tn0, tm1) == (e1, tn1, tm0 + 1)
        C = np.random.default_rng(8).integers(0, 65535, (p.M, p.N)).astype(np.uint16)
        outs = cm.reorder_back_a2a(p, cm.consume_a2a(p, cm.pre_reorder(p, C)), k)
        for rho in range(p.M):
            t, q = int(tok[rho]), int(sl[rho])
            assert np.array_equal(outs[t % D][(t // D) * k + q], C[rho])
    with pytest.raises(ValueError):   # an All-to-All option only
        P.build_plan([256], 128, 64, 128, 64, 2, 2, (1, 1), P.LAYOUT_TILE,
                     pad_expert_tile_rows=True)


def _padded_routing(capacity, n_tok=40, E=3, k=2, D=4, seed=0):
    """The routing of ``_tiny_routing`` with every expert's rows padded to a
    fixed capacity by rows that hold no token (token -1): the static layout a
    dynamic router fills at run time."""
    er, tok, sl = _tiny_routing(n_tok, E, k, D, seed)
    T, S = [], []
    r = 0
    for m in er:
        assert m <= capacity
        T += tok[r:r + m].tolist() + [-1] * (capacity - m)
        S += sl[r:r + m].tolist() + [0] * (capacity - m)
        r += m
    return [capacity] * E, np.array(T), np.array(S), n_tok


def test_a2a_padding_rows_go_nowhere():
    """Rows the routing leaves empty (token -1) are sent to no rank: C_r holds
    exactly the routed rows, each lands once at its token's place, and the
    sentinel written into every empty row appears in no received buffer."""
    D, k = 4, 2
    er, tok, sl, n_tok = _padded_routing(capacity=40, D=D)
    p = _tiny_plan(P.LAYOUT_A2A, R=D, N=3 * 64, tokens=(er, tok, sl))
    valid = tok >= 0
    assert p.n_units == int(valid.sum()) * p.tiles_n < p.M * p.tiles_n
    pad_rows = np.nonzero(~valid)[0]
    for s in range(p.tiles):
        g = p.tile_row0(s) + np.arange(p.tile_rows(s))
        assert (p.unit[s, :p.tile_rows(s)][~valid[g]] == -1).all()
    assert sorted(p.unit[p.unit >= 0].tolist()) == list(range(p.n_units))
    rng = np.random.default_rng(6)
    C = rng.integers(0, 0x7F00, (p.M, p.N)).astype(np.uint16)
    C[pad_rows] = 0xFFFF                         # a NaN nothing else carries
    recv = cm.consume_a2a(p, cm.pre_reorder(p, C))
    assert sum(r.shape[0] for r in recv) == p.n_units
    assert not any((r == 0xFFFF).any() for r in recv)
    outs = cm.reorder_back_a2a(p, recv, k, n_tokens=n_tok)
    assert sum(o.shape[0] for o in outs) == n_tok * k
    for rho in np.nonzero(valid)[0]:
        t, q = int(tok[rho]), int(sl[rho])
        assert np.array_equal(outs[t % D][(t // D) * k + q], C[rho])
    # the same tokens routed without padding give the same received rows
    er0, tok0, sl0 = _tiny_routing(D=D)
    p0 = _tiny_plan(P.LAYOUT_A2A, R=D, N=3 * 64, tokens=(er0, tok0, sl0))
    C0 = C[valid]
    outs0 = cm.reorder_back_a2a(p0, cm.consume_a2a(p0, cm.pre_reorder(p0, C0)), k)
    for a, b in zip(outs, outs0):
        assert np.array_equal(a, b)


# ---------------------------------------------------------------- GEMM pins

def _exact_gemm(A, Bm):
    """Exact rational product, rounded to bf16 by the value's definition."""
    M, K = A.shape
    N = Bm.shape[1]
    out = np.empty((M, N), dtype=np.float64)
    for i in range(M):
        for j in range(N):
            out[i, j] = float(sum(Fraction(float(A[i, k])) * Fraction(float(Bm[k, j]))
                                  for k in range(K)))
    return out


@pytest.mark.parametrize("M,K,N", [(3, 5, 7), (7, 2, 4), (1, 9, 2)])
def test_gemm_brute_force_non_square(M, K, N):
    """A non-square A . B against an exact rational brute force; integer
    inputs make the fp64 sums exact, so results match bit for bit after
    rounding (sums reach a few hundred, so bf16 rounding is exercised)."""
    rng = np.random.default_rng(M * 100 + K * 10 + N)
    A = B.round_to_bf16(rng.integers(-40, 40, (M, K)).astype(np.float64))
    Bm = B.round_to_bf16(rng.integers(-40, 40, (K, N)).astype(np.float64))
    want = B.round_to_bf16(_exact_gemm(B.bits_to_f64(A), B.bits_to_f64(Bm)))
    assert np.array_equal(G.gemm_bf16(A, Bm), want)


def test_gemm_unit_entries_exact_and_identity():
    rng = np.random.default_rng(7)
    A = B.round_to_bf16(rng.integers(-1, 2, (64, 256)).astype(np.float64))
    Bm = B.round_to_bf16(rng.integers(-1, 2, (256, 96)).astype(np.float64))
    got = B.bits_to_f64(G.gemm_bf16(A, Bm))
    ints = B.bits_to_f64(A).astype(np.int64) @ B.bits_to_f64(Bm).astype(np.int64)
    assert np.array_equal(got, ints.astype(np.float64))
    eye = B.round_to_bf16(np.eye(96))
    Bx = B.round_to_bf16(rng.standard_normal((96, 40)))
    assert np.array_equal(G.gemm_bf16(eye, Bx), Bx)


def test_grouped_gemm_uses_each_experts_B():
    rng = np.random.default_rng(8)
    rows = [3, 0, 5]
    A = B.round_to_bf16(rng.standard_normal((8, 16)))
    Bs = [B.round_to_bf16(rng.standard_normal((16, 4))) for _ in range(3)]
    C = G.grouped_gemm_bf16(A, Bs, rows)
    assert np.array_equal(C[:3], G.gemm_bf16(A[:3], Bs[0]))
    assert np.array_equal(C[3:], G.gemm_bf16(A[3:], Bs[2]))
    assert np.array_equal(G.gemm_rows_bf16(A, Bs, rows, [4, 0]), C[[4, 0]])


# ---------------------------------------------------------------- sums

def test_sum_order_and_single_rounding():
    """Own buffer first, then the partials in order, fp32 adds, one rounding:
    (1 + 2**24) - 2**24 is 0 in fp32 but 1 in another order."""
    bits = B.round_to_bf16
    own = bits(np.array([[1.0]]))
    p1 = bits(np.array([[2.0 ** 24]]))
    p2 = bits(np.array([[-(2.0 ** 24)]]))
    got = cm._fp32_sum_then_round(own, [p1, p2])
    assert B.bits_to_f64(got)[0, 0] == 0.0
    got2 = cm._fp32_sum_then_round(p1, [p2, own])
    assert B.bits_to_f64(got2)[0, 0] == 1.0


def test_sum_within_fp32_bound():
    rng = np.random.default_rng(9)
    own = B.round_to_bf16(rng.standard_normal((64, 32)))
    parts = [B.round_to_bf16(rng.standard_normal((64, 32))) for _ in range(7)]
    exact = B.bits_to_f64(own) + sum(B.bits_to_f64(q) for q in parts)
    got = B.bits_to_f64(cm._fp32_sum_then_round(own, parts))
    # seven fp32 roundings (rel 2**-24 each) and one bf16 rounding (2**-8)
    tol = np.abs(exact) * 2.0 ** -8 + 8 * 2.0 ** -24 * 8 * np.abs(exact).max()
    assert (np.abs(got - exact) <= tol).all()


# ---------------------------------------------------------------- planted mistakes

def test_planted_transposed_operand_is_caught(monkeypatch):
    monkeypatch.setattr(G, "gemm_f64",
                        lambda A, Bm: B.bits_to_f64(Bm).T @ B.bits_to_f64(A).T)
    with pytest.raises((AssertionError, ValueError)):
        test_gemm_brute_force_non_square(3, 5, 7)
    with pytest.raises((AssertionError, ValueError)):
        test_gemm_brute_force_non_square(7, 2, 4)


def test_planted_wave_mistakes_are_caught(monkeypatch):
    # the page's own counts divide evenly, so the ceiling hides an off-by-one
    # there; the brute force over tiny ragged grids does not
    monkeypatch.setattr(P, "wave_count", lambda n, w: -(-n // (w + 1)))
    with pytest.raises((AssertionError, IndexError, ValueError)):
        test_every_partition_brute_force(3, 5, 2, 4)
    monkeypatch.undo()
    monkeypatch.setattr(P, "wave_count", lambda n, w: n // w)   # drops a partial wave
    with pytest.raises((AssertionError, IndexError, ValueError)):
        test_every_partition_brute_force(3, 5, 2, 4)
    monkeypatch.undo()
    monkeypatch.setattr(P, "wave_of_slot", lambda s, w: (s + 1) // w)
    with pytest.raises((AssertionError, IndexError, ValueError)):
        test_every_partition_brute_force(3, 5, 2, 4)


def test_planted_round_half_away_is_caught(monkeypatch):
    monkeypatch.setattr(B, "_round_half_even",
                        lambda q: np.floor(q + 0.5))
    with pytest.raises(AssertionError):
        test_bf16_ties_subnormals_overflow_signed_zero()


def test_planted_dropped_partial_is_caught(monkeypatch):
    real = cm._fp32_sum_then_round
    monkeypatch.setattr(cm, "_fp32_sum_then_round",
                        lambda own, parts: real(own, parts[:-1]))
    with pytest.raises(AssertionError):
        test_sum_within_fp32_bound()
    with pytest.raises(AssertionError):
        test_sum_order_and_single_rounding()


def test_planted_subtile_index_is_caught(monkeypatch):
    real = P._assign_units

    def wrong(p):      # subtile k of a group placed in the wrong part order
        real(p)
        if p.layout == P.LAYOUT_RS_SUBTILE:
            p.part_start[:, [0, 1]] = p.part_start[:, [1, 0]]
    monkeypatch.setattr(P, "_assign_units", wrong)
    with pytest.raises((AssertionError, IndexError)):
        test_rs_subtile_kth_subtiles_form_whole_rows()


def test_planted_padding_routed_by_modulo_is_caught(monkeypatch):
    def wrong(plan, slot):   # token -1 taken modulo D like a real token
        g = plan.tile_row0(slot) + np.arange(plan.tile_rows(slot))
        return plan.row_token[g] % plan.n_dest
    monkeypatch.setattr(P, "_row_dests", wrong)
    with pytest.raises((AssertionError, IndexError)):
        test_a2a_padding_rows_go_nowhere()


def test_planted_swapped_group_order_is_caught(monkeypatch):
    real = P.build_plan

    def wrong(*a, **k):
        p = real(*a, **k)
        p.group_tiles = np.roll(p.group_tiles, 1)   # sizes off by one group
        return p
    monkeypatch.setattr(P, "build_plan", wrong)
    with pytest.raises(AssertionError):
        test_worked_example_counting_table()


# ---------------------------------------------------------------- pipeline

def test_pipeline_worked_example_end_to_end():
    rng = np.random.default_rng(11)
    A = B.round_to_bf16(rng.uniform(-1, 1, (256, 256)))
    Bm = B.round_to_bf16(rng.uniform(-1, 1, (256, 512)))
    res = pipeline.run([256], 512, 256, 128, 128, 2, 2, (1, 2, 1), P.LAYOUT_TILE,
                       "copy", A, [Bm])
    assert res.counting == [2, 4, 2]
    assert res.fired == [0, 1, 2]
    assert np.array_equal(res.final, res.C)
    assert np.array_equal(res.C, G.gemm_bf16(A, Bm))
