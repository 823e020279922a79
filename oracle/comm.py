"""Pre-comm reorder, the communication stand-ins and the post-comm reorder
(TEST INFRASTRUCTURE ONLY).

Pages (full titles in ``oracle/__init__``): [P1] 二、重排机制 -- the mapping
table makes each group's data contiguous so a collective can be called on
it directly (ncclAllReduce(contiguous_buf, ...)), and the inverse mapping
table puts the results back; Figure 6 gives the AllReduce (tile), the
ReduceScatter (subtile) and the All-to-All (sub-token) patterns.  [P2]
Figure 5 caption: reorder, then signal, then communicate, then reorder back.

On one GPU each collective is replaced by what it computes for this rank:
  copy  -- the received buffer equals the sent one (a plain transfer)
  sum   -- AllReduce: own data plus the other ranks' partial buffers
  rs    -- ReduceScatter: the sum, and part k of every group to rank k
  a2a   -- All-to-All: part d of every group to rank d

Units: ``C_r`` and every received buffer are arrays [units, tile_n] of bf16
bits; ``plan.unit[slot, r]`` is the unit of row r of the tile at ``slot``.
"""
import numpy as np

from .bf16 import bits_to_f64, f32_round_to_bf16
from . import plan as P


def _groups(p, groups):
    return range(p.n_groups) if groups is None else groups


def _slots(p, groups):
    for j in _groups(p, groups):
        s0, s1 = p.group_slots[j]
        yield from range(s0, s1)


def pre_reorder(p, C_bits, groups=None, out=None):
    """C_r[unit(slot, r)] = C[row0(slot) + r, col0(slot) : col0 + tile_n]
    for every valid row of every tile ([P1] 二 "预通信重排"); with ``groups``,
    only the tiles of those groups."""
    C_r = np.zeros((p.n_units, p.tile_n), dtype=np.uint16) if out is None else out
    for s in _slots(p, groups):
        rows = p.tile_rows(s)
        r0, c0 = p.tile_row0(s), p.tile_col0(s)
        u = p.unit[s, :rows]
        keep = u >= 0                 # rows that hold no token are not sent
        C_r[u[keep]] = C_bits[r0:r0 + rows, c0:c0 + p.tile_n][keep]
    return C_r


def group_units(p, j):
    """The contiguous unit range [first, last) of group j in C_r."""
    first = int(p.part_start[j, 0])
    return first, first + int(np.sum(p.part_len[j]))


def consume_copy(p, C_r, groups=None, out=None):
    """Plain transfer of each group's contiguous range."""
    recv = np.zeros_like(C_r) if out is None else out
    for j in _groups(p, groups):
        a, b = group_units(p, j)
        recv[a:b] = C_r[a:b]
    return recv


def _fp32_sum_then_round(own, partials):
    """bf16_rn(((own + P1) + P2) + ...) with every addition in fp32.

    The pages do not fix the summation order of an AllReduce; the reading
    taken is: own buffer first, then the partial buffers in order, each
    addition an IEEE fp32 add, one round to bf16 at the end."""
    acc = bits_to_f64(own).astype(np.float32)
    for q in partials:
        acc = acc + bits_to_f64(q).astype(np.float32)
    return f32_round_to_bf16(acc)


def consume_sum(p, C_r, partials, groups=None, out=None):
    """AllReduce stand-in over each group's range; partials are in the same
    reordered layout as C_r (they stand for the other ranks' C_r)."""
    S = np.zeros_like(C_r) if out is None else out
    for j in _groups(p, groups):
        a, b = group_units(p, j)
        S[a:b] = _fp32_sum_then_round(C_r[a:b], [q[a:b] for q in partials])
    return S


def consume_rs(p, C_r, partials, groups=None, out=None):
    """ReduceScatter stand-in: the group's sum, then part k of the group is
    appended (group after group) to slice k.  Returns n_dest arrays."""
    R = p.n_dest
    slices = out if out is not None else [
        np.zeros((P.dest_rows(p, k), p.tile_n), dtype=np.uint16) for k in range(R)]
    for j in _groups(p, groups):
        a, b = group_units(p, j)
        S = _fp32_sum_then_round(C_r[a:b], [q[a:b] for q in partials])
        for k in range(R):
            st = int(p.part_start[j, k]) - a
            n = int(p.part_len[j, k])
            d = int(p.part_dst[j, k])
            slices[k][d:d + n] = S[st:st + n]
    return slices


def consume_a2a(p, C_r, groups=None, out=None):
    """All-to-All stand-in: part d of each group is appended, group after
    group, to rank d's receive buffer.  Returns n_dest arrays."""
    D = p.n_dest
    recv = out if out is not None else [
        np.zeros((P.dest_rows(p, d), p.tile_n), dtype=np.uint16) for d in range(D)]
    for j in _groups(p, groups):
        for d in range(D):
            st, n, o = (int(p.part_start[j, d]), int(p.part_len[j, d]),
                        int(p.part_dst[j, d]))
            recv[d][o:o + n] = C_r[st:st + n]
    return recv


def reorder_back_tile(p, recv, groups=None, out=None):
    """Inverse mapping for the tile layout: unit(slot, r) of the received
    buffer goes back to row row0 + r, columns col0.. of the M x N output
    ([P1] 二 "通信后重排")."""
    C = np.zeros((p.M, p.N), dtype=np.uint16) if out is None else out
    for s in _slots(p, groups):
        rows = p.tile_rows(s)
        r0, c0 = p.tile_row0(s), p.tile_col0(s)
        C[r0:r0 + rows, c0:c0 + p.tile_n] = recv[p.unit[s, :rows]]
    return C


def _positions_in_dest(p, s):
    """For every valid row r of the tile at slot s: (k, index) of unit(s, r)
    inside destination buffer k -- the part's offset there plus the unit's
    place inside its part."""
    rows = p.tile_rows(s)
    u = p.unit[s, :rows]
    j = int(p.slot_group[s])
    k = np.full(rows, -1, dtype=np.int64)
    idx = np.full(rows, -1, dtype=np.int64)
    for d in range(p.part_start.shape[1]):
        st, n = int(p.part_start[j, d]), int(p.part_len[j, d])
        inside = (u >= st) & (u < st + n)
        k[inside] = d
        idx[inside] = int(p.part_dst[j, d]) + (u[inside] - st)
    assert ((k >= 0) | (u < 0)).all(), "unit outside its group's parts"
    return k, idx


def reorder_back_rs(p, slices, groups=None, out=None):
    """Inverse mapping inside each ReduceScatter slice: slice k becomes the
    row-major (M / R) x N block of the rows rank k owns.

    rs_subtile: slice row of tile-row tm's subtile k, row i, is h*tm + i
      (h = tile_m / R); it holds global row tile_m*tm + h*k + i ([P1] 二 (2):
      all k-th subtiles together form whole rows).
    rs_rowblock: slice k holds global rows [k M/R, (k+1) M/R) in order.
    """
    R = p.n_dest
    rows_per = p.M // R
    outs = out if out is not None else [
        np.zeros((rows_per, p.N), dtype=np.uint16) for _ in range(R)]
    h = p.tile_m // R
    for s in _slots(p, groups):
        _, tm, _ = p.slot_tile[s]
        c0 = p.tile_col0(s)
        k, idx = _positions_in_dest(p, s)
        r = np.arange(p.tile_rows(s))
        if p.layout == P.LAYOUT_RS_SUBTILE:
            rho = h * tm + (r - h * k)
        else:
            rho = p.tile_row0(s) + r - k * rows_per
        for d in range(R):
            sel = k == d
            outs[d][rho[sel], c0:c0 + p.tile_n] = slices[d][idx[sel]]
    return outs


def reorder_back_a2a(p, recv, top_k, groups=None, out=None, n_tokens=None):
    """Inverse mapping after the All-to-All: on rank d, the sub-token of
    routed row rho (token t, top-k slot q), column block c0, goes to row
    (t // D) * top_k + q, columns c0.. of rank d's output.  Each rank
    receives the tokens t with t mod D == d, all their top-k rows."""
    D = p.n_dest
    n_tok = int(p.row_token.max()) + 1 if n_tokens is None else n_tokens
    outs = out if out is not None else [
        np.zeros((len(range(d, n_tok, D)) * top_k, p.N), dtype=np.uint16)
        for d in range(D)]
    for s in _slots(p, groups):
        c0 = p.tile_col0(s)
        r0 = p.tile_row0(s)
        rows = p.tile_rows(s)
        k, idx = _positions_in_dest(p, s)
        t = p.row_token[r0:r0 + rows].astype(np.int64)
        q = p.row_slot[r0:r0 + rows].astype(np.int64)
        final_row = (t // D) * top_k + q
        for d in range(D):           # rows without a token (k = -1) match no d
            sel = k == d
            outs[d][final_row[sel], c0:c0 + p.tile_n] = recv[d][idx[sel]]
    return outs
