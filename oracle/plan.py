"""Tile order, waves, wave groups, counting table, mapping tables and the
reordered layouts -- the oracle's plan (TEST INFRASTRUCTURE ONLY).

Pages (full titles in ``oracle/__init__``):
  [P1] FlashOverlap deep-dive, 一、信号机制 (waves, block swizzling, wave
       groups, the counting table and its worked example), 二、重排机制 (mapping
       table, inverse mapping table, the AllReduce / ReduceScatter /
       All-to-All reordering patterns of Figure 6), 三、Wave Group 划分设计空间
       (the 2**(T-1) design space), 四、实时调优 Algorithm 1 (T = tiles / SMs
       left to the GEMM).
  [P2] Efficient and Adaptable Overlapping ... , captions of Figures 3 and 5.

Everything here is written as the plain definition: loops that walk slots in
order and concatenate, so that each table can be checked by eye.  Nothing is
shared with the CUDA path's planner.

Readings taken where the pages are silent (each is also stated where used):
  R1  block swizzle: bands of ``swizzle`` tile-rows, walked column by column
      (left to right; with the serpentine band order, an explicit plan
      input, the odd bands of each expert walk right to left)
  R2  wave(slot) = slot // W, W = number of persistent GEMM workers
  R3  |G_j| is counted in tiles, partitions are given in waves
  R6  intra-tile order is row-major; a "unit" is one tile row (tile_n values)
  R16 an expert's grid has ceil(m_e / tile_m) tile rows, the GEMM's output
      tiles.  Only when the plan asks for it (``pad_expert_tile_rows``, an
      explicit input, All-to-All layout only) is an odd count padded with
      one empty tile row (no valid rows), so that every band has an even
      height; empty tiles then take slots and count in |G_j| like others.
      The pages know no such padding: it is an input, never inferred.
"""
from dataclasses import dataclass, field
from itertools import product
import math

import numpy as np

LAYOUT_TILE = "tile"                # AllReduce / plain copy: whole tiles
LAYOUT_RS_SUBTILE = "rs_subtile"    # ReduceScatter: R row-subtiles per tile
LAYOUT_RS_ROWBLOCK = "rs_rowblock"  # ReduceScatter, literal row-block reading
LAYOUT_A2A = "a2a"                  # All-to-All: sub-tokens by destination


# --------------------------------------------------------------------------
# tile order, waves, groups

def launch_order(tiles_m, tiles_n, swizzle, serpentine=False):
    """Launch order of a tiles_m x tiles_n grid as a list of (tm, tn).

    [P1] 一 "Block Swizzling 的影响" and 二 "挑战: 不规则的 Tile 执行顺序": tiles are
    dispatched interleaved so a wave's tiles are not contiguous in memory.
    The pages never define the swizzle.  Reading R1: tile-rows form bands of
    ``swizzle`` rows (the last band may be shorter); bands are taken in
    order, and inside a band the tiles are taken column by column, top to
    bottom.  Columns go left to right; with ``serpentine`` (a plan input, not
    the pages') the odd bands (second, fourth, ...) go right to left.
    """
    order = []
    top, band = 0, 0
    while top < tiles_m:
        h = min(swizzle, tiles_m - top)
        cols = range(tiles_n)
        if serpentine and band % 2 == 1:
            cols = reversed(cols)
        for tn in cols:
            for dm in range(h):
                order.append((top + dm, tn))
        top += h
        band += 1
    return order


def wave_count(n_tiles, wave_width):
    """T = ceil(tiles / W): [P1] 一 "关键洞察" (512 tiles / 128 SMs = 4 waves) and
    四 Algorithm 1 (T = tile_num / (sm_num - comm sm_num)).  Reading R2: the
    last wave may be partial, hence the ceiling."""
    return -(-n_tiles // wave_width)


def wave_of_slot(slot, wave_width):
    """Reading R2: with W persistent workers taking slots round-robin, the
    k-th tile of every worker forms wave k, i.e. wave = slot // W."""
    return slot // wave_width


def design_space(T):
    """All wave-group partitions of T waves ([P1] 三 "设计空间大小"): after
    every wave but the last choose communicate (1) or not (0); the last wave
    always communicates.  Returns tuples of group sizes in waves."""
    out = []
    for bits in product((0, 1), repeat=T - 1):
        sizes, run = [], 0
        for b in bits + (1,):
            run += 1
            if b:
                sizes.append(run)
                run = 0
        out.append(tuple(sizes))
    return out


def one_then_two(T):
    """The partition "one wave, then groups of two, the last takes what is
    left" used by the workloads (a reading; the tuned choice is the job of
    [P1] 四's predictive search)."""
    if T <= 0:
        return ()
    parts = [1]
    left = T - 1
    while left > 0:
        parts.append(min(2, left))
        left -= parts[-1]
    return tuple(parts)


# --------------------------------------------------------------------------
# the plan

@dataclass
class Plan:
    # problem
    expert_rows: list          # rows per expert; one entry for a plain GEMM
    N: int
    K: int
    tile_m: int
    tile_n: int
    swizzle: int
    wave_width: int
    partition: tuple           # waves per group
    layout: str
    n_dest: int = 1
    row_token: np.ndarray = None   # A2A: token of each routed row
    row_slot: np.ndarray = None    # A2A: top-k slot of each routed row
    # derived
    tiles_n: int = 0
    expert_tiles_m: list = field(default_factory=list)
    expert_row0: list = field(default_factory=list)
    tiles: int = 0
    waves: int = 0
    slot_tile: list = field(default_factory=list)     # slot -> (e, tm, tn)
    slot_to_tile: np.ndarray = None                   # inverse mapping table
    tile_to_slot: np.ndarray = None                   # mapping table
    slot_group: np.ndarray = None
    group_tiles: np.ndarray = None                    # |G_j| in tiles
    group_slots: list = field(default_factory=list)   # [first, last+1) per group
    unit: np.ndarray = None       # [slot, tile_m] -> unit index in C_r, -1 if no row
    part_start: np.ndarray = None # [group, dest] first unit of the part in C_r
    part_len: np.ndarray = None   # [group, dest] units in the part
    part_dst: np.ndarray = None   # [group, dest] offset of the part in buffer dest
    n_units: int = 0

    def tile_id(self, e, tm, tn):
        """Row-major tile id, experts one after another."""
        base = sum(self.expert_tiles_m[:e]) * self.tiles_n
        return base + tm * self.tiles_n + tn

    def tile_rows(self, slot):
        """Valid rows of the tile at ``slot`` (the last tile-row of an expert
        may be ragged; a padding tile row (R16) has none)."""
        e, tm, _ = self.slot_tile[slot]
        return max(0, min(self.tile_m, self.expert_rows[e] - tm * self.tile_m))

    def tile_row0(self, slot):
        """First row of the tile at ``slot`` in the stacked GEMM output."""
        e, tm, _ = self.slot_tile[slot]
        return self.expert_row0[e] + tm * self.tile_m

    def tile_col0(self, slot):
        return self.slot_tile[slot][2] * self.tile_n

    @property
    def M(self):
        return sum(self.expert_rows)

    @property
    def n_groups(self):
        return len(self.partition)


def _row_dests(plan, slot):
    """Destination rank of every valid row of the tile at ``slot``, for the
    layouts that route rows: a2a sends row rho to rank token(rho) mod n_dest;
    rs_rowblock sends global row g to rank g // (M / n_dest).

    A2A rows whose token is negative hold no token (an expert's capacity left
    unfilled by the routing) and go nowhere: destination -1.  Reading of
    [P1] 二 (3) "映射表需要考虑动态路由模式": the mapping follows the routing,
    and a row the routing leaves empty has nothing to send."""
    rows = plan.tile_rows(slot)
    g = plan.tile_row0(slot) + np.arange(rows)
    if plan.layout == LAYOUT_A2A:
        t = plan.row_token[g].astype(np.int64)
        return np.where(t >= 0, t % plan.n_dest, -1)
    if plan.layout == LAYOUT_RS_ROWBLOCK:
        return g // (plan.M // plan.n_dest)
    raise ValueError(plan.layout)


def build_plan(expert_rows, N, K, tile_m, tile_n, swizzle, wave_width,
               partition, layout, n_dest=1, row_token=None, row_slot=None,
               pad_expert_tile_rows=False, serpentine=False):
    """Build every table of the path for one problem.

    * launch slots: experts in order, each expert's ceil(m_e/tile_m) x
      (N/tile_n) grid in the swizzled order of ``launch_order``, slots
      numbered consecutively across experts.
    * mapping table tile -> slot and inverse slot -> tile ([P1] 二
      "解决方案: 映射表重排"; the illustration there sends tile_0 -> 0,
      tile_3 -> 1, ... and back).
    * groups: group j holds the waves partition[j] after the earlier groups'
      ([P1] 一 "Wave Group 设计"); |G_j| counts its tiles (reading R3).
    * the reordered layout ``unit[slot, r]`` (see ``_assign_units``).

    pad_expert_tile_rows (reading R16; All-to-All only): give each expert's
    grid an even number of tile rows by adding one empty tile row when odd.
    Off by default: the grid is then exactly the GEMM's output tiles.

    serpentine (reading R1, a plan input): the odd bands of each expert walk
    their columns right to left.
    """
    if N % tile_n:
        raise ValueError("N must be a multiple of tile_n")
    p = Plan(list(expert_rows), N, K, tile_m, tile_n, swizzle, wave_width,
             tuple(partition), layout, n_dest,
             None if row_token is None else np.asarray(row_token),
             None if row_slot is None else np.asarray(row_slot))
    p.tiles_n = N // tile_n
    # Reading R16: padding only when asked for, and only in the A2A layout
    if pad_expert_tile_rows and layout != LAYOUT_A2A:
        raise ValueError("expert grid padding is an All-to-All option")
    pad_even = bool(pad_expert_tile_rows)
    row0 = 0
    for m_e in p.expert_rows:
        p.expert_row0.append(row0)
        tm = -(-m_e // tile_m)
        p.expert_tiles_m.append(tm + (tm % 2) if pad_even else tm)
        row0 += m_e
    for e, tm_count in enumerate(p.expert_tiles_m):
        for tm, tn in launch_order(tm_count, p.tiles_n, swizzle, serpentine):
            p.slot_tile.append((e, tm, tn))
    p.tiles = len(p.slot_tile)
    p.waves = wave_count(p.tiles, wave_width)
    if sum(p.partition) != p.waves or min(p.partition, default=0) < 1:
        raise ValueError("partition must be positive and sum to the wave count")

    p.slot_to_tile = np.array([p.tile_id(*t) for t in p.slot_tile], dtype=np.int64)
    p.tile_to_slot = np.empty(p.tiles, dtype=np.int64)
    for s, t in enumerate(p.slot_to_tile):
        p.tile_to_slot[t] = s

    # wave -> group, then slot -> group
    wave_group = []
    for j, g in enumerate(p.partition):
        wave_group += [j] * g
    p.slot_group = np.array([wave_group[wave_of_slot(s, wave_width)]
                             for s in range(p.tiles)], dtype=np.int64)
    p.group_tiles = np.array([int(np.sum(p.slot_group == j))
                              for j in range(p.n_groups)], dtype=np.int64)
    first = 0
    for j in range(p.n_groups):
        p.group_slots.append((first, first + int(p.group_tiles[j])))
        first += int(p.group_tiles[j])
    _assign_units(p)
    return p


def _assign_units(p):
    """Lay out the reordered buffer C_r as a sequence of units (one tile row
    of tile_n values each), group after group, so that every group -- and
    every (group, destination) part of it -- is one contiguous range.

    [P1] 二 "动机: 通信需要连续地址": a single NCCL call needs contiguous send
    and receive buffers, so both intra-tile and inter-tile data of a group
    are made contiguous.  Inside a group (Figure 6 of [P1] 二):

    * tile (AllReduce, copy): the group's tiles in slot order, each tile's
      rows in order -- tiles stay whole, rows stay whole.
    * rs_subtile (ReduceScatter): each tile is cut along rows into n_dest
      equal subtiles; part k of the group is the k-th subtile of each of the
      group's tiles, in slot order (subtile k always goes to rank k).
    * rs_rowblock (the literal "row block of M/R" reading): part k is the
      group's whole tiles whose rows fall in rank k's block of M/R rows.
    * a2a (All-to-All): part d is, over the group's tiles in slot order, the
      tile rows (sub-tokens) whose token goes to rank d, in row order.
    """
    R = p.n_dest if p.layout != LAYOUT_TILE else 1
    p.unit = np.full((p.tiles, p.tile_m), -1, dtype=np.int64)
    p.part_start = np.zeros((p.n_groups, R), dtype=np.int64)
    p.part_len = np.zeros((p.n_groups, R), dtype=np.int64)
    u = 0
    for j in range(p.n_groups):
        s0, s1 = p.group_slots[j]
        for k in range(R):
            p.part_start[j, k] = u
            for s in range(s0, s1):
                rows = p.tile_rows(s)
                if p.layout == LAYOUT_TILE:
                    sel = np.arange(rows)
                elif p.layout == LAYOUT_RS_SUBTILE:
                    h = p.tile_m // R
                    sel = np.arange(k * h, min((k + 1) * h, rows))
                else:
                    sel = np.nonzero(_row_dests(p, s) == k)[0]
                p.unit[s, sel] = u + np.arange(len(sel))
                u += len(sel)
            p.part_len[j, k] = u - p.part_start[j, k]
    p.n_units = u
    # a part (j, k) is appended, group after group, to destination buffer k
    p.part_dst = np.zeros_like(p.part_start)
    for k in range(R):
        off = 0
        for j in range(p.n_groups):
            p.part_dst[j, k] = off
            off += p.part_len[j, k]


def dest_rows(p, k):
    """Rows of destination buffer k (units it receives over all groups)."""
    return int(np.sum(p.part_len[:, k]))


# --------------------------------------------------------------------------
# the counting table

def simulate_counting(p):
    """Sequential simulation of the counting table ([P1] 一 "实现方法: 组级
    Tile 计数"): P counters start at 0; every finished tile adds 1 to the
    entry of its group (the tile's index identifies the group); when entry j
    reaches |G_j|, G_j's communication starts.  Tiles finish wave by wave, in
    slot order.

    Returns (snapshots, fired): the table after each wave, and for each wave
    the groups whose count became full in it.
    """
    table = [0] * p.n_groups
    snapshots, fired = [], []
    for w in range(p.waves):
        now = []
        for s in range(w * p.wave_width, min(p.tiles, (w + 1) * p.wave_width)):
            j = int(p.slot_group[s])
            table[j] += 1
            if table[j] == p.group_tiles[j]:
                now.append(j)
        snapshots.append(list(table))
        fired.append(now)
    return snapshots, fired
