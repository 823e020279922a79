"""Workload shapes and seeded synthetic inputs.

This module holds no arithmetic of the method: it only names the five
workloads and draws their inputs.  Both the CUDA path's tests/benchmark and
the CPU oracle receive the very same bf16 bit arrays from here.

Workloads (the shapes of the pages' workloads; synthetic data, no weights):
  worked_example  C[256x512] = A[256x256] B[256x512], U[-1,1] inputs,
                  128x128 tiles (8 tiles), wave width 2 -> 4 waves, groups
                  {W1},{W2,W3},{W4}; consumer: copy + reorder back
  wave_pattern    M=2048 N=8192 K=8192 (the shape whose tile completion
                  times show four waves); consumer: copy + reorder back
  allreduce       M=4096 N=8192 K=3584 (tensor-parallel down-projection of a
                  70B-class MLP, TP=8); consumer: sum with 7 partial buffers
  reducescatter   M=8192 N=4096 K=2752 (7B-class backward GEMM, R=4);
                  consumer: sum with 3 partials, scatter to 4 slices
  alltoall        16384 tokens x top-2 = 32768 routed rows over 8 experts,
                  N=14336 K=4096 (Mixtral-8x7B-shaped expert up-projection);
                  consumer: bucket rows by token mod 8 into 8 buffers; each
                  expert's grid is padded to an even number of tile rows
                  (an explicit plan input) so the GEMM runs as CTA pairs
  Every workload but the worked example launches its bands in serpentine
  order (odd bands right to left; an explicit plan input).
  alltoall_dynamic  the same layer with a fixed capacity of 5120 rows per
                  expert (1.25 x the mean load, a multiple of 128): the GEMM
                  shape never changes, each step draws a new routing, and the
                  rows an expert does not fill hold no token (token -1)

Seeds: ``numpy.random.default_rng(1000 * index + stream)`` with stream 0 for
A (or the token matrix X), 1 for B, 2 for the partial buffers and 9 for the
routing (9 + step for the routing of step ``step`` of the dynamic workload).  Values are drawn in fp32 and rounded once to bf16 (round to
nearest even, by torch's conversion).  Distributions: the worked example
U[-1,1]; the others N(0,1)/sqrt(K) for A and B and N(0,1) for partials.
"""
from dataclasses import dataclass
import math

import numpy as np
import torch

LAYOUT_TILE, LAYOUT_RS_SUBTILE, LAYOUT_RS_ROWBLOCK, LAYOUT_A2A = 0, 1, 2, 3
CONS_COPY, CONS_SUM, CONS_RS, CONS_A2A = 0, 1, 2, 3


@dataclass(frozen=True)
class Workload:
    name: str
    index: int            # seed base: 1000 * index
    M: int                # rows (routed rows for the grouped workload)
    N: int
    K: int
    tile_m: int = 128
    tile_n: int = 256
    swizzle: int = 8
    wave_width: int = 148
    layout: int = LAYOUT_TILE
    consumer: int = CONS_COPY
    n_dest: int = 1
    n_partials: int = 0
    uniform: bool = False
    # grouped (All-to-All) workload
    n_tokens: int = 0
    n_experts: int = 0
    top_k: int = 0
    capacity: int = 0     # rows per expert (0: exactly the routed rows)
    # each expert's grid padded to an even number of tile rows (one empty
    # tile row when odd), so the GEMM can run as CTA pairs; a plan input
    pad_expert_tile_rows: bool = False
    # launch order: the odd bands (of each expert) walk their columns right
    # to left (serpentine) instead of left to right; a plan input
    serpentine: bool = False

    @property
    def grouped(self):
        return self.n_experts > 0

    def gemm_flops(self):
        return 2.0 * self.M * self.N * self.K


# The large workloads launch their bands in serpentine order (measured: the
# GEMM 0.7-2.7% shorter, fewer re-reads of B); the worked example has one
# band, where both orders are the same.
#
# Band heights (swizzle): the wave-pattern shape is defined with swizzle 8.
# The others are free; B is read from DRAM about once per band, and the
# GEMM's main loop is bound by load latency, so fewer DRAM misses make it
# faster.  AllReduce takes one band of all 32 tile rows, and the All-to-All
# layer one band per expert (64 is above any expert's tile rows).  Measured
# against swizzle 8, interleaved: the AllReduce step 190.6 -> 185.8 us, the
# All-to-All step 2493 -> 2333 us.  The dynamic layer's experts hold 40 tile
# rows of capacity, and a routing fills at most 34 of them (4096 +- ~60
# tokens per expert, 34 x 128 = 4352): bands of 34 hold every row a routing
# can fill, and the short band of the 6 rows none reaches is skipped in whole
# waves.  Every CTA then gets the same number of live tiles (its busiest CTA
# 0.3 % above the mean, against 5 % in bands of 32, whose short band leaves
# its live tiles to every fourth CTA).  Interleaved: the step 2785 us in bands
# of 8, 2683 us in one band, 2610 us in bands of 32, 2519 us in bands of 34.
# ReduceScatter's B (22.5 MB) stays in L2 at any band height (106.2 us at 8,
# 107.4 us at 32), so it keeps 8.
WORKLOADS = {
    "worked_example": Workload("worked_example", 1, 256, 512, 256, tile_n=128,
                               swizzle=2, wave_width=2, uniform=True),
    "wave_pattern": Workload("wave_pattern", 2, 2048, 8192, 8192, serpentine=True),
    "allreduce": Workload("allreduce", 3, 4096, 8192, 3584, swizzle=32,
                          consumer=CONS_SUM, n_partials=7, serpentine=True),
    "reducescatter": Workload("reducescatter", 4, 8192, 4096, 2752,
                              layout=LAYOUT_RS_SUBTILE, consumer=CONS_RS,
                              n_dest=4, n_partials=3, serpentine=True),
    "alltoall": Workload("alltoall", 5, 32768, 14336, 4096, swizzle=64,
                         layout=LAYOUT_A2A, consumer=CONS_A2A, n_dest=8,
                         n_tokens=16384, n_experts=8, top_k=2, pad_expert_tile_rows=True,
                         serpentine=True),
    "alltoall_dynamic": Workload("alltoall_dynamic", 6, 8 * 5120, 14336, 4096, swizzle=34,
                                 layout=LAYOUT_A2A, consumer=CONS_A2A, n_dest=8,
                                 n_tokens=16384, n_experts=8, top_k=2, capacity=5120,
                                 serpentine=True),
}


def scaled(w: Workload, **changes) -> Workload:
    """A copy of a workload with some fields changed (smaller parity cases)."""
    d = dict(w.__dict__)
    d.update(changes)
    return Workload(**d)


def _rng(w, stream):
    return np.random.default_rng(1000 * w.index + stream)


def to_bf16_bits(x32: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16) by torch's round-to-nearest-even."""
    t = torch.from_numpy(np.ascontiguousarray(x32, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _draw(w, rng, shape, scale):
    if w.uniform:
        x = rng.uniform(-1.0, 1.0, size=shape).astype(np.float32)
    else:
        x = rng.standard_normal(size=shape, dtype=np.float32) * np.float32(scale)
    return to_bf16_bits(x)


@dataclass
class Inputs:
    A: np.ndarray                 # [M, K] bf16 bits (routed rows for grouped)
    B: list                       # n_experts (or 1) arrays [K, N] bf16 bits
    partials: list                # n_partials arrays [M * N / tile_n, tile_n]
    expert_rows: list             # rows per expert ([M] for a plain GEMM)
    row_token: np.ndarray = None  # grouped: token of each routed row
    row_slot: np.ndarray = None   # grouped: top-k slot of each routed row


def routing(w: Workload, step=0):
    """Top-k routing: every token draws n_experts i.i.d. U(0,1) keys and
    picks the experts with the k smallest keys (distinct), in key order; the
    first pick is slot 0.  Routed rows are sorted by (expert, token, slot).
    Returns (expert_rows, row_token, row_slot).

    With a capacity, every expert has exactly ``capacity`` rows: its routed
    rows in that order, those past the capacity dropped (the router's
    capacity limit), then empty rows (token -1, slot 0)."""
    if w.capacity:
        er, tok, sl = routing(scaled(w, capacity=0), step)
        T, S, r = [], [], 0
        for m in er:
            keep = min(m, w.capacity)
            T.append(tok[r:r + keep])
            S.append(sl[r:r + keep])
            T.append(np.full(w.capacity - keep, -1, np.int32))
            S.append(np.zeros(w.capacity - keep, np.int32))
            r += m
        return ([w.capacity] * w.n_experts, np.concatenate(T).astype(np.int32),
                np.concatenate(S).astype(np.int32))
    rng = _rng(w, 9 + step)
    keys = rng.random((w.n_tokens, w.n_experts))
    picks = np.argsort(keys, axis=1, kind="stable")[:, :w.top_k]
    tok = np.repeat(np.arange(w.n_tokens), w.top_k)
    slot = np.tile(np.arange(w.top_k), w.n_tokens)
    exp = picks.reshape(-1)
    order = np.lexsort((slot, tok, exp))
    expert_rows = np.bincount(exp, minlength=w.n_experts).tolist()
    return expert_rows, tok[order].astype(np.int32), slot[order].astype(np.int32)


def make_inputs(w: Workload, with_partials=True) -> Inputs:
    scale = 1.0 / math.sqrt(w.K)
    if w.grouped:
        expert_rows, row_token, row_slot = routing(w)
        X = _draw(w, _rng(w, 0), (w.n_tokens, w.K), scale)
        A = gather_rows(X, row_token)
        rb = _rng(w, 1)
        B = [_draw(w, rb, (w.K, w.N), scale) for _ in range(w.n_experts)]
    else:
        expert_rows, row_token, row_slot = [w.M], None, None
        A = _draw(w, _rng(w, 0), (w.M, w.K), scale)
        B = [_draw(w, _rng(w, 1), (w.K, w.N), scale)]
    partials = []
    if with_partials and w.n_partials:
        rp = _rng(w, 2)
        units = w.M * w.N // w.tile_n
        for _ in range(w.n_partials):
            x = rp.standard_normal(size=(units, w.tile_n), dtype=np.float32)
            partials.append(to_bf16_bits(x))
    return Inputs(A, B, partials, expert_rows, row_token, row_slot)


def gather_rows(X, row_token):
    """The dispatch gather that forms the routed A: row r is X[token(r)], an
    empty row (token < 0) is zero."""
    A = np.zeros((len(row_token), X.shape[1]), dtype=X.dtype)
    valid = row_token >= 0
    A[valid] = X[row_token[valid]]
    return A


def token_matrix(w: Workload):
    """The grouped workload's token matrix X (n_tokens x K bf16 bits)."""
    return _draw(w, _rng(w, 0), (w.n_tokens, w.K), 1.0 / math.sqrt(w.K))
