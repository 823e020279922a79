"""Device buffers, streams and the per-iteration call sequence of the path.

Plumbing only: torch provides device memory, streams and events; every
step of the path is a libfo.so call (see ``fo.py``).  One iteration is, on
one stream:

  fo_signaled_gemm(epoch) (which resets the counting table itself),
  fo_consume_group(all groups, epoch)   -- a programmatic dependent launch:
                                           runs alongside the GEMM
  fo_reorder_back(all groups)

so the consumer processes each wave group as soon as the GEMM's epilogue
raises that group's flag, while the GEMM keeps computing the rest.  With
overlap off the consumer is an ordinary launch and starts after the GEMM
(the serial baseline).
"""
from dataclasses import dataclass

import numpy as np
import torch

from . import fo
from .workloads import Workload, Inputs

_CONSUMER_OF = {0: fo.FO_CONS_COPY, 1: fo.FO_CONS_SUM, 2: fo.FO_CONS_RS, 3: fo.FO_CONS_A2A}


def _dev_bf16(bits: np.ndarray, device) -> torch.Tensor:
    """uint16 bit array -> device tensor of the same bits (int16 storage)."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device)


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy().view(np.uint16)


@dataclass
class Buffers:
    A: torch.Tensor
    B: list
    partials: list
    C_r: torch.Tensor
    count: torch.Tensor
    flags: torch.Tensor
    status: torch.Tensor
    comm: list        # consumer outputs
    final: list       # post-reorder outputs


class Pipeline:
    """One workload planned and resident on the device."""

    def __init__(self, w: Workload, inp: Inputs, device="cuda", partition=None,
                 wave_width=None, consumer_ctas=0, reorder_ctas=0, upload=True,
                 gemm_variant=None, reserved_consumer_sms=False):
        self.w = w
        self.device = torch.device(device)
        W = w.wave_width if wave_width is None else wave_width
        self.desc_args = dict(
            M=w.M, N=w.N, K=w.K, tile_m=w.tile_m, tile_n=w.tile_n, swizzle=w.swizzle,
            wave_width=W, layout=w.layout, n_dest=w.n_dest,
            expert_rows=inp.expert_rows if w.grouped else None,
            row_token=inp.row_token, row_slot=inp.row_slot,
            pad_expert_tile_rows=w.pad_expert_tile_rows,
            band_order=fo.FO_BAND_SERPENTINE if w.serpentine else fo.FO_BAND_FORWARD)
        probe = fo.make_desc(**self.desc_args, host_only=True)
        self.tiles, self.waves = fo.fo_wave_count(probe)
        self.partition = list(partition) if partition else fo.partition_one_then_two(self.waves)
        self.desc = fo.make_desc(**self.desc_args, group_waves=self.partition)
        self.plan = fo.fo_plan_groups(self.desc)
        self.gemm_variant = fo.FO_GEMM_AUTO if gemm_variant is None else gemm_variant
        self.pairable, self.pair_capacity = fo.fo_plan_set_gemm(self.plan, self.gemm_variant)
        # consumer CTAs only on the SMs the GEMM leaves free (see fo.h)
        self.reserved_consumer_sms = reserved_consumer_sms
        if reserved_consumer_sms:
            fo.fo_plan_set_consumer_placement(self.plan, fo.FO_CONSUMER_RESERVED)
        self.consumer_ctas, self.reorder_ctas = consumer_ctas, reorder_ctas
        self._overlap = None
        _, _, self.group_tiles, _ = fo.fo_plan_info(self.plan)
        self.P = len(self.partition)
        self.kind = _CONSUMER_OF[w.consumer]
        self.dest_units = fo.fo_plan_table(self.plan, fo.FO_TAB_DEST_UNITS)
        self.final_rows = fo.fo_plan_table(self.plan, fo.FO_TAB_FINAL_ROWS)
        self.dest_capacity = fo.fo_plan_table(self.plan, fo.FO_TAB_DEST_CAPACITY)
        if w.grouped:
            # buffers for any routing of the workload's tokens (fo_plan_route)
            R, TN = w.n_dest, w.N // w.tile_n
            self.final_rows = [max(f, len(range(d, w.n_tokens, R)) * w.top_k)
                               for d, f in enumerate(self.final_rows)]
            self.dest_capacity = [max(c, f * TN)
                                  for c, f in zip(self.dest_capacity, self.final_rows)]
        self.s0 = torch.cuda.Stream(device=self.device)
        self.s1 = self.s0   # the consumer follows the GEMM on its stream
        self.epoch = 0
        self.buf = self._alloc(inp) if upload else None

    def _alloc(self, inp):
        d, w = self.device, self.w
        A = _dev_bf16(inp.A, d)
        B = [_dev_bf16(b, d) for b in inp.B]
        partials = [_dev_bf16(p, d) for p in inp.partials]
        C_r = torch.empty((w.M * w.N,), dtype=torch.int16, device=d)
        count = torch.zeros((self.P,), dtype=torch.int32, device=d)
        flags = torch.zeros((self.P,), dtype=torch.int32, device=d)
        status = torch.zeros((1,), dtype=torch.int32, device=d)
        comm = [torch.empty((u * w.tile_n,), dtype=torch.int16, device=d)
                for u in self.dest_capacity]
        # (zeroed: a routing need not fill every row of an All-to-All output)
        final = [torch.zeros((r, w.N), dtype=torch.int16, device=d) for r in self.final_rows]
        return Buffers(A, B, partials, C_r, count, flags, status, comm, final)

    def close(self):
        fo.fo_plan_destroy(self.plan)
        self.plan = None

    def replan(self, partition):
        """Switch to another wave-group partition, keeping the data buffers
        (their sizes do not depend on the partition).  The new plan starts
        from the routing the pipeline was built with."""
        torch.cuda.synchronize(self.device)
        fo.fo_plan_destroy(self.plan)
        self.partition = list(partition)
        self.desc = fo.make_desc(**self.desc_args, group_waves=self.partition)
        self.plan = fo.fo_plan_groups(self.desc)
        fo.fo_plan_set_gemm(self.plan, self.gemm_variant)
        if self.reserved_consumer_sms:
            fo.fo_plan_set_consumer_placement(self.plan, fo.FO_CONSUMER_RESERVED)
        self._overlap = None
        _, _, self.group_tiles, _ = fo.fo_plan_info(self.plan)
        self.P = len(self.partition)
        assert all(u <= c for u, c in zip(fo.fo_plan_table(self.plan, fo.FO_TAB_DEST_UNITS),
                                          self.dest_capacity))
        d = self.device
        self.buf.count = torch.zeros((self.P,), dtype=torch.int32, device=d)
        self.buf.flags = torch.zeros((self.P,), dtype=torch.int32, device=d)
        self.buf.status.zero_()

    def route(self, row_token, row_slot, stream=None):
        """A new routing (device int32 tensors [M]) for the grouped workload:
        fo_plan_route rebuilds the plan's routing tables on the device, in
        stream order before the next step's GEMM."""
        w, st = self.w, stream or self.s0
        assert row_token.dtype == torch.int32 and row_token.numel() == w.M
        assert row_slot.dtype == torch.int32 and row_slot.numel() == w.M
        fo.fo_plan_route(self.plan, row_token.data_ptr(), row_slot.data_ptr(), w.n_tokens,
                         w.top_k, self.buf.status.data_ptr(), st.cuda_stream)
        self._routed = (row_token, row_slot)   # alive until the kernels have read them

    def set_A(self, bits):
        """Replace the routed activations A (uint16 bf16 bits, M x K)."""
        self.buf.A.copy_(_dev_bf16(bits, self.device))

    # ------------------------------------------------------------ calls
    def gemm(self, stream, epoch, signal=True):
        # (the kernel resets the counting table itself before counting)
        b = self.buf
        fo.fo_signaled_gemm(self.plan, b.A.data_ptr(), [x.data_ptr() for x in b.B],
                            b.C_r.data_ptr(), b.count.data_ptr() if signal else 0,
                            b.flags.data_ptr() if signal else 0, epoch, stream.cuda_stream)

    def consume(self, stream, epoch, group=-1, spin_limit_ns=0):
        b = self.buf
        fo.fo_consume_group(self.plan, group, self.kind, b.C_r.data_ptr(),
                            [p.data_ptr() for p in b.partials],
                            [c.data_ptr() for c in b.comm], b.flags.data_ptr(), epoch,
                            spin_limit_ns, b.status.data_ptr(), stream.cuda_stream)

    def reorder(self, stream, g0=0, g1=None):
        b = self.buf
        fo.fo_reorder_back(self.plan, g0, self.P if g1 is None else g1,
                           [c.data_ptr() for c in b.comm], [f.data_ptr() for f in b.final],
                           stream.cuda_stream)

    def consume_reorder(self, stream, epoch, group=-1, spin_limit_ns=0, bias=0,
                        act=fo.FO_ACT_NONE, direct=False):
        """direct: no communication buffers; every unit goes straight to
        its final place."""
        b = self.buf
        fo.fo_consume_reorder(self.plan, group, self.kind, b.C_r.data_ptr(),
                              [p.data_ptr() for p in b.partials],
                              None if direct else [c.data_ptr() for c in b.comm],
                              [f.data_ptr() for f in b.final],
                              bias, act, b.flags.data_ptr(), epoch, spin_limit_ns,
                              b.status.data_ptr(), stream.cuda_stream)

    def set_overlap(self, overlap):
        if overlap != self._overlap:
            fo.fo_plan_set_launch(self.plan, self.consumer_ctas, self.reorder_ctas, overlap)
            self._overlap = overlap

    def step(self, overlap=True, sync_current=True, fused=False, direct=False):
        """One pass of the whole path with a fresh epoch, on stream s0.  With
        overlap the consumer runs alongside the GEMM (dependent launch);
        without, it starts after the GEMM (the serial baseline).  fused: the
        consumer and the post-communication reorder in one kernel; direct
        (with fused): without the communication buffers."""
        self.set_overlap(overlap)
        self.epoch = (self.epoch + 1) & 0xffffffff or 1
        e = self.epoch
        cur = torch.cuda.current_stream(self.device)
        if sync_current:
            self.s0.wait_stream(cur)
        self.gemm(self.s0, e)
        if fused:
            self.consume_reorder(self.s0, e, direct=direct)
        else:
            self.consume(self.s0, e)
            self.reorder(self.s0)
        if sync_current:
            cur.wait_stream(self.s0)
        return e

    # ------------------------------------------------------------ results
    def results(self):
        torch.cuda.synchronize(self.device)
        b = self.buf
        w = self.w
        # the units each destination holds now (after fo_plan_route: as the
        # device tables say)
        self.dest_units = fo.fo_plan_table(self.plan, fo.FO_TAB_DEST_UNITS)
        return dict(
            C_r=_bits(b.C_r).reshape(-1, w.tile_n),
            count=b.count.cpu().numpy().tolist(),
            flags=b.flags.cpu().numpy().view(np.uint32).tolist(),
            status=int(b.status.item()),
            comm=[_bits(c).reshape(-1, w.tile_n)[:u] for c, u in zip(b.comm, self.dest_units)],
            final=[_bits(f) for f in b.final],
        )
