"""Benchmark of the signaled-GEMM + reorder path (one JSON line on rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--per-workload LIST|none]

A step is one pass of the whole path on a workload, inputs resident in HBM:
the signaled GEMM (it resets its own counting table), then the consumer and
the post-communication reorder, by default as one kernel that stores every
unit straight to its final place (a programmatic dependent launch running
alongside the GEMM; ``--step-kernels`` picks the others).  ``value`` is the
GEMM's FLOPs per step divided by the step time (TFLOPS of the whole
overlapped step); for the All-to-All layers only the rows that hold a token
count (2 x routed rows x N x K).  L2 is flushed (a 256 MiB write) before
every timed step, outside the timed events.

The headline workload (default: alltoall, the largest one, 16384 tokens x
top-2 over 8 experts, N=14336, K=4096) gets every measurement: the GEMM
alone (signals on and off), the consumer and the reorder alone, the serial
step (the same kernels, the consumer as an ordinary launch after the GEMM),
the overlap ratio, the GEMM's in-kernel duration inside the step and its
slowdown, the consumer's in-kernel bandwidth inside the step, ``roofline``
of the dominant kernel (the GEMM) against the measured and the nominal
peak, ``e2e`` through the C ABI with host buffers (every step's inputs
copied in from pinned host memory and its output copied back, pipelined
over two buffer sets), and ``cpu_baseline`` (the CPU oracle on a bounded
sample).  Every other workload (``--per-workload``) is timed in the same
process, one after another, with the same step and a compact set of the
same measurements, under ``per_workload``.

For N > 1 (torchrun) every rank runs its own replica of the headline
workload (the path has no data exchange on one node: "replicas only");
value sums the ranks' FLOPs over the slowest rank's time.

``--ncu-gemm`` runs only a few GEMM launches of the workload (the grouped
one optionally cut to ``--experts`` experts): the small case for ncu
captures of the GEMM.
"""
import argparse
import hashlib
import json
import os
import statistics
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np

METRIC = "signaled GEMM TFLOPS (% of bf16 peak); overlap time vs serial GEMM+consumer"
HEADLINE = "alltoall"
PER_WORKLOAD = "wave_pattern,allreduce,reducescatter,alltoall_dynamic"
# Nominal GB300 figures, for fractions beside the measured ones: dense bf16
# tensor throughput (NVIDIA's figures with 2:4 sparsity are twice this) and
# the HBM3e bandwidth.
NOMINAL_BF16_TFLOPS = 2250.0
NOMINAL_HBM_GBS = 8000.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=HEADLINE)
    ap.add_argument("--per-workload", default=PER_WORKLOAD,
                    help="comma-separated workloads timed after the headline in the same "
                         "process ('none': skip)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="target CPU time of the oracle sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-tune", action="store_true",
                    help="skip the tuned-partition report (Algorithm 1)")
    ap.add_argument("--trace-out", default="", help="write per-tile stamps (json)")
    ap.add_argument("--consumer-ctas", type=int, default=0,
                    help="consumer grid (0: library default, by consumer kind)")
    ap.add_argument("--step-kernels", default="auto",
                    choices=["auto", "fused", "separate", "direct"],
                    help="consumer and reorder as one kernel (fo_consume_reorder) or two; "
                         "direct: the fused kernel without communication buffers; "
                         "auto: direct")
    ap.add_argument("--reorder-ctas", type=int, default=0,
                    help="reorder grid (0: library default, 3 per SM)")
    ap.add_argument("--band-order", default="workload",
                    choices=["workload", "forward", "serpentine"],
                    help="column order inside the launch order's bands (default: each "
                         "workload's own)")
    ap.add_argument("--swizzle", type=int, default=0,
                    help="band height of the launch order in tile rows (default: each "
                         "workload's own; e.g. 8 for the bands every workload used before "
                         "the taller ones)")
    ap.add_argument("--wave-width", type=int, default=0,
                    help="W, the GEMM's persistent CTAs and the wave width (default: each "
                         "workload's own, 148)")
    ap.add_argument("--consumer-sms", default="shared", choices=["shared", "reserved"],
                    help="the consumer's CTAs beside the GEMM's (shared) or only on the SMs "
                         "the GEMM leaves free (reserved: [P1] 四's communication SMs)")
    ap.add_argument("--partition", default="workload", choices=["workload", "tuned"],
                    help="the headline's wave-group partition: the workload's own (one wave, "
                         "then groups of two) or Algorithm 1's with the interference factors, "
                         "tuned in this run before the timed steps")
    ap.add_argument("--ncu-gemm", action="store_true",
                    help="only GEMM launches (warm-up + --steps), for ncu captures")
    ap.add_argument("--ncu-step", action="store_true",
                    help="only overlapped steps of the workload (warm-up + --steps), the "
                         "grouped one optionally cut to --experts experts: the small case for "
                         "ncu captures of the consumer")
    ap.add_argument("--ncu-matmul", action="store_true",
                    help="only torch.matmul (cuBLAS) on the workload's operands (warm-up + "
                         "--steps calls), the library reference point for ncu captures")
    ap.add_argument("--experts", type=int, default=0,
                    help="with --ncu-gemm / --ncu-matmul: the grouped workload cut to its "
                         "first experts")
    return ap.parse_args()


def workload(args, name):
    """The named workload, with the launch order's band order and band
    height if given."""
    from communication_overlap_gb300 import workloads as W
    w = W.WORKLOADS[name]
    if args.band_order != "workload":
        w = W.scaled(w, serpentine=args.band_order == "serpentine")
    if getattr(args, "swizzle", 0) > 0:
        w = W.scaled(w, swizzle=args.swizzle)
    if getattr(args, "wave_width", 0) > 0:
        w = W.scaled(w, wave_width=args.wave_width)
    return w


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


# ----------------------------------------------------------------- peaks / clocks

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d["hbm_gbs"], d["bf16_tflops"], d["bf16_tflops_sustained"], "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


class Clocks:
    """SM clock and clock-event reasons sampled DURING the timed region.

    Polls NVML (libnvidia-ml, read-only queries) from a thread every ~2 ms,
    so even a timed region of a few milliseconds gets samples.  Changes no
    setting of the GPU."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, cuda_index):
        import ctypes
        import threading
        self.ctypes, self.threading = ctypes, threading
        self.samples, self.max_mhz, self.handle, self.nvml = [], None, None, None
        try:
            nvml = ctypes.CDLL("libnvidia-ml.so.1")
            if nvml.nvmlInit_v2() != 0:
                return
            count = ctypes.c_uint()
            nvml.nvmlDeviceGetCount_v2(ctypes.byref(count))
            handle = ctypes.c_void_p()
            index = self._nvml_index(nvml, count.value, cuda_index)
            if nvml.nvmlDeviceGetHandleByIndex_v2(index, ctypes.byref(handle)) != 0:
                return
            mx = ctypes.c_uint()
            if nvml.nvmlDeviceGetMaxClockInfo(handle, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = float(mx.value)
            try:
                self.reasons_fn = nvml.nvmlDeviceGetCurrentClocksEventReasons
            except AttributeError:
                self.reasons_fn = nvml.nvmlDeviceGetCurrentClocksThrottleReasons
            self.nvml, self.handle = nvml, handle
        except (OSError, AttributeError):
            pass

    def _nvml_index(self, nvml, count, cuda_index):
        """Match the CUDA device to an NVML device by UUID when possible."""
        ct = self.ctypes
        try:
            import torch
            want = str(torch.cuda.get_device_properties(cuda_index).uuid)
            for i in range(count):
                h = ct.c_void_p()
                buf = ct.create_string_buffer(96)
                if nvml.nvmlDeviceGetHandleByIndex_v2(i, ct.byref(h)) == 0 and \
                        nvml.nvmlDeviceGetUUID(h, buf, 96) == 0 and \
                        want.replace("GPU-", "") in buf.value.decode():
                    return i
        except Exception:
            pass
        return cuda_index if cuda_index < count else 0

    def _poll(self):
        ct = self.ctypes
        clk, reasons = ct.c_uint(), ct.c_ulonglong()
        while not self._stop.is_set():
            if self.nvml.nvmlDeviceGetClockInfo(self.handle, 1, ct.byref(clk)) == 0:
                r = 0
                if self.reasons_fn(self.handle, ct.byref(reasons)) == 0:
                    r = reasons.value
                self.samples.append((float(clk.value), r))
            self._stop.wait(0.002)

    def __enter__(self):
        if self.nvml is not None:
            self._stop = self.threading.Event()
            self._thread = self.threading.Thread(target=self._poll, daemon=True)
            self._thread.start()
        return self

    def __exit__(self, *exc):
        if self.nvml is not None:
            self._stop.set()
            self._thread.join()

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["unsampled"]}
        reasons = set()
        for _, r in self.samples:
            for bit, name in self.REASONS.items():
                if r & bit:
                    reasons.add(name)
        return {"sm_mhz": statistics.median(c for c, _ in self.samples),
                "sm_max_mhz": self.max_mhz, "reasons": sorted(reasons),
                "samples": len(self.samples), "source": "NVML, every ~2 ms"}


# ----------------------------------------------------------------- timing helpers

def timed(torch, stream, fn, steps, flush=None):
    """Run fn() `steps` times on `stream`; CUDA events around each call,
    L2 flushed before each (outside the events).  Returns per-call ms."""
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    torch.cuda.synchronize()
    for a, b in evs:
        if flush is not None:
            with torch.cuda.stream(stream):
                flush()
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def launch_order_key(w):
    """The plan inputs that fix the GEMM's launch order, as the committed ncu
    summaries record them."""
    return (f"swizzle={w.swizzle} serpentine={int(w.serpentine)} "
            f"pad={int(w.pad_expert_tile_rows)}")


def traffic_from_profile(w, kernel_src):
    """Per-launch DRAM bytes of the GEMM on workload `w` from the committed
    ncu summary (profiles/signaled_gemm_<workload>_ncu.md), if it was taken
    on the current source of the kernel and the workload's launch order
    (else None)."""
    path = os.path.join(ROOT, "profiles", f"signaled_gemm_{w.name}_ncu.md")
    try:
        txt = open(path).read()
    except OSError:
        return None
    h = hashlib.sha256(open(kernel_src, "rb").read()).hexdigest()[:16]
    src, order, traffic = None, None, None
    for line in txt.splitlines():
        if line.startswith("source_sha256_16:"):
            src = line.split(":", 1)[1].strip()
        if line.startswith("launch_order:"):
            order = line.split(":", 1)[1].strip()
        if line.startswith("traffic_bytes_per_launch:"):
            try:
                traffic = float(line.split(":", 1)[1].strip())
            except ValueError:
                traffic = None
    return traffic if src == h and order == launch_order_key(w) else None


# ----------------------------------------------------------------- CPU oracle leg

def calibrate_rows(w, inp, cpu_seconds):
    """Output rows of the oracle's GEMM sample: grown by 4x until one GEMM
    on them takes about a quarter of the CPU budget."""
    from oracle import gemm as OG
    rows = 128
    while rows < w.M:
        t0 = time.perf_counter()
        OG.gemm_rows_bf16(inp.A, inp.B, inp.expert_rows, np.arange(rows))
        if time.perf_counter() - t0 > cpu_seconds / 16:
            break
        rows = min(w.M, rows * 4)
    return rows


_LAYOUT_NAMES = {0: "tile", 1: "rs_subtile", 2: "rs_rowblock", 3: "a2a"}


def oracle_plan(w, inp, partition):
    from oracle import plan as OPN
    return OPN.build_plan(inp.expert_rows, w.N, w.K, w.tile_m, w.tile_n, w.swizzle,
                          w.wave_width, partition, _LAYOUT_NAMES[w.layout], w.n_dest,
                          inp.row_token, inp.row_slot,
                          pad_expert_tile_rows=w.pad_expert_tile_rows,
                          serpentine=w.serpentine)


def oracle_rest(w, inp, p, C, groups):
    """Pre-reorder, consumer and post-reorder of the oracle over `groups`
    (None: all), on the GEMM output C."""
    from oracle import comm as OC
    C_r = OC.pre_reorder(p, C, groups)
    if w.consumer == 0:
        recv = OC.consume_copy(p, C_r, groups)
    elif w.consumer == 1:
        recv = OC.consume_sum(p, C_r, inp.partials, groups)
    elif w.consumer == 2:
        recv = OC.consume_rs(p, C_r, inp.partials, groups)
    else:
        recv = OC.consume_a2a(p, C_r, groups)
    if w.layout == 0:
        OC.reorder_back_tile(p, recv, groups)
    elif w.layout in (1, 2):
        OC.reorder_back_rs(p, recv, groups)
    else:
        OC.reorder_back_a2a(p, recv, w.top_k or 2, groups, n_tokens=w.n_tokens or None)


def oracle_sample(w, inp, partition, rows, rest_seconds):
    """Time the CPU oracle on a bounded sample of the workload: the fp64 GEMM
    on the first `rows` output rows, plus pre-reorder, consumer and
    post-reorder on the first wave groups (all of them when that fits in
    about `rest_seconds`), each scaled to the full step.  The plan is built
    once per shape and not counted, except with a routing that changes every
    step.  Returns (seconds per full step estimate, description, cores)."""
    from oracle import gemm as OG

    t0 = time.perf_counter()
    OG.gemm_rows_bf16(inp.A, inp.B, inp.expert_rows, np.arange(rows))
    t_rows = time.perf_counter() - t0
    gemm_full = t_rows * (w.M / rows)
    t0 = time.perf_counter()
    p = oracle_plan(w, inp, partition)
    t_plan = time.perf_counter() - t0
    # the rest of the path (values do not matter for the time): group 0
    # first, then as many leading groups as the budget allows
    C = np.zeros((w.M, w.N), dtype=np.uint16)
    units = [int(p.part_len[j].sum()) for j in range(p.n_groups)]
    t0 = time.perf_counter()
    oracle_rest(w, inp, p, C, [0])
    t0_rest = time.perf_counter() - t0
    per_unit = t0_rest / max(1, units[0])
    g = 1
    while g < p.n_groups and sum(units[:g + 1]) * per_unit <= rest_seconds:
        g += 1
    if g > 1:
        t0 = time.perf_counter()
        oracle_rest(w, inp, p, C, list(range(g)))
        t_rest = time.perf_counter() - t0
    else:
        t_rest = t0_rest
    rest_full = t_rest * p.n_units / max(1, sum(units[:g]))
    plan_s = t_plan if w.capacity else 0.0
    plan_note = (f"plan ({t_plan:.2f} s) included: the routing changes every step"
                 if w.capacity else f"plan ({t_plan:.2f} s) excluded")
    desc = (f"fp64 GEMM on {rows} of {w.M} output rows ({t_rows:.2f} s, scaled x"
            f"{w.M / rows:.1f}) + pre-reorder, consumer and post-reorder on the first "
            f"{g} of {p.n_groups} wave groups ({t_rest:.2f} s, scaled x"
            f"{p.n_units / max(1, sum(units[:g])):.2f}); {plan_note}")
    return gemm_full + rest_full + plan_s, desc, os.cpu_count()


def run_reference(args):
    """--impl reference: the CPU oracle, as it stands, on this host's cores."""
    rank, _, world = dist_env()
    if rank != 0:
        return 0
    from communication_overlap_gb300 import workloads as W
    from oracle import plan as OPN
    w = workload(args, args.workload)
    inp = W.make_inputs(w)
    tiles_m = [-(-m // w.tile_m) for m in inp.expert_rows]
    if w.pad_expert_tile_rows:
        tiles_m = [t + t % 2 for t in tiles_m]
    tiles = sum(tiles_m) * (w.N // w.tile_n)
    partition = OPN.one_then_two(OPN.wave_count(tiles, w.wave_width))
    per = []
    # a few seconds of CPU work per step, so the whole run ends in minutes
    budget = max(2.0, 150.0 / max(1, args.steps + args.warmup))
    rows = calibrate_rows(w, inp, budget / 2)
    desc = ""
    for i in range(args.warmup + args.steps):
        secs, desc, cores = oracle_sample(w, inp, partition, rows, budget / 2)
        if i >= args.warmup:
            per.append(secs)
    step_s = statistics.mean(per)
    value = 2.0 * moved_rows(w, inp) * w.N * w.K / step_s / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOPS",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": step_s * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_name(w)},
        "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": os.cpu_count(),
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def workload_name(w):
    if w.grouped:
        cap = (f", capacity {w.capacity} rows per expert (M={w.M}), a new routing built on "
               f"the device every step" if w.capacity else "")
        pad = (", expert grids padded to even tile-row counts (CTA pairs)"
               if w.pad_expert_tile_rows else "")
        pad += ", serpentine bands" if w.serpentine else ""
        return (f"{w.name}: grouped bf16 GEMM {w.n_tokens} tokens x top-{w.top_k} over "
                f"{w.n_experts} experts, N={w.N} K={w.K}, {w.tile_m}x{w.tile_n} tiles, "
                f"W={w.wave_width}, swizzle {w.swizzle}{cap}{pad}")
    return (f"{w.name}: bf16 GEMM M={w.M} N={w.N} K={w.K}, {w.tile_m}x{w.tile_n} tiles, "
            f"W={w.wave_width}, swizzle {w.swizzle}"
            + (", serpentine bands" if w.serpentine else ""))


# ----------------------------------------------------------------- our path

STEP_KERNELS = {
    "direct": "signaled GEMM + one consumer kernel that stores every unit straight to "
              "its final place (communication and post-communication reorder fused)",
    "fused": "signaled GEMM + one consumer kernel that writes the communication buffers "
             "and moves each chunk on to its final place",
    "separate": "signaled GEMM + consumer + post-communication reorder",
}


class Bench:
    """One workload planned and resident, with the step and the timing legs
    the headline and the per-workload records share."""

    def __init__(self, ctx, w, args, inp=None, routes=None):
        from communication_overlap_gb300 import workloads as W
        from communication_overlap_gb300.pipeline import Pipeline
        self.ctx, self.w, self.args = ctx, w, args
        torch, dev = ctx["torch"], ctx["dev"]
        # (inputs and routings of another Bench of the same workload may be
        # passed in: they do not depend on the launch order)
        self.inp = W.make_inputs(w) if inp is None else inp
        self.pipe = Pipeline(w, self.inp, device=dev, consumer_ctas=args.consumer_ctas,
                             reorder_ctas=args.reorder_ctas,
                             reserved_consumer_sms=getattr(args, "consumer_sms",
                                                           "shared") == "reserved")
        self.s = self.pipe.s0
        # FLOPs of the rows that hold a token: with fixed expert capacities
        # the empty rows are not work (the GEMM skips tiles that have none)
        self.flops = 2.0 * moved_rows(w, self.inp) * w.N * w.K
        self.kernels = "direct" if args.step_kernels == "auto" else args.step_kernels
        self.fused = self.kernels in ("fused", "direct")
        self.direct = self.kernels == "direct"
        # Dynamic routing (expert capacities fixed): every step takes the
        # next of a few routings resident in HBM, with its routed A (the
        # dispatch gather, outside the path), and rebuilds the routing tables
        # on the device (fo_plan_route) before its GEMM.
        self.dyn = w.capacity > 0
        self.routes = list(routes) if routes else []
        if self.dyn and not self.routes:
            X = W.token_matrix(w)
            for k in range(1, 5):
                _, tok, sl = W.routing(w, k)
                self.routes.append((torch.from_numpy(tok).to(dev),
                                    torch.from_numpy(sl).to(dev),
                                    torch.from_numpy(W.gather_rows(X, tok).view(np.int16))
                                    .to(dev)))
            del X
        self.turn = 0

    def step(self, **kw):
        if self.dyn:
            tok, sl, A = self.routes[self.turn % len(self.routes)]
            self.turn += 1
            self.pipe.buf.A = A
            self.pipe.route(tok, sl)
        return self.pipe.step(**kw)

    def ovl(self):
        self.step(overlap=True, sync_current=False, fused=self.fused, direct=self.direct)

    def timed(self, fn, steps=None):
        return timed(self.ctx["torch"], self.s, fn, steps or self.args.steps, self.ctx["flush"])

    def close(self):
        self.pipe.close()

    # ------------------------------------------------------------------ legs
    def warm(self):
        torch = self.ctx["torch"]
        for _ in range(max(3, self.args.warmup)):
            self.step(overlap=True, fused=self.fused, direct=self.direct)
        torch.cuda.synchronize()
        assert int(self.pipe.buf.status.item()) == 0, "consumer wait timed out"
        assert self.pipe.buf.count.cpu().tolist() == self.pipe.group_tiles

    def consumer_bytes(self):
        return consumer_bytes(self.w, self.inp)

    def gemm_spans(self):
        """The GEMM's in-kernel duration (first CTA start to last tile, from
        the per-tile globaltimer stamps) alone and inside the overlapped
        step, `steps` times each, L2 flushed before each."""
        torch, fo = self.ctx["torch"], self.ctx["fo"]
        pipe, w = self.pipe, self.w
        trace = torch.zeros(pipe.tiles + 3 * w.wave_width, dtype=torch.int64,
                            device=pipe.device)
        fo.fo_plan_set_trace(pipe.plan, trace.data_ptr())

        def span():
            t = trace.cpu().numpy().astype(np.int64)
            starts = t[pipe.tiles:pipe.tiles + min(w.wave_width, pipe.tiles)]
            return (t[:pipe.tiles].max() - starts.min()) / 1e6

        alone, in_step = [], []
        for _ in range(self.args.steps):
            with torch.cuda.stream(self.s):
                self.ctx["flush"]()
            pipe.gemm(self.s, pipe.epoch)
            torch.cuda.synchronize()
            alone.append(span())
            with torch.cuda.stream(self.s):
                self.ctx["flush"]()
            self.step(overlap=True, fused=self.fused, direct=self.direct)
            torch.cuda.synchronize()
            in_step.append(span())
        fo.fo_plan_set_trace(pipe.plan, 0)
        return statistics.median(alone), statistics.median(in_step)

    def consumer_in_step(self, reps=3):
        """The consumer's bandwidth inside the overlapped step, from one
        traced step: group j's flag rises with its last tile (GEMM stamps);
        its consumer is busy from max(flag_j, end of group j-1) to the end of
        its last chunk (consumer stamps).  Bytes are the consumer's
        algorithmic bytes of the group (sources read once, output written
        once).  Median over `reps` steps of: all groups, the groups that
        complete while the GEMM still runs, and the last group (after it)."""
        torch, fo = self.ctx["torch"], self.ctx["fo"]
        pipe, w = self.pipe, self.w
        sm = self.ctx["sm_count"]
        trace = torch.zeros(pipe.tiles + 3 * w.wave_width, dtype=torch.int64,
                            device=pipe.device)
        ctrace = torch.zeros(2 * pipe.P + 4 * 4 * sm, dtype=torch.int64, device=pipe.device)
        per_unit = self.consumer_bytes() / max(1, moved_rows(w, self.inp) * (w.N // w.tile_n))
        out = {"all": [], "during_gemm": [], "last_group": [], "busy_us": []}
        for _ in range(reps):
            fo.fo_plan_set_trace(pipe.plan, trace.data_ptr(), ctrace.data_ptr())
            with torch.cuda.stream(self.s):
                self.ctx["flush"]()
                ctrace.zero_()
            self.step(overlap=True, fused=self.fused, direct=self.direct)
            torch.cuda.synchronize()
            fo.fo_plan_set_trace(pipe.plan, 0, 0)
            st = trace.cpu().numpy().astype(np.int64)
            cs = ctrace.cpu().numpy().astype(np.int64)
            slot_group = np.asarray(fo.fo_plan_table(pipe.plan, fo.FO_TAB_SLOT_GROUP))
            part_len = np.asarray(fo.fo_plan_table(pipe.plan, fo.FO_TAB_PART_LEN))
            units = part_len.reshape(pipe.P, -1).sum(axis=1)
            tile_done = st[:pipe.tiles]
            gemm_end = tile_done.max()
            # groups with units (a group of empty All-to-All tiles has none
            # and leaves no consumer stamp)
            live = np.nonzero(units > 0)[0]
            if live.size == 0 or (cs[live] == 0).any():
                continue
            flag = np.array([tile_done[slot_group == j].max() for j in live])
            done = cs[live]
            start = np.maximum(flag, np.concatenate(([flag[0]], done[:-1])))
            busy = np.maximum(done - start, 1)
            nbytes = units[live] * per_unit
            during = flag < gemm_end
            out["all"].append(nbytes.sum() / busy.sum())
            if during.any():
                out["during_gemm"].append(nbytes[during].sum() / busy[during].sum())
            if busy[-1] >= 3000:   # a group that short is not timed by its stamps
                out["last_group"].append(nbytes[-1] / busy[-1])
            out["busy_us"].append(busy.sum() / 1e3)
        res = {}
        for k, v in out.items():
            res[k] = statistics.median(v) if v else None
        hbm = self.ctx["hbm"]
        return {"gbs": res["all"], "gbs_groups_during_gemm": res["during_gemm"],
                "gbs_last_group": res["last_group"], "busy_us": res["busy_us"],
                "frac_of_measured": res["all"] / hbm if res["all"] else None,
                "frac_of_nominal": res["all"] / NOMINAL_HBM_GBS if res["all"] else None,
                "how": "per group: algorithmic bytes / (end of its last chunk - max(its "
                       "flag, end of the previous group)), from globaltimer stamps of one "
                       "traced overlapped step (median of 3)"}

    def alone_legs(self):
        """Consumer and reorder alone (flags of the last epoch already raised;
        ordinary launches so nothing overlaps the flush before them)."""
        fo, pipe, s = self.ctx["fo"], self.pipe, self.s
        torch = self.ctx["torch"]
        sm = self.ctx["sm_count"]
        pipe.step(overlap=True)
        torch.cuda.synchronize()
        pipe.set_overlap(False)
        r = {}
        r["direct"] = self.timed(lambda: pipe.consume_reorder(s, pipe.epoch, direct=True))
        r["consumer"] = self.timed(lambda: pipe.consume(s, pipe.epoch))
        r["reorder"] = self.timed(lambda: pipe.reorder(s))
        # a full grid (4 CTAs per SM): the bandwidth roofline figure; the step
        # uses the library's default grid for running beside the GEMM
        fo.fo_plan_set_launch(pipe.plan, 4 * sm, self.args.reorder_ctas, False)
        r["direct_full"] = self.timed(lambda: pipe.consume_reorder(s, pipe.epoch, direct=True))
        r["consumer_full"] = self.timed(lambda: pipe.consume(s, pipe.epoch))
        fo.fo_plan_set_launch(pipe.plan, self.args.consumer_ctas, self.args.reorder_ctas, False)
        pipe.set_overlap(True)
        # The reorder's bytes moved by a plain device-to-device copy
        # (torch.Tensor.copy_), timed the same way: the event-timed ceiling
        # of a move of this size, launch ramp and tail included.
        n = moved_rows(self.w, self.inp) * self.w.N * 2
        src = torch.empty(n, dtype=torch.uint8, device=self.ctx["dev"])
        dst = torch.empty_like(src)

        def plain_copy():
            with torch.cuda.stream(s):
                dst.copy_(src)
        plain_copy()
        r["plain_copy"] = self.timed(plain_copy)
        del src, dst
        return {k: statistics.mean(v) for k, v in r.items()}

    def torch_mm(self):
        """torch.matmul (cuBLAS) on the same operands, one call per expert."""
        torch, w = self.ctx["torch"], self.w
        A_bf = self.pipe.buf.A.view(torch.bfloat16).view(w.M, w.K)
        B_bf = [b.view(torch.bfloat16).view(w.K, w.N) for b in self.pipe.buf.B]
        rows = np.cumsum([0] + list(self.inp.expert_rows))

        def mm():
            with torch.cuda.stream(self.s):
                for e, Bm in enumerate(B_bf):
                    torch.matmul(A_bf[rows[e]:rows[e + 1]], Bm)
        for _ in range(3):   # cuBLAS handle, workspace and kernel choice
            mm()
        return statistics.mean(self.timed(mm))

    def record(self, ms_ov, ms_ser, ms_gemm, clk):
        """The per-workload record (shared by the headline's detail)."""
        w, pipe = self.w, self.pipe
        ctx = self.ctx
        hbm, peak = ctx["hbm"], ctx["peak_burst"]
        alone = self.alone_legs()
        span_alone, span_step = self.gemm_spans()
        cb = self.consumer_bytes()
        reo_bytes = 2 * moved_rows(w, self.inp) * w.N * 2
        ms_mm = self.torch_mm()
        gemm_tf = self.flops / (ms_gemm * 1e-3) / 1e12

        floor = ctx["event_floor_ms"]

        def bw(nbytes, ms):
            g = nbytes / (ms * 1e-3) / 1e9
            out = {"ms": ms, "gbs": g, "frac_of_measured": g / hbm,
                   "frac_of_nominal": g / NOMINAL_HBM_GBS}
            if ms > 2 * floor:   # the kernel's own time: the launch and event floor taken out
                gk = nbytes / ((ms - floor) * 1e-3) / 1e9
                out.update({"gbs_floor_removed": gk, "frac_of_measured_floor_removed": gk / hbm})
            return out
        return {
            "config": workload_name(w),
            "partition": pipe.partition, "groups_tiles": pipe.group_tiles,
            "consumer": consumer_name(w), "gemm_pairs": bool(pipe.pairable),
            "value_tflops": self.flops / (ms_ov * 1e-3) / 1e12,
            "ms_overlapped_step": ms_ov, "ms_serial_step": ms_ser,
            "overlap_speedup": ms_ser / ms_ov,
            "ms_gemm_alone": ms_gemm, "gemm_tflops_alone": gemm_tf,
            "gemm_frac_of_measured_peak": gemm_tf / peak,
            "gemm_frac_of_nominal_peak": gemm_tf / NOMINAL_BF16_TFLOPS,
            "ms_torch_matmul": ms_mm,
            "torch_matmul_tflops": self.flops / (ms_mm * 1e-3) / 1e12,
            "gemm_in_kernel_ms_alone": span_alone, "gemm_in_kernel_ms_in_step": span_step,
            "gemm_slowdown": span_step / span_alone,
            # DRAM bytes per GEMM launch from the committed ncu summary taken
            # on this kernel source and launch order (None if there is none)
            "gemm_traffic_bytes": traffic_from_profile(
                w, os.path.join(ROOT, "communication_overlap_gb300", "csrc", "gemm.cu")),
            "consumer_bytes": cb,
            "direct_alone_step_grid": bw(cb, alone["direct"]),
            "direct_alone_full_grid": bw(cb, alone["direct_full"]),
            "consumer_in_step": self.consumer_in_step(),
            "consumer_alone_step_grid": bw(cb, alone["consumer"]),
            "consumer_alone_full_grid": bw(cb, alone["consumer_full"]),
            "reorder_alone": bw(reo_bytes, alone["reorder"]),
            "plain_copy_same_bytes": bw(reo_bytes, alone["plain_copy"]),
            "reorder_frac_of_plain_copy": alone["plain_copy"] / alone["reorder"],
            "clocks": clk,
            "status_ok": int(pipe.buf.status.item()) == 0,
        }


def band8_leg(ctx, b, args, reps=3):
    """The workload on the same inputs with bands of 8 tile rows (swizzle
    8, the per-configuration launch order every workload used before the
    taller bands), timed alternately with its own launch order: the GEMM
    alone and the overlapped step, medians over 2 * `reps` runs of --steps
    steps each, the order reversed every other time.  None for a workload whose bands are already 8
    high."""
    from communication_overlap_gb300 import workloads as W_
    if b.w.swizzle == 8:
        return None
    torch = ctx["torch"]
    b8 = Bench(ctx, W_.scaled(b.w, swizzle=8), args, inp=b.inp, routes=b.routes)
    try:
        b8.warm()
        g8, g, st8, st = [], [], [], []

        def legs(x, out_step, out_gemm):
            out_step.append(statistics.mean(x.timed(x.ovl)))
            out_gemm.append(statistics.mean(x.timed(lambda: x.pipe.gemm(x.s, x.pipe.epoch))))
        with Clocks(ctx["local"]) as clk:
            # the order alternates, so that a clock that drifts (the power
            # cap) favours neither launch order
            for r in range(2 * reps):
                if r % 2 == 0:
                    legs(b8, st8, g8)
                    legs(b, st, g)
                else:
                    legs(b, st, g)
                    legs(b8, st8, g8)
        torch.cuda.synchronize()
        return {"swizzle": 8, "workload_swizzle": b.w.swizzle,
                "ms_overlapped_step": statistics.median(st8),
                "ms_overlapped_step_workload_swizzle": statistics.median(st),
                "value_tflops": b.flops / (statistics.median(st8) * 1e-3) / 1e12,
                "ms_gemm_alone": statistics.median(g8),
                "ms_gemm_alone_workload_swizzle": statistics.median(g),
                "clocks": clk.summary(),
                "status_ok": int(b8.pipe.buf.status.item()) == 0,
                "note": "the same inputs, GEMM and consumer; only the launch order's band "
                        "height differs; timed alternately in one loop"}
    finally:
        b8.close()
        del b8
        torch.cuda.empty_cache()


def measure_compact(ctx, w, args):
    """A workload other than the headline: the overlapped and serial steps,
    the GEMM alone, the GEMM's slowdown, the consumer's bandwidth (alone and
    inside the step) and the clocks of the overlapped steps."""
    torch = ctx["torch"]
    b = Bench(ctx, w, args)
    try:
        b.warm()
        with Clocks(ctx["local"]) as clk:
            t_ov = b.timed(b.ovl)
        t_ser = b.timed(lambda: b.step(overlap=False, sync_current=False, fused=b.fused,
                                       direct=b.direct))
        t_gemm = b.timed(lambda: b.pipe.gemm(b.s, b.pipe.epoch))
        rec = b.record(statistics.mean(t_ov), statistics.mean(t_ser), statistics.mean(t_gemm),
                       clk.summary())
        rec["step_kernels"] = b.kernels
        rec["swizzle_8"] = band8_leg(ctx, b, args)
        return rec
    finally:
        b.close()
        del b
        torch.cuda.empty_cache()


def ncu_case(args):
    """The workload of an ncu capture and its inputs, the grouped workload
    optionally cut to its first --experts experts."""
    from communication_overlap_gb300 import workloads as W
    w = workload(args, args.workload)
    inp = W.make_inputs(w)
    if w.grouped and args.experts:
        e = args.experts
        rows = int(sum(inp.expert_rows[:e]))
        tok = np.asarray(inp.row_token[:rows])
        w = W.scaled(w, M=rows, n_experts=e, n_tokens=int(tok.max()) + 1)
        inp.A, inp.B = inp.A[:rows], inp.B[:e]
        inp.expert_rows = inp.expert_rows[:e]
        inp.row_token, inp.row_slot = inp.row_token[:rows], inp.row_slot[:rows]
    return w, inp


def run_ncu_gemm(args):
    """Only GEMM launches of the workload (optionally its first --experts
    experts): the small case for ncu captures of the GEMM."""
    import torch
    from communication_overlap_gb300.pipeline import Pipeline
    w, inp = ncu_case(args)
    pipe = Pipeline(w, inp)
    for _ in range(args.warmup):
        pipe.gemm(pipe.s0, 1)
    for _ in range(args.steps):
        pipe.gemm(pipe.s0, 1)
    torch.cuda.synchronize()
    ok = pipe.buf.count.cpu().tolist() == pipe.group_tiles
    print(json.dumps({"ncu_gemm": w.name, "M": w.M, "experts": w.n_experts,
                      "tiles": pipe.tiles, "launches": args.warmup + args.steps,
                      "flops_per_launch": 2.0 * moved_rows(w, inp) * w.N * w.K,
                      "count_ok": ok}))
    pipe.close()
    return 0 if ok else 1


def run_ncu_step(args):
    """Only overlapped steps (the benchmark's step kernels) of the workload,
    optionally cut to its first --experts experts."""
    import torch
    from communication_overlap_gb300.pipeline import Pipeline
    w, inp = ncu_case(args)
    pipe = Pipeline(w, inp)
    kernels = "direct" if args.step_kernels == "auto" else args.step_kernels
    kw = dict(fused=kernels in ("fused", "direct"), direct=kernels == "direct")
    for _ in range(args.warmup + args.steps):
        pipe.step(overlap=True, **kw)
    torch.cuda.synchronize()
    ok = int(pipe.buf.status.item()) == 0 and pipe.buf.count.cpu().tolist() == pipe.group_tiles
    print(json.dumps({"ncu_step": w.name, "M": w.M, "experts": w.n_experts,
                      "steps": args.warmup + args.steps, "step_kernels": kernels, "ok": ok}))
    pipe.close()
    return 0 if ok else 1


def run_ncu_matmul(args):
    """torch.matmul (cuBLAS) on the workload's operands, one call per
    expert: the library reference point of an ncu capture."""
    import torch
    w, inp = ncu_case(args)
    A = torch.from_numpy(inp.A.view(np.int16)).cuda().view(torch.bfloat16)
    B = [torch.from_numpy(b.view(np.int16)).cuda().view(torch.bfloat16) for b in inp.B]
    rows = np.cumsum([0] + list(inp.expert_rows))
    for _ in range(args.warmup + args.steps):
        for e, Bm in enumerate(B):
            torch.matmul(A[rows[e]:rows[e + 1]], Bm)
    torch.cuda.synchronize()
    print(json.dumps({"ncu_matmul": w.name, "M": w.M, "experts": len(B),
                      "calls": (args.warmup + args.steps) * len(B)}))
    return 0


def run_ours(args):
    import torch
    import torch.distributed as dist
    from communication_overlap_gb300 import fo
    from communication_overlap_gb300 import workloads as W

    rank, local, world = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    hbm, peak_burst, peak_sust, peak_kind = measured_peaks()
    flush_buf = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    ctx = dict(torch=torch, fo=fo, dev=dev, local=local, hbm=hbm, peak_burst=peak_burst,
               sm_count=torch.cuda.get_device_properties(dev).multi_processor_count,
               flush=lambda: flush_buf.fill_(1))
    # the launch and event floor: a one-element kernel timed like every leg
    # (events on the stream around it, after the flush)
    tiny = torch.zeros(1, device=dev)
    s_tiny = torch.cuda.Stream(dev)
    for _ in range(3):
        with torch.cuda.stream(s_tiny):
            tiny.add_(1)

    def one_tiny():
        with torch.cuda.stream(s_tiny):
            tiny.add_(1)
    ctx["event_floor_ms"] = statistics.median(timed(torch, s_tiny, one_tiny, args.steps,
                                                    ctx["flush"]))
    w = workload(args, args.workload)
    b = Bench(ctx, w, args)
    pipe, s, flops, inp = b.pipe, b.s, b.flops, b.inp
    fused, direct, dyn, kernels = b.fused, b.direct, b.dyn, b.kernels
    sm_count = ctx["sm_count"]

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    # --partition tuned: Algorithm 1 (with the interference factors) picks the
    # headline's partition, its offline inputs measured here first
    pre_tuned = None
    if args.partition == "tuned":
        b.warm()
        ms_g = statistics.mean(b.timed(lambda: pipe.gemm(s, pipe.epoch)))
        pre_tuned = tune_partition(w, inp, ms_gemm_for_tuning=ms_g, partition=pipe.partition,
                                   steps=max(10, args.steps // 2))
        pipe.replan(pre_tuned["partition_interference"])

    # warm-up (also the first correctness evidence: status and counting table)
    b.warm()

    # the headline: overlapped steps
    barrier()
    with Clocks(local) as clk:
        t_ov = b.timed(b.ovl)
    barrier()
    ms_ov = statistics.mean(t_ov)
    status_ok = int(pipe.buf.status.item()) == 0

    # every overlapped variant: separate kernels, fused, fused direct
    t_var, clk_var = {}, {}
    for name, kw in (("separate", dict(fused=False)), ("fused", dict(fused=True)),
                     ("direct", dict(fused=True, direct=True))):
        with Clocks(local) as c_:
            t_var[name] = b.timed(lambda: b.step(overlap=True, sync_current=False, **kw))
        clk_var[name] = c_.summary()
    # serial = the same kernels as the overlapped step, the consumer as an
    # ordinary launch after the GEMM; and the separate kernels serially
    t_ser = b.timed(lambda: b.step(overlap=False, sync_current=False, fused=fused,
                                   direct=direct))
    t_ser_sep = b.timed(lambda: b.step(overlap=False, sync_current=False))
    t_route = []
    if dyn:   # the two routing kernels alone
        t_route = b.timed(lambda: pipe.route(*b.routes[0][:2]))
    # GEMM alone (signals on, as in the step; and off)
    t_gemm = b.timed(lambda: pipe.gemm(s, pipe.epoch))
    t_gemm_nosig = b.timed(lambda: pipe.gemm(s, pipe.epoch, signal=False))
    ms_gemm_local = statistics.mean(t_gemm)
    rec = b.record(ms_ov, statistics.mean(t_ser), ms_gemm_local, clk.summary())

    # the overlapped step again after about a second of back-to-back steps:
    # the power-limited steady state of a long run
    n_hot = max(args.steps, int(1000.0 / max(ms_ov, 1e-3)))
    for _ in range(n_hot):
        b.ovl()
    with Clocks(local) as clk_hot:
        t_hot = b.timed(b.ovl)
    sustained = {"ms_overlapped_step": statistics.mean(t_hot),
                 "value_tflops": flops / (statistics.mean(t_hot) * 1e-3) / 1e12,
                 "steps_before": n_hot, "clocks": clk_hot.summary(),
                 "note": "the same overlapped step timed after about 1 s of back-to-back "
                         "steps (no flush between them); the headline is timed after the "
                         "warm-up"}

    # reading of the wave: W = the GEMM's persistent CTAs; the workloads fix
    # W = 148, and where the device has another SM count the same path with
    # W = that count is timed beside it
    w_sm = None
    # (with the reserved placement W = the SM count leaves the consumer no SM)
    if sm_count != w.wave_width and world == 1 and args.consumer_sms == "shared":
        from communication_overlap_gb300 import workloads as W_
        b_sm = Bench(ctx, W_.scaled(w, wave_width=sm_count), args)
        try:
            b_sm.warm()
            t_gemm_sm = b_sm.timed(lambda: b_sm.pipe.gemm(b_sm.s, b_sm.pipe.epoch))
            t_step_sm = b_sm.timed(b_sm.ovl)
            w_sm = {"wave_width": sm_count, "waves": b_sm.pipe.waves,
                    "gemm_pairs": bool(b_sm.pipe.pairable),
                    "ms_gemm_alone": statistics.mean(t_gemm_sm),
                    "ms_overlapped_step": statistics.mean(t_step_sm),
                    "value_tflops": flops / (statistics.mean(t_step_sm) * 1e-3) / 1e12,
                    "status_ok": int(b_sm.pipe.buf.status.item()) == 0}
        finally:
            b_sm.close()
            del b_sm
            torch.cuda.empty_cache()

    # the launch order every workload used before the taller bands, on the
    # same inputs, alternated with the workload's own
    band8 = band8_leg(ctx, b, args) if world == 1 else None

    if args.trace_out:
        write_trace(ctx, b, args.trace_out)

    e2e = measure_e2e(ctx, b, args)

    # Algorithm 1 on this workload: the offline inputs (this run's GEMM time
    # and the consumer's latency curve, sampled) and the exact search; then
    # the overlapped step with the tuned partition against the workload's
    # own, alternating.  Reported beside the headline, which keeps the
    # workload's partition.
    tuned = None
    if not args.no_tune and pre_tuned is None:
        try:
            tuned = tune_partition(w, inp, ms_gemm_for_tuning=ms_gemm_local,
                                   partition=pipe.partition, steps=max(10, args.steps // 2))
        except Exception as e:   # a report, not the benchmark: keep the line
            tuned = {"error": f"{type(e).__name__}: {e}"}
    group_tiles, partition = pipe.group_tiles, pipe.partition
    b.close()
    del b
    torch.cuda.empty_cache()

    # every other workload, in the same process (one GPU, one replica)
    per = {}
    names = [] if args.per_workload in ("", "none") else args.per_workload.split(",")
    if world == 1:
        for name in names:
            if name == args.workload:
                continue
            try:
                per[name] = measure_compact(ctx, workload(args, name), args)
            except Exception as e:   # keep the headline line
                per[name] = {"error": f"{type(e).__name__}: {e}"}

    # max over ranks
    def rmax(x):
        return max_over_ranks(x, dist if world > 1 else None, dev)

    ms_ov = rmax(ms_ov)
    ms_ser = rmax(statistics.mean(t_ser))
    ms_gemm = rmax(ms_gemm_local)
    ms_e2e = rmax(e2e["ms_pipelined"])
    ms_e2e_serial = rmax(e2e["ms_one_step_at_a_time"])

    gemm_tflops = flops / (ms_gemm * 1e-3) / 1e12
    traffic = traffic_from_profile(w, os.path.join(ROOT, "communication_overlap_gb300",
                                                         "csrc", "gemm.cu"))
    out = None
    if rank == 0:
        cpu = None
        if not args.no_cpu_baseline:
            rows = calibrate_rows(w, inp, args.cpu_seconds / 2)
            secs, desc, cores = oracle_sample(w, inp, partition, rows, args.cpu_seconds / 2)
            cpu = {"value": flops / secs / 1e12, "unit": "TFLOPS", "cores": cores,
                   "kind": "oracle", "sample": desc}
        headline = dict(rec)
        headline.update({
            "overlapped_step_kernels": kernels,
            "ms_overlapped_step_median": statistics.median(t_ov),
            "ms_overlapped_step_by_kernels": {k: statistics.mean(v) for k, v in t_var.items()},
            "clocks_by_kernels": clk_var,
            "sustained": sustained,
            "partition_mode": args.partition,
            "w_sm_count": w_sm,
            "swizzle_8": band8,
            "partition_tuned_before_timing": pre_tuned,
            "ms_serial_step_separate_kernels": statistics.mean(t_ser_sep),
            "ms_gemm_alone_no_signal": statistics.mean(t_gemm_nosig),
            "gemm_frac_of_sustained": gemm_tflops / peak_sust,
            "hbm_peak_gbs": hbm, "nominal_hbm_gbs": NOMINAL_HBM_GBS,
            "event_floor_ms": ctx["event_floor_ms"],
            "nominal_bf16_tflops": NOMINAL_BF16_TFLOPS,
            "status_ok": status_ok,
            "tuned_partition": tuned,
        })
        if dyn:
            headline.update({"ms_route_alone": statistics.mean(t_route),
                             "routings": "4 routings resident in HBM, taken in turn, one "
                                         "per step"})
        out = {
            "metric": METRIC,
            "value": whole_job_tflops(world, flops, ms_ov),
            "unit": "TFLOPS",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms_ov, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": workload_name(w), "partition": partition,
                       "groups_tiles": group_tiles, "consumer": consumer_name(w),
                       "l2": "flushed before every timed step (256 MiB write)",
                       "consumer_ctas": args.consumer_ctas or "library default",
                       "consumer_sms": args.consumer_sms,
                       "step_kernels": STEP_KERNELS[kernels],
                       "parallelism": f"replicas x{world}"},
            "roofline": {"bound": "tensor", "achieved": gemm_tflops, "peak": peak_burst,
                         "unit": "TFLOP/s", "frac": gemm_tflops / peak_burst,
                         "frac_nominal": gemm_tflops / NOMINAL_BF16_TFLOPS,
                         "nominal_peak": NOMINAL_BF16_TFLOPS,
                         "traffic": traffic,
                         "kernel": "signaled_gemm_kernel (alone, signals on)",
                         "peak_source": f"{peak_kind} bf16 burst (frac); nominal GB300 "
                                        "dense bf16 (frac_nominal)"},
            "clocks": clk.summary(),
            "e2e": {"value": whole_job_tflops(world, flops, ms_e2e), "unit": "TFLOPS",
                    "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"],
                    "ms_per_step": ms_e2e,
                    "pipelined": "two sets of device inputs and outputs: step k+1's "
                                 "host-to-device copies and step k-1's device-to-host copy "
                                 "overlap step k",
                    "value_one_step_at_a_time": whole_job_tflops(world, flops, ms_e2e_serial),
                    "ms_per_step_one_step_at_a_time": ms_e2e_serial},
            "gpu_launches": ((2 if fused else 3) + (2 if dyn else 0)) * args.steps,
            "cpu_baseline": cpu,
            "detail": headline,
            "per_workload": {k: compact_view(v) for k, v in per.items()},
        }
        print(json.dumps(out))
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def compact_view(rec):
    """The per-workload record as printed: times, fractions and clocks."""
    if "error" in rec:
        return rec
    keep = ("config", "partition", "gemm_pairs", "consumer", "value_tflops",
            "ms_overlapped_step", "ms_serial_step", "overlap_speedup", "ms_gemm_alone",
            "gemm_tflops_alone", "gemm_frac_of_measured_peak", "gemm_frac_of_nominal_peak",
            "ms_torch_matmul", "gemm_slowdown", "gemm_in_kernel_ms_alone",
            "gemm_in_kernel_ms_in_step", "consumer_bytes", "direct_alone_step_grid",
            "direct_alone_full_grid", "consumer_in_step", "reorder_alone",
            "plain_copy_same_bytes", "reorder_frac_of_plain_copy", "gemm_traffic_bytes",
            "swizzle_8", "clocks", "status_ok", "step_kernels")
    out = {k: rec[k] for k in keep if k in rec}
    if isinstance(out.get("consumer_in_step"), dict):
        out["consumer_in_step"] = {k: v for k, v in out["consumer_in_step"].items()
                                   if k != "how"}
    return out


def write_trace(ctx, b, path):
    """One more overlapped step with the GEMM's and the consumer's stamps."""
    torch, fo = ctx["torch"], ctx["fo"]
    pipe, w = b.pipe, b.w
    sm_count = ctx["sm_count"]
    trace = torch.zeros(pipe.tiles + 3 * w.wave_width, dtype=torch.int64, device=pipe.device)
    ctrace = torch.zeros(2 * pipe.P + 16 * sm_count, dtype=torch.int64, device=pipe.device)
    fo.fo_plan_set_trace(pipe.plan, trace.data_ptr(), ctrace.data_ptr())
    with torch.cuda.stream(b.s):
        ctx["flush"]()
    b.step(overlap=True, fused=b.fused, direct=b.direct)
    torch.cuda.synchronize()
    fo.fo_plan_set_trace(pipe.plan, 0, 0)
    stamps = trace.cpu().numpy().astype(np.int64)
    cst = ctrace.cpu().numpy().astype(np.int64)
    t0 = stamps[pipe.tiles:pipe.tiles + w.wave_width].min()
    rec = cst[2 * pipe.P:].reshape(-1, 4)
    rec = rec[rec[:, 1] > 0]

    def rel(x):
        return [(float(v) - t0) / 1e3 if v > 0 else None for v in x]
    n_split = fo.fo_plan_set_split(pipe.plan, True)
    split = stamps[pipe.tiles + w.wave_width:pipe.tiles + w.wave_width + 2 * n_split]
    with open(path, "w") as f:
        json.dump({"tile_done_us": ((stamps[:pipe.tiles] - t0) / 1e3).tolist(),
                   "gemm_cta_start_us": rel(stamps[pipe.tiles:pipe.tiles + w.wave_width]),
                   "split_tiles": n_split,
                   "split_helper_done_us": rel(split[0::2]),
                   "split_owner_half_done_us": rel(split[1::2]),
                   "group_consumed_us": rel(cst[:pipe.P]),
                   "group_reordered_us": rel(cst[pipe.P:2 * pipe.P]),
                   "consumer_cta": [{"sm": int(r[0]), "start_us": (r[1] - t0) / 1e3,
                                     "end_us": (r[2] - t0) / 1e3, "chunks": int(r[3])}
                                    for r in rec],
                   "step_kernels": b.kernels,
                   "wave_width": w.wave_width, "partition": pipe.partition}, f)


def measure_e2e(ctx, b, args):
    """End to end through the C ABI with host buffers: every step copies its
    inputs in from pinned host memory and its output back.  One step at a
    time, and pipelined as a serving loop runs it."""
    torch = ctx["torch"]
    pipe, w, s, inp, dyn = b.pipe, b.w, b.s, b.inp, b.dyn
    fused, direct = b.fused, b.direct
    dev = pipe.device
    hA = torch.from_numpy(inp.A.view(np.int16)).pin_memory()
    h_route = []
    d_tok = d_sl = None
    if dyn:   # each step's routing and routed A come from the host
        h_route = [(t.cpu().pin_memory(), q.cpu().pin_memory(), a.cpu().pin_memory())
                   for t, q, a in b.routes]
        d_tok, d_sl = torch.empty_like(b.routes[0][0]), torch.empty_like(b.routes[0][1])
        pipe.buf.A = torch.empty_like(b.routes[0][2])
    hB = [torch.from_numpy(x.view(np.int16)).pin_memory() for x in inp.B]
    hP = [torch.from_numpy(p.view(np.int16)).pin_memory() for p in inp.partials]
    hOut = [torch.empty(f.shape, dtype=torch.int16).pin_memory() for f in pipe.buf.final]
    h2d = hA.numel() * 2 + sum(x.numel() * 2 for x in hB) + sum(p.numel() * 2 for p in hP)
    h2d += 2 * w.M * 4 if dyn else 0
    d2h = sum(o.numel() * 2 for o in hOut)
    turn = [0]

    def e2e_step():
        with torch.cuda.stream(s):
            if dyn:
                t_, q_, a_ = h_route[turn[0] % len(h_route)]
                turn[0] += 1
                pipe.buf.A.copy_(a_, non_blocking=True)
                d_tok.copy_(t_, non_blocking=True)
                d_sl.copy_(q_, non_blocking=True)
            else:
                pipe.buf.A.copy_(hA, non_blocking=True)
            for d_, h_ in zip(pipe.buf.B, hB):
                d_.copy_(h_, non_blocking=True)
            for d_, h_ in zip(pipe.buf.partials, hP):
                d_.copy_(h_, non_blocking=True)
        if dyn:
            pipe.route(d_tok, d_sl)
        pipe.step(overlap=True, sync_current=False, fused=fused, direct=direct)
        with torch.cuda.stream(s):
            for h_, d_ in zip(hOut, pipe.buf.final):
                h_.copy_(d_, non_blocking=True)
    # one step at a time: its copies in, the step, its copy out
    t_serial = b.timed(e2e_step)

    # pipelined: two sets of device inputs and outputs; step k+1's inputs are
    # copied in (one copy stream) and step k-1's output copied out (another)
    # while step k computes.  Every step still copies all its inputs in and
    # its output out; the region is timed from before the first copy to
    # after the last, over all steps.  Each step's copies write more than L2
    # holds (no flush between steps).
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    sets = [dict(A=pipe.buf.A, B=pipe.buf.B, partials=pipe.buf.partials,
                 final=pipe.buf.final, hOut=hOut)]
    sets.append(dict(A=torch.empty_like(pipe.buf.A), B=[torch.empty_like(x) for x in pipe.buf.B],
                     partials=[torch.empty_like(x) for x in pipe.buf.partials],
                     final=[torch.empty_like(x) for x in pipe.buf.final],
                     hOut=[torch.empty_like(x).pin_memory() for x in hOut]))
    if dyn:
        for st_ in sets:
            st_["tok"], st_["sl"] = torch.empty_like(d_tok), torch.empty_like(d_sl)
    ev = [{k: torch.cuda.Event() for k in ("h2d", "comp", "d2h")} for _ in sets]

    def pipelined(n):
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        s_in.wait_stream(s)
        s_out.wait_stream(s)
        for k in range(n):
            st_, e = sets[k & 1], ev[k & 1]
            if k >= 2:
                s_in.wait_event(e["comp"])   # step k-2 has read this set's inputs
            with torch.cuda.stream(s_in):
                if dyn:
                    t_, q_, a_ = h_route[k % len(h_route)]
                    st_["A"].copy_(a_, non_blocking=True)
                    st_["tok"].copy_(t_, non_blocking=True)
                    st_["sl"].copy_(q_, non_blocking=True)
                else:
                    st_["A"].copy_(hA, non_blocking=True)
                for d_, h_ in zip(st_["B"], hB):
                    d_.copy_(h_, non_blocking=True)
                for d_, h_ in zip(st_["partials"], hP):
                    d_.copy_(h_, non_blocking=True)
                e["h2d"].record(s_in)
            s.wait_event(e["h2d"])
            if k >= 2:
                s.wait_event(e["d2h"])      # step k-2's output has left this set
            pipe.buf.A, pipe.buf.B = st_["A"], st_["B"]
            pipe.buf.partials, pipe.buf.final = st_["partials"], st_["final"]
            if dyn:
                pipe.route(st_["tok"], st_["sl"])
            pipe.step(overlap=True, sync_current=False, fused=fused, direct=direct)
            e["comp"].record(s)
            s_out.wait_event(e["comp"])
            with torch.cuda.stream(s_out):
                for h_, d_ in zip(st_["hOut"], st_["final"]):
                    h_.copy_(d_, non_blocking=True)
                e["d2h"].record(s_out)
        s.wait_stream(s_in)
        s.wait_stream(s_out)
        e1.record(s)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n
    pipelined(2)   # warm-up of the streams and events
    ms_pipe = pipelined(args.steps)
    assert int(pipe.buf.status.item()) == 0
    pipe.buf.A, pipe.buf.B = sets[0]["A"], sets[0]["B"]
    pipe.buf.partials, pipe.buf.final = sets[0]["partials"], sets[0]["final"]
    del sets
    return {"ms_pipelined": ms_pipe, "ms_one_step_at_a_time": statistics.mean(t_serial),
            "h2d": h2d, "d2h": d2h}


def tune_partition(w, inp, ms_gemm_for_tuning, partition, steps):
    """The pages' predictive search (Algorithm 1) for this workload, with its
    offline inputs measured here: the GEMM alone (this run), the direct
    consumer's in-kernel latency for first groups of sampled sizes, and the
    interference factors (the GEMM's slowdown beside the consumer and the
    consumer's beside the GEMM, from traced steps with the workload's
    partition).  Returns the tuned partitions with and without the
    interference factors, their predictions, and the measured overlapped
    steps (median, L2 flushed) of the tuned and the workload's partitions,
    alternated."""
    from communication_overlap_gb300 import fo
    from communication_overlap_gb300.tuning import Tuner, sample_waves
    t = Tuner(w, inp, reps=10)
    try:
        gemm_us = ms_gemm_for_tuning * 1e3
        waves = sample_waves(t.pipe.waves)
        curve = t.curve(waves)
        curve_l = t.curve_in_launch(waves)
        sigma, rho = t.interference(gemm_us, partition)
        parts, pred = fo.fo_tune_partition(t.desc(), gemm_us, curve)
        parts_i, pred_i = fo.fo_tune_partition(t.desc(), gemm_us, curve_l, sigma, rho)
        t.reps = steps
        cands = {"tuned": parts, "tuned_interference": parts_i, "workload": partition}
        meas = {k: [] for k in cands}
        for _ in range(2):      # alternate, to share drift between them
            for k, c in cands.items():
                meas[k].append(t.step_us(c))
        ms = {k: statistics.median(v) / 1e3 for k, v in meas.items()}
        pw = fo.fo_predict_partition(t.desc(partition), gemm_us, curve)
        pw_i = fo.fo_predict_partition(t.desc(partition), gemm_us, curve_l, sigma, rho)
        return {"partition": parts, "predicted_us": pred, "ms_step": ms["tuned"],
                "gemm_slowdown": sigma, "comm_slowdown": rho,
                "partition_interference": parts_i, "predicted_interference_us": pred_i,
                "ms_step_interference": ms["tuned_interference"],
                "ms_step_workload_partition": ms["workload"],
                "predicted_us_workload_partition": pw,
                "predicted_interference_us_workload_partition": pw_i,
                "prediction_error_workload_partition": pw / (ms["workload"] * 1e3) - 1.0,
                "prediction_error_tuned": pred / (ms["tuned"] * 1e3) - 1.0,
                "prediction_error_interference_tuned":
                    pred_i / (ms["tuned_interference"] * 1e3) - 1.0,
                "interference_fit": "comm_slowdown fitted on the workload partition's "
                                    "measured step; the tuned partitions' steps are "
                                    "predictions",
                "curve_group_waves": waves,
                "note": "Algorithm 1 with offline inputs measured in this run, without and "
                        "with the interference factors; the headline keeps the workload's "
                        "partition unless --partition tuned"}
    finally:
        t.close()


def max_over_ranks(x, dist=None, device=None):
    """The slowest rank's value (every rank gets it); identity on one rank."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(world, flops_per_rank, ms_slowest):
    """Every rank runs its own replica: the job's FLOPs over the slowest
    rank's time per step."""
    return world * flops_per_rank / (ms_slowest * 1e-3) / 1e12


def consumer_name(w):
    return {0: "copy", 1: f"sum with {w.n_partials} partials",
            2: f"sum with {w.n_partials} partials + scatter to {w.n_dest} slices",
            3: f"bucket by token mod {w.n_dest}"}[w.consumer]


def moved_rows(w, inp):
    """Rows the consumer and the reorder move: all of them, except the empty
    rows of an expert capacity that the routing left unfilled."""
    if inp.row_token is None:
        return w.M
    return int((np.asarray(inp.row_token) >= 0).sum())


def consumer_bytes(w, inp):
    """Algorithmic bytes of the consumer: every source read once, every
    output written once."""
    c = moved_rows(w, inp) * w.N * 2
    if w.consumer in (1, 2):
        return c * (1 + w.n_partials) + c
    return 2 * c


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    if args.ncu_gemm:
        return run_ncu_gemm(args)
    if args.ncu_matmul:
        return run_ncu_matmul(args)
    if args.ncu_step:
        return run_ncu_step(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
