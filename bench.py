"""Benchmark of the signaled-GEMM + reorder path (one JSON line on rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME]

A step is one pass of the whole path on the workload (default: the
wave-pattern GEMM M=2048, N=8192, K=8192, 128x256 tiles, 148-CTA waves,
groups of 1 then 2 waves, copy consumer + reorder back), inputs resident in
HBM: signaled GEMM (it resets its own counting table), then the consumer
and the post-communication reorder, by default as one kernel that stores
every unit straight to its final place (a programmatic dependent launch
running alongside the GEMM; ``--step-kernels`` picks the others).  ``value`` is the GEMM's FLOPs per step divided by the step time
(TFLOPS of the whole overlapped step); for the dynamic-routing workload
only the rows that hold a token count (2 x routed rows x N x K).  L2 is flushed (a 256 MiB write)
before every timed step, outside the timed events.

Extra keys: the GEMM alone (signals on and off), the consumer+reorder alone
(flags already raised), the serial step (the same kernels, the consumer as an
ordinary launch after the GEMM; also with the separate kernels), the
overlap ratio serial/overlapped, the GEMM's in-kernel duration inside the
overlapped step (per-tile globaltimer stamps) and its slowdown against the
GEMM alone, ``roofline`` of the dominant kernel (the GEMM), ``e2e`` through
the C ABI with host buffers (every step's inputs copied in from pinned host
memory and its output copied back, pipelined over two buffer sets), and ``cpu_baseline`` (the CPU oracle on a
bounded sample).

For N > 1 (torchrun) every rank runs its own replica of the workload (the
path has no data exchange on one node: "replicas only"); value sums the
ranks' FLOPs over the slowest rank's time.
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


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="wave_pattern")
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
    return ap.parse_args()


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


def traffic_from_profile(kernel_src):
    """Per-launch DRAM bytes of the GEMM from the committed ncu summary, if
    it was taken on the current source of the kernel (else None)."""
    path = os.path.join(ROOT, "profiles", "signaled_gemm_wave_pattern_ncu.md")
    try:
        txt = open(path).read()
    except OSError:
        return None
    h = hashlib.sha256(open(kernel_src, "rb").read()).hexdigest()[:16]
    src, traffic = None, None
    for line in txt.splitlines():
        if line.startswith("source_sha256_16:"):
            src = line.split(":", 1)[1].strip()
        if line.startswith("traffic_bytes_per_launch:"):
            try:
                traffic = float(line.split(":", 1)[1].strip())
            except ValueError:
                traffic = None
    return traffic if src == h else None


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


def oracle_sample(w, inp, partition, rows):
    """Time the CPU oracle on a bounded sample of the workload: the fp64 GEMM
    on the first `rows` output rows, plus pre-reorder, consumer and
    post-reorder on the full output (the plan is built once per shape and
    not counted).  Returns (seconds per full step estimate, description,
    cores)."""
    from oracle import gemm as OG
    from oracle import pipeline as OPL

    t0 = time.perf_counter()
    OG.gemm_rows_bf16(inp.A, inp.B, inp.expert_rows, np.arange(rows))
    t_rows = time.perf_counter() - t0
    gemm_full = t_rows * (w.M / rows)
    # the rest of the path on the full output (values do not matter for time)
    C = np.zeros((w.M, w.N), dtype=np.uint16)
    cons = {0: "copy", 1: "sum", 2: "rs", 3: "a2a"}[w.consumer]
    res = OPL.run(inp.expert_rows, w.N, w.K, w.tile_m, w.tile_n, w.swizzle, w.wave_width,
                  partition, _LAYOUT_NAMES[w.layout], cons, inp.A, inp.B, inp.partials,
                  w.n_dest, inp.row_token, inp.row_slot, w.top_k or 2, C_given=C)
    # with dynamic routing the routing tables are rebuilt every step: the
    # plan is part of the step
    skip = ("gemm",) if w.capacity else ("gemm", "plan")
    rest = sum(v for k, v in res.seconds.items() if k not in skip)
    plan_note = (f"plan ({res.seconds['plan']:.2f} s) included: the routing changes every step"
                 if w.capacity else f"plan ({res.seconds['plan']:.2f} s) excluded")
    desc = (f"fp64 GEMM on {rows} of {w.M} output rows ({t_rows:.2f} s, scaled x"
            f"{w.M / rows:.1f}) + pre-reorder, consumer and post-reorder on the full "
            f"output ({rest:.2f} s); {plan_note}")
    return gemm_full + rest, desc, os.cpu_count()


def run_reference(args):
    """--impl reference: the CPU oracle, as it stands, on this host's cores."""
    rank, _, world = dist_env()
    if rank != 0:
        return 0
    from communication_overlap_gb300 import workloads as W
    from oracle import plan as OPN
    w = W.WORKLOADS[args.workload]
    inp = W.make_inputs(w)
    tiles = sum(-(-m // w.tile_m) for m in inp.expert_rows) * (w.N // w.tile_n)
    partition = OPN.one_then_two(OPN.wave_count(tiles, w.wave_width))
    per = []
    budget = max(2.0, 150.0 / max(1, args.steps + args.warmup))
    rows = calibrate_rows(w, inp, budget)
    desc = ""
    for i in range(args.warmup + args.steps):
        secs, desc, cores = oracle_sample(w, inp, partition, rows)
        if i >= args.warmup:
            per.append(secs)
    step_s = statistics.mean(per)
    value = 2.0 * moved_rows(w, inp) * w.N * w.K / step_s / 1e12
    line = {
        "impl": "reference", "metric": "signaled GEMM TFLOPS (% of bf16 peak); "
        "overlap time vs serial GEMM+consumer", "value": value, "unit": "TFLOPS",
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
        return (f"{w.name}: grouped bf16 GEMM {w.n_tokens} tokens x top-{w.top_k} over "
                f"{w.n_experts} experts, N={w.N} K={w.K}, {w.tile_m}x{w.tile_n} tiles, "
                f"W={w.wave_width}, swizzle {w.swizzle}{cap}")
    return (f"{w.name}: bf16 GEMM M={w.M} N={w.N} K={w.K}, {w.tile_m}x{w.tile_n} tiles, "
            f"W={w.wave_width}, swizzle {w.swizzle}")


# ----------------------------------------------------------------- our path

STEP_KERNELS = {
    "direct": "signaled GEMM + one consumer kernel that stores every unit straight to "
              "its final place (communication and post-communication reorder fused)",
    "fused": "signaled GEMM + one consumer kernel that writes the communication buffers "
             "and moves each chunk on to its final place",
    "separate": "signaled GEMM + consumer + post-communication reorder",
}

def run_ours(args):
    import torch
    import torch.distributed as dist
    from communication_overlap_gb300 import fo
    from communication_overlap_gb300 import workloads as W
    from communication_overlap_gb300.pipeline import Pipeline

    rank, local, world = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    w = W.WORKLOADS[args.workload]
    inp = W.make_inputs(w)
    pipe = Pipeline(w, inp, device=dev, consumer_ctas=args.consumer_ctas,
                    reorder_ctas=args.reorder_ctas)
    s = pipe.s0
    # FLOPs of the rows that hold a token: with fixed expert capacities the
    # empty rows are not work (the GEMM skips tiles that have none)
    flops = 2.0 * moved_rows(w, inp) * w.N * w.K
    flush_buf = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def flush():
        flush_buf.fill_(1)

    # tile stamps, CTA starts, and two stamps per split tile of the last wave
    trace = torch.zeros(pipe.tiles + 3 * w.wave_width, dtype=torch.int64, device=dev)

    # Dynamic routing (expert capacities fixed): every step takes the next of
    # a few routings resident in HBM, with its routed A (the dispatch gather,
    # outside the path), and rebuilds the routing tables on the device
    # (fo_plan_route) before its GEMM.
    dyn = w.capacity > 0
    routes = []
    if dyn:
        X = W.token_matrix(w)
        for k in range(1, 5):
            _, tok, sl = W.routing(w, k)
            routes.append((torch.from_numpy(tok).to(dev), torch.from_numpy(sl).to(dev),
                           torch.from_numpy(W.gather_rows(X, tok).view(np.int16)).to(dev)))
        del X
    turn = [0]

    def step(**kw):
        if dyn:
            tok, sl, A = routes[turn[0] % len(routes)]
            turn[0] += 1
            pipe.buf.A = A
            pipe.route(tok, sl)
        return pipe.step(**kw)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    # warm-up (also the first correctness evidence: status and counting table)
    # measured (all three variants timed in one process, interleaved): the
    # direct fused kernel gives the shortest step on every workload; the
    # fused kernel that writes the communication buffers and the separate
    # kernels are timed below as well
    kernels = "direct" if args.step_kernels == "auto" else args.step_kernels
    fused = kernels in ("fused", "direct")
    direct = kernels == "direct"
    for _ in range(max(3, args.warmup)):
        step(overlap=True, fused=fused, direct=direct)
    torch.cuda.synchronize()
    assert int(pipe.buf.status.item()) == 0, "consumer wait timed out"
    assert pipe.buf.count.cpu().tolist() == pipe.group_tiles

    # the headline: overlapped steps
    barrier()
    with Clocks(local) as clk:
        t_ov = timed(torch, s,
                     lambda: step(overlap=True, sync_current=False, fused=fused, direct=direct),
                     args.steps, flush)
    barrier()
    ms_ov = statistics.mean(t_ov)
    status_ok = int(pipe.buf.status.item()) == 0

    # the same step captured once in a CUDA graph and replayed (same epoch
    # and kernel parameters every time; the kernels clear their own signals)
    t_graph = []
    if not dyn:
        g_epoch = pipe.epoch + 1
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            pipe.gemm(s, g_epoch)
            if fused:
                pipe.consume_reorder(s, g_epoch, direct=direct)
            else:
                pipe.consume(s, g_epoch)
                pipe.reorder(s)
        pipe.epoch = g_epoch
        def replay():
            with torch.cuda.stream(s):   # replay on the step's stream
                graph.replay()
        t_graph = timed(torch, s, replay, args.steps, flush)
        assert int(pipe.buf.status.item()) == 0
        assert pipe.buf.count.cpu().tolist() == pipe.group_tiles
        del graph

    # every overlapped variant: separate kernels, fused, fused direct (no
    # communication buffers, each unit stored straight to its final place)
    t_var = {}
    for name, kw in (("separate", dict(fused=False)), ("fused", dict(fused=True)),
                     ("direct", dict(fused=True, direct=True))):
        t_var[name] = timed(torch, s, lambda: step(overlap=True, sync_current=False, **kw),
                            args.steps, flush)
    # serial = the same kernels as the overlapped step, the consumer as an
    # ordinary launch after the GEMM; and the separate kernels serially
    t_ser = timed(torch, s,
                  lambda: step(overlap=False, sync_current=False, fused=fused, direct=direct),
                  args.steps, flush)
    t_ser_sep = timed(torch, s, lambda: step(overlap=False, sync_current=False),
                      args.steps, flush)
    t_route = []
    if dyn:   # the two routing kernels alone
        t_route = timed(torch, s, lambda: pipe.route(*routes[0][:2]), args.steps, flush)
    # GEMM alone (signals on, as in the step; and off)
    t_gemm = timed(torch, s, lambda: pipe.gemm(s, pipe.epoch), args.steps, flush)
    t_gemm_nosig = timed(torch, s, lambda: pipe.gemm(s, pipe.epoch, signal=False),
                         args.steps, flush)
    # library reference point: torch.matmul (cuBLAS) on the same operands,
    # one call per expert for the grouped workload
    A_bf = pipe.buf.A.view(torch.bfloat16).view(w.M, w.K)
    B_bf = [b.view(torch.bfloat16).view(w.K, w.N) for b in pipe.buf.B]
    rows = np.cumsum([0] + list(inp.expert_rows))

    def torch_mm():
        with torch.cuda.stream(s):
            for e, Bm in enumerate(B_bf):
                torch.matmul(A_bf[rows[e]:rows[e + 1]], Bm)
    for _ in range(3):   # cuBLAS handle, workspace and kernel choice
        torch_mm()
    t_mm = timed(torch, s, torch_mm, args.steps, flush)

    # the same path with W = this device's SM count (the workloads fix W)
    sm_count = torch.cuda.get_device_properties(dev).multi_processor_count
    w_sm = None
    if sm_count != w.wave_width:
        pipe_sm = Pipeline(w, inp, device=dev, wave_width=sm_count)
        t_gemm_sm = timed(torch, pipe_sm.s0, lambda: pipe_sm.gemm(pipe_sm.s0, pipe_sm.epoch),
                          args.steps, flush)
        for _ in range(3):
            pipe_sm.step(overlap=True, fused=fused, direct=direct)
        t_step_sm = timed(torch, pipe_sm.s0,
                          lambda: pipe_sm.step(overlap=True, sync_current=False, fused=fused,
                                               direct=direct),
                          args.steps, flush)
        torch.cuda.synchronize()
        w_sm = {"wave_width": sm_count, "waves": pipe_sm.waves,
                "partition": pipe_sm.partition, "gemm_pairs": bool(pipe_sm.pairable),
                "ms_gemm_alone": statistics.mean(t_gemm_sm),
                "ms_overlapped_step": statistics.mean(t_step_sm),
                "status_ok": int(pipe_sm.buf.status.item()) == 0}
        pipe_sm.close()
        del pipe_sm

    # consumer + reorder alone: the flags of the last epoch are already raised;
    # ordinary launches so nothing overlaps the flush before them
    pipe.step(overlap=True)
    torch.cuda.synchronize()
    pipe.set_overlap(False)

    def cons_alone():
        pipe.consume(s, pipe.epoch)
        pipe.reorder(s)
    t_cons = timed(torch, s, cons_alone, args.steps, flush)

    def cons_only():
        pipe.consume(s, pipe.epoch)
    t_cons_only = timed(torch, s, cons_only, args.steps, flush)
    t_reo = timed(torch, s, lambda: pipe.reorder(s), args.steps, flush)
    t_direct_alone = timed(torch, s, lambda: pipe.consume_reorder(s, pipe.epoch, direct=True),
                           args.steps, flush)
    # the consumer's bandwidth with a full grid (4 CTAs per SM): its roofline
    # figure; the step uses the library's default grid for running beside the
    # GEMM, which for copies is smaller and slower alone
    fo.fo_plan_set_launch(pipe.plan, 4 * sm_count, args.reorder_ctas, False)
    t_cons_full = timed(torch, s, cons_only, args.steps, flush)
    t_direct_full = timed(torch, s, lambda: pipe.consume_reorder(s, pipe.epoch, direct=True),
                          args.steps, flush)
    fo.fo_plan_set_launch(pipe.plan, args.consumer_ctas, args.reorder_ctas, False)
    pipe.set_overlap(True)

    # in-kernel GEMM duration (per-tile stamps) alone and inside the step
    fo.fo_plan_set_trace(pipe.plan, trace.data_ptr())

    def gemm_span():
        t = trace.cpu().numpy().astype(np.int64)
        starts = t[pipe.tiles:pipe.tiles + min(w.wave_width, pipe.tiles)]
        return (t[:pipe.tiles].max() - starts.min()) / 1e6, t

    span_alone, span_step = [], []
    for _ in range(args.steps):
        with torch.cuda.stream(s):
            flush()
        pipe.gemm(s, pipe.epoch)
        torch.cuda.synchronize()
        span_alone.append(gemm_span()[0])
        with torch.cuda.stream(s):
            flush()
        pipe.step(overlap=True, fused=fused, direct=direct)
        torch.cuda.synchronize()
        sp, stamps = gemm_span()
        span_step.append(sp)
    fo.fo_plan_set_trace(pipe.plan, 0)
    if args.trace_out:
        # one more overlapped step with the consumer's stamps as well
        ctrace = torch.zeros(2 * pipe.P + 16 * sm_count, dtype=torch.int64, device=dev)
        fo.fo_plan_set_trace(pipe.plan, trace.data_ptr(), ctrace.data_ptr())
        with torch.cuda.stream(s):
            flush()
        pipe.step(overlap=True, fused=fused, direct=direct)
        torch.cuda.synchronize()
        fo.fo_plan_set_trace(pipe.plan, 0, 0)
        stamps = trace.cpu().numpy().astype(np.int64)
        cst = ctrace.cpu().numpy().astype(np.int64)
        t0 = stamps[pipe.tiles:pipe.tiles + w.wave_width].min()
        rec = cst[2 * pipe.P:].reshape(-1, 4)
        rec = rec[rec[:, 1] > 0]

        def rel(x):
            return [(float(v) - t0) / 1e3 if v > 0 else None for v in x]
        with open(args.trace_out, "w") as f:
            n_split = fo.fo_plan_set_split(pipe.plan, True)
            split = stamps[pipe.tiles + w.wave_width:pipe.tiles + w.wave_width + 2 * n_split]
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
                       "step_kernels": kernels,
                       "wave_width": w.wave_width, "partition": pipe.partition}, f)

    # end to end through the C ABI with host buffers
    hA = torch.from_numpy(inp.A.view(np.int16)).pin_memory()
    h_route = []
    if dyn:   # each step's routing and routed A come from the host
        h_route = [(t.cpu().pin_memory(), q.cpu().pin_memory(), a.cpu().pin_memory())
                   for t, q, a in routes]
        d_tok, d_sl = torch.empty_like(routes[0][0]), torch.empty_like(routes[0][1])
        pipe.buf.A = torch.empty_like(routes[0][2])
    hB = [torch.from_numpy(b.view(np.int16)).pin_memory() for b in inp.B]
    hP = [torch.from_numpy(p.view(np.int16)).pin_memory() for p in inp.partials]
    hOut = [torch.empty(f.shape, dtype=torch.int16).pin_memory() for f in pipe.buf.final]
    h2d = hA.numel() * 2 + sum(b.numel() * 2 for b in hB) + sum(p.numel() * 2 for p in hP)
    h2d += 2 * w.M * 4 if dyn else 0
    d2h = sum(o.numel() * 2 for o in hOut)

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
    t_e2e_serial = timed(torch, s, e2e_step, args.steps, flush)

    # pipelined, as a serving loop runs it: two sets of device inputs and
    # outputs; step k+1's inputs are copied in (one copy stream) and step
    # k-1's output copied out (another) while step k computes.  Every step
    # still copies all its inputs in and its output out; the region is timed
    # from before the first copy to after the last, over all steps.  Each
    # step's copies write more than L2 holds (no flush between steps).
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

    def e2e_pipelined(n):
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
    e2e_pipelined(2)   # warm-up of the streams and events
    ms_e2e_pipe = e2e_pipelined(args.steps)
    assert int(pipe.buf.status.item()) == 0
    for st_ in sets[1:]:
        for kk in ("A", "B", "partials", "final"):
            st_[kk] = None
    pipe.buf.A, pipe.buf.B = sets[0]["A"], sets[0]["B"]
    pipe.buf.partials, pipe.buf.final = sets[0]["partials"], sets[0]["final"]
    del sets

    # Algorithm 1 on this workload: the offline inputs (this run's GEMM time
    # and the consumer's latency curve, sampled) and the exact search; then
    # the overlapped step with the tuned partition against the workload's
    # own, in one pipeline, alternating.  Reported beside the headline, which
    # keeps the workload's partition.
    tuned = None
    if not args.no_tune:
        try:
            tuned = tune_partition(w, inp, ms_gemm_for_tuning=statistics.mean(t_gemm),
                                   partition=pipe.partition, steps=max(10, args.steps // 5))
        except Exception as e:   # a report, not the benchmark: keep the line
            tuned = {"error": f"{type(e).__name__}: {e}"}

    # max over ranks
    def rmax(x):
        return max_over_ranks(x, dist if world > 1 else None, dev)

    ms_ov = rmax(ms_ov)
    ms_ser = rmax(statistics.mean(t_ser))
    ms_gemm = rmax(statistics.mean(t_gemm))
    ms_e2e = rmax(ms_e2e_pipe)
    ms_e2e_serial = rmax(statistics.mean(t_e2e_serial))

    hbm, peak_burst, peak_sust, peak_kind = measured_peaks()
    gemm_tflops = flops / (ms_gemm * 1e-3) / 1e12
    traffic = traffic_from_profile(os.path.join(ROOT, "communication_overlap_gb300",
                                                "csrc", "gemm.cu"))
    cons_bytes = consumer_bytes(w, inp)
    reo_bytes = 2 * moved_rows(w, inp) * w.N * 2
    out = None
    if rank == 0:
        cpu = None
        if not args.no_cpu_baseline:
            rows = calibrate_rows(w, inp, args.cpu_seconds)
            secs, desc, cores = oracle_sample(w, inp, pipe.partition, rows)
            cpu = {"value": flops / secs / 1e12, "unit": "TFLOPS", "cores": cores,
                   "kind": "oracle", "sample": desc}
        out = {
            "metric": "signaled GEMM TFLOPS (% of bf16 peak); overlap time vs serial "
                      "GEMM+consumer",
            "value": whole_job_tflops(world, flops, ms_ov),
            "unit": "TFLOPS",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms_ov, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": workload_name(w), "partition": pipe.partition,
                       "groups_tiles": pipe.group_tiles, "consumer": consumer_name(w),
                       "l2": "flushed before every timed step (256 MiB write)",
                       "consumer_ctas": args.consumer_ctas or "library default",
                       "step_kernels": STEP_KERNELS[kernels],
                       "parallelism": f"replicas x{world}"},
            "roofline": {"bound": "tensor", "achieved": gemm_tflops, "peak": peak_burst,
                         "unit": "TFLOP/s", "frac": gemm_tflops / peak_burst,
                         "traffic": traffic,
                         "kernel": "signaled_gemm_kernel<256> (alone, signals on)",
                         "peak_source": f"{peak_kind} bf16 burst"},
            "clocks": clk.summary(),
            "e2e": {"value": whole_job_tflops(world, flops, ms_e2e), "unit": "TFLOPS",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": ms_e2e,
                    "pipelined": "two sets of device inputs and outputs: step k+1's "
                                 "host-to-device copies and step k-1's device-to-host copy "
                                 "overlap step k",
                    "value_one_step_at_a_time": whole_job_tflops(world, flops, ms_e2e_serial),
                    "ms_per_step_one_step_at_a_time": ms_e2e_serial},
            "gpu_launches": ((2 if fused else 3) + (2 if dyn else 0)) * args.steps,
            "cpu_baseline": cpu,
            "detail": {
                "ms_overlapped_step": ms_ov,
                "ms_overlapped_step_median": statistics.median(t_ov),
                "ms_serial_step_median": statistics.median(t_ser),
                "ms_gemm_alone_median": statistics.median(t_gemm),
                "overlapped_step_kernels": kernels,
                "ms_overlapped_step_by_kernels": {k: statistics.mean(v) for k, v in t_var.items()},
                "ms_overlapped_step_graph_replay": statistics.mean(t_graph) if t_graph else None,
                "ms_serial_step": ms_ser,
                "serial_step_kernels": kernels,
                "ms_serial_step_separate_kernels": statistics.mean(t_ser_sep),
                "overlap_speedup": ms_ser / ms_ov,
                "ms_gemm_alone": ms_gemm,
                "ms_gemm_alone_no_signal": statistics.mean(t_gemm_nosig),
                "gemm_tflops_alone": gemm_tflops,
                "gemm_frac_of_sustained": gemm_tflops / peak_sust,
                "ms_torch_matmul": statistics.mean(t_mm),
                "torch_matmul_tflops": flops / (statistics.mean(t_mm) * 1e-3) / 1e12,
                "torch_matmul_note": "library reference point: torch.matmul on the same "
                                     "operands (one call per expert), no reorder or signal",
                "w_sm_count": w_sm,
                "ms_consumer_plus_reorder_alone": statistics.mean(t_cons),
                "ms_consumer_alone": statistics.mean(t_cons_only),
                "ms_reorder_alone": statistics.mean(t_reo),
                "consumer_gbs": cons_bytes / (statistics.mean(t_cons_only) * 1e-3) / 1e9,
                "ms_consumer_alone_full_grid": statistics.mean(t_cons_full),
                "consumer_gbs_full_grid": cons_bytes / (statistics.mean(t_cons_full) * 1e-3) / 1e9,
                "reorder_gbs": reo_bytes / (statistics.mean(t_reo) * 1e-3) / 1e9,
                "ms_direct_alone": statistics.mean(t_direct_alone),
                "direct_gbs": cons_bytes / (statistics.mean(t_direct_alone) * 1e-3) / 1e9,
                "ms_direct_alone_full_grid": statistics.mean(t_direct_full),
                "direct_gbs_full_grid": cons_bytes / (statistics.mean(t_direct_full) * 1e-3) / 1e9,
                "hbm_peak_gbs": hbm,
                "gemm_in_kernel_ms_alone": statistics.median(span_alone),
                "gemm_in_kernel_ms_in_step": statistics.median(span_step),
                "gemm_slowdown": statistics.median(span_step) / statistics.median(span_alone),
                "status_ok": status_ok,
                "tuned_partition": tuned,
                **({"ms_route_alone": statistics.mean(t_route),
                    "routings": "4 routings resident in HBM, taken in turn, one per step"}
                   if dyn else {}),
            },
        }
        print(json.dumps(out))
    pipe.close()
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def tune_partition(w, inp, ms_gemm_for_tuning, partition, steps):
    """The pages' predictive search (Algorithm 1) for this workload, with its
    offline inputs measured here: the GEMM alone (this run) and the direct
    consumer's in-kernel latency for first groups of sampled sizes.  Returns
    the tuned partition, its prediction, and the measured overlapped steps
    (median, L2 flushed) of the tuned and the workload's partitions."""
    from communication_overlap_gb300 import fo
    from communication_overlap_gb300.tuning import Tuner, sample_waves
    t = Tuner(w, inp, reps=10)
    try:
        gemm_us = ms_gemm_for_tuning * 1e3
        waves = sample_waves(t.pipe.waves)
        curve = t.curve(waves)
        parts, pred = fo.fo_tune_partition(t.desc(), gemm_us, curve)
        t.reps = steps
        meas = {"tuned": [], "workload": []}
        for _ in range(2):      # alternate, to share drift between the two
            meas["tuned"].append(t.step_us(parts))
            meas["workload"].append(t.step_us(partition))
        return {"partition": parts, "predicted_us": pred,
                "predicted_us_workload_partition":
                    fo.fo_predict_partition(t.desc(partition), gemm_us, curve),
                "ms_step": statistics.median(meas["tuned"]) / 1e3,
                "ms_step_workload_partition": statistics.median(meas["workload"]) / 1e3,
                "curve_group_waves": waves,
                "note": "Algorithm 1 with offline inputs measured in this run; the headline "
                        "keeps the workload's partition"}
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
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
