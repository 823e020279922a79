"""Algorithm 1 on one GB300: offline measurements, the predictive search,
and a check of the prediction against measured step times.

  python -m communication_overlap_gb300.tuning --workload allreduce [--validate]

Offline ([P1] "FlashOverlap: 信号驱动计算通信重叠论文详解", 四、实时调优, 离线阶段):
  * GEMM configuration: our own signaled GEMM, its duration timed alone;
  * "bandwidth curve": on one GPU the communication is the consumer
    stand-in (by default the direct consumer+reorder the benchmark's step
    runs), so the curve is the consumer's latency against group bytes,
    sampled on a first group of k waves (k = 1 .. T), its flag already
    raised.  The latency is taken inside the kernel (first CTA start to last
    CTA end, from the consumer's globaltimer trace): in the overlapped step
    one consumer launch serves every group, so no group pays a launch;
  * SM contention: W = the GEMM's persistent CTAs, fixed by the workload.
Online: fo_tune_partition (exact over all 2^(T-1) candidates).

Interference (one GPU: the GEMM and the consumer share memory and SMs and
slow each other while both run), from the workload's own partition:
  * gemm_slowdown: the GEMM's in-kernel duration in the overlapped step
    over its duration alone (per-tile stamps);
  * comm_slowdown: fitted so that the model reproduces that partition's
    measured step (one calibration point; every other candidate is a
    prediction).
The interference model takes the consumer's latency per group inside one
persistent launch (curve_in_launch: no launch or ramp-up per group, as in
the step), the pages' model the latency of a launch per group (curve).
fo_tune_partition_ex / fo_predict_partition_ex take both.

--validate runs the overlapped step for every candidate partition (T <= 8)
and reports how the predicted best compares with the measured best, with
and without the interference factors.
"""
import argparse
import json
import statistics
import sys

import torch

from . import fo
from . import workloads as W
from .pipeline import Pipeline


def _design_space(T):
    """All partitions of T waves into consecutive groups (2^(T-1))."""
    out = []
    for mask in range(1 << (T - 1)):
        parts, run = [], 0
        for k in range(T):
            run += 1
            if k == T - 1 or (mask >> (T - 2 - k)) & 1:
                parts.append(run)
                run = 0
        out.append(parts)
    return out


def _time(fn, stream, reps, flush):
    ms = []
    for _ in range(reps):
        flush()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        torch.cuda.synchronize()
        ms.append(a.elapsed_time(b))
    return statistics.median(ms) * 1e3   # us


def sample_waves(T):
    """Group sizes at which to sample the curve for a GEMM of T waves: every
    size up to 8, then about four per doubling, and T itself (the predictor
    interpolates between them)."""
    ks, k = [], 1
    while k < T:
        ks.append(k)
        k = k + 1 if k < 8 else k + max(1, k // 4)
    return ks + [T]


class Tuner:
    """kernels: the step's consumer kernels, "direct" (the consumer+reorder
    storing straight to the final layout, the benchmark's default) or
    "separate" (consumer, then reorder); the curve and the validation steps
    both use them."""

    def __init__(self, w, inp=None, reps=20, kernels="direct"):
        self.w = w
        self.inp = inp or W.make_inputs(w)
        self.reps = reps
        self.direct = kernels == "direct"
        self.pipe = Pipeline(w, self.inp)
        self.flush_buf = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
        self.tile_bytes = w.tile_m * w.tile_n * 2

    def flush(self):
        with torch.cuda.stream(self.pipe.s0):
            self.flush_buf.fill_(1)

    def close(self):
        self.pipe.close()

    def gemm_us(self):
        p = self.pipe
        for _ in range(3):
            p.gemm(p.s0, p.epoch)
        return _time(lambda: p.gemm(p.s0, p.epoch), p.s0, self.reps, self.flush)

    def curve(self, waves=None):
        """[(bytes, us)] for first groups of k waves (in-kernel time), k in
        `waves` (default every k = 1 .. T)."""
        p = self.pipe
        T = p.waves
        ctas = 4 * torch.cuda.get_device_properties(p.device).multi_processor_count
        pts = []
        for k in (waves or range(1, T + 1)):
            p.replan([k, T - k] if k < T else [T])
            p.step(overlap=False)
            torch.cuda.synchronize()
            p.set_overlap(False)
            trace = torch.zeros(2 * p.P + 4 * ctas, dtype=torch.int64, device=p.device)
            fo.fo_plan_set_trace(p.plan, 0, trace.data_ptr())
            spans = []
            for _ in range(self.reps):
                self.flush()
                trace.zero_()
                if self.direct:
                    p.consume_reorder(p.s0, p.epoch, group=0, direct=True)
                else:
                    p.consume(p.s0, p.epoch, group=0)
                torch.cuda.synchronize()
                rec = trace[2 * p.P:].view(-1, 4).cpu()
                ran = rec[rec[:, 1] > 0]
                spans.append(float(ran[:, 2].max() - ran[:, 1].min()) / 1e3)
            fo.fo_plan_set_trace(p.plan, 0, 0)
            pts.append((float(p.group_tiles[0] * self.tile_bytes), statistics.median(spans)))
        self.last_curve = pts
        return pts

    def curve_in_launch(self, waves=None):
        """[(bytes, us)]: the consumer's latency per group inside one
        persistent launch, as the overlapped step runs it.  For group size
        k: plan the waves as groups of k (the remainder last), raise every
        flag with a step, then run the consumer over all groups alone;
        each full group after the first takes the time between its last
        chunk and the previous group's (consumer stamps), no launch or
        ramp-up in it; median over groups and repetitions.  Sizes with
        fewer than two full groups are skipped (the predictor extrapolates
        from the last two samples)."""
        p = self.pipe
        T = p.waves
        sm = torch.cuda.get_device_properties(p.device).multi_processor_count
        pts = []
        for k in (waves or range(1, T + 1)):
            if T // k < 2:
                continue
            part = [k] * (T // k) + ([T % k] if T % k else [])
            p.replan(part)
            p.step(overlap=False)
            torch.cuda.synchronize()
            p.set_overlap(False)
            trace = torch.zeros(2 * p.P + 16 * sm, dtype=torch.int64, device=p.device)
            fo.fo_plan_set_trace(p.plan, 0, trace.data_ptr())
            lat = []
            for _ in range(self.reps):
                self.flush()
                trace.zero_()
                if self.direct:
                    p.consume_reorder(p.s0, p.epoch, direct=True)
                else:
                    p.consume(p.s0, p.epoch)
                torch.cuda.synchronize()
                done = trace[:p.P].cpu().tolist()
                lat += [(done[j] - done[j - 1]) / 1e3 for j in range(1, T // k)]
            fo.fo_plan_set_trace(p.plan, 0, 0)
            pts.append((float(p.group_tiles[1] * self.tile_bytes), statistics.median(lat)))
        if len(pts) < 2:   # too few waves: the stand-alone curve
            return self.curve(waves)
        self.last_curve = pts
        return pts

    def interference(self, gemm_us, partition=None, reps=5):
        """(gemm_slowdown, comm_slowdown) for the interference model, from
        `partition` (default: the workload's one wave then groups of two):
        gemm_slowdown is the GEMM's in-kernel duration inside the
        overlapped step over its duration alone (per-tile stamps, median of
        `reps`); comm_slowdown is then fitted (bisection) so that the
        model, with this run's GEMM time `gemm_us` and latency curve (call
        self.curve first), reproduces that partition's measured step."""
        p = self.pipe
        part = list(partition or fo.partition_one_then_two(p.waves))
        p.replan(part)
        kw = dict(fused=True, direct=True) if self.direct else {}
        for _ in range(3):
            p.step(overlap=True, **kw)
        torch.cuda.synchronize()
        W = p.desc_args["wave_width"]
        trace = torch.zeros(p.tiles + 3 * W, dtype=torch.int64, device=p.device)
        fo.fo_plan_set_trace(p.plan, trace.data_ptr())

        def span():
            st = trace.cpu()
            return float(st[:p.tiles].max() - st[p.tiles:p.tiles + min(W, p.tiles)].min())
        sig = []
        for _ in range(reps):
            self.flush()
            p.gemm(p.s0, p.epoch)
            torch.cuda.synchronize()
            alone = span()
            self.flush()
            p.step(overlap=True, **kw)
            torch.cuda.synchronize()
            sig.append(span() / alone)
        fo.fo_plan_set_trace(p.plan, 0)
        sigma = statistics.median(sig)
        measured = self.step_us(part)
        desc = self.desc(part)

        def pred(rho):
            return fo.fo_predict_partition(desc, gemm_us, self.last_curve, sigma, rho)
        lo, hi = 0.25, 8.0
        if pred(lo) >= measured:
            return sigma, lo
        if pred(hi) <= measured:
            return sigma, hi
        for _ in range(50):
            mid = 0.5 * (lo + hi)
            if pred(mid) > measured:
                hi = mid
            else:
                lo = mid
        return sigma, 0.5 * (lo + hi)

    def step_us(self, partition):
        p = self.pipe
        p.replan(partition)
        kw = dict(fused=True, direct=True) if self.direct else {}
        for _ in range(3):
            p.step(overlap=True, **kw)
        torch.cuda.synchronize()
        assert int(p.buf.status.item()) == 0
        return _time(lambda: p.step(overlap=True, sync_current=False, **kw), p.s0, self.reps,
                     self.flush)

    def desc(self, partition=()):
        return fo.make_desc(**self.pipe.desc_args, group_waves=partition, host_only=True)


def run(name, validate=False, reps=20, kernels="direct"):
    w = W.WORKLOADS[name]
    t = Tuner(w, reps=reps, kernels=kernels)
    try:
        gemm = t.gemm_us()
        curve = t.curve()                  # the pages' model: one launch per group
        curve_l = t.curve_in_launch()      # the interference model: groups in one launch
        sigma, rho = t.interference(gemm)
        best, pred = fo.fo_tune_partition(t.desc(), gemm, curve)
        best_i, pred_i = fo.fo_tune_partition(t.desc(), gemm, curve_l, sigma, rho)
        out = {"workload": name, "kernels": kernels, "waves": t.pipe.waves, "gemm_us": gemm,
               "curve": curve, "curve_in_launch": curve_l,
               "gemm_slowdown": sigma, "comm_slowdown": rho,
               "tuned": best, "tuned_predicted_us": pred,
               "tuned_interference": best_i, "tuned_interference_predicted_us": pred_i}
        base = fo.partition_one_then_two(t.pipe.waves)
        out["one_then_two_predicted_us"] = fo.fo_predict_partition(t.desc(base), gemm, curve)
        out["one_then_two_predicted_interference_us"] = fo.fo_predict_partition(
            t.desc(base), gemm, curve_l, sigma, rho)
        if validate:
            rows = []
            for cand in _design_space(t.pipe.waves):
                rows.append({"partition": cand,
                             "predicted_us": fo.fo_predict_partition(t.desc(cand), gemm, curve),
                             "predicted_interference_us": fo.fo_predict_partition(
                                 t.desc(cand), gemm, curve_l, sigma, rho),
                             "measured_us": t.step_us(cand)})
            meas_best = min(rows, key=lambda r: r["measured_us"])
            by_part = {tuple(r["partition"]): r for r in rows}
            tuned_meas = by_part[tuple(best)]["measured_us"]
            tuned_i_meas = by_part[tuple(best_i)]["measured_us"]
            finest = by_part[tuple([1] * t.pipe.waves)]
            coarsest = by_part[(t.pipe.waves,)]
            ranked = sorted(r["measured_us"] for r in rows)

            def err(key):
                e = [abs(r[key] / r["measured_us"] - 1.0) for r in rows]
                return {"mean": statistics.mean(e), "max": max(e)}
            out.update({
                "candidates": len(rows),
                "measured_best": meas_best,
                "tuned_measured_us": tuned_meas,
                "tuned_regret": tuned_meas / meas_best["measured_us"] - 1.0,
                "rank_of_tuned": 1 + ranked.index(tuned_meas),
                "tuned_interference_measured_us": tuned_i_meas,
                "tuned_interference_regret": tuned_i_meas / meas_best["measured_us"] - 1.0,
                "rank_of_tuned_interference": 1 + ranked.index(tuned_i_meas),
                "prediction_error": err("predicted_us"),
                "prediction_error_interference": err("predicted_interference_us"),
                "finest_measured_us": finest["measured_us"],
                "finest_loss": finest["measured_us"] / meas_best["measured_us"] - 1.0,
                "coarsest_measured_us": coarsest["measured_us"],
                "all": rows,
            })
        return out
    finally:
        t.close()


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="allreduce")
    ap.add_argument("--validate", action="store_true")
    ap.add_argument("--reps", type=int, default=20)
    ap.add_argument("--out", default="")
    ap.add_argument("--kernels", default="direct", choices=["direct", "separate"])
    a = ap.parse_args(argv)
    res = run(a.workload, a.validate, a.reps, a.kernels)
    text = json.dumps(res)
    if a.out:
        with open(a.out, "w") as f:
            f.write(text)
    summary = {k: v for k, v in res.items() if k not in ("all", "curve")}
    print(json.dumps(summary))
    return 0


if __name__ == "__main__":
    sys.exit(main())
