"""Predictive wave-group tuning, Algorithm 1 (TEST INFRASTRUCTURE ONLY).

[P1] 四、实时调优 (see ``oracle/__init__`` for the page title): offline, take
the GEMM's duration and the communication latency curve (latency against
message size); online, for every candidate partition of the T waves into
groups, predict the latency of computing and communicating them and keep
the partition with the smallest prediction.

For each group G_i in order: t_p = duration / T * |G_i| (|G_i| in waves);
the group's communication latency t_m comes from interpolating the curve at
the group's data size; accumulated compute t_acc_p and communication
t_acc_m advance as t_acc_m = max(t_acc_p, t_acc_m) + t_m and
t_acc_p += t_p.

Reading of the printed pseudo-code, whose indices are garbled (it takes the
data size of G_{i-1} at i = 0 and adds the last group's communication
without a max): a group's communication starts once its own compute is done
and the previous group's communication has ended, i.e.

    C_i = sum_{k <= i} t_p(k)               (end of compute of G_1..G_i)
    E_i = max(C_i, E_{i-1}) + t_m(G_i),  E_{-1} = 0
    predicted latency = E_{P-1}

Curve interpolation: piecewise linear in bytes between the samples (sorted
by size); below the smallest sample its latency (a fixed floor); above the
largest, the slope of the last two samples.  Candidates: all 2**(T-1)
partitions, enumerated by ``plan.design_space``.

Interference (not in the pages, whose compute and communication run on
separate hardware): on one GPU the GEMM and the consumer share memory and
SMs, so each slows the other while both run (reading R19).  Two measured
factors: while a communication runs, the GEMM advances at 1 / sigma of its
alone rate (gemm_slowdown); while the GEMM runs, a communication advances at
1 / rho of the curve's rate (comm_slowdown).  A group's communication still
starts once its own waves are computed and the previous group's
communication has ended; everything else is the pages' loop.  The schedule
is simulated event by event (wave completions and communication ends), with
both rates constant between events.  With sigma = rho = 1 the events give
back the pages' recurrence exactly.
"""
from . import plan as P


def interp_latency(curve, nbytes):
    """Latency at `nbytes` from [(bytes, latency), ...] (see module doc)."""
    pts = sorted(curve)
    if nbytes <= pts[0][0]:
        return pts[0][1]
    for (b0, t0), (b1, t1) in zip(pts, pts[1:]):
        if nbytes <= b1:
            return t0 + (t1 - t0) * (nbytes - b0) / (b1 - b0)
    (b0, t0), (b1, t1) = pts[-2], pts[-1]
    return t1 + (t1 - t0) * (nbytes - b1) / (b1 - b0)


def group_bytes(partition, wave_width, tiles, tile_bytes):
    """Bytes each group communicates: its tiles (the last wave may be
    partial) times the bytes of one tile."""
    out, wave0 = [], 0
    for g in partition:
        first = wave0 * wave_width
        last = min(tiles, (wave0 + g) * wave_width)
        out.append((last - first) * tile_bytes)
        wave0 += g
    return out


def predict(partition, duration, curve, wave_width, tiles, tile_bytes,
            gemm_slowdown=1.0, comm_slowdown=1.0):
    """Predicted latency of one candidate: Algorithm 1's loop, with the
    mutual slowdown of the module doc when a factor is not 1."""
    T = sum(partition)
    sizes = group_bytes(partition, wave_width, tiles, tile_bytes)
    if gemm_slowdown == 1.0 and comm_slowdown == 1.0:
        t_acc_p = 0.0
        t_acc_m = 0.0
        for g, nbytes in zip(partition, sizes):
            t_p = duration / T * g
            t_m = interp_latency(curve, nbytes)
            t_acc_p = t_acc_p + t_p                  # this group's compute is done
            t_acc_m = max(t_acc_p, t_acc_m) + t_m    # then its communication runs
        return t_acc_m
    # event by event: GEMM work done (in alone microseconds), the running
    # communication's remaining work (in curve microseconds)
    ready = []                 # GEMM work at which each group is computed
    w = 0
    for g in partition:
        w += g
        ready.append(duration / T * w)
    t, gemm_done = 0.0, 0.0
    j, comm_left = 0, None
    while True:
        gemm_on = gemm_done < duration
        if comm_left is None and j < len(partition) and gemm_done >= ready[j]:
            comm_left = interp_latency(curve, sizes[j])
        comm_on = comm_left is not None
        if not gemm_on and not comm_on:
            return t
        gemm_rate = (1.0 / gemm_slowdown if comm_on else 1.0) if gemm_on else 0.0
        comm_rate = (1.0 / comm_slowdown if gemm_on else 1.0) if comm_on else 0.0
        dt = float("inf")
        if gemm_on:            # the next group computed, or the GEMM's end
            nxt = min([r for r in ready if r > gemm_done] + [duration])
            dt = (nxt - gemm_done) / gemm_rate
        if comm_on:
            dt = min(dt, comm_left / comm_rate)
        t += dt
        if gemm_on:
            gemm_done = min(duration, gemm_done + gemm_rate * dt)
            # snap to a boundary reached within rounding
            for r in ready + [duration]:
                if abs(gemm_done - r) <= 1e-9 * max(1.0, duration):
                    gemm_done = r
        if comm_on:
            comm_left -= comm_rate * dt
            if comm_left <= 1e-9 * max(1.0, duration):
                comm_left = None
                j += 1


def best_partition(T, duration, curve, wave_width, tiles, tile_bytes,
                   gemm_slowdown=1.0, comm_slowdown=1.0):
    """Algorithm 1's online search: the candidate with the smallest
    prediction (the first one in enumeration order on ties)."""
    best, t_min = None, float("inf")
    for cand in P.design_space(T):
        t = predict(cand, duration, curve, wave_width, tiles, tile_bytes,
                    gemm_slowdown, comm_slowdown)
        if t < t_min:
            best, t_min = cand, t
    return best, t_min
