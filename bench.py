#!/usr/bin/env python3
"""Benchmark: differentiable Fourier-slice projection, forward + fused backward.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-e2e] [--no-cpu-baseline]

A step is one pass of the hot path over one batch: the forward projection of B poses
(tp_project_3d_to_2d) and the fused backward for an upstream gradient
(tp_project_backward: volume, rotation and shift gradients).  The default workload is
D = 128 volume (128 x 128 x 65 complex64), B = 16384 uniform-SO(3) poses, shifts U(-5, 5)
px, Catmull-Rom cubic, cutoff 64, centered layout.  Inputs are seeded and synthetic.

Under torchrun (N > 1) every rank runs its own batch on its own GPU (weak scaling); the
volume gradient is summed over ranks with one NCCL all-reduce per step.  Rank 0 prints one
JSON line.  ``--impl reference`` times the fp64 CPU oracle on the host cores instead, on a
bounded sample of the same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time
from pathlib import Path

import numpy as np

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

METRIC = "projections/sec fwd+bwd at D=128 cubic; achieved GB/s vs HBM/L2 roofline"
DEFAULT_WORKLOAD = "fwdbwd3d_d128_cubic_b16384"
TRAFFIC_FILE = ROOT / "profiles" / "traffic.json"
KERNEL_SOURCES = ["back_projection_fourier_b300/csrc/kernels.cu",
                  "back_projection_fourier_b300/csrc/tp_device.cuh",
                  "back_projection_fourier_b300/csrc/gather.cuh",
                  "back_projection_fourier_b300/csrc/scatter.cuh"]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--fused-backward", action="store_true",
                    help="the step's backward as one kernel pass (tp_project_backward_fused; "
                         "no e2e leg)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-sample", type=int, default=16384, help="poses in the oracle sample")
    ap.add_argument("--batch", type=int, default=None,
                    help="override the workload's batch (small cases for profiling only)")
    ap.add_argument("--e2e-chunks", type=int, default=2,
                    help="pose chunks of the end-to-end step that reads back the gradients")
    ap.add_argument("--e2e-proj-chunks", type=int, default=8,
                    help="pose chunks of the end-to-end step that also reads back the projections")
    ap.add_argument("--interp", choices=["linear", "cubic"], default=None,
                    help="override the workload's interpolation (insertion: both are asked for)")
    ap.add_argument("--study", choices=["oversampling"], default=None,
                    help="instead of the step: time the on-the-fly oversampling comparison")
    ap.add_argument("--study-poses", default="1,16,256,4096,16384",
                    help="pose counts of the oversampling study")
    return ap.parse_args()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def kernel_hash() -> str:
    """Hash of the kernel sources without comments and blank lines: a counter capture stays
    valid across comment edits and is dropped by any change to the code itself."""
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        for line in (ROOT / rel).read_text().splitlines():
            code = line.split("//", 1)[0].rstrip()
            if code:
                h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


# ----------------------------------------------------------------- oracle ----

def metric_for(wl) -> str:
    """The headline metric for the headline workload; the same wording for the others."""
    if wl.name == DEFAULT_WORKLOAD:
        return METRIC
    what = {"fwd": "forward", "insert": "insertion with weights", "fwdbwd": "fwd+bwd"}[wl.op]
    if wl.ndim == 2:
        what = "2D rotation " + what
    recs = f", {wl.n_rec} reconstructions" if wl.ndim == 3 and wl.n_rec > 1 else ""
    return f"projections/sec {what} at D={wl.D} {'cubic' if wl.interp else 'linear'}{recs}"


def oracle_rate(wl, n_poses: int, nthreads: int) -> tuple[float, str]:
    """Projections/s of the fp64 oracle on the workload's own operation, over the first
    n_poses poses of every reconstruction (3D) or the first n_poses images (2D)."""
    import oracle

    kw = dict(interp=wl.interp, layout=wl.layout, cutoff=wl.rc, nthreads=nthreads)
    if wl.ndim == 3:
        n = min(n_poses, wl.n_pose)
        take = lambda a: None if a is None else np.ascontiguousarray(a[:, :n])  # noqa: E731
        rec, items = wl.rec, wl.n_rec * n
        per = f" of each of {wl.n_rec} reconstructions" if wl.n_rec > 1 else ""
        what = f"first {n} of {wl.n_pose} poses{per}"
    else:
        n = min(n_poses, wl.n_rec)
        take = lambda a: None if a is None else np.ascontiguousarray(a[:n])  # noqa: E731
        rec, items = take(wl.rec), n
        what = f"first {n} of {wl.n_rec} images"
    rot, sh, g = take(wl.rot), take(wl.shift), take(wl.grad)
    t0 = time.perf_counter()
    if wl.op == "insert":
        w = take(np.ascontiguousarray(wl.weights))
        oracle.backproject(wl.ndim, g, rot, weights=w, shift=sh, Dv=wl.D, **kw)
        op = "insertion with weights"
    else:
        oracle.project(wl.ndim, rec, rot, sh, **kw)
        op = "forward"
        if wl.op == "fwdbwd":
            oracle.project_backward(wl.ndim, rec, rot, g, sh, **kw)
            op = "forward + full backward"
    dt = time.perf_counter() - t0
    return items / dt, f"{what}, {op}, fp64, {dt:.1f} s"


def run_reference(args, wl):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    nthreads = cores()
    n_units = wl.n_pose if wl.ndim == 3 else wl.n_rec
    per_step = max(8, min(args.cpu_sample // 4 // (wl.n_rec if wl.ndim == 3 else 1), n_units))
    items = per_step * (wl.n_rec if wl.ndim == 3 else 1)
    import oracle

    oracle.build()
    for _ in range(args.warmup):
        oracle_rate(wl, per_step, nthreads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_rate(wl, per_step, nthreads)
    dt = time.perf_counter() - t0
    value = items * args.steps / dt
    sample = (f"each timed step is the first {items} of the workload's {wl.B} projections "
              f"({wl.op}, fp64); ms_per_step is that step's own time")
    line = {
        "impl": "reference", "metric": metric_for(wl), "value": value, "unit": "projections/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * dt / args.steps, "items_per_step": items,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(wl, l2_policy(wl)[1]),
        "cpu_baseline": {"value": value, "unit": "projections/s", "cores": nthreads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "projections/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------- clocks ----

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.proc = None
        self.path = None
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                   "-lms", "200"]
            if uuid:
                cmd += ["-i", uuid]
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(cmd, stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        rows = []
        for line in Path(self.path).read_text().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[4:8]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for _, _, r in rows for k in range(4) if r[k].lower() == "active"})
        sm = [r[0] for r in rows]
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------ ours ----

def l2_policy(wl) -> tuple[bool, str]:
    """(flush, note): inputs smaller than twice the 126 MB L2 get a 256 MB write between timed
    steps; larger ones stream through L2 anyway.  Both arms state the same policy for a
    workload, so that their config dicts are equal."""
    img = wl.D * wl.H * 8
    if wl.op == "insert":
        step = wl.B * img * 3 // 2
    elif wl.op == "fwd":
        step = wl.B * img
    else:
        step = 2 * wl.B * img
    step += (wl.rec.nbytes if wl.rec is not None else 0)
    if step < (256 << 20):
        return True, "L2 flushed between steps (256 MB write; step time = sum of the calls' events)"
    return False, (f"inputs larger than L2 ({wl.B * img / 1e9:.2f} GB of images read or written "
                   f"per kernel); no flush")


def workload_config(wl, l2: str, fused: bool = False) -> dict:
    world = dist_env()[0]
    par = "dp1" if world == 1 else f"dp{world} (pose shards of {wl.B} per rank, one volume all-reduce)"
    step = ("forward + one-pass backward (tp_project_backward_fused)" if fused else
            "forward + backward (volume, rotation and shift gradients)")
    return {"workload": wl.name, "D": wl.D, "batch": wl.B, "n_rec": wl.n_rec, "parallelism": par,
            "interp": "cubic" if wl.interp else "linear",
            "cutoff": wl.rc, "shift_amp": wl.extra["shift_amp"],
            "layout": "centered" if wl.layout else "fftw", "step": step, "l2": l2}


def hbm_bytes(wl):
    """Algorithmic HBM bytes per launch of each kernel: each unique input read once, each
    output written once.  Per projection: Do*(Do/2+1)*8 B of image (written by the forward,
    read by each backward kernel) and 4*(k*k+2) B of pose (read; the pose gradients are
    written by the pose-gradient kernel); per launch: the volume (read by the gathers, the
    volume gradient written by the scatter)."""
    img = wl.D * wl.H * 8
    k = wl.ndim
    pose = 4 * (k * k + 2)
    vol = wl.rec.nbytes
    return {"forward": wl.B * (img + pose) + vol,
            "grad_pose": wl.B * (img + 2 * pose) + vol,
            "grad_volume": wl.B * (img + pose) + vol,
            # one pass: the upstream gradient read once, the volume read, its gradient written
            "backward_fused": wl.B * (img + 2 * pose) + 2 * vol}


def measure_peaks(dev) -> dict | None:
    """The microbenchmarks of libtp_peaks.so on `dev` (None if that library is missing)."""
    try:
        from back_projection_fourier_b300 import peaks
    except ImportError:
        return None
    return peaks.measure(dev)


def onchip_work(wl) -> dict:
    """Algorithmic on-chip work per launch of each kernel of the step.  Taps = kept pixels x
    (4^3 cubic, 2^3 linear), in rows of 4 (cubic) / 2 (linear) consecutive x taps.
    Gathers read 8 B per tap.  Separable sums: the forward forms per row a complex sum
    weighted by the x weights (one complex FMA per tap) and adds it with the y-z weight
    (one per row): 4 flop per tap + 4 per row.  The pose gradients also form the
    x-derivative row sum (one more complex FMA per tap) and add value, x-, y- and
    z-derivative terms per row: 8 flop per tap + 16 per row.  Scatter: one float2
    read-modify-write and one complex FMA per tap."""
    nt = 4 if wl.interp else 2
    taps = kept_pixels(wl) * wl.B * nt ** wl.ndim
    rows = taps // nt
    gather = {"taps": taps, "bytes": 8 * taps, "rows": rows, "flop": 4 * taps + 4 * rows}
    scatter = {"taps": taps, "rmw": taps, "flop": 4 * taps}
    # the insertion with weights adds a float read-modify-write per tap: half the shared
    # bytes of a float2 one, counted as half of one
    insertion = {"taps": taps, "rmw": taps * 3 // 2, "flop": 6 * taps}
    if wl.ndim == 3 and not wl.interp:
        # the linear 3D scatter adds each tap with shared float atomics (two pixels of a
        # warp may share a voxel): 2 per tap, 3 with the weights
        scatter = dict(scatter, smem_red=2 * taps)
        insertion = dict(insertion, smem_red=3 * taps)
    return {"forward": gather, "grad_pose": dict(gather, flop=8 * taps + 16 * rows),
            "grad_volume": scatter, "grad_image": scatter, "insertion": insertion}


def relevant_roofline(wl, kms, hbm, hbm_peak, pk, sm_mhz) -> dict | None:
    """Per kernel: T_roof = max(HBM bytes / HBM peak, tap bytes / L1 load peak, flops / FP32
    peak, scatter read-modify-writes / shared-memory read-modify-write peak), every peak
    measured (HBM by the driver's copy; the rest by the microbenchmarks of this run);
    frac = T_roof / measured kernel time.  As context, `row_gather_frac` sets the gathers' tap
    rows against the measured rate of random 32-byte L1 loads (the gathers' access pattern),
    and `smem_red_frac` the linear 3D scatter's shared float atomics against the measured
    shared atomic rate (the operation that kernel issues)."""
    if not pk:
        return None
    work = onchip_work(wl)
    out = {}
    for k, ms in kms.items():
        w = work.get(k)
        if w is None:
            continue
        t = {"hbm": hbm[k] / (hbm_peak * 1e9),
             "fp32": w["flop"] / pk["fma"]["ops_per_s"]}
        if "bytes" in w:
            t["l1_load"] = w["bytes"] / pk["l1_load"]["bytes_per_s"]
        if "rmw" in w:
            t["smem_rmw"] = w["rmw"] / pk["smem_rmw"]["ops_per_s"]
        bound = max(t, key=t.get)
        ent = {"bound": bound, "t_roof_ms": 1e3 * t[bound], "kernel_ms": ms,
               "frac": 1e3 * t[bound] / ms, "t_ms": {u: 1e3 * v for u, v in t.items()}}
        if "rows" in w:
            ent["row_gather_frac"] = w["rows"] / pk["l1_gather32"]["ops_per_s"] / (ms * 1e-3)
        if "smem_red" in w:
            ent["smem_red_frac"] = w["smem_red"] / pk["smem_red"]["ops_per_s"] / (ms * 1e-3)
        out[k] = ent
    sms = pk.get("sms")
    if sm_mhz and sms:
        hz = sm_mhz * 1e6 * sms
        out["per_sm_per_clk"] = {"l1_load_B": pk["l1_load"]["bytes_per_s"] / hz,
                                 "l1_gather32_loads": pk["l1_gather32"]["ops_per_s"] / hz,
                                 "l1_gather8_loads": pk["l1_gather8"]["ops_per_s"] / hz,
                                 "smem_rmw": pk["smem_rmw"]["ops_per_s"] / hz,
                                 "smem_rmw_random": pk["smem_rmw_random"]["ops_per_s"] / hz,
                                 "smem_red": pk["smem_red"]["ops_per_s"] / hz,
                                 "l2_red": pk["l2_red"]["ops_per_s"] / hz,
                                 "fma_flop": pk["fma"]["ops_per_s"] / hz}
    out["peak_source"] = ("measured in this run: libtp_peaks.so microbenchmarks (CUDA events, best "
                          "of 3) on the same GPU; HBM: MEASURED_PEAKS.json copy bandwidth")
    return out


def kept_pixels(wl) -> int:
    ky = np.arange(wl.D) - wl.D // 2
    kx = np.arange(wl.H)
    return int(((kx[None, :] ** 2 + ky[:, None] ** 2) <= wl.rc ** 2).sum())


def host_link(b, hG, s_in, s_out, h2d, d2h, step_s) -> dict:
    """Host-link rates on the end-to-end step's own pinned buffers, best of three: the
    upstream gradient in alone, the projections out alone, and both at once.  A step that
    moves h2d bytes in and d2h bytes out takes at least the two-way time scaled to them."""
    import torch

    n_in = hG.numel() * hG.element_size()
    n_out = b["Y"].numel() * b["Y"].element_size()

    def timed(copy_in, copy_out):
        best = float("inf")
        for _ in range(3):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            if copy_in:
                with torch.cuda.stream(s_in):
                    b["dG"].copy_(hG, non_blocking=True)
            if copy_out:
                with torch.cuda.stream(s_out):
                    b["oY"].copy_(b["Y"], non_blocking=True)
            torch.cuda.synchronize()
            best = min(best, time.perf_counter() - t0)
        return best

    t_in, t_out, t_both = timed(True, False), timed(False, True), timed(True, True)
    # each direction at its own rate, and the overlapped part at the shared two-way rate
    floor_s = max(t_in * h2d / n_in, t_out * d2h / n_out, t_both * min(h2d / n_in, d2h / n_out))
    return {"h2d_GBps": n_in / t_in / 1e9, "d2h_GBps": n_out / t_out / 1e9,
            "both_ways_GBps": [n_in / t_both / 1e9, n_out / t_both / 1e9],
            "floor_ms_per_step": 1e3 * floor_s, "frac": floor_s / step_s}


def run_ours(args, wl):
    import torch
    import torch.distributed as dist

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    from back_projection_fourier_b300 import shard, tp

    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    op = tp.make_opts(wl.interp, wl.layout, 1.0, wl.rc)
    V = torch.from_numpy(wl.rec).to(dev)
    R = torch.from_numpy(wl.rot).to(dev)
    S = torch.from_numpy(wl.shift).to(dev) if wl.shift is not None else None
    G = torch.from_numpy(wl.grad).to(dev)
    Y = torch.empty_like(G)
    gV = torch.empty_like(V)
    gR = torch.empty_like(R)
    gS = torch.empty((1 if S is None else S.shape[0], wl.n_pose, 2), device=dev)
    # workspace of the gathers: each _ws call writes the grouped copy of the volume into it
    # (one short kernel) before its gather
    WS = tp.workspace_for(V, op)

    # The backward is issued as two C-ABI calls (pose gradients, then the volume gradient):
    # the same outputs as one tp_project_backward call, but each call is one gather or one
    # scatter, so CUDA events give every kernel's own duration.  With --fused-backward it is
    # one tp_project_backward_fused call (one kernel).  The step is the package's
    # data-parallel step: on N ranks each holds its own pose shard and the volume gradient
    # is summed with one all-reduce (a no-op on one rank).
    cur_ev = [None]

    def mark(k):
        if cur_ev[0] is not None:
            cur_ev[0][k].record(stream)

    def project(V_, R_, S_):
        mark(0)
        tp.tp_project_3d_to_2d_ws(V_, R_, S_, Y, WS, op, stream)
        mark(1)
        return Y

    def backward(V_, R_, S_, G_):
        if args.fused_backward:
            mark(2)
            tp.tp_project_backward_fused(3, V_, R_, S_, G_, gV, gR, gS, op, stream)
        else:
            tp.tp_project_backward_ws(3, V_, R_, S_, G_, None, gR, gS, WS, op, stream)
            mark(2)
            tp.tp_project_backward(3, V_, R_, S_, G_, gV, None, None, op, stream)
        mark(3)
        return gV, gR, gS

    def step(ev=None):
        cur_ev[0] = ev
        shard.shard_step(project, backward, V, R, S, G)

    flush_l2, l2_note = l2_policy(wl)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if flush_l2 else None

    # on-chip peaks of this GPU, measured now, before the step (the relevant roofline)
    onchip_peaks = measure_peaks(dev) if rank == 0 else None

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
        uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        uuid = None
    sampler = ClockSampler(uuid) if rank == 0 else None
    time.sleep(0.3 if sampler else 0)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    start.record(stream)
    for k in range(args.steps):
        if flush is not None:
            flush.zero_()
        step(evs[k])
    end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop() if sampler else None
    ms = start.elapsed_time(end)
    if world > 1:
        t = torch.tensor([ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    kms = {"forward": statistics.mean(e[0].elapsed_time(e[1]) for e in evs)}
    if args.fused_backward:
        kms["backward_fused"] = statistics.mean(e[2].elapsed_time(e[3]) for e in evs)
    else:
        kms["grad_pose"] = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
        kms["grad_volume"] = statistics.mean(e[2].elapsed_time(e[3]) for e in evs)
    # with an L2 flush between steps the step time is the sum of the calls' own events
    ms_step = ms / args.steps if flush is None else sum(kms.values())
    if flush is not None and world > 1:
        t = torch.tensor([ms_step], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms_step = float(t.item())
    value = wl.B * world / (ms_step * 1e-3)

    # e2e: host (pinned) inputs -> device -> forward + backward -> host outputs, every step
    e2e = None
    if not args.no_e2e and not args.fused_backward:
        hV, hR, hG = V.cpu().pin_memory(), R.cpu().pin_memory(), G.cpu().pin_memory()
        hS = S.cpu().pin_memory() if S is not None else None

        # Two buffer sets, device and host side, used by alternate steps, so that one step's
        # host->device copies and the previous step's device->host copies overlap the kernels
        # of their neighbours instead of waiting for them.
        def buffer_set(first):
            b = {"Y": Y, "gV": gV, "gR": gR, "gS": gS, "WS": WS} if first else {
                "Y": torch.empty_like(Y), "gV": torch.empty_like(gV), "gR": torch.empty_like(gR),
                "gS": torch.empty_like(gS), "WS": None if WS is None else torch.empty_like(WS)}
            b.update(dV=torch.empty_like(V), dR=torch.empty_like(R), dG=torch.empty_like(G),
                     dS=torch.empty_like(S) if S is not None else None)
            b.update(oY=torch.empty(Y.shape, dtype=Y.dtype, pin_memory=True),
                     ogV=torch.empty(gV.shape, dtype=gV.dtype, pin_memory=True),
                     ogR=torch.empty(gR.shape, dtype=gR.dtype, pin_memory=True),
                     ogS=torch.empty(gS.shape, dtype=gS.dtype, pin_memory=True))
            return b
        bufs = [buffer_set(True), buffer_set(False)]

        # Pipelined over chunks of poses on three streams: the host->device copy of chunk c+1
        # and the device->host copy of chunk c-1 overlap the kernels of chunk c.  Per chunk:
        # forward, pose gradients, and the chunk's share of the volume gradient, accumulated
        # by the insertion call (the transpose of the projection, the same kernel as the
        # backward's volume gradient).  One reconstruction: chunks are contiguous pose ranges.
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev_v = torch.cuda.Event()
        ev_vol = torch.cuda.Event()
        # per buffer set: its inputs were last read (kernels done) / its outputs last copied out
        ev_read = [torch.cuda.Event() for _ in bufs]
        ev_out = [torch.cuda.Event() for _ in bufs]
        sl = lambda t, a, b: None if t is None else t[:, a:b]  # noqa: E731
        n_e2e = [0]

        def e2e_step(copy_proj, bounds, ev_in, ev_done):
            k = n_e2e[0] % 2
            n_e2e[0] += 1
            b = bufs[k]
            dV, dR, dG, dS = b["dV"], b["dR"], b["dG"], b["dS"]
            with torch.cuda.stream(s_in):
                s_in.wait_event(ev_read[k])
                dV.copy_(hV, non_blocking=True)
                dR.copy_(hR, non_blocking=True)
                if dS is not None:
                    dS.copy_(hS, non_blocking=True)
                ev_v.record(s_in)
                for c, (a, bb) in enumerate(bounds):
                    dG[:, a:bb].copy_(hG[:, a:bb], non_blocking=True)
                    ev_in[c].record(s_in)
            stream.wait_event(ev_v)
            stream.wait_event(ev_out[k])
            for c, (a, bb) in enumerate(bounds):
                stream.wait_event(ev_in[c])
                Rc, Sc, Gc = sl(dR, a, bb), sl(dS, a, bb), sl(dG, a, bb)
                tp.tp_project_3d_to_2d_ws(dV, Rc, Sc, b["Y"][:, a:bb], b["WS"], op, stream)
                tp.tp_project_backward_ws(3, dV, Rc, Sc, Gc, None, b["gR"][:, a:bb],
                                          b["gS"][:, a:bb], b["WS"], op, stream)
                tp.tp_backproject_2d_to_3d(Gc, None, Rc, Sc, b["gV"], None, wl.D, c > 0, op,
                                           stream)
                ev_done[c].record(stream)
            ev_read[k].record(stream)
            shard.volume_allreduce(b["gV"])
            ev_vol.record(stream)
            with torch.cuda.stream(s_out):
                for c, (a, bb) in enumerate(bounds):
                    s_out.wait_event(ev_done[c])
                    if copy_proj:
                        b["oY"][:, a:bb].copy_(b["Y"][:, a:bb], non_blocking=True)
                    b["ogR"][:, a:bb].copy_(b["gR"][:, a:bb], non_blocking=True)
                    b["ogS"][:, a:bb].copy_(b["gS"][:, a:bb], non_blocking=True)
                s_out.wait_event(ev_vol)
                b["ogV"].copy_(b["gV"], non_blocking=True)
                ev_out[k].record(s_out)

        def timed_e2e(copy_proj, n_chunk):
            n_chunk = max(1, min(n_chunk, wl.n_pose)) if wl.n_rec == 1 else 1
            bounds = [(wl.n_pose * c // n_chunk, wl.n_pose * (c + 1) // n_chunk) for c in range(n_chunk)]
            ev_in = [torch.cuda.Event() for _ in bounds]
            ev_done = [torch.cuda.Event() for _ in bounds]
            for _ in range(max(1, args.warmup)):
                e2e_step(copy_proj, bounds, ev_in, ev_done)
            torch.cuda.synchronize()
            if world > 1:
                dist.barrier()
            t0 = time.perf_counter()
            for _ in range(args.steps):
                e2e_step(copy_proj, bounds, ev_in, ev_done)
            torch.cuda.synchronize()
            dt = time.perf_counter() - t0
            if world > 1:
                t = torch.tensor([dt], device=dev)
                dist.all_reduce(t, op=dist.ReduceOp.MAX)
                dt = float(t.item())
            return dt

        h2d = sum(x.numel() * x.element_size() for x in (hV, hR, hG) + ((hS,) if hS is not None else ()))
        # the step's result is its gradients (volume, rotations, shifts); the projections stay
        # on the device, where a loss would consume them
        dt = timed_e2e(False, args.e2e_chunks)
        d2h = sum(bufs[0][n].numel() * bufs[0][n].element_size() for n in ("ogV", "ogR", "ogS"))
        e2e = {"value": wl.B * world / (dt / args.steps), "unit": "projections/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "result_read_back": "volume, rotation and shift gradients",
               "pose_chunks": args.e2e_chunks}
        e2e["host_link"] = host_link(bufs[0], hG, s_in, s_out, h2d, d2h, dt / args.steps)
        # the same step reading the 1.09 GB of projections back as well
        dt_all = timed_e2e(True, args.e2e_proj_chunks)
        d2h_all = d2h + bufs[0]["oY"].numel() * bufs[0]["oY"].element_size()
        e2e["with_projections"] = {
            "value": wl.B * world / (dt_all / args.steps), "d2h_bytes_per_step": d2h_all,
            "pose_chunks": args.e2e_proj_chunks,
            "host_link": host_link(bufs[0], hG, s_in, s_out, h2d, d2h_all, dt_all / args.steps)}
        # both buffer sets ran the same inputs: their host results must agree (the forward
        # exactly, the gradients up to the order of their float sums)
        if n_e2e[0] >= 2:
            h0, h1 = bufs[0], bufs[1]
            rel = lambda n: float((h0[n] - h1[n]).abs().max()  # noqa: E731
                                  / h0[n].abs().max().clamp_min(1e-30))
            errs = {n: rel(n) for n in ("ogV", "ogR", "ogS")}
            if not torch.equal(h0["oY"], h1["oY"]) or max(errs.values()) > 1e-5:
                raise RuntimeError(f"e2e buffer sets disagree: {errs}")

    # roofline of the dominant kernel
    dom = max(kms, key=kms.get)
    dom_ms = kms[dom]
    peaks = {}
    try:
        peaks = json.loads((ROOT / "MEASURED_PEAKS.json").read_text())
    except (OSError, ValueError):
        pass
    peak = peaks.get("hbm_gbs")
    peak_src = "measured"
    if peak is None:
        peak, peak_src = 6400.0, "fallback"
    hbm = hbm_bytes(wl)
    achieved = hbm[dom] / (dom_ms * 1e-3) / 1e9
    traffic = None
    try:
        tr = json.loads(TRAFFIC_FILE.read_text())
        ent = tr.get(wl.name, {}).get(dom)
        if ent and ent.get("kernel_hash") == kernel_hash():
            traffic = ent["dram_bytes_per_launch"] * (wl.B / ent["batch"])
    except (OSError, ValueError, KeyError, ZeroDivisionError):
        pass
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": traffic, "kernel": dom,
                "peak_source": peak_src, "kernel_ms": dom_ms}
    relevant = relevant_roofline(wl, kms, hbm, peak, onchip_peaks, (clocks or {}).get("sm_mhz"))

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, sample = oracle_rate(wl, args.cpu_sample, cores())
        cpu = {"value": rate, "unit": "projections/s", "cores": cores(), "kind": "oracle",
               "sample": sample}
        # the same oracle on one host thread, on a sixteenth of the sample
        rate1, sample1 = oracle_rate(wl, max(64, args.cpu_sample // 16), 1)
        cpu["one_core"] = {"value": rate1, "unit": "projections/s", "cores": 1,
                           "sample": sample1}

    if rank == 0:
        line = {
            "metric": metric_for(wl), "value": value, "unit": "projections/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "ms_per_step_median": statistics.median(e[0].elapsed_time(e[3]) for e in evs),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded rfft of N(0,1) volume, uniform SO(3), CN(0,1) upstream grad)",
            "config": workload_config(wl, l2_note, args.fused_backward),
            "gpu_launches": ((2 + (WS is not None)) if args.fused_backward else
                             (3 + 2 * (WS is not None))) * args.steps,
            "kernel_ms": kms,
            "roofline": roofline, "roofline_relevant": relevant, "peaks_measured": onchip_peaks,
            "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_workload(args, wl):
    """One GPU, any other workload: the forward-only 3D workload, the insertion (with its
    CTF-like weights) and the 2D rotation workload (forward + backward).  Each C-ABI call of
    the step is timed with CUDA events on the launch stream; inputs smaller than L2 are
    followed, between steps, by a 256 MB write that flushes L2 (outside the timed calls)."""
    import torch
    from back_projection_fourier_b300 import tp

    world, _, local = dist_env()
    if world > 1:
        raise SystemExit("the non-headline workloads run on one GPU")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    op = tp.make_opts(wl.interp, wl.layout, 1.0, wl.rc)
    up = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    R, S = up(wl.rot), up(wl.shift)
    img = wl.D * wl.H * 8
    n_img = wl.n_rec * wl.n_pose
    calls, launches = {}, 0
    if wl.op == "fwd":
        V = up(wl.rec)
        Y = torch.empty((wl.n_rec, wl.n_pose, wl.D, wl.H), dtype=torch.complex64, device=dev)
        WS = tp.workspace_for(V, op)
        calls["forward"] = lambda: tp.tp_project_3d_to_2d_ws(V, R, S, Y, WS, op, stream)
        launches = 1 + (WS is not None)
        hbm = {"forward": n_img * img + V.numel() * 8}
        what = "forward"
    elif wl.op == "insert":
        P, W = up(wl.grad), up(np.ascontiguousarray(wl.weights))
        vol = torch.empty((1, wl.D, wl.D, wl.H), dtype=torch.complex64, device=dev)
        wvol = torch.empty((1, wl.D, wl.D, wl.H), device=dev)
        calls["insertion"] = lambda: tp.tp_backproject_2d_to_3d(P, W, R, S, vol, wvol, wl.D, False,
                                                                op, stream)
        launches = 1
        hbm = {"insertion": n_img * (img + img // 2) + vol.numel() * 12}
        what = "insertion with weights"
    elif wl.op == "fwdbwd" and wl.ndim == 2:
        V, G = up(wl.rec), up(wl.grad)
        Y, gV, gR = torch.empty_like(G), torch.empty_like(V), torch.empty_like(R)
        gS = torch.empty((S.shape[0], wl.n_pose, 2), device=dev)
        calls["forward"] = lambda: tp.tp_project_2d_to_2d(V, R, S, Y, op, stream)
        calls["grad_pose"] = lambda: tp.tp_project_backward(2, V, R, S, G, None, gR, gS, op, stream)
        calls["grad_image"] = lambda: tp.tp_project_backward(2, V, R, S, G, gV, None, None, op,
                                                             stream)
        launches = 3
        hbm = {"forward": 2 * n_img * img, "grad_pose": 2 * n_img * img,
               "grad_image": 2 * n_img * img}
        what = "2D rotation forward + backward"
    else:
        raise SystemExit(f"no timing recipe for workload {wl.name}")
    flush_l2, l2_note = l2_policy(wl)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if flush_l2 else None
    onchip_peaks = measure_peaks(dev)
    clock_sampler = ClockSampler(None)
    names = list(calls)
    ev = {k: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for k in names}
    tot = {k: 0.0 for k in names}
    for it in range(args.warmup + args.steps):
        if flush is not None:
            flush.zero_()
        for k in names:
            ev[k][0].record(stream)
            calls[k]()
            ev[k][1].record(stream)
        torch.cuda.synchronize()
        if it >= args.warmup:
            for k in names:
                tot[k] += ev[k][0].elapsed_time(ev[k][1])
    clocks = clock_sampler.stop()
    kms = {k: v / args.steps for k, v in tot.items()}
    ms_step = sum(kms.values())
    dom = max(kms, key=kms.get)
    peaks = {}
    try:
        peaks = json.loads((ROOT / "MEASURED_PEAKS.json").read_text())
    except (OSError, ValueError):
        pass
    peak = float(peaks.get("hbm_gbs") or 6400.0)
    achieved = hbm[dom] / (kms[dom] * 1e-3) / 1e9
    line = {
        "metric": metric_for(wl), "value": n_img / (ms_step * 1e-3),
        "unit": "projections/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": dict(workload_config(wl, l2_note), step=what),
        "gpu_launches": launches * args.steps, "kernel_ms": kms,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": None, "kernel": dom,
                     "peak_source": "measured" if peaks.get("hbm_gbs") else "fallback"},
        "roofline_relevant": relevant_roofline(wl, kms, hbm, peak, onchip_peaks,
                                               (clocks or {}).get("sm_mhz")),
        "peaks_measured": onchip_peaks, "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_oversampling_study(args):
    """On-the-fly oversampling against cubic interpolation without it, at D = 128: a real-space
    volume is zero-padded by 2 and transformed on every pass, then projected with linear
    weights at c = 2 R q; the alternative transforms the unpadded volume and projects with
    cubic weights.  'offline' variants start from a precomputed spectrum (projection only).
    Forward: images from the real-space volume; fwd+bwd adds the gradient of the real-space
    volume (projection backward, FFT backward, crop).  One JSON line per pose count."""
    import numpy as np
    import torch
    from back_projection_fourier_b300 import synth, tp

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    D = 128
    rng = np.random.default_rng(12345)
    vol = torch.from_numpy(rng.standard_normal((1, D, D, D)).astype(np.float32)).to(dev)
    variants = {"cubic_o1": (1, tp.TP_CUBIC), "linear_o2": (2, tp.TP_LINEAR)}
    bufs = {}
    for name, (f, interp) in variants.items():
        P = f * D
        X = torch.empty((1, P, P, P), device=dev)
        tp.tp_pad_volume(3, vol, f, X, stream)
        S = torch.fft.rfftn(X, dim=(-3, -2, -1))
        bufs[name] = dict(f=f, X=X, S=S, gS=torch.empty_like(S), gvol=torch.empty_like(vol),
                          op=tp.make_opts(interp, tp.TP_LAYOUT_FFTW, float(f), -1.0))
    for n_pose in [int(x) for x in args.study_poses.split(",")]:
        rot = torch.from_numpy(synth.rotations_3d(rng, n_pose)[None]).to(dev)
        sh = torch.from_numpy(rng.uniform(-5, 5, (1, n_pose, 2)).astype(np.float32)).to(dev)
        Y = torch.empty((1, n_pose, D, D // 2 + 1), dtype=torch.complex64, device=dev)
        G = torch.randn((1, n_pose, D, D // 2 + 1), dtype=torch.complex64, device=dev)
        res = {}
        for name, b in bufs.items():
            def fly_fwd(b=b):
                tp.tp_pad_volume(3, vol, b["f"], b["X"], stream)
                b["S"] = torch.fft.rfftn(b["X"], dim=(-3, -2, -1))
                tp.tp_project_3d_to_2d(b["S"], rot, sh, Y, b["op"], stream)

            def fly_fwdbwd(b=b):
                X = b["X"]
                tp.tp_pad_volume(3, vol, b["f"], X, stream)
                Xg = X.detach().requires_grad_(True)
                S = torch.fft.rfftn(Xg, dim=(-3, -2, -1))
                tp.tp_project_3d_to_2d(S.detach(), rot, sh, Y, b["op"], stream)
                tp.tp_project_backward(3, S.detach(), rot, sh, G, b["gS"], None, None, b["op"],
                                       stream)
                (gX,) = torch.autograd.grad(S, Xg, b["gS"])
                tp.tp_crop_volume(3, gX.contiguous(), b["f"], b["gvol"], stream)

            def off_fwd(b=b):
                tp.tp_project_3d_to_2d(b["S"], rot, sh, Y, b["op"], stream)

            def off_fwdbwd(b=b):
                tp.tp_project_3d_to_2d(b["S"], rot, sh, Y, b["op"], stream)
                tp.tp_project_backward(3, b["S"], rot, sh, G, b["gS"], None, None, b["op"], stream)

            for tag, fn in (("fly_fwd", fly_fwd), ("fly_fwdbwd", fly_fwdbwd),
                            ("offline_fwd", off_fwd), ("offline_fwdbwd", off_fwdbwd)):
                for _ in range(args.warmup):
                    fn()
                torch.cuda.synchronize()
                t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                t0.record(stream)
                for _ in range(args.steps):
                    fn()
                t1.record(stream)
                torch.cuda.synchronize()
                res[f"{name}_{tag}"] = t0.elapsed_time(t1) / args.steps
        line = {"study": "oversampling", "D": D, "n_pose": n_pose, "unit": "ms per pass",
                "ms": {k: round(v, 4) for k, v in res.items()},
                "ratio_fly_fwd": res["linear_o2_fly_fwd"] / res["cubic_o1_fly_fwd"],
                "ratio_fly_fwdbwd": res["linear_o2_fly_fwdbwd"] / res["cubic_o1_fly_fwdbwd"],
                "ratio_offline_fwd": res["linear_o2_offline_fwd"] / res["cubic_o1_offline_fwd"],
                "note": "ratios are linear o=2 time / cubic o=1 time; L2 not flushed (the "
                        "volumes are re-read every pass, as in training)"}
        print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse()
    if args.study == "oversampling":
        return run_oversampling_study(args)
    from back_projection_fourier_b300 import synth

    if args.impl == "reference":
        world, rank, _ = dist_env()
        if rank != 0:
            return 0
        interp = None if args.interp is None else (1 if args.interp == "cubic" else 0)
        return run_reference(args, synth.make_workload(args.workload, interp=interp))
    interp = None if args.interp is None else (1 if args.interp == "cubic" else 0)
    world, rank, _ = dist_env()
    if world > 1:
        # weak scaling: rank r draws and runs only its own shard of a batch of
        # (workload batch) x N poses
        from back_projection_fourier_b300 import shard
        wl = shard.workload_shard(args.workload, args.batch, rank, world, interp=interp)
    else:
        wl = synth.make_workload(args.workload, B=args.batch, interp=interp)
    if wl.op != "fwdbwd" or wl.ndim != 3:
        return run_workload(args, wl)
    return run_ours(args, wl)


if __name__ == "__main__":
    sys.exit(main())
