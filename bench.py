"""RMSNorm-for-training benchmark on GB300: one step = forward + backward over one batch.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--T 65536] [--H 4096] [--nondet]

Workload (default): plain rows T=65536, H=4096, BF16 x and dy ~ N(0,1), BF16 weight
1 + 0.1*N(0,1), eps 1e-6 (the pages' plain-rows configuration at its largest T); the
backward runs deterministic=True unless --nondet.  Inputs are 512 MiB per tensor, larger
than the 129 MB L2, so no flush is needed between iterations.

`value` is whole-job HBM throughput in GB/s: the algorithmic bytes of a step (forward
4*R*H + 4*R + |w|, backward 6*R*H + 4*R + |w| + 4*H; R = T*nh rows) times the steps of
all ranks, over the slowest rank's device time (CUDA events, inputs resident in HBM).
`e2e` is the same metric through the public C ABI with pinned host buffers, the
host->device input copies and the device->host result copies inside the timed region.
`roofline` is for the backward (the dominant op: its dx row pass with fused dw partials
plus the dw finish), timed by events around it on its launch stream.
`cpu_baseline` times the FP64 oracle on a bounded row sample on this host's cores.

With --gpus N under torchrun each rank runs an independent replica (the op has no
exchange step); timings are max-reduced over ranks on the host (gloo).

`--sweep` instead times every op of every workload family (isolated and back to back, one
JSON line each); `--sweep --sweep-once` runs each op once, untimed, for a profiler;
`--sweep --sweep-layernorm` does the same for the LayerNorm ops on the shapes of the
normalization tables.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "RMSNorm fwd/bwd µs and HBM GB/s per (T,H) vs GB300 peak; max dw err / budget"
FALLBACK_HBM_GBS = 6800.0
CSRC = os.path.join(ROOT, "rmsnorm_fwd_02_gb300", "csrc")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


# ---- byte model ----------------------------------------------------------------------

def fwd_bytes(R: int, H: int, wbytes: int) -> int:
    return 4 * R * H + 4 * R + wbytes * H


def bwd_bytes(R: int, H: int, wbytes: int) -> int:
    return 6 * R * H + 4 * R + wbytes * H + 4 * H


def kernel_source_hash() -> str:
    """Hash of the RMSNorm kernel sources (the rmsn_* files): the key that ties a recorded
    traffic figure to the kernels it was measured on.  The LayerNorm sources beside them
    (ln_*) build into the same library but no RMSNorm launch runs their code."""
    h = hashlib.sha256()
    for fn in sorted(os.listdir(CSRC)):
        if not fn.startswith("rmsn_"):
            continue
        with open(os.path.join(CSRC, fn), "rb") as f:
            h.update(fn.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        for key in ("hbm_gbs", "hbm_GBs", "hbm_gb_s"):
            if key in d:
                return float(d[key]), "measured"
    except (OSError, ValueError):
        pass
    return FALLBACK_HBM_GBS, "fallback"


def traffic_for(workload_key: str):
    """DRAM bytes per backward launch from the committed ncu summary, if it was taken on
    the current kernel sources; else None."""
    try:
        with open(TRAFFIC_FILE) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    ent = d.get(workload_key)
    if not ent or ent.get("source_hash") != kernel_source_hash():
        return None
    return ent.get("dram_bytes_per_op")


# ---- distributed replicas --------------------------------------------------------------

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def dist_init(ws: int):
    if ws <= 1:
        return None
    import torch.distributed as dist
    if not dist.is_initialized():
        dist.init_process_group("gloo")
    return dist


def reduce_max(value: float, dist) -> float:
    """Max of a host scalar over ranks (host-side gloo; not a data-path collective)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


# ---- clocks during the timed region -----------------------------------------------------

class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,"
              "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.lines = []
        self.proc = None
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "200"]
        if gpu_id:
            cmd += ["-i", gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ts, line in self.lines:
            if ts < t0 or ts > t1 + 0.25:
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                sm.append(float(parts[2]))
                mx.append(float(parts[3]))
            except ValueError:
                continue
            for name, val in zip(names, parts[6:10]):
                if val.lower() in ("active", "1"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def gpu_uuid(dev: int):
    import torch
    try:
        u = torch.cuda.get_device_properties(dev).uuid
        s = str(u)
        return s if s.startswith("GPU-") else "GPU-" + s
    except Exception:
        return None


def d2d_copy_gbps(torch, dev, stream, nbytes: int = 1 << 30, reps: int = 10) -> float:
    """Read+write bandwidth of a plain 1 GiB device-to-device copy (context only)."""
    src = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    dst = torch.empty_like(src)
    for _ in range(3):
        dst.copy_(src)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(reps):
        dst.copy_(src)
    b.record(stream)
    torch.cuda.synchronize()
    gbs = 2.0 * nbytes * reps / (a.elapsed_time(b) * 1e-3) / 1e9
    del src, dst
    return gbs


# ---- the CPU oracle baseline ------------------------------------------------------------

def oracle_step(case, rows: np.ndarray):
    """One forward + backward of the FP64 oracle over the rows `rows` of `case`."""
    import oracle
    H = case.H
    sub_x = case.x.reshape(-1, H)[rows].reshape(-1)
    sub_dy = case.dy.reshape(-1, H)[rows].reshape(-1)
    n = rows.size
    _, r64, _ = oracle.fwd(sub_x, case.w, case.eps, n, 1, H, H, H)
    r_in = r64.astype(np.float32).astype(np.float64)
    oracle.bwd_dx(sub_x, sub_dy, r_in, case.w, n, 1, H, H, H)
    oracle.bwd_dw(sub_x, sub_dy, r_in, n, 1, H, H, H)


def cpu_baseline(case, wbytes: int, budget_s: float = 10.0, rows_per_step: int = 64):
    rng = np.random.default_rng(1)
    rows = np.sort(rng.choice(case.R, size=min(rows_per_step, case.R), replace=False))
    n_steps = 0
    t0 = time.perf_counter()
    while True:
        oracle_step(case, rows)
        n_steps += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    nbytes = (fwd_bytes(rows.size, case.H, wbytes) + bwd_bytes(rows.size, case.H, wbytes))
    return {
        "value": nbytes * n_steps / el / 1e9,
        "unit": "GB/s",
        "cores": 1,
        "kind": "oracle",
        "sample": (f"{n_steps} x forward+backward of {rows.size} random rows of the "
                   f"[{case.T},{case.H}] workload, {el:.1f} s single-threaded FP64"),
    }


# ---- the reference arm: the oracle, as it stands ---------------------------------------

def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    from rmsnorm_fwd_02_gb300 import synth
    case = synth.make_case(0, args.T, args.H)
    wbytes = 2
    rows = np.arange(min(64, case.R), dtype=np.int64)
    for _ in range(args.warmup):
        oracle_step(case, rows)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(case, rows)
    el = time.perf_counter() - t0
    nbytes = fwd_bytes(rows.size, case.H, wbytes) + bwd_bytes(rows.size, case.H, wbytes)
    value = nbytes * args.steps / el / 1e9
    sample = f"each step: forward+backward of {rows.size} rows of [{args.T},{args.H}]"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": el / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(args),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def workload_config(args):
    mode = "non-deterministic" if args.nondet else "deterministic"
    return {
        "workload": (f"plain rows T={args.T} H={args.H}: BF16 x, dy ~ N(0,1), BF16 w = "
                     f"1+0.1*N(0,1), eps 1e-6; step = forward + backward ({mode})"),
        "T": args.T, "H": args.H, "nh": 1, "w": "bf16", "storage": "bf16",
        "deterministic": not args.nondet,
        "l2": "inputs larger than L2 (no flush): 2*T*H bytes per tensor",
    }


# ---- our arm -------------------------------------------------------------------------------

def run_ours(args):
    import torch
    from rmsnorm_fwd_02_gb300 import _native as N
    from rmsnorm_fwd_02_gb300 import synth

    ws, rank, local = dist_env()
    dist = dist_init(ws)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    det = not args.nondet

    case = synth.make_case(0, args.T, args.H)
    R, H, T = case.R, case.H, case.T
    wbytes = 2

    def dbf(bits):
        return torch.from_numpy(bits.view(np.int16)).to(dev).view(torch.bfloat16)

    x, dy, w = dbf(case.x), dbf(case.dy), dbf(case.w)
    y = torch.empty(R * H, dtype=torch.bfloat16, device=dev)
    dx = torch.empty_like(y)
    rstd = torch.empty(R, dtype=torch.float32, device=dev)
    dw = torch.empty(H, dtype=torch.float32, device=dev)
    nws = N.rmsnorm_train_bwd_workspace_bytes(T, 1, H, det)
    wsb = torch.empty(max(nws, 16), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    lib = N.lib()

    def fwd_call(xp, wp, yp, rp):
        st = lib.rmsnorm_train_fwd(xp, None, wp, 0, yp, None, rp, T, 1, H, H, H, 1e-6, sh)
        if st:
            raise N.RmsnError("rmsnorm_train_fwd", st)

    def bwd_call(xp, dyp, wp, dxp, rp, dwp):
        st = lib.rmsnorm_train_bwd(xp, dyp, None, rp, wp, 0, dxp, dwp, wsb.data_ptr(), nws,
                                   T, 1, H, H, H, int(det), sh)
        if st:
            raise N.RmsnError("rmsnorm_train_bwd", st)

    xp, dyp, wp = x.data_ptr(), dy.data_ptr(), w.data_ptr()
    yp, dxp, rp, dwp = y.data_ptr(), dx.data_ptr(), rstd.data_ptr(), dw.data_ptr()

    def step():
        fwd_call(xp, wp, yp, rp)
        bwd_call(xp, dyp, wp, dxp, rp, dwp)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    # ---- device-timed region 1: K whole steps back to back (the headline) ----
    sampler = ClockSampler(gpu_uuid(local)) if rank == 0 else None
    time.sleep(0.5 if sampler else 0.0)
    t_begin = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    barrier(dist)
    torch.cuda.synchronize()
    wall0 = time.time()
    t_begin.record(stream)
    for _ in range(args.steps):
        step()
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(dist)
    total_ms = t_begin.elapsed_time(t_end)

    # ---- device-timed region 2: the same steps with events around each op ----
    k2 = min(args.steps, 500)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(k2)]
    torch.cuda.synchronize()
    for i in range(k2):
        ev[i][0].record(stream)
        fwd_call(xp, wp, yp, rp)
        ev[i][1].record(stream)
        bwd_call(xp, dyp, wp, dxp, rp, dwp)
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    wall1 = time.time()
    fwd_ms = [e[0].elapsed_time(e[1]) for e in ev]
    bwd_ms = [e[1].elapsed_time(e[2]) for e in ev]
    clocks = sampler.summary(wall0, wall1) if sampler else None
    if sampler:
        sampler.stop()
    max_ms = reduce_max(total_ms, dist)

    # ---- context: the device-to-device copy bandwidth of this GPU (cudaMemcpyAsync) ----
    copy_gbs = d2d_copy_gbps(torch, dev, stream)

    step_bytes = fwd_bytes(R, H, wbytes) + bwd_bytes(R, H, wbytes)
    value = step_bytes * args.steps * ws / (max_ms * 1e-3) / 1e9
    fwd_us = statistics.mean(fwd_ms) * 1e3
    bwd_us = statistics.mean(bwd_ms) * 1e3

    # ---- end to end through the C ABI with pinned host buffers ----
    e2e_steps = max(3, min(args.steps, args.e2e_steps))
    hx = torch.from_numpy(case.x.view(np.int16)).view(torch.bfloat16).pin_memory()
    hdy = torch.from_numpy(case.dy.view(np.int16)).view(torch.bfloat16).pin_memory()
    hw = torch.from_numpy(case.w.view(np.int16)).view(torch.bfloat16).pin_memory()
    hy = torch.empty(R * H, dtype=torch.bfloat16).pin_memory()
    hdx = torch.empty(R * H, dtype=torch.bfloat16).pin_memory()
    hr = torch.empty(R, dtype=torch.float32).pin_memory()
    hdw = torch.empty(H, dtype=torch.float32).pin_memory()
    def e2e_step():
        x.copy_(hx, non_blocking=True)
        dy.copy_(hdy, non_blocking=True)
        w.copy_(hw, non_blocking=True)
        step()
        hy.copy_(y, non_blocking=True)
        hr.copy_(rstd, non_blocking=True)
        hdx.copy_(dx, non_blocking=True)
        hdw.copy_(dw, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    barrier(dist)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = reduce_max(e0.elapsed_time(e1), dist)
    h2d = 2 * R * H * 2 + H * wbytes
    d2h = 2 * R * H * 2 + 4 * R + 4 * H
    e2e_value = step_bytes * e2e_steps * ws / (e2e_ms * 1e-3) / 1e9

    # ---- dw error vs the oracle (outside every timed region) ----
    dw_ratio = None
    if rank == 0 and not args.skip_dw_check:
        import oracle
        _, r64, _ = oracle.fwd(case.x, case.w, case.eps, T, 1, H, H, H, want_y=False)
        r32 = r64.astype(np.float32)
        rin = torch.from_numpy(r32).to(dev)
        x.copy_(hx)
        dy.copy_(hdy)
        w.copy_(hw)
        st = lib.rmsnorm_train_bwd(x.data_ptr(), dy.data_ptr(), None, rin.data_ptr(),
                                   w.data_ptr(), 0, dx.data_ptr(), dw.data_ptr(),
                                   wsb.data_ptr(), nws, T, 1, H, H, H, int(det), sh)
        assert st == 0
        dw64 = oracle.bwd_dw(case.x, case.dy, r32.astype(np.float64), T, 1, H, H, H)
        err = np.abs(dw.cpu().numpy().astype(np.float64) - dw64)
        dw_ratio = float((err / (1e-4 + 1e-4 * np.abs(dw64))).max())

    if rank != 0:
        return 0
    peak, peak_kind = measured_peak()
    bwd_achieved = bwd_bytes(R, H, wbytes) / (bwd_us * 1e-6) / 1e9
    fwd_achieved = fwd_bytes(R, H, wbytes) / (fwd_us * 1e-6) / 1e9
    wkey = f"bwd_plain_T{T}_H{H}_{'det' if det else 'nondet'}"
    cpu = cpu_baseline(case, wbytes, budget_s=args.cpu_seconds) if ws == 1 else None
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "GB/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": max_ms / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": workload_config(args),
        "roofline": {
            "bound": "hbm",
            "kernel": "backward op (dx row pass with fused dw partials + dw finish)",
            "achieved": bwd_achieved,
            "peak": peak,
            "peak_kind": f"{peak_kind} HBM copy bandwidth",
            "unit": "GB/s",
            "frac": bwd_achieved / peak,
            "traffic": traffic_for(wkey),
        },
        "fwd": {"us": fwd_us, "GBps": fwd_achieved, "frac": fwd_achieved / peak},
        "bwd": {"us": bwd_us, "GBps": bwd_achieved, "frac": bwd_achieved / peak},
        "dw_err_over_budget": dw_ratio,
        "d2d_copy_GBps": copy_gbs,
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps},
        "gpu_launches": 3 * args.steps,  # fwd + bwd row pass + dw finish per step
        "clocks": clocks,
        "source_hash": kernel_source_hash(),
    }
    print(json.dumps(line))
    return 0


# ---- per-workload sweep (one JSON line per op and workload; not the headline) -----------

SWEEP = [
    # label, T, H, nh, buf_heads, w_fp32, residual
    ("plain", 16384, 4096, 1, None, False, False),
    ("plain", 65536, 4096, 1, None, False, False),
    ("stress", 32768, 1536, 1, None, True, False),
    ("stress", 65536, 1536, 1, None, True, False),
    ("stress", 131072, 1536, 1, None, True, False),
    ("stress", 32768, 2048, 1, None, True, False),
    ("stress", 131072, 2048, 1, None, True, False),
    ("stress", 32768, 5120, 1, None, True, False),
    ("stress", 131072, 5120, 1, None, True, False),
    ("residual", 30720, 6144, 1, None, False, True),
    ("residual", 65536, 6144, 1, None, False, True),
    ("heads24of32", 4096, 256, 24, 32, True, False),
    ("heads24of32", 16384, 256, 24, 32, True, False),
    ("heads24of32", 65536, 256, 24, 32, True, False),
    ("heads4", 65536, 256, 4, None, True, False),
]


def _sweep_timers(torch, stream, flush):
    """The sweep's two clocks (see run_sweep): isolated launches after a read-based L2
    flush, and launches back to back over rotating input sets."""

    def timed(fn, reps):
        out = []
        for _ in range(3):
            fn(0)
        for _ in range(reps):
            flush.sum()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn(0)
            b.record(stream)
            torch.cuda.synchronize()
            out.append(a.elapsed_time(b) * 1e3)
        # the event clock ticks in steps of about 2 us on this part: a median would be one
        # of those steps, the mean of the middle 80 % resolves below it
        out.sort()
        cut = len(out) // 10
        return statistics.fmean(out[cut:len(out) - cut])

    def timed_stream(fn, nsets, reps):
        n = max(reps, 2 * nsets)
        for i in range(nsets):
            fn(i)
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for i in range(n):
            fn(i % nsets)
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) * 1e3 / n

    return timed, timed_stream


def run_sweep(args):
    """Times each op of each workload (forward; backward in both modes, with and without dh
    in the residual form; the checkpointed step 2xfwd+bwd = forward, forward recompute,
    deterministic backward) two ways, CUDA events on the launch stream:

    isolated  `reps` launches, each after an L2 flush outside the events; trimmed mean.
              The flush READS a 512 MiB buffer, so L2 is cold but clean (a write-based
              flush would leave dirty lines whose write-back lands inside the next timed
              kernel).  Includes the launch's ramp-up and tail and the gap before the first
              CTA starts.
    stream    `reps` launches back to back inside one event pair, rotating over copies of
              the inputs and outputs so that every launch finds its inputs out of L2 (the
              sets in between exceed twice the L2); time / launches.  This is the op as a
              training step runs it, queued behind other work."""
    import torch
    from rmsnorm_fwd_02_gb300 import _native as N
    from rmsnorm_fwd_02_gb300 import synth

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    lib = N.lib()
    flush = torch.ones(128 << 20, dtype=torch.int32, device=dev)
    peak, peak_kind = measured_peak()
    l2_bytes = 129 << 20

    def dbf(bits):
        return torch.from_numpy(bits.view(np.int16)).to(dev).view(torch.bfloat16)

    timed, timed_stream = _sweep_timers(torch, stream, flush)

    for label, T, H, nh, bh, w32, res in SWEEP:
        if args.sweep_filter and args.sweep_filter != f"{label}_{T}_{H}":
            continue
        c = synth.make_case(0, T, H, nh=nh, buf_heads=bh, w_fp32=w32, residual=res, dh=res)
        R = c.R
        wbytes = 4 if w32 else 2
        wd = 1 if w32 else 0
        base = {"x": dbf(c.x), "dy": dbf(c.dy)}
        if res:
            base["rr"], base["dh"] = dbf(c.residual), dbf(c.dh)
        w = torch.from_numpy(c.w).to(dev) if w32 else dbf(c.w)
        set_bytes = sum(t.numel() * t.element_size() for t in base.values()) + 3 * R * H * 2
        nsets = 1 if args.sweep_once else max(2, -(-2 * l2_bytes // set_bytes) + 1)
        sets = []
        for i in range(nsets):
            st = {k: (v if i == 0 else v.clone()) for k, v in base.items()}
            st["y"] = torch.empty(R * H, dtype=torch.bfloat16, device=dev)
            st["h"] = torch.empty_like(st["y"]) if res else None
            st["dx"] = torch.empty_like(st["y"])
            st["rstd"] = torch.empty(R, dtype=torch.float32, device=dev)
            st["dw"] = torch.empty(H, dtype=torch.float32, device=dev)
            sets.append(st)

        def fwd(i):
            q = sets[i]
            st = lib.rmsnorm_train_fwd(q["x"].data_ptr(), q["rr"].data_ptr() if res else None,
                                       w.data_ptr(), wd, q["y"].data_ptr(),
                                       q["h"].data_ptr() if res else None,
                                       q["rstd"].data_ptr(), T, nh, H, c.s_tok, c.s_head,
                                       1e-6, sh)
            assert st == 0, st

        for i in range(1 if args.sweep_once else nsets):
            fwd(i)
        s_tok, s_head = (nh * H, H) if res else (c.s_tok, c.s_head)
        rows = [("fwd", fwd, (8 if res else 4) * R * H + 4 * R + wbytes * H)]
        for det in (1, 0):
            for use_dh in ((False, True) if res else (False,)):
                nws = N.rmsnorm_train_bwd_workspace_bytes(T, nh, H, det)
                ws = torch.empty(max(nws, 16), dtype=torch.uint8, device=dev)

                def bwd(i, det=det, use_dh=use_dh, ws=ws, nws=nws):
                    q = sets[i]
                    xs = q["h"] if res else q["x"]
                    st = lib.rmsnorm_train_bwd(xs.data_ptr(), q["dy"].data_ptr(),
                                               q["dh"].data_ptr() if use_dh else None,
                                               q["rstd"].data_ptr(), w.data_ptr(), wd,
                                               q["dx"].data_ptr(), q["dw"].data_ptr(),
                                               ws.data_ptr(), nws, T, nh, H, s_tok, s_head,
                                               det, sh)
                    assert st == 0, st

                name = ("bwd_det" if det else "bwd_nondet") + ("+dh" if use_dh else "")
                bwd_bytes_ = (8 if use_dh else 6) * R * H + 4 * R + wbytes * H + 4 * H
                rows.append((name, bwd, bwd_bytes_))
                if det and not use_dh:
                    # the checkpointed step: forward, forward recompute, backward
                    def ckpt(i, bwd=bwd):
                        fwd(i)
                        fwd(i)
                        bwd(i)

                    rows.append(("2xfwd+bwd_det", ckpt, 2 * rows[0][2] + bwd_bytes_))
        if args.sweep_once:
            torch.cuda.synchronize()
            for name, fn, nbytes in rows:
                if name.startswith("2x") or "nondet" in name or name == "fwd":
                    continue   # the forward already ran once, for the backward's rstd
                fn(0)
                torch.cuda.synchronize()
                print(json.dumps({"sweep": label, "op": name, "T": T, "H": H, "nh": nh,
                                  "ran_once": True}), flush=True)
            del sets, base, w
            torch.cuda.empty_cache()
            continue
        for name, fn, nbytes in rows:
            us = timed(fn, args.sweep_reps)
            us_s = timed_stream(fn, nsets, args.sweep_reps)
            gbs = nbytes / (us * 1e-6) / 1e9
            gbs_s = nbytes / (us_s * 1e-6) / 1e9
            print(json.dumps({"sweep": label, "op": name, "T": T, "H": H, "nh": nh,
                              "w": "fp32" if w32 else "bf16", "us": round(us, 2),
                              "GBps": round(gbs, 1), "frac": round(gbs / peak, 4),
                              "stream_us": round(us_s, 2), "stream_GBps": round(gbs_s, 1),
                              "stream_frac": round(gbs_s / peak, 4), "input_sets": nsets,
                              "peak": peak, "peak_kind": peak_kind,
                              "bytes": nbytes}), flush=True)
        del sets, base, w
        torch.cuda.empty_cache()
    return 0


# ---- LayerNorm sweep (the normalization tables' shapes: M rows of hidden_size, BF16) ------

LN_SWEEP = [(M, H) for H in (3584, 4096, 8192, 16384) for M in (1024, 2048, 4096, 8192)] + [
    (32768, 4096), (65536, 4096), (16384, 8192)]


def ln_fwd_bytes(R: int, H: int, wbytes: int) -> int:
    """x read, y written (BF16), mean and rstd written (FP32), w and b read."""
    return 4 * R * H + 8 * R + 2 * wbytes * H


def ln_bwd_bytes(R: int, H: int, wbytes: int) -> int:
    """x, dy read and dx written (BF16), mean and rstd read, w read, dw and db written."""
    return 6 * R * H + 8 * R + wbytes * H + 8 * H


def run_ln_sweep(args):
    """The LayerNorm forward and backward (both modes) on the normalization tables' shapes
    (M in 1024..8192 at hidden 3584, 4096, 8192, 16384) and a few larger M, with RMSNorm's
    forward and deterministic backward on the same inputs beside them (H <= 8192), timed
    like run_sweep:
    isolated (L2 flushed by a read) and back to back over rotating input sets."""
    import torch
    from rmsnorm_fwd_02_gb300 import _native as N
    from rmsnorm_fwd_02_gb300 import synth

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    lib = N.lib()
    flush = torch.ones(128 << 20, dtype=torch.int32, device=dev)
    peak, peak_kind = measured_peak()
    l2_bytes = 129 << 20
    timed, timed_stream = _sweep_timers(torch, stream, flush)

    def dbf(bits):
        return torch.from_numpy(bits.view(np.int16)).to(dev).view(torch.bfloat16)

    for M, H in LN_SWEEP:
        if args.sweep_filter and args.sweep_filter != f"layernorm_{M}_{H}":
            continue
        c = synth.make_ln_case(0, M, H)
        wbytes = 4 if c.wb_fp32 else 2
        wd = N.RMSN_W_FP32 if c.wb_fp32 else N.RMSN_W_BF16
        w = torch.from_numpy(c.w).to(dev) if c.wb_fp32 else dbf(c.w)
        b = torch.from_numpy(c.b).to(dev) if c.wb_fp32 else dbf(c.b)
        base = {"x": dbf(c.x), "dy": dbf(c.dy)}
        set_bytes = 4 * M * H * 2
        nsets = 1 if args.sweep_once else max(2, -(-2 * l2_bytes // set_bytes) + 1)
        sets = []
        for i in range(nsets):
            st = {k: (v if i == 0 else v.clone()) for k, v in base.items()}
            st["y"] = torch.empty(M * H, dtype=torch.bfloat16, device=dev)
            st["dx"] = torch.empty_like(st["y"])
            st["mean"] = torch.empty(M, dtype=torch.float32, device=dev)
            st["rstd"] = torch.empty(M, dtype=torch.float32, device=dev)
            st["dw"] = torch.empty(H, dtype=torch.float32, device=dev)
            st["db"] = torch.empty(H, dtype=torch.float32, device=dev)
            sets.append(st)

        def fwd(i):
            q = sets[i]
            st = lib.layernorm_train_fwd(q["x"].data_ptr(), w.data_ptr(), b.data_ptr(), wd,
                                         q["y"].data_ptr(), q["mean"].data_ptr(),
                                         q["rstd"].data_ptr(), M, H, c.eps, sh)
            assert st == 0, st

        for i in range(1 if args.sweep_once else nsets):
            fwd(i)
        rows = [("ln_fwd", fwd, ln_fwd_bytes(M, H, wbytes))]
        for det in (1, 0):
            nws = N.layernorm_train_bwd_workspace_bytes(M, H, det)
            ws = torch.empty(max(nws, 16), dtype=torch.uint8, device=dev)

            def bwd(i, det=det, ws=ws, nws=nws):
                q = sets[i]
                st = lib.layernorm_train_bwd(q["x"].data_ptr(), q["dy"].data_ptr(),
                                             q["mean"].data_ptr(), q["rstd"].data_ptr(),
                                             w.data_ptr(), wd, q["dx"].data_ptr(),
                                             q["dw"].data_ptr(), q["db"].data_ptr(),
                                             ws.data_ptr(), nws, M, H, det, sh)
                assert st == 0, st

            rows.append(("ln_bwd_det" if det else "ln_bwd_nondet", bwd,
                         ln_bwd_bytes(M, H, wbytes)))
        if H <= 8192:
            # RMSNorm on the same rows, weight and gradient (the tables put the two norms
            # side by side): forward, and the deterministic backward on its rstd
            nws_r = N.rmsnorm_train_bwd_workspace_bytes(M, 1, H, 1)
            ws_r = torch.empty(max(nws_r, 16), dtype=torch.uint8, device=dev)

            def rms_fwd(i):
                q = sets[i]
                st = lib.rmsnorm_train_fwd(q["x"].data_ptr(), None, w.data_ptr(), wd,
                                           q["y"].data_ptr(), None, q["rstd"].data_ptr(),
                                           M, 1, H, H, H, 1e-6, sh)
                assert st == 0, st

            def rms_bwd(i):
                q = sets[i]
                st = lib.rmsnorm_train_bwd(q["x"].data_ptr(), q["dy"].data_ptr(), None,
                                           q["rstd"].data_ptr(), w.data_ptr(), wd,
                                           q["dx"].data_ptr(), q["dw"].data_ptr(),
                                           ws_r.data_ptr(), nws_r, M, 1, H, H, H, 1, sh)
                assert st == 0, st

            rows.append(("rms_fwd", rms_fwd, fwd_bytes(M, H, wbytes)))
            rows.append(("rms_bwd_det", rms_bwd, bwd_bytes(M, H, wbytes)))
        if args.sweep_once:
            torch.cuda.synchronize()
            rows[1][1](0)
            torch.cuda.synchronize()
            print(json.dumps({"sweep": "layernorm", "op": "ln_fwd+ln_bwd_det", "M": M, "H": H,
                              "ran_once": True}), flush=True)
            del sets, base, w, b
            torch.cuda.empty_cache()
            continue
        for name, fn, nbytes in rows:
            us = timed(fn, args.sweep_reps)
            us_s = timed_stream(fn, nsets, args.sweep_reps)
            gbs = nbytes / (us * 1e-6) / 1e9
            gbs_s = nbytes / (us_s * 1e-6) / 1e9
            print(json.dumps({"sweep": "layernorm", "op": name, "M": M, "H": H,
                              "w": "fp32" if c.wb_fp32 else "bf16", "us": round(us, 2),
                              "GBps": round(gbs, 1), "frac": round(gbs / peak, 4),
                              "stream_us": round(us_s, 2), "stream_GBps": round(gbs_s, 1),
                              "stream_frac": round(gbs_s / peak, 4), "input_sets": nsets,
                              "peak": peak, "peak_kind": peak_kind,
                              "bytes": nbytes}), flush=True)
        del sets, base, w, b
        torch.cuda.empty_cache()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--T", type=int, default=65536)
    ap.add_argument("--H", type=int, default=4096)
    ap.add_argument("--nondet", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--skip-dw-check", action="store_true")
    ap.add_argument("--sweep", action="store_true",
                    help="time each op on every workload family (one line each) instead")
    ap.add_argument("--sweep-reps", type=int, default=30)
    ap.add_argument("--sweep-filter", default="",
                    help="only the sweep entry LABEL_T_H (e.g. stress_131072_1536)")
    ap.add_argument("--sweep-layernorm", action="store_true",
                    help="with --sweep: the LayerNorm ops on the normalization tables' shapes "
                         "(filter entries as layernorm_M_H)")
    ap.add_argument("--sweep-once", action="store_true",
                    help="with --sweep: run each op of each selected workload once, untimed "
                         "(one launch of each kernel, for a profiler)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    if args.sweep:
        return run_ln_sweep(args) if args.sweep_layernorm else run_sweep(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
