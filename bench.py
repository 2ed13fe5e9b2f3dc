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
    """One forward + backward of the FP64 oracle over the rows `rows` of `case` (plain
    rows).  Returns the block's dw (the sum over its rows)."""
    import oracle
    H = case.H
    sub_x = case.x.reshape(-1, H)[rows].reshape(-1)
    sub_dy = case.dy.reshape(-1, H)[rows].reshape(-1)
    n = rows.size
    _, r64, _ = oracle.fwd(sub_x, case.w, case.eps, n, 1, H, H, H)
    r_in = r64.astype(np.float32).astype(np.float64)
    oracle.bwd_dx(sub_x, sub_dy, r_in, case.w, n, 1, H, H, H)
    return oracle.bwd_dw(sub_x, sub_dy, r_in, n, 1, H, H, H)


class OracleRunner:
    """Times the oracle as it stands on this host's cores: one thread per row block (the
    oracle's C functions run without the GIL), each block's forward, dx and dw by the
    oracle itself, the blocks' dw added in block order afterwards.  The row blocks split
    a fixed random sample of the workload's rows."""

    def __init__(self, case, rows_per_thread: int, threads: int | None = None):
        from concurrent.futures import ThreadPoolExecutor
        self.case = case
        self.threads = max(1, threads or (os.cpu_count() or 1))
        n = min(rows_per_thread * self.threads, case.R)
        rng = np.random.default_rng(1)
        rows = np.sort(rng.choice(case.R, size=n, replace=False))
        self.blocks = [b for b in np.array_split(rows, self.threads) if b.size]
        self.rows = int(rows.size)
        self.pool = ThreadPoolExecutor(max_workers=self.threads) if self.threads > 1 else None

    def step(self):
        if self.pool is None:
            parts = [oracle_step(self.case, b) for b in self.blocks]
        else:
            parts = list(self.pool.map(lambda b: oracle_step(self.case, b), self.blocks))
        dw = parts[0]
        for p in parts[1:]:
            dw = dw + p
        return dw

    def close(self):
        if self.pool is not None:
            self.pool.shutdown()


def cpu_baseline(case, wbytes: int, budget_s: float = 10.0, rows_per_thread: int = 64):
    """The oracle's forward + backward throughput on this host, single-threaded and on all
    cores (each for about half of `budget_s`)."""
    out = {}
    for threads in (1, os.cpu_count() or 1):
        runner = OracleRunner(case, rows_per_thread, threads)
        n_steps = 0
        t0 = time.perf_counter()
        while True:
            runner.step()
            n_steps += 1
            el = time.perf_counter() - t0
            if el >= budget_s / 2:
                break
        runner.close()
        nbytes = fwd_bytes(runner.rows, case.H, wbytes) + bwd_bytes(runner.rows, case.H, wbytes)
        out[threads] = (nbytes * n_steps / el / 1e9, n_steps, runner.rows, el)
    cores = max(out)
    v, n_steps, rows, el = out[cores]
    v1, n1, rows1, el1 = out[1]
    return {
        "value": v,
        "unit": "GB/s",
        "cores": cores,
        "host_cpu_count": os.cpu_count(),
        "single_thread_value": v1,
        "kind": "oracle",
        "sample": (f"{n_steps} x forward+backward of {rows} random rows of the "
                   f"[{case.T},{case.H}] workload in {cores} row blocks on {cores} threads "
                   f"({el:.1f} s); single-threaded: {n1} x {rows1} rows ({el1:.1f} s); FP64"),
    }


# ---- the reference arm: the oracle, as it stands ---------------------------------------

def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    from rmsnorm_fwd_02_gb300 import synth
    case = synth.make_case(0, args.T, args.H)
    wbytes = 2
    runner = OracleRunner(case, rows_per_thread=64)
    for _ in range(args.warmup):
        runner.step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        runner.step()
    el = time.perf_counter() - t0
    runner.close()
    nbytes = fwd_bytes(runner.rows, case.H, wbytes) + bwd_bytes(runner.rows, case.H, wbytes)
    value = nbytes * args.steps / el / 1e9
    sample = (f"each step: forward+backward of {runner.rows} random rows of "
              f"[{args.T},{args.H}] in {runner.threads} row blocks on {runner.threads} threads")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": el / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(args),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": runner.threads,
                         "kind": "oracle", "sample": sample},
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


def target_summary(configs, target=0.75):
    """The cells at T >= 8192 whose forward or backward (either mode, either clock) falls
    below `target` of the peak; the configurations' stated goal is none."""
    if not configs:
        return None
    below, n = [], 0
    for name, ops in configs.items():
        T = int(name.split("_T")[1].split("_")[0])
        if T < 8192:
            continue
        for op, r in ops.items():
            n += 1
            worst = min(r["frac"], r["stream_frac"])
            if worst < target:
                below.append({"cell": name, "op": op, "frac": r["frac"],
                              "stream_frac": r["stream_frac"]})
    return {"target_frac": target, "ops_checked": n, "below": below}


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

    # ---- device-timed region 2: the same steps with events around each op (at least
    # about a second of them, so the clock sampler sees the GPU under load) ----
    k2 = max(min(args.steps, 500), int(args.min_op_seconds / max(total_ms / args.steps * 1e-3,
                                                                  1e-6)))
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(k2)]
    torch.cuda.synchronize()
    for i in range(k2):
        ev[i][0].record(stream)
        fwd_call(xp, wp, yp, rp)
        ev[i][1].record(stream)
        bwd_call(xp, dyp, wp, dxp, rp, dwp)
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    fwd_ms = [e[0].elapsed_time(e[1]) for e in ev]
    bwd_ms = [e[1].elapsed_time(e[2]) for e in ev]

    # ---- every configuration's cells at T >= 8192 (and the tiny one), each op timed
    # isolated and back to back (time_cell); rank 0 only, still under the clock sampler ----
    configs = None
    if rank == 0 and not args.skip_configs:
        env = _cell_env(torch, N, dev, stream)
        configs = {}
        for cell in CONFIG_CELLS:
            configs[cell_name(cell)] = {r.pop("op"): r for r in time_cell(env, cell,
                                                                          args.config_reps)}
        del env
        torch.cuda.empty_cache()
    wall2 = time.time()
    clocks = sampler.summary(wall0, wall2) if sampler else None
    if sampler:
        sampler.stop()
    max_ms = reduce_max(total_ms, dist)

    # ---- context: the device-to-device copy bandwidth of this GPU (cudaMemcpyAsync) ----
    copy_gbs = d2d_copy_gbps(torch, dev, stream)

    step_bytes = fwd_bytes(R, H, wbytes) + bwd_bytes(R, H, wbytes)
    value = step_bytes * args.steps * ws / (max_ms * 1e-3) / 1e9
    fwd_us = statistics.mean(fwd_ms) * 1e3
    bwd_us = statistics.mean(bwd_ms) * 1e3

    # ---- end to end through the C ABI with pinned host buffers: every step uploads its
    # inputs (x, dy, w) and downloads its results (y, rstd, dx, dw).  Three streams and two
    # device buffer sets overlap step i's upload with step i-1's compute and download (the
    # two copy directions run at once); events keep a set's inputs until its compute has
    # read them and its outputs until they are downloaded ----
    e2e_steps = max(3, min(args.steps, args.e2e_steps))
    hx = torch.from_numpy(case.x.view(np.int16)).view(torch.bfloat16).pin_memory()
    hdy = torch.from_numpy(case.dy.view(np.int16)).view(torch.bfloat16).pin_memory()
    hw = torch.from_numpy(case.w.view(np.int16)).view(torch.bfloat16).pin_memory()
    hy = torch.empty(R * H, dtype=torch.bfloat16).pin_memory()
    hdx = torch.empty(R * H, dtype=torch.bfloat16).pin_memory()
    hr = torch.empty(R, dtype=torch.float32).pin_memory()
    hdw = torch.empty(H, dtype=torch.float32).pin_memory()
    sets = [dict(x=x, dy=dy, w=w, y=y, dx=dx, rstd=rstd, dw=dw)]
    sets.append({k: torch.empty_like(v) for k, v in sets[0].items()})
    for b in sets:
        b.update(in_ready=torch.cuda.Event(), comp_done=torch.cuda.Event(),
                 out_done=torch.cuda.Event())
    s_in = torch.cuda.Stream(dev)
    s_out = torch.cuda.Stream(dev)

    def e2e_step(i):
        b = sets[i % 2]
        s_in.wait_event(b["comp_done"])      # step i-2's compute has read this set
        with torch.cuda.stream(s_in):
            b["x"].copy_(hx, non_blocking=True)
            b["dy"].copy_(hdy, non_blocking=True)
            b["w"].copy_(hw, non_blocking=True)
        b["in_ready"].record(s_in)
        stream.wait_event(b["in_ready"])
        stream.wait_event(b["out_done"])     # step i-2's results are downloaded
        bxp, bdyp, bwp = b["x"].data_ptr(), b["dy"].data_ptr(), b["w"].data_ptr()
        brp = b["rstd"].data_ptr()
        fwd_call(bxp, bwp, b["y"].data_ptr(), brp)
        bwd_call(bxp, bdyp, bwp, b["dx"].data_ptr(), brp, b["dw"].data_ptr())
        b["comp_done"].record(stream)
        s_out.wait_event(b["comp_done"])
        with torch.cuda.stream(s_out):
            hy.copy_(b["y"], non_blocking=True)
            hr.copy_(b["rstd"], non_blocking=True)
            hdx.copy_(b["dx"], non_blocking=True)
            hdw.copy_(b["dw"], non_blocking=True)
        b["out_done"].record(s_out)

    e2e_step(0)
    e2e_step(1)
    torch.cuda.synchronize()
    barrier(dist)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for i in range(e2e_steps):
        e2e_step(i)
    e1.record(s_out)  # after the last download, which follows every earlier step's work
    torch.cuda.synchronize()
    e2e_ms = reduce_max(e0.elapsed_time(e1), dist)
    h2d = 2 * R * H * 2 + H * wbytes
    d2h = 2 * R * H * 2 + 4 * R + 4 * H
    e2e_value = step_bytes * e2e_steps * ws / (e2e_ms * 1e-3) / 1e9
    del sets[1]

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
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "overlap": "upload, compute and download on three streams, two buffer sets"},
        "gpu_launches": 3 * args.steps,  # fwd + bwd row pass + dw finish per step
        "clocks": clocks,
        "configs": configs,
        "configs_target": target_summary(configs),
        "source_hash": kernel_source_hash(),
    }
    print(json.dumps(line))
    return 0


# ---- per-cell timing: the default run's per-configuration table and the sweep ----------

# The configurations' cells with T >= 8192 (where the 75 %-of-peak target applies) and the
# tiny one: name, T, H, heads, buffer heads, FP32 weight, residual form, outlier rows.
CONFIG_CELLS = (
    [("tiny", 64, 256, 1, None, True, False, 0.0)]
    + [("plain", T, 4096, 1, None, False, False, 0.0) for T in (16384, 65536)]
    + [("stress", T, H, 1, None, True, False, 0.01)
       for H in (1536, 2048, 5120) for T in (32768, 65536, 98304, 131072)]
    + [("residual", T, 6144, 1, None, False, True, 0.0) for T in (30720, 65536)]
    + [("heads24of32", 65536, 256, 24, 32, True, False, 0.0),
       ("heads4", 65536, 256, 4, None, True, False, 0.0)]
)

# --sweep: the same families at more row counts (label, T, H, nh, buf_heads, w_fp32,
# residual, outlier rows)
SWEEP = [
    ("plain", 16384, 4096, 1, None, False, False, 0.0),
    ("plain", 65536, 4096, 1, None, False, False, 0.0),
    ("stress", 32768, 1536, 1, None, True, False, 0.01),
    ("stress", 65536, 1536, 1, None, True, False, 0.01),
    ("stress", 131072, 1536, 1, None, True, False, 0.01),
    ("stress", 32768, 2048, 1, None, True, False, 0.01),
    ("stress", 131072, 2048, 1, None, True, False, 0.01),
    ("stress", 32768, 5120, 1, None, True, False, 0.01),
    ("stress", 131072, 5120, 1, None, True, False, 0.01),
    ("residual", 30720, 6144, 1, None, False, True, 0.0),
    ("residual", 65536, 6144, 1, None, False, True, 0.0),
    ("heads24of32", 4096, 256, 24, 32, True, False, 0.0),
    ("heads24of32", 16384, 256, 24, 32, True, False, 0.0),
    ("heads24of32", 65536, 256, 24, 32, True, False, 0.0),
    ("heads4", 65536, 256, 4, None, True, False, 0.0),
]

L2_BYTES = 129 << 20


def device_case(torch, dev, T, H, nh=1, buf_heads=None, w_fp32=False, residual=False,
                outlier_frac=0.0, seed=0):
    """Timing inputs drawn on the device by torch's seeded generator, with the
    configurations' distributions (x, residual, dy, dh ~ N(0,1) rounded to BF16; w =
    1 + 0.1*N(0,1); outlier rows x16).  Parity is the tests' job: these only need the
    shapes and value ranges, and drawing them on the device keeps the run short."""
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    bh = buf_heads or nh

    def draw(n):
        return torch.randn(n, generator=g, device=dev, dtype=torch.float32)

    x = draw(T * bh * H)
    if outlier_frac > 0.0 and T > 0:
        n = max(1, int(round(outlier_frac * T * nh)))
        rows = torch.randperm(T * nh, generator=g, device=dev)[:n]
        xv = x.view(T, bh, H)
        xv[rows // nh, rows % nh] *= 16.0
    d = {"x": x.to(torch.bfloat16)}
    del x
    if residual:
        d["res"] = draw(T * bh * H).to(torch.bfloat16)
    d["dy"] = draw(T * nh * H).to(torch.bfloat16)
    if residual:
        d["dh"] = draw(T * nh * H).to(torch.bfloat16)
    w = 1.0 + 0.1 * draw(H)
    d["w"] = w if w_fp32 else w.to(torch.bfloat16)
    return d


def _cell_timers(torch, stream, flush):
    """Three clocks, CUDA events on the launch stream:

    graph     (the "frac" of a cell) the pages' method: the op captured once into a CUDA
              graph, `reps` replays, each after an L2 flush outside the events; trimmed
              mean.  The flush READS a 512 MiB buffer, so L2 is cold but clean (a
              write-based flush would leave dirty lines whose write-back lands inside the
              next timed kernel).  Includes the op's ramp-up and tail and the gap before
              its first CTA starts.
    eager     the same, launching the op directly instead of replaying a graph.
    stream    `reps` launches back to back inside one event pair, rotating over copies of
              the inputs and outputs so that every launch finds its inputs out of L2 (the
              sets in between exceed twice the L2); time / launches.  This is the op as a
              training step runs it, queued behind other work."""

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

    def timed_graph(fn, reps, cur):
        """isolated, the pages' way: the op captured once into a CUDA graph (fn launches on
        the stream handle cur["sh"]), each replay after the same L2 flush"""
        cs = torch.cuda.Stream()
        cs.wait_stream(stream)
        old = cur["sh"]
        cur["sh"] = cs.cuda_stream
        try:
            with torch.cuda.stream(cs):
                fn(0)   # warm-up on the capture stream
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cs):
                fn(0)
        finally:
            cur["sh"] = old
        torch.cuda.synchronize()
        for _ in range(3):
            g.replay()
        out = []
        for _ in range(reps):
            flush.sum()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            g.replay()
            b.record(stream)
            torch.cuda.synchronize()
            out.append(a.elapsed_time(b) * 1e3)
        del g
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

    return timed, timed_stream, timed_graph


def time_cell(env, cell, reps, ckpt=False, once=False, only=None):
    """Times every op of one cell (forward; backward in both modes, with and without dh in
    the residual form; with ckpt the checkpointed step 2xfwd+bwd = forward, forward
    recompute, deterministic backward) with both clocks of _cell_timers.  Returns one
    record per op.  With once, runs each op once, untimed (for a profiler)."""
    torch, N, lib, dev, stream, flush, peak, peak_kind = env
    _, T, H, nh, bh, w32, res, outl = cell
    cur = {"sh": stream.cuda_stream}   # the stream the ops launch on (graph capture swaps it)
    R = T * nh
    wbytes = 4 if w32 else 2
    wd = N.RMSN_W_FP32 if w32 else N.RMSN_W_BF16
    base = device_case(torch, dev, T, H, nh, bh, w32, res, outl)
    w = base.pop("w")
    s_tok_in, s_head_in = (bh or nh) * H, H
    set_bytes = sum(t.numel() * t.element_size() for t in base.values()) + 3 * R * H * 2
    nsets = 1 if once or set_bytes >= 2 * L2_BYTES else -(-2 * L2_BYTES // set_bytes) + 1
    sets = []
    for i in range(nsets):
        q = {k: (v if i == 0 else v.clone()) for k, v in base.items()}
        q["y"] = torch.empty(R * H, dtype=torch.bfloat16, device=dev)
        q["h"] = torch.empty_like(q["y"]) if res else None
        q["dx"] = torch.empty_like(q["y"])
        q["rstd"] = torch.empty(R, dtype=torch.float32, device=dev)
        q["dw"] = torch.empty(H, dtype=torch.float32, device=dev)
        sets.append(q)

    def fwd(i):
        q = sets[i]
        st = lib.rmsnorm_train_fwd(q["x"].data_ptr(), q["res"].data_ptr() if res else None,
                                   w.data_ptr(), wd, q["y"].data_ptr(),
                                   q["h"].data_ptr() if res else None, q["rstd"].data_ptr(),
                                   T, nh, H, s_tok_in, s_head_in, 1e-6, cur["sh"])
        assert st == 0, st

    for i in range(nsets):
        fwd(i)
    s_tok, s_head = (nh * H, H) if res else (s_tok_in, s_head_in)
    fwd_b = (8 if res else 4) * R * H + 4 * R + wbytes * H
    ops = [("fwd", fwd, fwd_b)]
    for det in (1, 0):
        nws = N.rmsnorm_train_bwd_workspace_bytes(T, nh, H, det)
        ws = torch.empty(max(nws, 16), dtype=torch.uint8, device=dev)
        for use_dh in ((False, True) if res else (False,)):
            def bwd(i, det=det, use_dh=use_dh, ws=ws, nws=nws):
                q = sets[i]
                xs = q["h"] if res else q["x"]
                st = lib.rmsnorm_train_bwd(xs.data_ptr(), q["dy"].data_ptr(),
                                           q["dh"].data_ptr() if use_dh else None,
                                           q["rstd"].data_ptr(), w.data_ptr(), wd,
                                           q["dx"].data_ptr(), q["dw"].data_ptr(),
                                           ws.data_ptr(), nws, T, nh, H, s_tok, s_head,
                                           det, cur["sh"])
                assert st == 0, st

            name = ("bwd_det" if det else "bwd_nondet") + ("+dh" if use_dh else "")
            bwd_b = (8 if use_dh else 6) * R * H + 4 * R + wbytes * H + 4 * H
            ops.append((name, bwd, bwd_b))
            if ckpt and det and not use_dh:
                def step(i, bwd=bwd):
                    fwd(i)
                    fwd(i)
                    bwd(i)

                ops.append(("2xfwd+bwd_det", step, 2 * fwd_b + bwd_b))

                # the backward that recomputes rstd (writing it to the set's rstd), and the
                # checkpointed step with it in place of the second forward
                def bwd_rc(i, ws=ws, nws=nws):
                    q = sets[i]
                    xs = q["h"] if res else q["x"]
                    st = lib.rmsnorm_train_bwd_recompute(xs.data_ptr(), q["dy"].data_ptr(), None,
                                                         w.data_ptr(), wd, q["dx"].data_ptr(),
                                                         q["dw"].data_ptr(), q["rstd"].data_ptr(),
                                                         ws.data_ptr(), nws, T, nh, H, s_tok,
                                                         s_head, 1e-6, 1, cur["sh"])
                    assert st == 0, st

                def step_rc(i, bwd_rc=bwd_rc):
                    fwd(i)
                    bwd_rc(i)

                ops.append(("bwd_det_rc", bwd_rc, bwd_b))
                ops.append(("fwd+bwd_det_rc", step_rc, fwd_b + bwd_b))
    timed, timed_stream, timed_graph = _cell_timers(torch, stream, flush)
    out = []
    if only:
        ops = [o for o in ops if o[0] in only]
    for name, fn, nbytes in ops:
        if once:
            fn(0)
            torch.cuda.synchronize()
            out.append({"op": name, "ran_once": True})
            continue
        us = timed_graph(fn, reps, cur)
        us_e = timed(fn, reps)
        us_s = timed_stream(fn, nsets, reps)
        gbs = nbytes / (us * 1e-6) / 1e9
        gbs_s = nbytes / (us_s * 1e-6) / 1e9
        out.append({"op": name, "us": round(us, 2), "GBps": round(gbs, 1),
                    "frac": round(gbs / peak, 4), "stream_us": round(us_s, 2),
                    "stream_GBps": round(gbs_s, 1), "stream_frac": round(gbs_s / peak, 4),
                    "eager_us": round(us_e, 2),
                    "eager_frac": round(nbytes / (us_e * 1e-6) / 1e9 / peak, 4),
                    "input_sets": nsets, "bytes": nbytes})
    del sets, base, w
    torch.cuda.empty_cache()
    return out


def cell_name(cell):
    label, T, H = cell[0], cell[1], cell[2]
    return f"{label}_T{T}_H{H}"


def _cell_env(torch, N, dev, stream):
    flush = torch.ones(128 << 20, dtype=torch.int32, device=dev)
    peak, peak_kind = measured_peak()
    return (torch, N, N.lib(), dev, stream, flush, peak, peak_kind)


def run_sweep(args):
    """Times each op of each workload of SWEEP (one JSON line per op) with time_cell's two
    clocks; --sweep-once runs each op once, untimed."""
    import torch
    from rmsnorm_fwd_02_gb300 import _native as N

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    env = _cell_env(torch, N, dev, torch.cuda.current_stream(dev))
    for cell in SWEEP:
        label, T, H, nh = cell[:4]
        if args.sweep_filter and args.sweep_filter != f"{label}_{T}_{H}":
            continue
        only = set(args.sweep_ops.split(",")) if args.sweep_ops else None
        for rec in time_cell(env, cell, args.sweep_reps, ckpt=True, once=args.sweep_once,
                             only=only):
            rec.update({"sweep": label, "T": T, "H": H, "nh": nh,
                        "w": "fp32" if cell[5] else "bf16", "peak": env[6],
                        "peak_kind": env[7]})
            print(json.dumps(rec), flush=True)
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
    l2_bytes = L2_BYTES
    timed, timed_stream, _ = _cell_timers(torch, stream, flush)

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
    ap.add_argument("--skip-configs", action="store_true",
                    help="leave out the per-configuration table")
    ap.add_argument("--config-reps", type=int, default=20)
    ap.add_argument("--min-op-seconds", type=float, default=1.0,
                    help="least duration of the per-op timing loop (clock samples)")
    ap.add_argument("--sweep", action="store_true",
                    help="time each op on every workload family (one line each) instead")
    ap.add_argument("--sweep-reps", type=int, default=30)
    ap.add_argument("--sweep-filter", default="",
                    help="only the sweep entry LABEL_T_H (e.g. stress_131072_1536)")
    ap.add_argument("--sweep-layernorm", action="store_true",
                    help="with --sweep: the LayerNorm ops on the normalization tables' shapes "
                         "(filter entries as layernorm_M_H)")
    ap.add_argument("--sweep-ops", default="",
                    help="with --sweep: only these ops (comma-separated: fwd, bwd_det, "
                         "bwd_nondet, bwd_det+dh, bwd_nondet+dh, 2xfwd+bwd_det, bwd_det_rc, "
                         "fwd+bwd_det_rc)")
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
