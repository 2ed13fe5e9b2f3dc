"""bench.py's host logic without a GPU: the byte model, the peak lookup, the traffic gate
on the kernel-source hash, the clock-sample summary, the reference arm's JSON line, and
the max-over-ranks timing reduction across two gloo ranks (the replicas' only
collective, host-side)."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_byte_model():
    R, H = 65536, 4096
    assert bench.fwd_bytes(R, H, 2) == 4 * R * H + 4 * R + 2 * H
    assert bench.bwd_bytes(R, H, 4) == 6 * R * H + 4 * R + 4 * H + 4 * H


def test_layernorm_byte_model():
    R, H = 8192, 4096
    # forward: x read, y written, w and b read, mean and rstd written
    assert bench.ln_fwd_bytes(R, H, 2) == 2 * R * H + 2 * R * H + 2 * 2 * H + 8 * R
    # backward: x, dy read, dx written, mean and rstd read, w read, dw and db written
    assert bench.ln_bwd_bytes(R, H, 4) == 6 * R * H + 8 * R + 4 * H + 8 * H
    assert all(H <= 16384 and H % 16 == 0 for _, H in bench.LN_SWEEP)


def test_peak_fallback_when_no_measured_file(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_peak() == (bench.FALLBACK_HBM_GBS, "fallback")
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 7000.0}))
    assert bench.measured_peak() == (7000.0, "measured")


def test_traffic_needs_matching_source_hash(tmp_path, monkeypatch):
    f = tmp_path / "traffic.json"
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    assert bench.traffic_for("k") is None
    f.write_text(json.dumps({"k": {"source_hash": "stale", "dram_bytes_per_op": 1.0}}))
    assert bench.traffic_for("k") is None
    f.write_text(json.dumps({"k": {"source_hash": bench.kernel_source_hash(),
                                   "dram_bytes_per_op": 123.0}}))
    assert bench.traffic_for("k") == 123.0


def test_clock_summary_filters_window_and_reasons():
    s = bench.ClockSampler.__new__(bench.ClockSampler)
    s.lines = [
        (10.0, "2026/01/01 00:00:00.000, 0, 1000, 2070, 500, 0x0, Not Active, Not Active, Not Active, Not Active"),
        (20.0, "2026/01/01 00:00:00.000, 0, 2070, 2070, 900, 0x4, Not Active, Not Active, Not Active, Active"),
        (20.2, "2026/01/01 00:00:00.000, 0, 2040, 2070, 950, 0x0, Not Active, Not Active, Not Active, Not Active"),
    ]
    out = s.summary(19.0, 21.0)
    assert out["samples"] == 2 and out["sm_mhz"] == 2055.0 and out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == ["sw_power_cap"]


def test_reference_arm_line(capsys):
    bench.main(["--impl", "reference", "--T", "64", "--H", "256", "--steps", "3",
                "--warmup", "3"])
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["cpu_baseline"]["cores"] == (os.cpu_count() or 1)
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
    assert line["higher_is_better"] is True


_WORKER = r"""
import os, sys
sys.path.insert(0, {root!r})
import bench
ws, rank, _ = bench.dist_env()
dist = bench.dist_init(ws)
bench.barrier(dist)
t = bench.reduce_max(10.0 + rank, dist)
print("RESULT", rank, t, flush=True)
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_max_over_two_gloo_ranks(tmp_path):
    script = tmp_path / "w.py"
    script.write_text(_WORKER.format(root=ROOT))
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, WORLD_SIZE="2", RANK=str(rank), LOCAL_RANK=str(rank),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, str(script)], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.STDOUT,
                                      text=True))
    outs = []
    for p in procs:
        try:
            out, _ = p.communicate(timeout=120)
        except subprocess.TimeoutExpired:
            p.kill()
            pytest.fail("gloo rank did not finish")
        outs.append(out)
        assert p.returncode == 0, out
    vals = sorted(float(l.split()[2]) for o in outs for l in o.splitlines()
                  if l.startswith("RESULT"))
    assert vals == [11.0, 11.0]


def test_target_summary_lists_cells_below_target():
    cfg = {
        "tiny_T64_H256": {"fwd": {"frac": 0.01, "stream_frac": 0.02}},
        "plain_T16384_H4096": {"fwd": {"frac": 0.80, "stream_frac": 0.85},
                               "bwd_det": {"frac": 0.74, "stream_frac": 0.80}},
        "residual_T65536_H6144": {"bwd_det+dh": {"frac": 0.9, "stream_frac": 0.7}},
    }
    out = bench.target_summary(cfg)
    assert out["ops_checked"] == 3          # the T=64 cell is outside the target's range
    assert [(b["cell"], b["op"]) for b in out["below"]] == [
        ("plain_T16384_H4096", "bwd_det"), ("residual_T65536_H6144", "bwd_det+dh")]
    assert bench.target_summary(None) is None


def test_config_cells_cover_every_configuration_at_t_8192_and_above():
    names = {bench.cell_name(c) for c in bench.CONFIG_CELLS}
    for T in (16384, 65536):
        assert f"plain_T{T}_H4096" in names
    for H in (1536, 2048, 5120):
        for T in (32768, 65536, 98304, 131072):
            assert f"stress_T{T}_H{H}" in names
    for T in (30720, 65536):
        assert f"residual_T{T}_H6144" in names
    assert {"heads24of32_T65536_H256", "heads4_T65536_H256", "tiny_T64_H256"} <= names


def test_cpu_baseline_reports_single_and_all_cores():
    from rmsnorm_fwd_02_gb300 import synth
    c = synth.make_case(0, 40, 64)
    out = bench.cpu_baseline(c, 2, budget_s=0.2, rows_per_thread=4)
    assert out["kind"] == "oracle" and out["cores"] == (os.cpu_count() or 1)
    assert out["value"] > 0 and out["single_thread_value"] > 0
    assert out["host_cpu_count"] == os.cpu_count()


def test_oracle_runner_blocks_sum_to_whole_sample_dw():
    # the threaded harness only splits rows: its dw equals the oracle's over the same rows
    import numpy as np
    import oracle
    from rmsnorm_fwd_02_gb300 import synth
    c = synth.make_case(3, 50, 32)
    r = bench.OracleRunner(c, rows_per_thread=5, threads=4)
    dw = r.step()
    r.close()
    rows = np.concatenate(r.blocks)
    sub_x = c.x.reshape(-1, 32)[rows].reshape(-1)
    sub_dy = c.dy.reshape(-1, 32)[rows].reshape(-1)
    _, r64, _ = oracle.fwd(sub_x, c.w, c.eps, rows.size, 1, 32, 32, 32)
    want = oracle.bwd_dw(sub_x, sub_dy, r64.astype(np.float32).astype(np.float64),
                         rows.size, 1, 32, 32, 32)
    np.testing.assert_allclose(dw, want, rtol=1e-12, atol=1e-12)
