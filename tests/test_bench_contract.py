"""The benchmark's reference arm on the CPU: `bench.py --impl reference` prints
exactly one JSON line with the keys and types of the benchmark line (the oracle
timed on the host cores, on a bounded sample of the workload), and nothing else
on standard output."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*extra):
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
           "--warmup", "1", "--ref-seconds", "4", *extra]
    env = dict(os.environ)
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        env.pop(k, None)
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, r.stdout
    return json.loads(lines[0])


def test_reference_arm_line():
    line = _run("--workload", "C5", "--heads", "1", "--seq", "4096")
    assert line["impl"] == "reference"
    assert line["metric"] and line["unit"] == "TFLOP/s"
    assert line["higher_is_better"] is True and line["scaling"] == "weak"
    assert line["n_gpus"] == 1 and line["steps"] == 1 and line["warmup"] == 1
    assert line["dtype"] == "f64" and line["data"] == "synthetic" and line["vs_baseline"] is None
    assert isinstance(line["value"], float) and line["value"] > 0
    assert line["ms_per_step"] >= 2000.0 * 0.9          # one bounded sample of about 2 s
    cfg = line["config"]
    assert "C5" in cfg["workload"] and cfg["S"] == 4096 and cfg["H"] == 1 and cfg["N"] == 16
    assert cfg["layout"] == "zigzag" and cfg["causal"] and cfg["backward"]
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == line["value"] and cb["unit"] == line["unit"]
    assert isinstance(cb["cores"], int) and cb["cores"] >= 1 and "query rows" in cb["sample"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_forward_only_workload():
    line = _run("--workload", "C3", "--heads", "1", "--seq", "2048")
    assert line["config"]["backward"] is False and line["config"]["N"] == 8
    assert "dQ rows" not in line["cpu_baseline"]["sample"]


@pytest.mark.gpu
def test_gpu_arm_line_small_case():
    """The GPU arm on a smaller case of the C5 step (2 heads, 16384 tokens): one
    line carrying the roofline, the end-to-end figure, the launch count, the clocks
    and the CPU baseline; no traffic figure, since the committed ncu record is for
    the full-size workload only."""
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "3", "--warmup", "3",
           "--heads", "2", "--seq", "16384", "--no-side-configs", "--cpu-seconds", "1"]
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["n_gpus"] == 1 and line["steps"] == 3 and line["warmup"] == 3
    assert line["value"] > 0 and line["ms_per_step"] > 0 and line["dtype"] == "bf16"
    assert line["config"]["S"] == 16384 and line["config"]["H"] == 2
    roof = line["roofline"]
    assert roof["bound"] in ("tensor", "hbm") and roof["unit"] in ("TFLOP/s", "GB/s")
    assert roof["achieved"] > 0 and roof["peak"] > 0
    assert abs(roof["frac"] - roof["achieved"] / roof["peak"]) < 1e-3
    assert roof["traffic"] is None
    e2e = line["e2e"]
    assert e2e["value"] > 0 and e2e["unit"] == "TFLOP/s"
    # Q, K, V, dO in; O, dQ, dK, dV out (bf16) plus the fp32 LSE
    nbytes = 2 * 16384 * 128 * 2
    assert e2e["h2d_bytes_per_step"] == 4 * nbytes
    assert e2e["d2h_bytes_per_step"] == 4 * nbytes + 2 * 16384 * 4
    assert line["gpu_launches"] >= 3 * 4            # permute, forward, backward, unpermute per step
    assert set(line["phase_ms"]) == {"permute", "forward", "backward", "unpermute"}
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] > 0
    if line["clocks"] is not None:                  # nvidia-smi samples during the timed region
        assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(line["clocks"])


def test_committed_traffic_is_keyed_by_workload_and_source(tmp_path, monkeypatch):
    """The DRAM traffic figure is reported only for the workload it was captured
    on, and only while the kernel sources hash as they did at capture time."""
    sys.path.insert(0, ROOT)
    import bench
    (tmp_path / "profiles").mkdir()
    src = tmp_path / "k.cu"
    src.write_text("kernel source\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h = bench.source_hash(["k.cu"])
    (tmp_path / "profiles" / "traffic.txt").write_text(
        "# kernel workload bytes_per_launch source_hash sources\n"
        f"bwd_tc_kernel C5 123456 {h} k.cu\n")
    assert bench.committed_traffic("bwd_tc_kernel", "C5") == {"dram_bytes_per_launch": 123456}
    assert bench.committed_traffic("bwd_tc_kernel", "C3") is None
    assert bench.committed_traffic("fwd_tc_kernel", "C5") is None
    src.write_text("kernel source, changed\n")
    assert bench.committed_traffic("bwd_tc_kernel", "C5") is None



def test_flop_counts_are_the_published_convention():
    """Useful attention flops (FlashAttention convention, causal-adjusted): 4·S²·D
    per head forward, half of it under causal, 2.5× that for the backward — the
    figures each workload's TFLOP/s is computed from."""
    sys.path.insert(0, ROOT)
    import bench
    from context_ra_forward_gb300 import inputs
    expect = {"C1": (2.684e8, 0.0), "C2": (1.759e13, 0.0), "C3": (3.518e13, 0.0), "C4": (3.518e13, 0.0),
              "C5": (2.815e14, 7.037e14)}
    for name, (fwd, bwd) in expect.items():
        f, b = bench.flops_of(inputs.WORKLOADS[name])
        assert abs(f - fwd) <= 1e-3 * fwd, name
        assert abs(b - bwd) <= 1e-3 * max(bwd, 1.0), name
    # the strided variants do the same work as their zig-zag twins
    assert bench.flops_of(inputs.WORKLOADS["C5S"]) == bench.flops_of(inputs.WORKLOADS["C5"])


def test_peak_fractions_name_their_denominators(tmp_path, monkeypatch):
    """Every fraction of a bf16 figure says which peak it divides by: the pool's
    measured sustained and burst cuBLAS rates (or the labelled fallback when the
    measurement is absent) and the datasheet's dense 2.25 PFLOP/s."""
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (tmp_path / "MEASURED_PEAKS.json").write_text('{"bf16_tflops": 2000.0, "bf16_tflops_sustained": 1600.0}')
    f = bench.peak_fractions(1200.0)
    assert f == {"of_measured_sustained": 0.75, "of_measured_burst": 0.6, "of_nominal_dense": round(1200 / 2250, 4)}
    (tmp_path / "MEASURED_PEAKS.json").unlink()
    f = bench.peak_fractions(1190.0)
    assert f["of_fallback_sustained"] == 0.7 and f["of_fallback_burst"] == round(1190 / 1900, 4)
