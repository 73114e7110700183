"""The JSON line `bench.py` prints: every key the benchmark contract names,
with sane values.  The reference arm (the CPU oracle) runs without a GPU;
the CUDA arm is checked on the small fp32 workload."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench(*args, timeout=900):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                       capture_output=True, text=True, timeout=timeout)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert lines, r.stdout[-2000:]
    return [json.loads(l) for l in lines]


def _common(d, steps, warmup):
    assert d["metric"] and d["unit"] == "tokens/s" and d["value"] > 0
    assert d["n_gpus"] == 1 and d["steps"] == steps and d["warmup"] == warmup
    assert d["ms_per_step"] > 0 and d["higher_is_better"] is True
    assert d["scaling"] == "weak" and d["data"] == "synthetic" and d["dtype"]
    assert isinstance(d["config"], dict) and d["config"]["workload"]
    e2e = d["e2e"]
    assert e2e["unit"] == d["unit"] and e2e["value"] > 0


def test_reference_arm_line():
    """`--impl reference` times the oracle on the host cores, on the headline
    workload, and prints the contract's line with its cpu_baseline and a
    copy-free e2e."""
    (d,) = _bench("--impl", "reference", "--steps", "1", "--warmup", "3")
    _common(d, 1, 3)
    assert d["impl"] == "reference" and d["config"]["workload"] == "skew"
    assert d["vs_baseline"] is None
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1
    assert cb["unit"] == d["unit"] and cb["sample"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


@pytest.mark.gpu
def test_cuda_arm_line():
    """The CUDA arm on the small workload: roofline with the measured peak,
    DRAM traffic from the committed capture, e2e with its copied bytes, the
    launch count, clocks sampled during the timed region, medians."""
    (d,) = _bench("--workload", "tiny", "--steps", "5", "--warmup", "3", "--no-cpu-baseline")
    _common(d, 5, 3)
    assert "impl" not in d and d["config"]["workload"] == "tiny"
    rf = d["roofline"]
    assert rf["bound"] in ("hbm", "tensor") and rf["unit"] in ("GB/s", "TFLOP/s")
    assert rf["achieved"] > 0 and rf["peak"] > 0 and rf["kernel_ms"] > 0
    assert rf["kernel_ms"] <= d["segments_ms"]["fc1_swiglu"] * 1.05
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-9
    assert rf["traffic"] is None or rf["traffic"] > 0
    e2e = d["e2e"]
    assert e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert d["gpu_launches"] > 0
    clk = d["clocks"]
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(clk)
    assert d["step_ms_median"] > 0 and set(d["segments_ms_median"]) == set(d["segments_ms"])
    assert d["counts"]["achieved_gbs"] > 0


def test_traffic_lookup_follows_the_kernel_source(tmp_path, monkeypatch):
    """roofline.traffic comes from a committed ncu figure only while the
    kernel's source (comments and blank space aside) is the one it was
    taken on; any other source gives null."""
    sys.path.insert(0, ROOT)
    import bench
    src = tmp_path / "k.cu"
    src.write_text("// a comment\n__global__ void k() { int a = 1; }\n")
    h = bench._src_hash(str(src))
    (tmp_path / "traffic.json").write_text(json.dumps(
        {"gmm_fc1:uniform": {"src_sha256_16": h, "dram_bytes_per_launch": 123}}))
    monkeypatch.setattr(bench, "PROFILE_DIR", str(tmp_path))
    assert bench._ncu_traffic("gmm_fc1", "uniform", str(src)) == 123
    assert bench._ncu_traffic("gmm_fc1", "skew", str(src)) is None
    src.write_text("/* another\n comment */\n\n    __global__ void k() { int a = 1; }  // end\n")
    assert bench._ncu_traffic("gmm_fc1", "uniform", str(src)) == 123   # comments, blank space
    src.write_text("__global__ void k() { int a = 2; }\n")
    assert bench._ncu_traffic("gmm_fc1", "uniform", str(src)) is None  # the code changed
