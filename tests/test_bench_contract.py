"""bench.py's JSON line: the reference arm (the fp64 oracle on the host cores)
on the CPU, within its time budget, and the timed arm on a GPU."""
import json
import os
import subprocess
import sys
import time

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_line():
    t0 = time.time()
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "500",
                          "--warmup", "3", "--ref-seconds", "3"], capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["steps"] == 500 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
    assert line["config"]["workload"] == "all"
    assert time.time() - t0 < 120          # the budget, not the step count, sets the time


@pytest.mark.gpu
def test_bench_line_on_the_gpu():
    """The timed arm on the decode workload: one JSON line with the contract's
    keys, a live roofline of the dominant kernel, an end-to-end number that
    moved bytes both ways, the oracle's CPU baseline and the sampled clocks."""
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--workload", "decode", "--steps", "10",
                          "--warmup", "3", "--cpu-seconds", "1", "--e2e-steps", "3"],
                         capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e", "clocks", "gpu_launches"):
        assert key in line, key
    assert line["n_gpus"] == 1 and line["steps"] == 10 and line["warmup"] == 3 and line["value"] > 0
    assert line["config"]["workload"] == "decode"
    roof = line["roofline"]
    assert roof["bound"] == "hbm" and roof["unit"] == "GB/s" and 0 < roof["frac"] < 1.5
    assert abs(roof["frac"] - roof["achieved"] / roof["peak"]) < 1e-9
    e2e = line["e2e"]
    assert e2e["value"] > 0 and e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert e2e["value"] < line["value"]                 # the copies cost time
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] > 0
    assert line["gpu_launches"] > 0
    assert line["clocks"]["sm_max_mhz"] > 0


def test_kernel_code_hash_ignores_comments(tmp_path):
    """The recorded ncu traffic stays valid across comment edits, and only those."""
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench_module", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    a, b, c = tmp_path / "a.cu", tmp_path / "b.cu", tmp_path / "c.cu"
    a.write_text("// one\nint f(int x) {  /* two */ return x + 1; }\n")
    b.write_text("// another comment,\n// over two lines\nint f(int x) {\n    return x + 1;   // the same code\n}\n")
    c.write_text("// one\nint f(int x) {  /* two */ return x + 2; }\n")
    assert bench.kernel_code_sha256(str(a)) == bench.kernel_code_sha256(str(b))
    assert bench.kernel_code_sha256(str(a)) != bench.kernel_code_sha256(str(c))
