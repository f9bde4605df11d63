"""The benchmark's JSON line on a GPU: one short run of bench.py (the timed
sandwich step, its end-to-end leg, decode and a short CPU-baseline sample),
checked key by key against the line's contract."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_line_contract():
    cmd = [sys.executable, "bench.py", "--steps", "40", "--warmup", "3", "--no-secondary",
           "--decode-calls", "128", "--e2e-steps", "2", "--cpu-seconds", "1"]
    res = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert res.returncode == 0, res.stderr[-2000:]
    line = json.loads(res.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "e2e", "gpu_launches", "clocks", "cpu_baseline", "decode"):
        assert key in line, key
    assert line["n_gpus"] == 1 and line["steps"] == 40 and line["warmup"] == 3
    assert line["higher_is_better"] is True and line["scaling"] == "weak"
    assert line["value"] > 0 and line["unit"] == "GB/s" and line["dtype"] == "f32"
    assert line["config"]["workload"] == "sandwich_f32_rows4096_n6656"
    assert line["gpu_launches"] == 40                # one kernel per timed step
    rf = line["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s" and rf["peak"] > 0
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-9
    assert rf["algorithmic_bytes_per_launch"] == 436260864
    assert rf["frac"] < 1.2                          # a copy-bandwidth peak cannot be far exceeded
    e2e = line["e2e"]
    assert e2e["unit"] == "GB/s" and 0 < e2e["value"] < line["value"]
    assert e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] == 2 * 4096 * 6656 * 4
    assert e2e["copies_only"] > 0   # the same steps without the call
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] > 0
    assert line["clocks"]["sm_max_mhz"] > 0
    assert line["decode"]["us_per_call_graph"] > 0
    # the compact per-workload summary closes the line (the end of the line is
    # what survives when only a tail of the output is kept)
    assert list(line)[-1] == "workloads"
    wk = line["workloads"]
    assert wk["3_sandwich_f32_rows4096_n6656"]["GB_per_s"] == round(line["value"], 1)
    assert wk["2_decode_sandwich_f32_rows1_n6656_us_per_call"]["graph"] > 0
    assert len(json.dumps(wk)) < 2000
