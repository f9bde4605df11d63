"""The benchmark's compact per-workload summary (the `workloads` key that closes
the JSON line), on the CPU: built from a synthetic line with every section the
full run fills, it carries one rounded entry per workload and stays short
enough to survive when only the end of the output is kept."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from dual_epsilon_sandwich_gb300 import workloads as wl  # noqa: E402


def synthetic_line():
    small = {f"{rows}x{n}": {"rmsnorm": 1.23456 + rows * 1e-5, "then_add": 2.34567, "sets": 2}
             for n, rows in wl.sweep_shapes() if rows * n < 2 ** 26}
    large = {f"rows{rows}_n{n}": {"rmsnorm": {"GB_per_s": 6512.34}, "then_add": {"GB_per_s": 6939.9}}
             for n, rows in wl.sweep_shapes() if rows * n >= 2 ** 26}
    sec = {"rmsnorm_f32_rows4_n6656": {"us_per_call_graph": 1.9601},
           "rmsnorm_bf16_rows16384_n4096": {"GB_per_s": 6458.12},
           "then_add_bf16_rows16384_n4096": {"GB_per_s": 6908.34},
           "sweep_large_f32": large, "sweep_small_f32_us_per_call_graph": small}
    for name in ("add_rmsnorm_f32_rows4096_n6656", "then_add_scale_bf16_rows16384_n4096",
                 "rmsnorm_q8_1_bf16_rows16384_n4096", "qk_norm_bf16_rows163840_n128",
                 "seam_f16_from_f32_rows4096_n6656", "seam_bf16_from_bf16_rows16384_n4096",
                 "sandwich_f32_rows4096_n6655", "rmsnorm_f32_rows4096_n6655"):
        sec[name] = {"GB_per_s": 6000.06}
    return {"value": 6500.33, "n_gpus": 1, "ms_per_step": 0.067112,
            "decode": {"us_per_call_graph": 2.1071, "us_per_call_graph_l2_hot": 1.6871,
                       "us_per_call_stream": 3.5861},
            "secondary": sec}


def test_summary_carries_every_workload():
    line = synthetic_line()
    wk = bench.workload_summary(line, 6785.2)
    assert wk["1_rmsnorm_f32_rows4_n6656_us_per_call_graph"] == 1.96
    assert wk["2_decode_sandwich_f32_rows1_n6656_us_per_call"] == {
        "graph": 2.107, "graph_l2_hot": 1.687, "stream": 3.586}
    assert wk["3_sandwich_f32_rows4096_n6656"] == {"GB_per_s": 6500.3, "pct_of_copy": 95.8,
                                                   "us_per_call": 67.11}
    assert wk["4_rmsnorm_bf16_rows16384_n4096_GB_per_s"] == 6458.1
    large = wk["5_sweep_f32_GB_per_s_rmsnorm_then_add"]
    small = wk["5_sweep_small_f32_us_per_call_graph_rmsnorm_then_add"]
    shapes = wl.sweep_shapes()
    assert len(large) + len(small) == len(shapes) == 35
    assert len(large) == 7 and large["rows65536_n6656"] == [6512.0, 6940.0]
    assert small["1x2"] == [1.23, 2.35] and small["65536x768"] == [1.89, 2.35]
    assert len(wk["next_GB_per_s"]) == 8
    assert len(json.dumps(wk)) < 2000


def test_summary_without_secondary():
    line = synthetic_line()
    line["secondary"] = {}
    wk = bench.workload_summary(line, 6785.2)
    assert wk["5_sweep_small_f32_us_per_call_graph_rmsnorm_then_add"] is None
    assert wk["5_sweep_f32_GB_per_s_rmsnorm_then_add"] is None
    assert wk["next_GB_per_s"] is None
