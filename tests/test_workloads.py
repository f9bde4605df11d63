"""The seeded input recipes: deterministic, the stated shapes and structure (no GPU)."""
import numpy as np

from dual_epsilon_sandwich_gb300 import workloads as wl


def test_seeded_and_deterministic():
    a = wl.sandwich_decode()
    b = wl.sandwich_decode()
    for k in a.arrays:
        assert np.array_equal(a.arrays[k], b.arrays[k])
    assert a.arrays["block_out"].dtype == np.float32
    assert a.rows == 1 and a.n == 6656 and a.eps == 1e-8 and a.eps_pre == 1e-5


def test_prefill_row_mean_squares_are_log_uniform():
    w = wl.sandwich_prefill(rows=256)
    b = w.arrays["block_out"].astype(np.float64)
    ms = np.mean(b * b, axis=1)
    assert ms.min() >= 1e-4 * (1 - 1e-5) and ms.max() <= 1e2 * (1 + 1e-5)
    assert np.log10(ms).std() > 1.0          # spread over the six decades


def test_bf16_workload_is_bit_patterns():
    w = wl.llama_bf16(rows=64)
    for k in ("x", "gamma", "residual"):
        assert w.arrays[k].dtype == np.uint16
    assert w.eps == 1e-6


def test_sweep_shapes_and_zero_rows():
    shapes = wl.sweep_shapes()
    assert len(shapes) == 35
    assert (65536, 65536) not in shapes and (16384, 65536) in shapes
    w = wl.sweep(768, 4096)
    assert len(w.zero_rows) == 41
    assert np.all(w.arrays["x"][w.zero_rows] == 0.0)
    nz = np.setdiff1d(np.arange(4096), w.zero_rows)
    assert np.all(np.any(w.arrays["x"][nz] != 0.0, axis=1))
    assert len(wl.sweep(7, 1).zero_rows) == 0 and len(wl.sweep(7, 64).zero_rows) == 1
