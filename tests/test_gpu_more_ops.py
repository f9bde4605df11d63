"""GPU parity of residual-add + RMSNorm (Hesper residualAddRmsNormKernel) and
post-norm, add, broadcast scale (Hesper rmsNormThenAddThenBroadcastScaleKernel):
tiny and ragged rows, batch shapes in the staged kernel, every geometry kind,
in-place aliasing and bf16."""
import numpy as np
import pytest
import torch

import gpu_util as gu
from dual_epsilon_sandwich_gb300 import mrn
from dual_epsilon_sandwich_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
DTYPES = ("f32", "bf16")


@pytest.fixture(autouse=True)
def _lib(gpu_lib):
    mrn.mrn_force_geometry(None)
    yield
    mrn.mrn_force_geometry(None)
    assert mrn.mrn_wait_timeouts() == 0


def both(d, dtype, what, sample=None, scale=0.625):
    gu.parity_add_rmsnorm(d["x"], d["residual"], d["gamma"], 1e-5, dtype, sample,
                          what=f"{what} add_rmsnorm")
    gu.parity_then_add_scale(d["x"], d["gamma"], d["residual"], scale, 1e-6, dtype, sample,
                             what=f"{what} then_add_scale")


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("n", [1, 2, 3, 7, 8, 33, 128, 129, 768, 1000, 4096, 6656, 16384])
def test_shapes(n, dtype):
    for rows in (1, 3, 64):
        both(wl.random_rows(3000 + n + rows, rows, n, dtype), dtype, f"{rows}x{n}")


@pytest.mark.parametrize("dtype", DTYPES)
def test_batches(dtype):
    """Batch shapes in the automatic geometry (the register kernel, except the
    f32 then-add-scale at 1664 loads per row, which stays staged) and both
    operations forced into the staged kernel."""
    for rows, n in ((4096, 6656), (2048, 4096)):
        assert mrn.mrn_query_geometry(3, rows, n, gu.code(dtype), True)["kind"] == mrn.MRN_GEOM_CTA
        want = mrn.MRN_GEOM_TMA if (dtype, n) == ("f32", 6656) else mrn.MRN_GEOM_CTA
        assert mrn.mrn_query_geometry(4, rows, n, gu.code(dtype), True)["kind"] == want
        d = wl.random_rows(rows + n, rows, n, dtype)
        sample = gu.sample_rows(rows, 128, seed=n)
        both(d, dtype, f"batch {rows}x{n}", sample=sample)
        nvec = n // (4 if dtype == "f32" else 8)
        k = -(-nvec // 416)
        assert mrn.mrn_force_geometry({"kind": 4, "k": k, "threads": 832, "stages": 2,
                                       "groups": 2}) == 0
        try:
            both(d, dtype, f"staged {rows}x{n}", sample=sample)
        finally:
            mrn.mrn_force_geometry(None)


GEOMS = [
    ({"kind": 1, "lanes_per_row": 32, "k": 8}, 250),
    ({"kind": 1, "lanes_per_row": 8, "k": 1}, 7),
    ({"kind": 2, "k": 3, "threads": 96, "cluster": 3}, 700),
    ({"kind": 2, "k": 8, "threads": 256, "cluster": 8}, 16000),
    ({"kind": 3, "threads": 128}, 1500),
    ({"kind": 4, "k": 4, "threads": 256, "stages": 4, "groups": 2, "ctas": 9}, 500),
    ({"kind": 4, "k": 2, "threads": 512, "stages": 1, "groups": 1}, 1000),
]


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("geom,nvec", GEOMS, ids=[str(i) for i in range(len(GEOMS))])
def test_forced_geometries(geom, nvec, dtype):
    n = nvec * (4 if dtype == "f32" else 8)
    assert mrn.mrn_force_geometry(geom) == 0
    both(wl.random_rows(n + 11, 37, n, dtype), dtype, f"forced {geom}", scale=-3.5)


@pytest.mark.parametrize("dtype", DTYPES)
def test_in_place(dtype):
    rows, n = 96, 2048
    d = wl.random_rows(17, rows, n, dtype)
    gu.parity_add_rmsnorm(d["x"], d["residual"], d["gamma"], 1e-5, dtype, inplace="a")
    gu.parity_add_rmsnorm(d["x"], d["residual"], d["gamma"], 1e-5, dtype, inplace="b")
    a, b, g = (gu.to_device(d[k], dtype) for k in ("x", "residual", "gamma"))
    s_ref, o_ref = torch.empty_like(a), torch.empty_like(a)
    assert gu.call_add_rmsnorm(a, b, g, s_ref, o_ref, rows, n, 1e-5, dtype) == 0
    a2, b2 = a.clone(), b.clone()
    assert gu.call_add_rmsnorm(a2, b2, g, b2, a2, rows, n, 1e-5, dtype) == 0   # both in place
    sc = gu.to_device(np.array([0.5], np.float32) if dtype == "f32"
                      else gu.oracle.bf16_from_double([0.5]), dtype)
    out_ref = torch.empty_like(a)
    assert gu.call_then_add_scale(a, g, b, sc, out_ref, rows, n, 1e-5, dtype) == 0
    r3 = b.clone()
    assert gu.call_then_add_scale(a, g, r3, sc, r3, rows, n, 1e-5, dtype) == 0
    torch.cuda.synchronize()
    view = torch.int32 if dtype == "f32" else torch.int16
    assert torch.equal(b2.view(view), s_ref.view(view))
    assert torch.equal(a2.view(view), o_ref.view(view))
    assert torch.equal(r3.view(view), out_ref.view(view))


def test_scale_reads_device_memory_each_call():
    """The broadcast scale is read by the kernel, so a graph replays with the
    current value (the layer's output scale can change without a relaunch)."""
    rows, n = 8, 4096
    d = wl.random_rows(19, rows, n, "f32")
    x, g, r = (gu.to_device(d[k], "f32") for k in ("x", "gamma", "residual"))
    sc = torch.tensor([1.0], device="cuda")
    out = torch.empty_like(x)
    assert gu.call_then_add_scale(x, g, r, sc, out, rows, n, 1e-5, "f32") == 0
    first = out.clone()
    sc.fill_(-2.0)
    assert gu.call_then_add_scale(x, g, r, sc, out, rows, n, 1e-5, "f32") == 0
    torch.cuda.synchronize()
    assert torch.equal(out, -2.0 * first)


def test_tensor_api():
    d = wl.random_rows(21, 6, 512, "bf16")
    a, b, g = (gu.to_device(d[k], "bf16") for k in ("x", "residual", "gamma"))
    s, o = mrn.add_rmsnorm(a, b, g, 1e-5)
    out = mrn.rmsnorm_then_add_scale(a, g, b, torch.ones(1, dtype=torch.bfloat16,
                                                         device="cuda"), 1e-5)
    ref = mrn.rmsnorm_then_add(a, g, b, 1e-5)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert s.shape == o.shape == a.shape


@pytest.mark.parametrize("dtype", DTYPES)
def test_per_head_qk_norm_shape(dtype):
    """Per-head QK-norm (Chapter 12, section 12.5: head_dim = 128, one norm per
    head): rows = tokens x heads, n = 128, gamma shared by all heads."""
    rows, n = 4096 * 40, 128
    d = wl.random_rows(23, rows, n, dtype)
    g = mrn.mrn_query_geometry(0, rows, n, gu.code(dtype), True)
    assert g["kind"] == mrn.MRN_GEOM_ROWS_PER_WARP
    sample = gu.sample_rows(rows, 512, seed=29)
    gu.parity_rmsnorm(d["x"], d["gamma"], 1e-6, dtype, sample, what="qk-norm")
    gu.parity_rmsnorm(d["x"], np.ones_like(d["gamma"]) if dtype == "f32"
                      else gu.oracle.bf16_from_double(np.ones(n)), 1e-6, dtype, sample,
                      what="qk-norm, constant gamma")
