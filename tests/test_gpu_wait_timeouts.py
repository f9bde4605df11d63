"""A bounded wait that runs out, driven on the GPU without a fault.  The test
launch option MRN_LAUNCH_TEST_WAIT_TIMEOUT makes the first wait of every CTA
expect 16 bytes more than ever arrive (every copy and message still lands, so
nothing is left in flight).  Each kernel family must then return after about
a second per wait, report the timeouts through mrn_wait_timeouts(), write
nothing where the staged kernels promise it, and leave the context usable: the
same call without the option matches the oracle afterwards."""
import time

import numpy as np
import pytest
import torch

import gpu_util as gu
from dual_epsilon_sandwich_gb300 import mrn
from dual_epsilon_sandwich_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _lib(gpu_lib):
    mrn.mrn_force_geometry(None)
    mrn.mrn_set_launch_options(mrn.MRN_LAUNCH_PDL)
    mrn.mrn_wait_timeouts()          # (the count since the previous read)
    yield
    mrn.mrn_set_launch_options(mrn.MRN_LAUNCH_PDL)
    mrn.mrn_wait_timeouts()


def stalled(call):
    """call() once with the test hook on: (status, seconds, timeouts counted)."""
    assert mrn.mrn_wait_timeouts() == 0
    torch.cuda.synchronize()
    assert mrn.mrn_set_launch_options(mrn.MRN_LAUNCH_PDL | mrn.MRN_LAUNCH_TEST_WAIT_TIMEOUT) == 0
    try:
        t0 = time.perf_counter()
        st = call()
        torch.cuda.synchronize()
        seconds = time.perf_counter() - t0
    finally:
        mrn.mrn_set_launch_options(mrn.MRN_LAUNCH_PDL)
    return st, seconds, mrn.mrn_wait_timeouts()


def untouched(g: gu.Guarded) -> bool:
    return bool((g.raw == g.sentinel).all())


@pytest.mark.parametrize("dtype,n", [("bf16", 6656), ("f32", 6655)])
def test_staged_kernel_stops_without_writing(dtype, n):
    """The staged sandwich (bf16: both gammas by bulk copy; f32 at n = 6655: the
    edge-staged kernel, whose threads place the gammas and arrive on the same
    barrier) stops at the gamma wait's timeout before writing anything."""
    rows = 304
    g = mrn.mrn_query_geometry(mrn.MRN_OP_SANDWICH, rows, n, gu.code(dtype), True)
    assert (g["kind"], g["cluster"], g["edge"]) == (mrn.MRN_GEOM_TMA, 1, int(dtype == "f32"))
    d = wl.random_rows(41, rows, n, dtype)
    b, r = gu.to_device(d["x"], dtype), gu.to_device(d["residual"], dtype)
    gp, gq = gu.to_device(d["gamma"], dtype), gu.to_device(d["gamma2"], dtype)
    s, o = gu.Guarded(rows, n, dtype), gu.Guarded(rows, n, dtype)
    st, seconds, count = stalled(
        lambda: gu.call_sandwich(b, r, gp, gq, s, o, rows, n, 1e-8, 1e-5, dtype))
    assert st == 0 and count >= 1 and seconds < 30, (st, count, seconds)
    assert untouched(s) and untouched(o)
    gu.parity_sandwich(d["x"], d["residual"], d["gamma"], d["gamma2"], 1e-8, 1e-5, dtype,
                       what="staged sandwich after a timeout")
    assert mrn.mrn_wait_timeouts() == 0


def test_staged_kernel_without_a_gamma_copy_stops_without_writing():
    """The seam reads its 16-bit gamma through L1: its staged kernel arms the
    gamma barrier for no bytes at all, and the hook's 16 bytes never come."""
    rows, n = 304, 6656
    g = mrn.mrn_query_geometry(mrn.MRN_OP_RMSNORM_SEAM, rows, n, mrn.MRN_F32, True)
    assert g["kind"] == mrn.MRN_GEOM_TMA
    d = wl.seam_rows(42, rows, n, "f32", "f16")
    x = gu.to_device(d["x"], "f32")
    gam = torch.from_numpy(np.ascontiguousarray(d["gamma"]).view(np.int16)).cuda()
    y = torch.full((rows * n,), 0x5A5A, dtype=torch.int16, device="cuda")
    st, seconds, count = stalled(
        lambda: mrn.mrn_rmsnorm_seam(x.data_ptr(), gam.data_ptr(), y.data_ptr(), rows, n, 1e-5,
                                     mrn.MRN_F32, mrn.MRN_F16, gu.stream_handle()))
    assert st == 0 and count >= 1 and seconds < 30, (st, count, seconds)
    assert bool((y == 0x5A5A).all())
    gu.parity_seam(d["x"], d["gamma"], 1e-5, "f32", "f16", what="seam after a timeout")
    assert mrn.mrn_wait_timeouts() == 0


def test_cluster_staged_kernel_stops_without_writing():
    rows, n = 160, 16384
    g = mrn.mrn_query_geometry(mrn.MRN_OP_THEN_ADD, rows, n, mrn.MRN_F32, True)
    assert (g["kind"], g["cluster"]) == (mrn.MRN_GEOM_TMA, 2)
    d = wl.random_rows(43, rows, n, "f32")
    x, r = gu.to_device(d["x"], "f32"), gu.to_device(d["residual"], "f32")
    gam = gu.to_device(d["gamma"], "f32")
    out = gu.Guarded(rows, n, "f32")
    st, seconds, count = stalled(lambda: gu.call_then_add(x, gam, r, out, rows, n, 1e-5, "f32"))
    assert st == 0 and count >= 1 and seconds < 30, (st, count, seconds)
    assert untouched(out)
    gu.parity_then_add(d["x"], d["gamma"], d["residual"], 1e-5, "f32",
                       what="cluster-staged then-add after a timeout")
    assert mrn.mrn_wait_timeouts() == 0


def test_staged_q8_1_kernel_stops_without_writing():
    rows, n = 304, 4096
    g = mrn.mrn_query_geometry(mrn.MRN_OP_RMSNORM_Q8_1, rows, n, mrn.MRN_BF16, True)
    assert g["kind"] == mrn.MRN_GEOM_Q8_BLOCKS and g["stages"] > 0
    d = wl.random_rows(44, rows, n, "bf16")
    x, gam = gu.to_device(d["x"], "bf16"), gu.to_device(d["gamma"], "bf16")
    blocks = torch.full((rows * (n // 32) * mrn.Q8_1_BLOCK_BYTES,), 0x3C, dtype=torch.uint8,
                        device="cuda")
    st, seconds, count = stalled(
        lambda: mrn.mrn_rmsnorm_q8_1(x.data_ptr(), gam.data_ptr(), blocks.data_ptr(), rows, n,
                                     1e-6, mrn.MRN_BF16, gu.stream_handle()))
    assert st == 0 and count >= 1 and seconds < 30, (st, count, seconds)
    assert bool((blocks == 0x3C).all())
    gu.parity_q8_1(d["x"], d["gamma"], 1e-6, "bf16", what="staged Q8_1 after a timeout")
    assert mrn.mrn_wait_timeouts() == 0


def test_cluster_reduction_of_the_register_kernel_times_out_and_recovers():
    """Decode: one row over a cluster of CTAs.  The first message exchange
    runs out (the outputs of that call are unspecified); the call returns and
    the next call is exact."""
    rows, n = 1, 6656
    g = mrn.mrn_query_geometry(mrn.MRN_OP_SANDWICH, rows, n, mrn.MRN_F32, True)
    assert g["kind"] == mrn.MRN_GEOM_CTA and g["cluster"] > 1
    d = wl.random_rows(45, rows, n, "f32")
    b, r = gu.to_device(d["x"], "f32"), gu.to_device(d["residual"], "f32")
    gp, gq = gu.to_device(d["gamma"], "f32"), gu.to_device(d["gamma2"], "f32")
    s, o = torch.empty_like(b), torch.empty_like(b)
    st, seconds, count = stalled(
        lambda: gu.call_sandwich(b, r, gp, gq, s, o, rows, n, 1e-8, 1e-5, "f32"))
    assert st == 0 and count >= 1 and seconds < 30, (st, count, seconds)
    gu.parity_sandwich(d["x"], d["residual"], d["gamma"], d["gamma2"], 1e-8, 1e-5, "f32",
                       what="decode sandwich after a timeout")
    assert mrn.mrn_wait_timeouts() == 0
