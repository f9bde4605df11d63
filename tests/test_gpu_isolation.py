"""Rows are independent, and so are callers.

* A row holding NaN or infinity gives non-finite outputs in that row only:
  every other row is bit-identical to a run without the poisoned row, in
  every kernel kind (the persistent kernels reduce many rows per CTA).
* The forced geometry and launch options are per thread: two threads calling
  the library at once with different forced geometries each get their own."""
import threading

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
    yield
    mrn.mrn_force_geometry(None)


def _run_all(x, r, g, g2, gh, rows, n, dtype):
    """Outputs of every operation as host arrays (bit patterns for 16-bit data)."""
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    dt, sh = gu.code(dtype), gu.stream_handle()
    y = torch.empty(rows, n, dtype=tdt, device="cuda")
    t = torch.empty_like(y)
    s, o = torch.empty_like(y), torch.empty_like(y)
    a_, b_ = torch.empty_like(y), torch.empty_like(y)
    sc = torch.full((1,), 0.5, device="cuda").to(tdt)
    ts = torch.empty_like(y)
    seam = torch.empty(rows, n, dtype=torch.float16, device="cuda")
    calls = [
        mrn.mrn_rmsnorm(x.data_ptr(), g.data_ptr(), y.data_ptr(), rows, n, 1e-5, dt, sh),
        mrn.mrn_rmsnorm_then_add(x.data_ptr(), g.data_ptr(), r.data_ptr(), t.data_ptr(), rows, n,
                                 1e-5, dt, sh),
        mrn.mrn_norm_residual_norm(x.data_ptr(), r.data_ptr(), g.data_ptr(), g2.data_ptr(),
                                   s.data_ptr(), o.data_ptr(), rows, n, 1e-8, 1e-5, dt, sh),
        mrn.mrn_add_rmsnorm(x.data_ptr(), r.data_ptr(), g.data_ptr(), a_.data_ptr(),
                            b_.data_ptr(), rows, n, 1e-5, dt, sh),
        mrn.mrn_rmsnorm_then_add_scale(x.data_ptr(), g.data_ptr(), r.data_ptr(), sc.data_ptr(),
                                       ts.data_ptr(), rows, n, 1e-5, dt, sh),
        mrn.mrn_rmsnorm_seam(x.data_ptr(), gh.data_ptr(), seam.data_ptr(), rows, n, 1e-5, dt,
                             mrn.MRN_F16, sh),
    ]
    assert all(c == 0 for c in calls), calls
    torch.cuda.synchronize()
    return [v.view(torch.int16 if v.element_size() == 2 else torch.int32).cpu().numpy()
            for v in (y, t, s, o, a_, b_, ts, seam)]


SHAPES = [(700, 128), (1000, 2048), (400, 6656), (3, 200000)]   # rows-per-warp, staged, cluster, looped


@pytest.mark.parametrize("dtype", ("f32", "bf16"))
@pytest.mark.parametrize("rows,n", SHAPES, ids=[f"{r}x{n}" for r, n in SHAPES])
@pytest.mark.parametrize("poison", (np.nan, np.inf))
def test_a_poisoned_row_stays_in_its_row(rows, n, dtype, poison):
    d = wl.random_rows(900 + n, rows, n, dtype)
    gh = torch.from_numpy(wl.to_f16_bits(1.0 + 0.01 * np.arange(n) / n).view(np.int16)).cuda()
    to = lambda a: gu.to_device(a, dtype)
    g, g2 = to(d["gamma"]), to(d["gamma2"])
    clean = _run_all(to(d["x"]), to(d["residual"]), g, g2, gh, rows, n, dtype)
    bad_row = rows // 2
    xp = d["x"].copy()
    xp[bad_row, n // 3] = np.float32(poison) if dtype == "f32" else wl.to_bf16_bits(
        np.array([poison]))[0]
    dirty = _run_all(to(xp), to(d["residual"]), g, g2, gh, rows, n, dtype)
    keep = np.ones(rows, bool)
    keep[bad_row] = False
    for i, (c, p) in enumerate(zip(clean, dirty)):
        assert np.array_equal(c[keep], p[keep]), f"output {i}: another row changed"
        assert not np.array_equal(c[bad_row], p[bad_row]), f"output {i}: the row did not change"


def test_forced_geometry_is_per_thread():
    """Thread A forces the one-row-per-CTA kernel, thread B a rows-per-warp
    geometry; both run interleaved calls and check parity; each thread then
    still sees its own forced geometry."""
    n_a, n_b = 2048, 128
    mine = mrn.mrn_query_geometry(mrn.MRN_OP_RMSNORM, 64, n_a, mrn.MRN_F32, True)
    errors = []
    start = threading.Barrier(2)

    def worker(geom, n, seed):
        try:
            assert mrn.mrn_force_geometry(geom) == 0
            start.wait(timeout=60)
            stream = torch.cuda.Stream()
            with torch.cuda.stream(stream):
                for i in range(5):
                    d = wl.random_rows(seed + i, 64, n, "f32")
                    gu.parity_rmsnorm(d["x"], d["gamma"], 1e-5, "f32", what=f"thread {seed}")
            got = mrn.mrn_query_geometry(mrn.MRN_OP_RMSNORM, 64, n, mrn.MRN_F32, True)
            assert got["kind"] == geom["kind"], got
            mrn.mrn_force_geometry(None)
        except BaseException as exc:   # reported by the main thread
            errors.append(exc)
            start.abort()              # never leave the other thread waiting

    ta = threading.Thread(target=worker,
                          args=({"kind": 2, "k": 2, "threads": 256, "cluster": 1}, n_a, 10))
    tb = threading.Thread(target=worker, args=({"kind": 1, "lanes_per_row": 8, "k": 4}, n_b, 20))
    ta.start()
    tb.start()
    ta.join(timeout=300)
    tb.join(timeout=300)
    assert not ta.is_alive() and not tb.is_alive(), "a worker thread did not finish"
    assert not errors, errors
    assert mrn.mrn_query_geometry(mrn.MRN_OP_RMSNORM, 64, n_a, mrn.MRN_F32, True) == mine
