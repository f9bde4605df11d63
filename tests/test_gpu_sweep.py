"""GPU parity over the f32 shape sweep: n in {2 .. 65536} x rows in {1 .. 65536}
(operands up to 4 GiB, so 64-bit offsets), 1% all-zero rows, eps 1e-5 and 1e-8,
plain and then-add.  Rows are compared with the oracle in full up to 2^25
elements; above that on a seeded sample of rows that includes every zero row,
with exactness of the zero rows and finiteness checked over the whole output."""
import numpy as np
import pytest
import torch

import gpu_util as gu
import oracle
from dual_epsilon_sandwich_gb300 import mrn
from dual_epsilon_sandwich_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

FULL_LIMIT = 1 << 25


@pytest.fixture(autouse=True)
def _lib(gpu_lib):
    mrn.mrn_force_geometry(None)


@pytest.mark.parametrize("n,rows", wl.sweep_shapes(), ids=lambda v: str(v))
def test_sweep_shape(n, rows):
    w = wl.sweep(n, rows)
    x, g, r = w.arrays["x"], w.arrays["gamma"], w.arrays["residual"]
    sample = None
    if rows * n > FULL_LIMIT:
        sample = gu.sample_rows(rows, 96, seed=rows * 131 + n, must=w.zero_rows[:64])
    dx, dg, dr = gu.to_device(x, "f32"), gu.to_device(g, "f32"), gu.to_device(r, "f32")
    zero = torch.from_numpy(w.zero_rows).cuda()
    for eps in wl.SWEEP_EPS:
        # plain
        y = gu.Guarded(rows, n, "f32")
        assert gu.call_rmsnorm(dx, dg, y, rows, n, eps, "f32") == 0
        torch.cuda.synchronize()
        y.check(f"rmsnorm {rows}x{n}")
        assert bool(torch.isfinite(y.tensor).all())
        if len(w.zero_rows):
            assert bool((y.tensor[zero] == 0).all()), "zero rows must give exact zeros"
        got = gu.to_host(y.tensor if sample is None else y.tensor[torch.from_numpy(sample).cuda()],
                         "f32")
        xs = x if sample is None else x[sample]
        want = oracle.rmsnorm(xs.astype(np.float64), g.astype(np.float64), float(np.float32(eps)))
        gu.check_f32_norm(got, want, f"rmsnorm {rows}x{n} eps={eps}")
        del y
        # then-add
        out = gu.Guarded(rows, n, "f32")
        assert gu.call_then_add(dx, dg, dr, out, rows, n, eps, "f32") == 0
        torch.cuda.synchronize()
        out.check(f"then_add {rows}x{n}")
        assert bool(torch.isfinite(out.tensor).all())
        if len(w.zero_rows):
            assert bool((out.tensor[zero] == dr[zero]).all()), "zero rows must return residual"
        got = gu.to_host(out.tensor if sample is None
                         else out.tensor[torch.from_numpy(sample).cuda()], "f32")
        rs = r if sample is None else r[sample]
        e = float(np.float32(eps))
        want = oracle.rmsnorm_then_add(xs.astype(np.float64), g.astype(np.float64),
                                       rs.astype(np.float64), e)
        scale = np.abs(oracle.rmsnorm(xs.astype(np.float64), g.astype(np.float64), e)) + np.abs(rs)
        gu.check_f32_sum(got, want, scale, f"then_add {rows}x{n} eps={eps}")
        del out
    del dx, dr
    torch.cuda.empty_cache()
