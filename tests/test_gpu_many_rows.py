"""More rows than one launch takes: the launchers split a call every 2^26 rows
(so that a grid dimension stays far below its limit).  Every output written,
nothing outside the output touched (guard bands), and the rows on both sides
of the split against the oracle, for the rows-per-warp kernel (n = 1) and the
persistent staged kernel (n = 4, forced)."""
import numpy as np
import pytest
import torch

import gpu_util as gu
import oracle
from dual_epsilon_sandwich_gb300 import mrn

pytestmark = pytest.mark.gpu
SPLIT = 1 << 26
ROWS = SPLIT + 3


@pytest.fixture(autouse=True)
def _lib(gpu_lib):
    mrn.mrn_force_geometry(None)
    yield
    mrn.mrn_force_geometry(None)


@pytest.mark.parametrize("n,geom", [(1, None),
                                    (4, {"kind": 4, "k": 1, "threads": 64, "stages": 2,
                                         "groups": 2})],
                         ids=["rows-per-warp", "staged"])
def test_rows_beyond_one_launch(n, geom):
    gen = torch.Generator(device="cuda")
    gen.manual_seed(2026 + n)
    x = torch.randn(ROWS, n, device="cuda", generator=gen)
    x[SPLIT - 1].zero_()                         # a zero row right before the split
    gamma = 1 + 0.1 * torch.randn(n, device="cuda", generator=gen)
    y = gu.Guarded(ROWS, n, "f32")
    assert mrn.mrn_force_geometry(geom) == 0
    before = mrn.mrn_launch_count()
    st = mrn.mrn_rmsnorm(x.data_ptr(), gamma.data_ptr(), y.ptr(), ROWS, n, 1e-5, mrn.MRN_F32,
                         gu.stream_handle())
    assert st == 0, mrn.STATUS.get(st)
    assert mrn.mrn_launch_count() - before == 2   # one launch per 2^26 rows
    torch.cuda.synchronize()
    y.check(f"{ROWS} rows")
    pick = np.array([0, 1, SPLIT - 2, SPLIT - 1, SPLIT, SPLIT + 1, ROWS - 1])
    got = y.tensor[torch.from_numpy(pick).cuda()].cpu().numpy()
    xs = x[torch.from_numpy(pick).cuda()].cpu().numpy().astype(np.float64)
    want = oracle.rmsnorm(xs, gamma.cpu().numpy().astype(np.float64), float(np.float32(1e-5)))
    gu.check_f32_norm(got, want, f"rows around the launch split, n={n}")
    assert np.all(got[3] == 0.0)                  # the zero row
