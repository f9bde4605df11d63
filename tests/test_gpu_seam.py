"""GPU parity of the split-norm seam ("Chapter 12 -- RMSNorm and the
dual-epsilon sandwich", section 12.7, the cross-vendor seam): the weightless
norm published in binary16 or bf16, then the weight multiply as a second
operation in that format.  Every case runs the split route (two kernels) and
the fused kernel; both are checked against the oracle, and the fused result
must equal the split route's bit for bit."""
import numpy as np
import pytest
import torch

import gpu_util as gu
from dual_epsilon_sandwich_gb300 import mrn
from dual_epsilon_sandwich_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
DTYPES = ("f32", "bf16")
SEAMS = ("f16", "bf16")


@pytest.fixture(autouse=True)
def _lib(gpu_lib):
    mrn.mrn_force_geometry(None)
    yield
    mrn.mrn_force_geometry(None)


@pytest.mark.parametrize("seam", SEAMS)
@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("n", [1, 2, 7, 64, 128, 1000, 2560, 4096, 6656])
def test_widths(n, dtype, seam):
    for rows in (1, 3, 64):
        d = wl.seam_rows(7000 + n + rows, rows, n, dtype, seam, scale=2.0)
        gu.parity_seam(d["x"], d["gamma"], 1e-5, dtype, seam, what=f"seam {rows}x{n}")


@pytest.mark.parametrize("seam", SEAMS)
@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("kernel", ["auto", "staged"])
def test_batch(dtype, seam, kernel):
    """Many rows (the register kernel by the automatic choice at this width, and
    the persistent staged kernel forced), rows of very different scales and a
    few zero rows."""
    rows, n = 4096, 2560
    g = np.random.Generator(np.random.PCG64(61))
    x = g.standard_normal((rows, n)) * 10.0 ** g.uniform(-3, 3, size=(rows, 1))
    x[[5, 700, 4000], :] = 0.0
    x = wl.to_f32(x) if dtype == "f32" else wl.to_bf16_bits(x)
    gamma = wl.to_seam_bits(1.0 + 0.1 * g.standard_normal(n), seam)
    assert mrn.mrn_query_geometry(mrn.MRN_OP_RMSNORM_SEAM, rows, n, gu.code(dtype), True)["kind"] \
        == mrn.MRN_GEOM_CTA
    if kernel == "staged":
        per_group = -(-(n // (4 if dtype == "f32" else 8) // 4) // 32) * 32
        assert mrn.mrn_force_geometry({"kind": 4, "k": 4, "threads": 2 * per_group, "stages": 2,
                                       "groups": 2}) == 0
    try:
        flips, near = gu.parity_seam(x, gamma, 1e-6, dtype, seam,
                                     what=f"seam batch {dtype}/{seam} {kernel}")
    finally:
        mrn.mrn_force_geometry(None)
    print(f"seam {dtype}->{seam} {kernel}: {flips} of {near} near-tie elements took the other side")


GEOMS = [
    {"kind": 1, "lanes_per_row": 1, "k": 8},
    {"kind": 1, "lanes_per_row": 4, "k": 2},
    {"kind": 1, "lanes_per_row": 32, "k": 1},
    {"kind": 2, "k": 3, "threads": 96, "cluster": 1},
    {"kind": 2, "k": 1, "threads": 64, "cluster": 4},
    {"kind": 3, "threads": 96},
    {"kind": 3, "threads": 64, "cluster": 4},
]


@pytest.mark.parametrize("seam", SEAMS)
@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("geom", GEOMS, ids=[str(i) for i in range(len(GEOMS))])
def test_forced_geometries(geom, dtype, seam):
    vec = 4 if dtype == "f32" else 8
    cover = {1: geom.get("lanes_per_row", 0) * geom.get("k", 0),
             2: geom.get("threads", 0) * geom.get("k", 0) * geom.get("cluster", 1),
             3: 10 ** 6}[geom["kind"]]
    n = min(cover, 300) * vec - 3 * (geom["kind"] == 3)
    assert mrn.mrn_force_geometry(geom) == 0
    d = wl.seam_rows(90 + n, 37, n, dtype, seam)
    gu.parity_seam(d["x"], d["gamma"], 1e-5, dtype, seam, what=f"seam forced {geom} n={n}")


STAGED = [   # persistent TMA-staged kernel: x staged, the 16-bit gamma read through L1
    {"kind": 4, "k": 4, "threads": 832, "stages": 2, "groups": 2},
    {"kind": 4, "k": 8, "threads": 448, "stages": 4, "groups": 2, "ctas": 9},
    {"kind": 4, "k": 8, "threads": 256, "stages": 2, "groups": 1, "ctas": 7},
    {"kind": 4, "k": 2, "threads": 192, "stages": 4, "groups": 2, "ctas": 3},
    {"kind": 4, "k": 1, "threads": 64, "stages": 4, "groups": 2, "ctas": 1},
    {"kind": 4, "k": 3, "threads": 96, "stages": 3, "groups": 1, "ctas": 5},
]


@pytest.mark.parametrize("seam", SEAMS)
@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("geom", STAGED, ids=[str(i) for i in range(len(STAGED))])
def test_forced_staged_geometries(geom, dtype, seam):
    vec = 4 if dtype == "f32" else 8
    cover = geom["threads"] // geom["groups"] * geom["k"]
    n = max(1, cover - 1) * vec            # some idle slots; for f32 often n % 8 != 0
    assert mrn.mrn_force_geometry(geom) == 0
    assert mrn.mrn_query_geometry(mrn.MRN_OP_RMSNORM_SEAM, 50, n, gu.code(dtype), True)["kind"] \
        == mrn.MRN_GEOM_TMA
    d = wl.seam_rows(95 + n, 50, n, dtype, seam)
    gu.parity_seam(d["x"], d["gamma"], 1e-5, dtype, seam, what=f"seam staged {geom} n={n}")
    assert mrn.mrn_wait_timeouts() == 0


@pytest.mark.parametrize("seam", SEAMS)
@pytest.mark.parametrize("dtype", DTYPES)
def test_unaligned_and_wide_rows(dtype, seam):
    d = wl.seam_rows(71, 5, 4096, dtype, seam)
    gu.parity_seam(d["x"], d["gamma"], 1e-5, dtype, seam, what="seam unaligned", x_offset=1)
    n = 200000 if dtype == "f32" else 300000
    d = wl.seam_rows(72, 3, n, dtype, seam)
    assert mrn.mrn_query_geometry(mrn.MRN_OP_RMSNORM_SEAM, 3, n, gu.code(dtype), True)["kind"] \
        == mrn.MRN_GEOM_STREAM
    gu.parity_seam(d["x"], d["gamma"], 1e-5, dtype, seam, what="seam wide")


@pytest.mark.parametrize("seam", SEAMS)
@pytest.mark.parametrize("dtype", DTYPES)
def test_extreme_gammas(dtype, seam):
    """Products that overflow the format to infinity, land in its subnormal
    range or underflow to zero; negative gammas (signed zeros of zero rows)."""
    rows, n = 8, 512
    g = np.random.Generator(np.random.PCG64(73))
    x = g.standard_normal((rows, n))
    x[3, :] = 0.0
    gamma = 1.0 + 0.1 * g.standard_normal(n)
    gamma[0:64] *= -1.0
    if seam == "f16":
        gamma[64:128] = 3.0e4 * (1 + g.uniform(0, 1, 64))      # |u| > ~2 overflows
        gamma[128:192] = 2.0 ** -14 * g.uniform(0.01, 1, 64)   # binary16 subnormal products
        gamma[192:200] = 2.0 ** -24                            # smallest subnormal
    else:
        gamma[64:128] = 3.0e38 * g.uniform(0.5, 1, 64)
        gamma[128:192] = 2.0 ** -126 * g.uniform(0.01, 1, 64)  # bf16 subnormal products
        gamma[192:200] = 2.0 ** -133
    x = wl.to_f32(x) if dtype == "f32" else wl.to_bf16_bits(x)
    gamma = wl.to_seam_bits(gamma, seam)
    gu.parity_seam(x, gamma, 1e-5, dtype, seam, what=f"seam extremes {dtype}/{seam}")


@pytest.mark.parametrize("seam", SEAMS)
def test_in_place(seam):
    """bf16 x overwritten by its own seam output, and the scale applied in place."""
    d = wl.seam_rows(74, 64, 2048, "bf16", seam)
    u, ys, yf = gu.run_seam(d["x"], d["gamma"], 1e-5, "bf16", seam)
    sc, sh = gu.seam_code(seam), gu.stream_handle()
    x = gu.to_device(d["x"], "bf16")
    g = torch.from_numpy(d["gamma"].view(np.int16)).cuda()
    assert mrn.mrn_rmsnorm_seam(x.data_ptr(), g.data_ptr(), x.data_ptr(), 64, 2048, 1e-5,
                                mrn.MRN_BF16, sc, sh) == 0
    torch.cuda.synchronize()
    assert np.array_equal(x.view(torch.int16).cpu().numpy().view(np.uint16), yf)
    x = gu.to_device(d["x"], "bf16")
    assert mrn.mrn_rmsnorm_unweighted(x.data_ptr(), x.data_ptr(), 64, 2048, 1e-5, mrn.MRN_BF16,
                                      sc, sh) == 0
    assert mrn.mrn_seam_scale(x.data_ptr(), g.data_ptr(), x.data_ptr(), 64, 2048, sc, sh) == 0
    torch.cuda.synchronize()
    assert np.array_equal(x.view(torch.int16).cpu().numpy().view(np.uint16), ys)


@pytest.mark.parametrize("seam", SEAMS)
def test_full_size_rows_sampled(seam):
    """The benchmark's shape (4096 rows of 6656, f32 in), oracle on sampled rows."""
    rows, n = 4096, 6656
    d = wl.seam_rows(75, rows, n, "f32", seam)
    gu.parity_seam(d["x"], d["gamma"], 1e-5, "f32", seam,
                   rows_sample=gu.sample_rows(rows, 64, 5), what=f"seam 4096x6656 {seam}")


def test_tensor_api():
    d = wl.seam_rows(76, 6, 384, "f32", "f16")
    x = gu.to_device(d["x"], "f32")
    g = torch.from_numpy(d["gamma"].view(np.float16)).cuda()
    y = mrn.rmsnorm_seam(x, g, 1e-5)
    u = mrn.rmsnorm_unweighted(x, 1e-5, torch.float16)
    y2 = mrn.seam_scale(u, g)
    torch.cuda.synchronize()
    assert y.dtype == torch.float16 and y.shape == (6, 384)
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))
    want = mrn.rmsnorm(x, torch.ones(384, device="cuda"), 1e-5).half()
    assert torch.equal(u.view(torch.int16), want.view(torch.int16))   # S(x * inv) itself
