"""GPU parity of RMSNorm fused with Q8_1 block quantisation (Hesper
fusedRMSNormQ8_1Kernel): the page's D = 2560 example, model widths, ragged
row counts, zero blocks, every geometry kind and unaligned rows."""
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


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("n", [32, 64, 128, 2560, 4096, 6656])
def test_widths(n, dtype):
    for rows in (1, 3, 64):
        d = wl.random_rows(5000 + n + rows, rows, n, dtype, scale=3.0)
        gu.parity_q8_1(d["x"], d["gamma"], 1e-6, dtype, what=f"q8 {rows}x{n}")


@pytest.mark.parametrize("dtype", DTYPES)
def test_batch_and_zero_blocks(dtype):
    rows, n = 4096, 2560
    g = np.random.Generator(np.random.PCG64(31))
    x = g.standard_normal((rows, n)) * 10.0 ** g.uniform(-2, 2, size=(rows, 1))
    x[5, :] = 0.0
    x[9, 32:64] = 0.0
    x[9, 100] = 1e-30
    x = wl.to_f32(x) if dtype == "f32" else wl.to_bf16_bits(x)
    gamma = wl.random_rows(32, 1, n, dtype)["gamma"]
    assert mrn.mrn_query_geometry(5, rows, n, gu.code(dtype), True)["kind"] == \
        mrn.MRN_GEOM_Q8_BLOCKS
    off, ties = gu.parity_q8_1(x, gamma, 1e-6, dtype,
                               rows_sample=gu.sample_rows(rows, 200, 3, must=(5, 9)))
    print(f"q8 {dtype}: {off} codes one off, all within {ties} near-tie codes")


@pytest.mark.parametrize("geom", [None, {"kind": 5, "k": 1, "threads": 32},
                                  {"kind": 5, "k": 1, "threads": 64, "stages": 2, "groups": 2,
                                   "ctas": 2}],
                         ids=["auto", "blocks", "staged blocks"])
@pytest.mark.parametrize("dtype", DTYPES)
def test_extreme_block_magnitudes(dtype, geom):
    """Blocks whose amax is far from 1: tiny (normed values near 1e-34),
    products that fall below the smallest normal f32, and huge ones (gamma
    1e33, so d overflows f16 to infinity) -- the codes of such blocks are
    formed by per-element division rather than by the block reciprocal."""
    rows, n = 6, 512
    g = np.random.Generator(np.random.PCG64(77))
    x = g.standard_normal((rows, n))
    x[0, :] = 0.0
    x[0, 0] = 1.0
    x[0, 32:64] = 1e-35 * g.uniform(0.5, 1.0, size=32)
    x[0, 64:96] = 3e-39 * g.uniform(0.5, 1.0, size=32)
    x[1, 96:128] *= 1e-33
    gamma = 1.0 + 0.1 * g.standard_normal(n)
    gamma[128:160] = 1e33
    gamma[160:192] *= 1e-30
    x = wl.to_f32(x) if dtype == "f32" else wl.to_bf16_bits(x)
    gamma = wl.to_f32(gamma) if dtype == "f32" else wl.to_bf16_bits(gamma)
    assert mrn.mrn_force_geometry(geom) == 0
    gu.parity_q8_1(x, gamma, 1e-6, dtype, what=f"q8 extreme magnitudes {dtype} {geom}")


GEOMS = [   # (geometry, n for f32, n for bf16); 0 = not coverable
    ({"kind": 1, "lanes_per_row": 32, "k": 8}, 1024, 2048),
    ({"kind": 1, "lanes_per_row": 8, "k": 2}, 64, 128),
    ({"kind": 1, "lanes_per_row": 4, "k": 4}, 0, 128),
    ({"kind": 2, "k": 2, "threads": 64, "cluster": 4}, 2048, 4096),
    ({"kind": 3, "threads": 96}, 2560, 2560),
    ({"kind": 3, "threads": 64, "cluster": 5}, 8192, 16384),   # blocks never straddle CTAs
    ({"kind": 4, "k": 1, "threads": 128, "stages": 2, "groups": 2, "ctas": 5}, 256, 512),
    ({"kind": 4, "k": 4, "threads": 256, "stages": 2, "groups": 2}, 2048, 4096),
    ({"kind": 5, "k": 1, "threads": 128}, 4096, 4096),
    ({"kind": 5, "k": 2, "threads": 64}, 4000, 4000),
    ({"kind": 5, "k": 2, "threads": 96}, 6144, 6112),
    ({"kind": 5, "k": 1, "threads": 32}, 32, 1024),
    ({"kind": 5, "k": 1, "threads": 256, "stages": 2, "groups": 2}, 4096, 4096),
    ({"kind": 5, "k": 2, "threads": 128, "stages": 2, "groups": 2, "ctas": 5}, 4000, 4064),
    ({"kind": 5, "k": 1, "threads": 96, "stages": 3, "groups": 1, "ctas": 3}, 3072, 2976),
    ({"kind": 5, "k": 2, "threads": 64, "stages": 4, "groups": 2, "ctas": 1}, 2048, 1024),
]


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("geom,n32,n16", GEOMS, ids=[str(i) for i in range(len(GEOMS))])
def test_forced_geometries(geom, n32, n16, dtype):
    n = n32 if dtype == "f32" else n16
    if n == 0:
        pytest.skip("4 lanes cannot hold an f32 block of 8 vectors")
    assert mrn.mrn_force_geometry(geom) == 0
    d = wl.random_rows(41 + n, 37, n, dtype, scale=0.01)
    gu.parity_q8_1(d["x"], d["gamma"], 1e-5, dtype, what=f"q8 forced {geom}")


def test_warp_geometry_must_hold_whole_blocks():
    assert mrn.mrn_force_geometry({"kind": 1, "lanes_per_row": 4, "k": 8}) == 0
    with pytest.raises(mrn.MrnError):        # 4 lanes cannot hold a block of 8 f32 vectors
        mrn.mrn_query_geometry(5, 64, 128, mrn.MRN_F32, True)


@pytest.mark.parametrize("dtype", DTYPES)
def test_unaligned_rows_and_wide_rows(dtype):
    d = wl.random_rows(43, 5, 4096, dtype)
    gu.parity_q8_1(d["x"], d["gamma"], 1e-6, dtype, what="q8 unaligned", x_offset=1)
    d = wl.random_rows(44, 3, 200000 if dtype == "f32" else 300000, dtype)
    assert mrn.mrn_query_geometry(5, 3, d["x"].shape[1], gu.code(dtype), True)["kind"] == \
        mrn.MRN_GEOM_STREAM
    gu.parity_q8_1(d["x"], d["gamma"], 1e-6, dtype, what="q8 wide")


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("y_offset", [4, 8, 12])
def test_staged_blocks_at_unaligned_output(dtype, y_offset):
    """Blocks written from 4 (8, 12) bytes past a 16-byte boundary: the staged
    kernel copies such rows out word by word rather than by one bulk copy."""
    rows, n = 300, 4096
    assert mrn.mrn_query_geometry(5, rows, n, gu.code(dtype), True)["stages"] > 0
    d = wl.random_rows(46 + y_offset, rows, n, dtype)
    gu.parity_q8_1(d["x"], d["gamma"], 1e-6, dtype, what=f"q8 output +{y_offset}",
                   y_offset=y_offset)


def test_tensor_api_layout():
    d = wl.random_rows(45, 4, 128, "f32")
    x, g = gu.to_device(d["x"], "f32"), gu.to_device(d["gamma"], "f32")
    blocks = mrn.rmsnorm_q8_1(x, g, 1e-6)
    torch.cuda.synchronize()
    assert blocks.shape == (4, 4, 36) and blocks.dtype == torch.uint8
    dq, sq, q = gu.decode_q8_1(blocks.cpu().numpy())
    dd = np.repeat(dq.view(np.float16).astype(np.float64), 32, axis=1)
    y = mrn.rmsnorm(x, g, 1e-6).cpu().numpy().astype(np.float64)
    assert np.all(np.abs(q * dd - y) <= 0.5 * dd * 1.01 + 1e-3 * np.abs(y))   # dequantised
