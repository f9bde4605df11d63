"""GPU parity on rows that are not 16-byte aligned: a row pitch n * s that is
not a multiple of 16 bytes on aligned buffers, and buffers offset by 1..3
elements (every row operand and output alike, or not).  Batches of the plain,
then-add, then-add-scale and sandwich operations whose row operands share one
offset take the edge-staged kernel (16-byte granules covering each row, edge
elements masked and stored one by one); the rest move element-wise.  Every
output is compared with the oracle element by element inside guard bands;
the edge-staged kernel on aligned rows is bit-identical to the aligned
staged kernel of the same shape."""
import numpy as np
import pytest
import torch

import gpu_util as gu
import oracle
from dual_epsilon_sandwich_gb300 import mrn
from dual_epsilon_sandwich_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DTYPES = ("f32", "bf16")
WIDTHS = (7, 4097, 5121, 6655)
ROWS = 304          # two persistent waves' worth of rows: the staged kernels serve it


@pytest.fixture(autouse=True)
def _lib(gpu_lib):
    mrn.mrn_force_geometry(None)
    yield
    mrn.mrn_force_geometry(None)
    assert mrn.mrn_wait_timeouts() == 0


def offset_device(a, dtype, off):
    """a copied to the device `off` elements past a 256-byte-aligned start."""
    flat = np.concatenate([np.zeros(off, a.dtype), a.ravel()])
    t = gu.to_device(flat, dtype)
    v = t[off:]
    return v.view(a.shape) if a.ndim == 2 else v


def scale_device(value, dtype):
    host = np.array([value], dtype=np.float32)
    if dtype == "bf16":
        host = oracle.bf16_from_double(host.astype(np.float64))
    return gu.to_device(host, dtype), float(gu.widen(host, dtype)[0])


def run_ops(d, dtype, off_in, off_out, what):
    """The four operations on offset inputs/outputs, checked against the oracle."""
    rows, n = d["x"].shape
    x = offset_device(d["x"], dtype, off_in)
    r = offset_device(d["residual"], dtype, off_in)
    g = offset_device(d["gamma"], dtype, (off_in + 1) % 4)     # gamma at another offset
    g2 = offset_device(d["gamma2"], dtype, (off_in + 3) % 4)
    X, R = gu.widen(d["x"], dtype), gu.widen(d["residual"], dtype)
    Gm, G2 = gu.widen(d["gamma"], dtype), gu.widen(d["gamma2"], dtype)
    e = float(np.float32(1e-5))
    p = oracle.rmsnorm(X, Gm, e)

    y = gu.Guarded(rows, n, dtype, offset_elems=off_out)
    assert gu.call_rmsnorm(x, g, y, rows, n, 1e-5, dtype) == 0
    out = gu.Guarded(rows, n, dtype, offset_elems=off_out)
    assert gu.call_then_add(x, g, r, out, rows, n, 1e-5, dtype) == 0
    sc_t, sc = scale_device(-0.75, dtype)
    outs = gu.Guarded(rows, n, dtype, offset_elems=off_out)
    assert gu.call_then_add_scale(x, g, r, sc_t, outs, rows, n, 1e-5, dtype) == 0
    s = gu.Guarded(rows, n, dtype, offset_elems=off_out)
    o = gu.Guarded(rows, n, dtype, offset_elems=off_out)
    assert gu.call_sandwich(x, r, g, g2, s, o, rows, n, 1e-8, 1e-5, dtype) == 0
    torch.cuda.synchronize()
    for buf, name in ((y, "rmsnorm"), (out, "then_add"), (outs, "then_add_scale"),
                      (s, "stream"), (o, "normed")):
        buf.check(f"{what} {name}")
    want_t = oracle.rmsnorm_then_add(X, Gm, R, e)
    want_ts = oracle.rmsnorm_then_add_scale(X, Gm, R, sc, e)
    summands = np.abs(p) + np.abs(R)
    if dtype == "f32":
        gu.check_f32_norm(y.host(), p, f"{what} rmsnorm")
        gu.check_f32_sum(out.host(), want_t, summands, f"{what} then_add")
        gu.check_f32_sum(outs.host(), want_ts, summands * abs(sc), f"{what} then_add_scale")
    else:
        gu.check_bf16(y.host(), p, np.abs(p), f"{what} rmsnorm")
        gu.check_bf16(out.host(), want_t, summands, f"{what} then_add")
        gu.check_bf16(outs.host(), want_ts, summands * abs(sc), f"{what} then_add_scale")
    gu.check_sandwich(s.host(), o.host(), d["x"], d["residual"], d["gamma"], d["gamma2"],
                      1e-8, 1e-5, dtype, f"{what} sandwich")


def expect_edge(op, n, dtype, same):
    """Whether the library picks the edge-staged kernel for this batch."""
    g = mrn.mrn_query_geometry(op, ROWS, n, gu.code(dtype), 2 if same else 0)
    return g["edge"] == 1


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("n", WIDTHS)
@pytest.mark.parametrize("off", (0, 1, 2, 3))
def test_rows_at_one_offset(n, off, dtype):
    """Every row operand and output at the same offset within 16 bytes (off = 0:
    aligned buffers, a pitch that is not a multiple of 16 bytes)."""
    if off == 0 and (n * gu.elem_bytes(dtype)) % 16 == 0:
        pytest.skip("aligned rows")
    d = wl.random_rows(9000 + n + off, ROWS, n, dtype)
    if n > 256:
        for op in (mrn.MRN_OP_RMSNORM, mrn.MRN_OP_THEN_ADD, mrn.MRN_OP_THEN_ADD_SCALE,
                   mrn.MRN_OP_SANDWICH):
            assert expect_edge(op, n, dtype, True), (op, n, dtype)
    run_ops(d, dtype, off, off, f"{ROWS}x{n} +{off}")


@pytest.mark.parametrize("dtype", DTYPES)
def test_inputs_and_outputs_at_different_offsets(dtype):
    """Row operands at one offset, outputs at another: element-wise path."""
    n = 5121
    assert not expect_edge(mrn.MRN_OP_SANDWICH, n, dtype, False)
    d = wl.random_rows(9101, ROWS, n, dtype)
    run_ops(d, dtype, 1, 0, f"{ROWS}x{n} in +1 out +0")
    run_ops(d, dtype, 0, 3, f"{ROWS}x{n} in +0 out +3")


@pytest.mark.parametrize("dtype", DTYPES)
def test_in_place_unaligned(dtype):
    """Exact aliasing on unaligned rows (out_stream == residual, y == x, out ==
    residual) gives the out-of-place bits."""
    rows, n, off = ROWS, 6655, 1
    d = wl.random_rows(9102, rows, n, dtype)
    x, r = offset_device(d["x"], dtype, off), offset_device(d["residual"], dtype, off)
    g, g2 = gu.to_device(d["gamma"], dtype), gu.to_device(d["gamma2"], dtype)
    assert expect_edge(mrn.MRN_OP_SANDWICH, n, dtype, True)
    ref_s = offset_device(np.zeros_like(d["x"]), dtype, off)
    ref_o = offset_device(np.zeros_like(d["x"]), dtype, off)
    assert gu.call_sandwich(x, r, g, g2, ref_s, ref_o, rows, n, 1e-8, 1e-5, dtype) == 0
    r1 = offset_device(d["residual"], dtype, off)
    o1 = offset_device(np.zeros_like(d["x"]), dtype, off)
    assert gu.call_sandwich(x, r1, g, g2, r1, o1, rows, n, 1e-8, 1e-5, dtype) == 0
    ref_y = offset_device(np.zeros_like(d["x"]), dtype, off)
    assert gu.call_rmsnorm(x, g, ref_y, rows, n, 1e-5, dtype) == 0
    x1 = offset_device(d["x"], dtype, off)
    assert gu.call_rmsnorm(x1, g, x1, rows, n, 1e-5, dtype) == 0
    ref_t = offset_device(np.zeros_like(d["x"]), dtype, off)
    assert gu.call_then_add(x, g, r, ref_t, rows, n, 1e-5, dtype) == 0
    r2 = offset_device(d["residual"], dtype, off)
    assert gu.call_then_add(x, g, r2, r2, rows, n, 1e-5, dtype) == 0
    torch.cuda.synchronize()
    it = torch.int16 if dtype == "bf16" else torch.int32
    for a, b, what in ((r1, ref_s, "stream == residual"), (o1, ref_o, "normed"),
                       (x1, ref_y, "y == x"), (r2, ref_t, "out == residual")):
        assert torch.equal(a.view(it), b.view(it)), what
    gu.check_sandwich(gu.to_host(ref_s, dtype), gu.to_host(ref_o, dtype), d["x"],
                      d["residual"], d["gamma"], d["gamma2"], 1e-8, 1e-5, dtype, "in place")


def _edge_geometry(threads, k, ctas=0):
    return {"kind": mrn.MRN_GEOM_TMA, "vec": 0, "k": k, "threads": threads, "cluster": 1,
            "lanes_per_row": 0, "stages": 2, "ctas": ctas, "groups": 2, "edge": 1}


@pytest.mark.parametrize("dtype", DTYPES)
def test_edge_kernel_on_aligned_rows_is_the_staged_kernel(dtype):
    """On 16-byte-aligned rows (offset 0, whole granules) the edge-staged kernel
    does the aligned staged kernel's arithmetic: with the same threads and
    register slots every thread sums the same elements in the same order, so
    the outputs are bit-identical."""
    rows = ROWS
    n, per, k = (6656, 224, 8) if dtype == "f32" else (8192, 160, 7)
    d = wl.random_rows(9103, rows, n, dtype)
    x, r = gu.to_device(d["x"], dtype), gu.to_device(d["residual"], dtype)
    g, g2 = gu.to_device(d["gamma"], dtype), gu.to_device(d["gamma2"], dtype)
    outs = {}
    for edge in (0, 1):
        geo = _edge_geometry(2 * per, k)
        geo["edge"] = edge
        assert mrn.mrn_force_geometry(geo) == 0, geo
        s, o = torch.empty_like(x), torch.empty_like(x)
        assert gu.call_sandwich(x, r, g, g2, s, o, rows, n, 1e-8, 1e-5, dtype) == 0
        y = torch.empty_like(x)
        assert gu.call_rmsnorm(x, g, y, rows, n, 1e-5, dtype) == 0
        torch.cuda.synchronize()
        outs[edge] = (s, o, y)
    mrn.mrn_force_geometry(None)
    it = torch.int16 if dtype == "bf16" else torch.int32
    for a, b in zip(outs[0], outs[1]):
        assert torch.equal(a.view(it), b.view(it))


@pytest.mark.parametrize("ctas", (100, 13, 8))
def test_edge_grid_is_a_multiple_of_eight(ctas):
    """A forced persistent grid that is not a multiple of 8 CTAs is rounded
    down (a CTA's rows must share one offset); results stay exact."""
    rows, n, dtype = 1000, 4097, "f32"
    d = wl.random_rows(9104 + ctas, rows, n, dtype)
    assert mrn.mrn_force_geometry(_edge_geometry(2 * 288, 4, ctas)) == 0
    try:
        run_ops(d, dtype, 2, 2, f"{rows}x{n} ctas {ctas}")
    finally:
        mrn.mrn_force_geometry(None)


def test_prefill_width_minus_one_full_size():
    """4096 x 6655 f32 sandwich (the benchmark's shape with a pitch of 26,620
    bytes), sampled rows against the oracle, the rest finite."""
    rows, n = 4096, 6655
    w = wl.sandwich_prefill(rows=rows, n=n)
    a = w.arrays
    assert expect_edge(mrn.MRN_OP_SANDWICH, n, "f32", True)
    sample = gu.sample_rows(rows, 96, 9105)
    gu.parity_sandwich(a["block_out"], a["residual"], a["gamma_post"], a["gamma_pre"], w.eps,
                       w.eps_pre, "f32", rows_sample=sample, what="4096x6655 sandwich")


@pytest.mark.parametrize("n,forced", [(6655, None), (6656, _edge_geometry(512, 7)),
                                      (6656, dict(_edge_geometry(832, 4), edge=0))])
def test_staged_sandwich_one_exchange_rows_that_cancel(n, forced):
    """The staged f32 sandwich reduces the stream's three first-pass sums with
    the first norm's (after each warp group's first row) and reduces the
    stored stream again only where those sums cancel.  1216 rows (four per
    warp group), every third row's block output nearly cancelling its
    residual: both kinds of rows, and first rows, against the oracle."""
    rows = 1216
    g = np.random.default_rng(4500 + n)
    r = g.standard_normal((rows, n))
    gp = 1 + 0.1 * g.standard_normal(n)
    gq = 1 + 0.1 * g.standard_normal(n)
    b = g.standard_normal((rows, n)) * 2.0
    for i in range(0, rows, 3):
        b[i] = -r[i] * (1 + 1e-3 * g.standard_normal(n)) / gp * 3.0
    f = [np.asarray(v, dtype=np.float32) for v in (b, r, gp, gq)]
    if forced is not None:
        assert mrn.mrn_force_geometry(forced) == 0
    geo = mrn.mrn_query_geometry(mrn.MRN_OP_SANDWICH, rows, n, mrn.MRN_F32, True)
    assert geo["kind"] == mrn.MRN_GEOM_TMA
    try:
        gu.parity_sandwich(*f, 1e-8, 1e-5, "f32", what=f"staged one exchange {rows}x{n}")
    finally:
        mrn.mrn_force_geometry(None)
