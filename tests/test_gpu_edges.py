"""GPU parity on edge cases: tiny and ragged rows (the d=2 silent-wrong-answer
class the dormouse page reports), misaligned rows, in-place aliasing, every
geometry variant forced on the same inputs, cluster sizes 1..16, the looped
fallback for very wide rows, epsilon routing, determinism and streams."""
import numpy as np
import pytest
import torch

import gpu_util as gu
import oracle
from dual_epsilon_sandwich_gb300 import mrn
from dual_epsilon_sandwich_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DTYPES = ("f32", "bf16")


@pytest.fixture(autouse=True)
def _lib(gpu_lib):
    mrn.mrn_force_geometry(None)
    yield
    mrn.mrn_force_geometry(None)


def rows_data(seed, rows, n, dtype, scale=1.0):
    return wl.random_rows(seed, rows, n, dtype, scale)


def all_ops(d, dtype, what, sample=None):
    x, r, g, g2 = d["x"], d["residual"], d["gamma"], d["gamma2"]
    gu.parity_rmsnorm(x, g, 1e-5, dtype, sample, what=f"{what} rmsnorm")
    gu.parity_then_add(x, g, r, 1e-6, dtype, sample, what=f"{what} then_add")
    gu.parity_sandwich(x, r, g, g2, 1e-8, 1e-5, dtype, sample, what=f"{what} sandwich")


SMALL_N = [1, 2, 3, 4, 5, 7, 8, 9, 15, 16, 17, 31, 32, 33, 63, 64, 65, 127, 128, 129, 255, 256,
           257, 260, 1000, 2049]


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("n", SMALL_N)
def test_small_and_ragged_rows_every_output_written(n, dtype):
    for rows in (1, 2, 3, 4, 5, 33):
        all_ops(rows_data(1000 * n + rows, rows, n, dtype), dtype, f"{rows}x{n}")


def test_two_element_rows_by_hand():
    """x = [3, 4] -> [3, 4] / sqrt(12.5 + eps); x = [1, -1] -> +-1/sqrt(1 + eps), at rows 1..4."""
    x = np.array([[3, 4], [1, -1], [0, 0], [-4, 3]], dtype=np.float32)
    for rows in (1, 2, 3, 4):
        dx = gu.to_device(x[:rows], "f32")
        dg = gu.to_device(np.ones(2, np.float32), "f32")
        y = gu.Guarded(rows, 2, "f32")
        assert gu.call_rmsnorm(dx, dg, y, rows, 2, 1e-5, "f32") == 0
        torch.cuda.synchronize()
        y.check(f"n=2 rows={rows}")
        e = float(np.float32(1e-5))
        want = np.array([[3, 4] / np.sqrt(12.5 + e), [1, -1] / np.sqrt(1 + e), [0, 0],
                         [-4, 3] / np.sqrt(12.5 + e)])[:rows]
        gu.check_f32_norm(y.host(), want, f"n=2 rows={rows}")


@pytest.mark.parametrize("dtype", DTYPES)
def test_rows_not_16_byte_aligned(dtype):
    """Pointers offset by one element: rows move element-wise, same results."""
    rows, n = 5, 6656
    d = rows_data(7, rows, n, dtype)
    e = gu.elem_bytes(dtype)

    def shifted(a):
        t = gu.to_device(np.concatenate([np.zeros(1, a.dtype), a.ravel()]), dtype)
        return t[1:].view(a.shape) if a.ndim == 2 else t[1:]

    x, r, g, g2 = (shifted(d[k]) for k in ("x", "residual", "gamma", "gamma2"))
    assert x.data_ptr() % 16 != 0
    y = gu.Guarded(rows, n, dtype, offset_elems=1)
    assert gu.call_rmsnorm(x, g, y, rows, n, 1e-5, dtype) == 0
    torch.cuda.synchronize()
    y.check("misaligned rmsnorm")
    want = oracle.rmsnorm(gu.widen(d["x"], dtype), gu.widen(d["gamma"], dtype),
                          float(np.float32(1e-5)))
    if dtype == "f32":
        gu.check_f32_norm(y.host(), want, "misaligned rmsnorm")
    else:
        gu.check_bf16(y.host(), want, np.abs(want), "misaligned rmsnorm")
    s = gu.Guarded(rows, n, dtype, offset_elems=1)
    o = gu.Guarded(rows, n, dtype, offset_elems=1)
    assert gu.call_sandwich(x, r, g, g2, s, o, rows, n, 1e-8, 1e-5, dtype) == 0
    torch.cuda.synchronize()
    s.check("misaligned stream")
    o.check("misaligned normed")
    gu.check_sandwich(s.host(), o.host(), d["x"], d["residual"], d["gamma"], d["gamma2"],
                      1e-8, 1e-5, dtype, "misaligned sandwich")
    assert e in (2, 4)


@pytest.mark.parametrize("dtype", DTYPES)
def test_in_place_aliasing(dtype):
    rows, n = 7, 2048
    d = rows_data(8, rows, n, dtype)
    x, r, g, g2 = (gu.to_device(d[k], dtype) for k in ("x", "residual", "gamma", "gamma2"))

    ref_y = torch.empty_like(x)
    assert gu.call_rmsnorm(x, g, ref_y, rows, n, 1e-5, dtype) == 0
    xi = x.clone()
    assert gu.call_rmsnorm(xi, g, xi, rows, n, 1e-5, dtype) == 0            # y == x
    ref_o = torch.empty_like(x)
    assert gu.call_then_add(x, g, r, ref_o, rows, n, 1e-5, dtype) == 0
    ri = r.clone()
    assert gu.call_then_add(x, g, ri, ri, rows, n, 1e-5, dtype) == 0        # out == residual
    xo = x.clone()
    assert gu.call_then_add(xo, g, r, xo, rows, n, 1e-5, dtype) == 0        # out == x
    ref_s, ref_n = torch.empty_like(x), torch.empty_like(x)
    assert gu.call_sandwich(x, r, g, g2, ref_s, ref_n, rows, n, 1e-8, 1e-5, dtype) == 0
    r1, n1 = r.clone(), torch.empty_like(x)
    assert gu.call_sandwich(x, r1, g, g2, r1, n1, rows, n, 1e-8, 1e-5, dtype) == 0   # stream == residual
    b2, n2 = x.clone(), torch.empty_like(x)
    assert gu.call_sandwich(b2, r, g, g2, b2, n2, rows, n, 1e-8, 1e-5, dtype) == 0   # stream == block_out
    b3, s3 = x.clone(), torch.empty_like(x)
    assert gu.call_sandwich(b3, r, g, g2, s3, b3, rows, n, 1e-8, 1e-5, dtype) == 0   # normed == block_out
    r4, s4 = r.clone(), torch.empty_like(x)
    assert gu.call_sandwich(x, r4, g, g2, s4, r4, rows, n, 1e-8, 1e-5, dtype) == 0   # normed == residual
    torch.cuda.synchronize()

    def same(a, b, what):
        assert torch.equal(a.view(torch.int16 if dtype == "bf16" else torch.int32),
                           b.view(torch.int16 if dtype == "bf16" else torch.int32)), what

    same(xi, ref_y, "y == x")
    same(ri, ref_o, "out == residual")
    same(xo, ref_o, "out == x")
    same(r1, ref_s, "stream == residual (stream)")
    same(n1, ref_n, "stream == residual (normed)")
    same(b2, ref_s, "stream == block_out (stream)")
    same(n2, ref_n, "stream == block_out (normed)")
    same(s3, ref_s, "normed == block_out (stream)")
    same(b3, ref_n, "normed == block_out (normed)")
    same(s4, ref_s, "normed == residual (stream)")
    same(r4, ref_n, "normed == residual (normed)")
    gu.parity_then_add(d["x"], d["gamma"], d["residual"], 1e-5, dtype)


# Every geometry variant on shapes it can cover, including ragged coverage.
FORCED = [
    ({"kind": 1, "lanes_per_row": 32, "k": 8}, 250),
    ({"kind": 1, "lanes_per_row": 32, "k": 3}, 90),
    ({"kind": 1, "lanes_per_row": 16, "k": 5}, 77),
    ({"kind": 1, "lanes_per_row": 4, "k": 7}, 25),
    ({"kind": 1, "lanes_per_row": 1, "k": 2}, 2),
    ({"kind": 2, "k": 1, "threads": 1024, "cluster": 1}, 1000),
    ({"kind": 2, "k": 2, "threads": 96, "cluster": 5}, 950),
    ({"kind": 2, "k": 3, "threads": 64, "cluster": 2}, 380),
    ({"kind": 2, "k": 4, "threads": 512, "cluster": 1}, 2048),
    ({"kind": 2, "k": 5, "threads": 256, "cluster": 3}, 3800),
    ({"kind": 2, "k": 6, "threads": 32, "cluster": 7}, 1300),
    ({"kind": 2, "k": 7, "threads": 224, "cluster": 1}, 1500),
    ({"kind": 2, "k": 8, "threads": 256, "cluster": 16}, 32768),
    ({"kind": 3, "threads": 32}, 1999),
    ({"kind": 3, "threads": 512}, 7000),
    ({"kind": 3, "threads": 64, "cluster": 3}, 1999),       # slices of 32-load multiples,
    ({"kind": 3, "threads": 256, "cluster": 16}, 7000),     # the last ones short or empty
    ({"kind": 3, "threads": 512, "cluster": 16}, 65536),
]


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("geom,nvec", FORCED, ids=[str(i) for i in range(len(FORCED))])
def test_forced_geometry(geom, nvec, dtype):
    vec = 4 if dtype == "f32" else 8
    for n, g in ((nvec * vec, geom), (nvec, dict(geom, vec=1))):
        assert mrn.mrn_force_geometry(g) == 0
        rows = 3 if n * 3 < (1 << 22) else 2
        all_ops(rows_data(n + rows, rows, n, dtype), dtype, f"forced {g} n={n}")
        mrn.mrn_force_geometry(None)


@pytest.mark.parametrize("cluster", [1, 2, 3, 4, 5, 6, 7, 8, 12, 16])
def test_cluster_split_decode_row(cluster):
    """One n=6656 row split over `cluster` CTAs with a DSMEM reduction."""
    per = -(-1664 // cluster)
    k = 1 if per <= 1024 else 2
    threads = -(-per // (32 * k)) * 32
    assert mrn.mrn_force_geometry({"kind": 2, "k": k, "threads": threads,
                                   "cluster": cluster}) == 0
    w = wl.sandwich_decode()
    a = w.arrays
    gu.parity_sandwich(a["block_out"], a["residual"], a["gamma_post"], a["gamma_pre"], w.eps,
                       w.eps_pre, "f32", what=f"cluster {cluster}")
    d = rows_data(9, 3, 6656, "bf16")
    gu.parity_sandwich(d["x"], d["residual"], d["gamma"], d["gamma2"], 1e-8, 1e-5, "bf16",
                       what=f"bf16 cluster {cluster}")


@pytest.mark.parametrize("dtype,n", [("f32", 200000), ("f32", 140001), ("bf16", 300000),
                                     ("bf16", 270001)])
def test_wide_rows_use_the_looped_fallback(dtype, n):
    g = mrn.mrn_query_geometry(0, 3, n, gu.code(dtype), True)
    assert g["kind"] == mrn.MRN_GEOM_STREAM and g["cluster"] == 16   # (few rows)
    all_ops(rows_data(n, 3, n, dtype), dtype, f"wide n={n}")


def test_widest_row_batch():
    """256 rows of 1 MB (f32, n = 262144): the looped kernel over clusters of 8,
    sampled rows of all three operations against the oracle, every output
    written (guard bands, sentinels)."""
    rows, n = 256, 262144
    g = mrn.mrn_query_geometry(2, rows, n, mrn.MRN_F32, True)
    assert g["kind"] == mrn.MRN_GEOM_STREAM and g["cluster"] == 8
    d = rows_data(262144, rows, n, "f32")
    sample = gu.sample_rows(rows, 12, 2621)
    all_ops(d, "f32", f"widest {rows}x{n}", sample)


@pytest.mark.parametrize("dtype,n,cluster", [("f32", 16384, 2), ("f32", 32768, 4),
                                             ("f32", 65536, 8), ("f32", 131072, 16),
                                             ("bf16", 65536, 4), ("bf16", 262144, 16)])
def test_wide_row_batches_use_the_cluster_staged_kernel(dtype, n, cluster):
    """Batches (rows >= the SM count) of rows of 2049 .. 16 x 2048 loads take the
    cluster-staged kernel, a cluster of 2 .. 16 CTAs per row, for the plain,
    then-add, then-add-scale and sandwich operations (the sandwich's cluster is
    doubled from 8); every output matches the oracle."""
    rows = 160
    for op in (0, 1, 2, 4):
        g = mrn.mrn_query_geometry(op, rows, n, gu.code(dtype), True)
        want = cluster * 2 if op == 2 and cluster == 8 else cluster
        assert (g["kind"], g["cluster"], g["groups"]) == (mrn.MRN_GEOM_TMA, want, 1), (op, g)
    d = rows_data(n + 11, rows, n, dtype)
    all_ops(d, dtype, f"cluster-staged {rows}x{n}")
    gu.parity_then_add_scale(d["x"], d["gamma"], d["residual"], 0.75, 1e-5, dtype,
                             what=f"cluster-staged {rows}x{n} then_add_scale")
    assert mrn.mrn_wait_timeouts() == 0


@pytest.mark.parametrize("rows,n,cluster", [(2048, 16384, 4), (2048, 10240, 3), (2048, 8196, 3)])
def test_plain_f32_wide_batches_in_register_clusters(rows, n, cluster):
    """Plain f32 batches of 2048+ rows wider than 2048 loads: the register kernel
    at eight slots per thread, a cluster of ceil(loads / 1024) CTAs per row (3 at
    n = 10240 and 8196: slices of 864 / 704 loads, the last one shorter); sampled
    rows against the oracle."""
    g = mrn.mrn_query_geometry(0, rows, n, mrn.MRN_F32, True)
    assert (g["kind"], g["cluster"], g["k"]) == (mrn.MRN_GEOM_CTA, cluster, 8)
    d = rows_data(n + 21, rows, n, "f32")
    gu.parity_rmsnorm(d["x"], d["gamma"], 1e-5, "f32", gu.sample_rows(rows, 48, n),
                      what=f"register cluster {rows}x{n}")
    assert mrn.mrn_wait_timeouts() == 0


def test_epsilon_routing_is_visible():
    """Block output of mean square 1e-8 and a stream of mean square ~1e-6:
    eps_post = 1e-8 and eps_pre = 1e-5 both move the outputs, and an oracle with
    the two swapped is far outside the tolerance the GPU meets."""
    g = np.random.Generator(np.random.PCG64(77))
    rows, n = 8, 4096
    b = (1e-4 * np.where(g.random((rows, n)) < 0.5, -1.0, 1.0)).astype(np.float32)
    r = (1e-3 * g.standard_normal((rows, n))).astype(np.float32)
    gp = (1e-3 * (1.0 + 0.1 * g.standard_normal(n))).astype(np.float32)
    gq = (1.0 + 0.1 * g.standard_normal(n)).astype(np.float32)
    gu.parity_sandwich(b, r, gp, gq, 1e-8, 1e-5, "f32", what="routing")
    db, dr, dgp, dgq = (gu.to_device(a, "f32") for a in (b, r, gp, gq))
    s, o = torch.empty_like(db), torch.empty_like(db)
    assert gu.call_sandwich(db, dr, dgp, dgq, s, o, rows, n, 1e-8, 1e-5, "f32") == 0
    torch.cuda.synchronize()
    ws, wo = oracle.norm_residual_norm(b, r, gp, gq, float(np.float32(1e-5)),
                                       float(np.float32(1e-8)))
    with pytest.raises(AssertionError):
        gu.check_f32_norm(gu.to_host(o, "f32"), wo, "swapped eps must be detectable")


@pytest.mark.parametrize("scale", [1e-20, 1e-9, 1e-3, 1e3, 1e15])
def test_row_magnitudes(scale):
    """From epsilon-dominated rows (mean square << eps) to large ones."""
    for dtype in DTYPES:
        all_ops(rows_data(5, 6, 6656, dtype, scale=scale), dtype, f"scale {scale}")


def test_all_ones_gamma_entry_norm():
    """The entry norm binds an all-ones gamma (Chapter 12, section 12.3)."""
    d = rows_data(10, 4, 6656, "f32")
    gu.parity_rmsnorm(d["x"], np.ones(6656, np.float32), 1e-5, "f32")


def test_deterministic_bits():
    d = rows_data(11, 64, 6656, "f32")
    x, r, g, g2 = (gu.to_device(d[k], "f32") for k in ("x", "residual", "gamma", "gamma2"))
    outs = []
    for _ in range(2):
        s, o = torch.empty_like(x), torch.empty_like(x)
        assert gu.call_sandwich(x, r, g, g2, s, o, 64, 6656, 1e-8, 1e-5, "f32") == 0
        outs.append((s, o))
    torch.cuda.synchronize()
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


def test_non_default_stream_and_launch_count():
    d = rows_data(12, 16, 4096, "bf16")
    x, g = gu.to_device(d["x"], "bf16"), gu.to_device(d["gamma"], "bf16")
    side = torch.cuda.Stream()
    before = mrn.mrn_launch_count()
    with torch.cuda.stream(side):
        y = torch.empty_like(x)
        assert gu.call_rmsnorm(x, g, y, 16, 4096, 1e-6, "bf16") == 0
    side.synchronize()
    assert mrn.mrn_launch_count() == before + 1
    want = oracle.rmsnorm(gu.widen(d["x"], "bf16"), gu.widen(d["gamma"], "bf16"),
                          float(np.float32(1e-6)))
    gu.check_bf16(gu.to_host(y, "bf16"), want, np.abs(want), "side stream")
    assert mrn.mrn_rmsnorm(0, 0, 0, 0, 4096, 1e-6, mrn.MRN_BF16, 0) == 0
    assert mrn.mrn_launch_count() == before + 1


def test_tensor_convenience_api():
    d = rows_data(13, 5, 768, "f32")
    x, r, g, g2 = (gu.to_device(d[k], "f32") for k in ("x", "residual", "gamma", "gamma2"))
    y = mrn.rmsnorm(x, g, 1e-5)
    s, o = mrn.norm_residual_norm(x, r, g, g2)
    torch.cuda.synchronize()
    want = oracle.rmsnorm(d["x"].astype(np.float64), d["gamma"].astype(np.float64),
                          float(np.float32(1e-5)))
    gu.check_f32_norm(y.cpu().numpy(), want, "tensor api")
    with pytest.raises(mrn.MrnError):
        mrn.rmsnorm(x, g, 0.0)
    base = torch.empty(5 * 768 + 1, device="cuda")
    x2 = base[:5 * 768].view(5, 768)
    x2.copy_(x)
    with pytest.raises(mrn.MrnError) as exc:          # output overlaps x by all but one element
        mrn.rmsnorm_then_add(x2, g, r, 1e-5, out=base[1:].view(5, 768))
    assert exc.value.status == mrn.MRN_ERR_ALIASING


# The persistent TMA-staged kernel: stages 1..4, persistent grids from one CTA
# (every row through one pipeline) to the full device, ragged register coverage.
FORCED_TMA = [
    ({"kind": 4, "k": 4, "threads": 416, "stages": 3}, 1664, 1000),
    ({"kind": 4, "k": 1, "threads": 1024, "stages": 1, "ctas": 7}, 1024, 50),
    ({"kind": 4, "k": 2, "threads": 96, "stages": 4, "ctas": 5}, 190, 333),
    ({"kind": 4, "k": 8, "threads": 256, "stages": 2}, 2000, 400),
    ({"kind": 4, "k": 3, "threads": 64, "stages": 2, "ctas": 1}, 150, 37),
    ({"kind": 4, "k": 5, "threads": 128, "stages": 3, "ctas": 300}, 600, 7),
    ({"kind": 4, "k": 7, "threads": 512, "stages": 2, "groups": 2}, 1664, 1000),
    ({"kind": 4, "k": 4, "threads": 832, "stages": 2, "groups": 2}, 1664, 300),
    ({"kind": 4, "k": 4, "threads": 256, "stages": 4, "groups": 2, "ctas": 19}, 250, 500),
    ({"kind": 4, "k": 2, "threads": 192, "stages": 2, "groups": 2, "ctas": 3}, 190, 101),
    ({"kind": 4, "k": 1, "threads": 64, "stages": 4, "groups": 2, "ctas": 1}, 20, 9),
    # a cluster per row, each CTA staging a slice of it
    ({"kind": 4, "k": 2, "threads": 128, "stages": 2, "cluster": 4}, 1024, 300),
    ({"kind": 4, "k": 1, "threads": 64, "stages": 3, "cluster": 2, "ctas": 6}, 128, 101),
    ({"kind": 4, "k": 4, "threads": 256, "stages": 2, "cluster": 8}, 8192, 64),
    ({"kind": 4, "k": 2, "threads": 64, "stages": 1, "cluster": 16}, 2048, 40),
    ({"kind": 4, "k": 8, "threads": 128, "stages": 3, "cluster": 8}, 8192, 200),
    ({"kind": 4, "k": 4, "threads": 256, "stages": 6, "cluster": 4}, 4096, 77),
    ({"kind": 4, "k": 8, "threads": 32, "stages": 8, "cluster": 16}, 4096, 300),
]


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("geom,nvec,rows", FORCED_TMA, ids=[str(i) for i in range(len(FORCED_TMA))])
def test_forced_staged_kernel(geom, nvec, rows, dtype):
    n = nvec * (4 if dtype == "f32" else 8)
    assert mrn.mrn_force_geometry(geom) == 0
    g = mrn.mrn_query_geometry(2, rows, n, gu.code(dtype), True)
    assert g["kind"] == mrn.MRN_GEOM_TMA
    all_ops(rows_data(n * 7 + rows, rows, n, dtype), dtype, f"staged {geom} {rows}x{n}")
    mrn.mrn_force_geometry(None)
    assert mrn.mrn_wait_timeouts() == 0


def test_batch_kernel_choice_and_both_kernels():
    """Batches of aligned rows take the register kernel where it measured faster
    (f32 plain, then-add and sandwich at n = 6656 from 2048 rows, every
    operation at 512 loads per row) and the staged kernel elsewhere (the bf16
    sandwich past 512 loads); the same 2048 x 6656 batch through the automatic
    choice and through the staged kernel forced, every operation against the
    oracle."""
    assert [mrn.mrn_query_geometry(op, 4096, 6656, mrn.MRN_F32, True)["kind"]
            for op in (0, 1, 2)] == [mrn.MRN_GEOM_CTA] * 3
    assert mrn.mrn_query_geometry(2, 4096, 8192, mrn.MRN_BF16, True)["kind"] == mrn.MRN_GEOM_TMA
    for op in (0, 1, 2):
        assert mrn.mrn_query_geometry(op, 16384, 4096, mrn.MRN_BF16, True)["kind"] == \
            mrn.MRN_GEOM_CTA
    assert mrn.mrn_query_geometry(2, 1, 6656, mrn.MRN_F32, True)["kind"] == mrn.MRN_GEOM_CTA
    d = rows_data(14, 2048, 6656, "f32")
    all_ops(d, "f32", "auto 2048x6656")
    assert mrn.mrn_force_geometry({"kind": 4, "k": 4, "threads": 832, "stages": 2,
                                   "groups": 2}) == 0
    try:
        all_ops(d, "f32", "staged 2048x6656")
    finally:
        mrn.mrn_force_geometry(None)
    assert mrn.mrn_wait_timeouts() == 0


@pytest.mark.parametrize("rows,n", [(1, 6656), (4, 6656), (2048, 6656), (300, 768), (64, 200000)])
def test_programmatic_launch_chain_matches(rows, n):
    """A chain of dependent sandwich calls (each call's normed is the next
    call's block_out, its stream the next residual, updated in place) gives the
    same bits with programmatic dependent launch as without."""
    d = rows_data(15 + n, rows, n, "f32")
    g1, g2 = gu.to_device(d["gamma"], "f32"), gu.to_device(d["gamma2"], "f32")

    def chain(options):
        assert mrn.mrn_set_launch_options(options) == 0
        b = gu.to_device(d["x"], "f32")
        r = gu.to_device(d["residual"], "f32")
        o = torch.empty_like(b)
        for _ in range(6):
            assert gu.call_sandwich(b, r, g1, g2, r, o, rows, n, 1e-8, 1e-5, "f32") == 0
            b, o = o, b
        torch.cuda.synchronize()
        assert mrn.mrn_set_launch_options(mrn.MRN_LAUNCH_PDL) == 0   # the default
        return b, r

    b0, r0 = chain(0)
    b1, r1 = chain(mrn.MRN_LAUNCH_PDL)
    assert torch.equal(b0, b1) and torch.equal(r0, r1)
    assert mrn.mrn_wait_timeouts() == 0


@pytest.mark.parametrize("rows", [1, 2, 4])
def test_decode_sandwich_stream_that_cancels(rows):
    """The f32 register kernel forms the stream's sum of squares from three
    first-pass sums when they do not cancel, and reduces the stored stream
    again when they do.  Rows whose block output nearly cancels the residual
    (the stream about 1/50 of its summands) take the second reduction; the
    rows between them do not; both match the oracle."""
    n = 6656
    g = np.random.default_rng(4401 + rows)
    r = g.standard_normal((rows, n))
    gp = 1 + 0.1 * g.standard_normal(n)
    gq = 1 + 0.1 * g.standard_normal(n)
    b = g.standard_normal((rows, n)) * 2.0
    for i in range(0, rows, 2):                  # every other row cancels
        b[i] = -r[i] * (1 + 1e-3 * g.standard_normal(n)) / gp * 3.0
    f = [np.asarray(v, dtype=np.float32) for v in (b, r, gp, gq)]
    geo = mrn.mrn_query_geometry(mrn.MRN_OP_SANDWICH, rows, n, mrn.MRN_F32, True)
    assert geo["kind"] == mrn.MRN_GEOM_CTA and geo["cluster"] > 1
    gu.parity_sandwich(*f, 1e-8, 1e-5, "f32", what=f"cancelling {rows}x{n}")
    e1, e2 = float(np.float32(1e-8)), float(np.float32(1e-5))
    s, _ = oracle.norm_residual_norm(*(v.astype(np.float64) for v in f), e1, e2)
    p = oracle.rmsnorm(f[0].astype(np.float64), f[2].astype(np.float64), e1)
    r64 = f[1].astype(np.float64)
    mag = np.sum(p * p, axis=1) + 2 * np.abs(np.sum(p * r64, axis=1)) + np.sum(r64 * r64, axis=1)
    ratio = np.sum(s * s, axis=1) / mag          # the kernel's test: at least 1/2 or not
    assert np.all(ratio[0::2] < 0.1) and np.all(ratio[1::2] > 0.9)   # both paths taken
