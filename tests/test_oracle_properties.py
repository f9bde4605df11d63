"""Randomised properties of the CPU oracle (no GPU): laws the definitions
imply, over random shapes (tails included), scales and epsilons, so that a
mistake that the fixed pins happen to miss still fails here.  Each property
follows from the mathematics of the operation or from another oracle
function; none restates the formula it checks."""
import numpy as np
import pytest

import oracle

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

EPS = st.sampled_from([1e-8, 1e-6, 1e-5, 1e-3, 1.0])
SETTINGS = settings(max_examples=60, deadline=None, derandomize=True)


def draw_rows(seed, rows, n, scale):
    g = np.random.Generator(np.random.PCG64(seed))
    x = scale * g.standard_normal((rows, n))
    gamma = 1.0 + 0.1 * g.standard_normal(n)
    res = g.standard_normal((rows, n))
    return x, gamma, res, g


shapes = st.tuples(st.integers(0, 2**31 - 1), st.integers(1, 5), st.integers(1, 70),
                   st.sampled_from([1e-3, 1.0, 1e3]))


def prop_scale_law(orc, shape, eps, alpha):
    """y(alpha x; alpha^2 eps) = y(x; eps): the norm sees only x / rms."""
    seed, rows, n, scale = shape
    x, gamma, _, _ = draw_rows(seed, rows, n, scale)
    y1 = orc.rmsnorm(x, gamma, eps)
    y2 = orc.rmsnorm(alpha * x, gamma, alpha * alpha * eps)
    assert np.allclose(y2, y1, rtol=1e-12, atol=0.0)


def prop_odd_symmetry_and_row_independence(orc, shape, eps):
    seed, rows, n, scale = shape
    x, gamma, _, g = draw_rows(seed, rows, n, scale)
    y = orc.rmsnorm(x, gamma, eps)
    assert np.array_equal(orc.rmsnorm(-x, gamma, eps), -y)
    perm = g.permutation(rows)
    assert np.array_equal(orc.rmsnorm(x[perm], gamma, eps), y[perm])


def prop_column_permutation_and_closed_forms(orc, shape, eps):
    """Permuting the columns of x and gamma together permutes y (up to the
    order of the sum); mean((y / gamma)^2) = ms / (ms + eps); and
    |y_j| <= |gamma_j| sqrt(n) since x_j^2 <= n ms."""
    seed, rows, n, scale = shape
    x, gamma, _, g = draw_rows(seed, rows, n, scale)
    y = orc.rmsnorm(x, gamma, eps)
    perm = g.permutation(n)
    assert np.allclose(orc.rmsnorm(x[:, perm], gamma[perm], eps), y[:, perm], rtol=1e-13,
                       atol=0.0)
    ms = np.mean(x * x, axis=1)
    assert np.allclose(np.mean((y / gamma) ** 2, axis=1), ms / (ms + eps), rtol=1e-12, atol=0.0)
    assert np.all(np.abs(y) <= np.abs(gamma) * np.sqrt(n) * (1 + 1e-12))


def prop_fused_operations_compose(orc, shape, eps1, eps2):
    """then-add is the norm plus the residual; add + norm is the norm of the
    sum; the sandwich's stream is then-add at eps_post and its normed output
    the norm of that stream at eps_pre (of its bf16 rounding when the stream
    is published in bf16)."""
    seed, rows, n, scale = shape
    x, gamma, res, g = draw_rows(seed, rows, n, scale)
    gamma2 = 1.0 + 0.1 * g.standard_normal(n)
    y = orc.rmsnorm(x, gamma, eps1)
    assert np.allclose(orc.rmsnorm_then_add(x, gamma, res, eps1), y + res, rtol=1e-15,
                       atol=1e-15)
    s, o = orc.add_rmsnorm(x, res, gamma, eps1)
    assert np.array_equal(s, x + res)
    assert np.allclose(o, orc.rmsnorm(x + res, gamma, eps1), rtol=1e-15, atol=0.0)
    s_b, o_b = orc.add_rmsnorm(x, res, gamma, eps1, sum_bf16=True)     # the bf16 sum is stored
    rounded_sum = orc.double_from_bf16(orc.bf16_from_double(x + res))
    assert np.array_equal(s_b, rounded_sum)
    assert np.allclose(o_b, orc.rmsnorm(rounded_sum, gamma, eps1), rtol=1e-15, atol=0.0)
    out = orc.rmsnorm_then_add_scale(x, gamma, res, -0.5, eps1)
    assert np.allclose(out, -0.5 * (y + res), rtol=1e-15, atol=1e-15)
    stream, normed = orc.norm_residual_norm(x, res, gamma, gamma2, eps1, eps2)
    assert np.allclose(stream, orc.rmsnorm_then_add(x, gamma, res, eps1), rtol=1e-15,
                       atol=1e-15)
    assert np.allclose(normed, orc.rmsnorm(stream, gamma2, eps2), rtol=1e-15, atol=0.0)
    stream_b, normed_b = orc.norm_residual_norm(x, res, gamma, gamma2, eps1, eps2,
                                                   stream_bf16=True)
    rounded = orc.double_from_bf16(orc.bf16_from_double(stream))
    assert np.array_equal(stream_b, rounded)
    assert np.allclose(normed_b, orc.rmsnorm(rounded, gamma2, eps2), rtol=1e-15, atol=0.0)


q8_shapes = st.tuples(st.integers(0, 2**31 - 1), st.integers(1, 4), st.integers(1, 4),
                      st.sampled_from([1e-3, 1.0, 1e3]))


def prop_q8_1_blocks(orc, shape, eps):
    """Per 32-element block of the normed row: d = amax / 127, every non-zero
    block reaches |q| = 127, d * q is within d / 2 of the normed value (plus
    nothing else: codes are the nearest integers), an all-zero block is zero."""
    seed, rows, nblocks, scale = shape
    n = 32 * nblocks
    x, gamma, _, g = draw_rows(seed, rows, n, scale)
    x[:, :32] *= (g.random(rows) < 0.3)[:, None]            # some all-zero first blocks
    d, qreal, q = orc.rmsnorm_q8_1(x, gamma, eps)
    normed = orc.rmsnorm(x, gamma, eps)
    blocks = normed.reshape(rows, nblocks, 32)
    amax = np.max(np.abs(blocks), axis=2)
    assert np.allclose(d, amax / 127.0, rtol=1e-14, atol=0.0)
    qb = q.reshape(rows, nblocks, 32).astype(np.int64)
    nonzero = amax > 0
    assert np.all(np.max(np.abs(qb), axis=2)[nonzero] == 127)
    assert np.all(qb[~nonzero] == 0) and np.all(d[~nonzero] == 0)
    err = np.abs(d[:, :, None] * qb - blocks)
    assert np.all(err <= d[:, :, None] * (0.5 + 1e-9) + 1e-15 * np.abs(blocks))


def prop_seam_roundings(orc, shape, eps, seam):
    """u is a value of the format within half a unit of x * inv (relative
    2^-11 for binary16, 2^-8 for bf16, plus half the smallest subnormal);
    y is a value of the format within half a unit of u * gamma; with
    gamma = 1, y = u."""
    seed, rows, n, scale = shape
    x, _, _, g = draw_rows(seed, rows, n, scale)
    if seam == "f16":
        to_bits, from_bits, rel, tiny = orc.f16_from_double, orc.double_from_f16, 2.0**-11, 2.0**-25
    else:
        to_bits, from_bits, rel, tiny = orc.bf16_from_double, orc.double_from_bf16, 2.0**-8, 2.0**-134
    gamma = from_bits(to_bits(1.0 + 0.1 * g.standard_normal(n)))
    u, y = orc.rmsnorm_seam(x, gamma, eps, seam)
    p = orc.rmsnorm(x, np.ones(n), eps)
    assert np.array_equal(from_bits(to_bits(u)), u)
    assert np.array_equal(from_bits(to_bits(y)), y)
    assert np.all(np.abs(u - p) <= rel * np.abs(p) + tiny)
    assert np.all(np.abs(y - u * gamma) <= rel * np.abs(u * gamma) + tiny)
    u1, y1 = orc.rmsnorm_seam(x, np.ones(n), eps, seam)
    assert np.array_equal(u1, u) and np.array_equal(y1, u1)


# -- the properties over drawn cases, on the oracle as built ----------------------------


@SETTINGS
@given(shapes, EPS, st.floats(1e-3, 1e3))
def test_scale_law(shape, eps, alpha):
    prop_scale_law(oracle.default(), shape, eps, alpha)


@SETTINGS
@given(shapes, EPS)
def test_odd_symmetry_and_row_independence(shape, eps):
    prop_odd_symmetry_and_row_independence(oracle.default(), shape, eps)


@SETTINGS
@given(shapes, EPS)
def test_column_permutation_and_closed_forms(shape, eps):
    prop_column_permutation_and_closed_forms(oracle.default(), shape, eps)


@SETTINGS
@given(shapes, EPS, EPS)
def test_fused_operations_compose_from_the_separate_ones(shape, eps1, eps2):
    prop_fused_operations_compose(oracle.default(), shape, eps1, eps2)


@SETTINGS
@given(q8_shapes, EPS)
def test_q8_1_blocks(shape, eps):
    prop_q8_1_blocks(oracle.default(), shape, eps)


@SETTINGS
@given(shapes, EPS, st.sampled_from(["f16", "bf16"]))
def test_seam_roundings(shape, eps, seam):
    prop_seam_roundings(oracle.default(), shape, eps, seam)
