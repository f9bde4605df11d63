"""Pins of the CPU oracle to facts other than the oracle itself.

Each ``check_*`` function takes an ``oracle.Oracle`` (the real one, or a mutant
compiled from an edited copy of its source) and raises AssertionError when the
oracle disagrees with:

* the worked example printed on "Chapter 12 -- RMSNorm and the dual-epsilon
  sandwich", section 12.3 (``golden/rmsnorm_worked_example.txt``);
* closed forms: a constant row, the two-element rows, the epsilon-dominated
  limit, the exact scale law y(a x; a^2 eps) = y(x; eps), a residual-free
  sandwich over rows of known mean square;
* library routines in float64: ``torch.nn.functional.rms_norm`` (the routine the
  dormouse page pins against, its section 6) and ``layer_norm`` on mean-centred
  rows (the identity mean(x^2) = sigma^2 + mu^2 of section 12.2);
* exact rational / 50-digit decimal arithmetic on tiny inputs;
* structural invariants (row and column permutations);
* torch's float32 -> bfloat16 conversion for the bf16 rounding routine;
* numpy's float64 -> float16 cast (correctly rounded, ties to even) and exact
  rational rounding for the split-norm seam of section 12.7.

``ALL_CHECKS`` lists them; the mutation test runs every check against each
planted mistake and expects at least one to fail.
"""
from __future__ import annotations

import os
from decimal import Decimal, getcontext
from fractions import Fraction

import numpy as np
import torch
import torch.nn.functional as F

GOLDEN_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load_golden(name: str) -> dict:
    """Parse ``<key> <values...> | <tol>`` lines into {key: (array, tol)}."""
    out = {}
    with open(os.path.join(GOLDEN_DIR, name)) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            lhs, tol = line.split("|")
            parts = lhs.split()
            out[parts[0]] = (np.array([float(v) for v in parts[1:]]), float(tol))
    return out


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def _assert_close(got, want, tol, what):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    err = np.abs(got - want)
    bad = ~(err <= tol)                    # a NaN anywhere fails
    assert not np.any(bad), (f"{what}: max err {np.nanmax(err):.3e} > tol, "
                             f"{int(np.isnan(err).sum())} NaN; "
                             f"got {got[bad][:4]} want {want[bad][:4]}")


def _assert_rel(got, want, rel, what, floor=0.0):
    want = np.asarray(want, dtype=np.float64)
    _assert_close(got, want, rel * np.abs(want) + floor, what)


def _torch_rms(x, gamma, eps):
    t = torch.from_numpy(np.asarray(x, dtype=np.float64))
    w = torch.from_numpy(np.asarray(gamma, dtype=np.float64))
    return F.rms_norm(t, (t.shape[-1],), weight=w, eps=float(eps)).numpy()


# ---------------------------------------------------------------------------
# RMSNorm
# ---------------------------------------------------------------------------
def check_worked_example(orc):
    """Section 12.3: x = [3, 4, 0, 0], eps = 1e-5, with both gammas printed."""
    g = load_golden("rmsnorm_worked_example.txt")
    eps = g["eps"][0][0]
    x = g["x"][0][None, :]
    y1 = orc.rmsnorm(x, g["gamma_ones"][0], eps)[0]
    y2 = orc.rmsnorm(x, g["gamma_shaped"][0], eps)[0]
    inv = y1[0] / x[0, 0]
    rms = 1.0 / inv
    mean_sq = rms * rms - eps
    _assert_close(inv, g["inv_rms"][0][0], g["inv_rms"][1], "inv_rms")
    _assert_close(rms, g["rms"][0][0], g["rms"][1], "rms")
    _assert_close(mean_sq, g["mean_sq"][0][0], 1e-12, "mean of squares")
    _assert_close(mean_sq * 4, g["sum_sq"][0][0], 1e-11, "sum of squares")
    _assert_close(y1, g["y_gamma_ones"][0], g["y_gamma_ones"][1], "y, gamma = 1")
    _assert_close(np.mean(y1 * y1), g["mean_sq_y_gamma_ones"][0][0],
                  g["mean_sq_y_gamma_ones"][1], "mean(y^2), gamma = 1")
    _assert_close(y2, g["y_gamma_shaped"][0], g["y_gamma_shaped"][1], "y, gamma shaped")


def check_constant_rows(orc):
    """x = c in every column  =>  y_j = c / sqrt(c^2 + eps) * gamma_j."""
    g = _rng(11)
    for n in (1, 2, 7, 64, 6656):
        gamma = 1.0 + 0.1 * g.standard_normal(n)
        for c in (1e-3, -0.5, 3.0, 1e3):
            for eps in (1e-5, 1e-8):
                x = np.full((2, n), c)
                y = orc.rmsnorm(x, gamma, eps)
                want = c / np.sqrt(c * c + eps) * gamma
                _assert_rel(y, np.broadcast_to(want, y.shape), 1e-12,
                            f"constant row c={c} n={n} eps={eps}")


def check_two_element_rows(orc):
    """n = 2 by hand: [3, 4] -> [3, 4] / sqrt(12.5 + eps); [1, -1] -> +-1/sqrt(1 + eps)."""
    eps = 1e-5
    x = np.array([[3.0, 4.0], [1.0, -1.0], [0.0, 0.0], [-4.0, 3.0]])
    for rows in (1, 2, 3, 4):
        y = orc.rmsnorm(x[:rows], np.ones(2), eps)
        want = np.array([[3.0, 4.0] / np.sqrt(12.5 + eps),
                         [1.0, -1.0] / np.sqrt(1.0 + eps),
                         [0.0, 0.0],
                         [-4.0, 3.0] / np.sqrt(12.5 + eps)])[:rows]
        _assert_rel(y, want, 1e-15, f"n=2 rows={rows}")
        if rows >= 3:
            assert np.all(y[2] == 0.0), "a zero row must give exact zeros"


def check_scale_law(orc):
    """y(a x; a^2 eps) = y(x; eps) exactly in real arithmetic; and y(a x; eps) ~ y(x; eps)
    when eps << mean(x^2), within eps / (2 mean(x^2))."""
    g = _rng(12)
    x = g.standard_normal((5, 300))
    gamma = 1.0 + 0.1 * g.standard_normal(300)
    eps = 1e-5
    base = orc.rmsnorm(x, gamma, eps)
    for a in (1e-3, 0.5, 10.0, 1e4):
        _assert_rel(orc.rmsnorm(a * x, gamma, a * a * eps), base, 1e-13,
                    f"exact scale law a={a}")
    for a in (3.0, 100.0):
        # mean squares here are ~1, so the eps effect is below ~1e-5 / 2 * 1.1
        _assert_rel(orc.rmsnorm(a * x, gamma, eps), base, 0.6e-5 * 1.2,
                    f"approximate scale invariance a={a}")


def check_eps_dominated(orc):
    """mean(x^2) << eps  =>  y ~ x * gamma / sqrt(eps) (relative deviation ~ ms/(2 eps))."""
    g = _rng(13)
    x = 1e-9 * g.standard_normal((3, 512))
    gamma = 1.0 + 0.1 * g.standard_normal(512)
    for eps in (1e-5, 1e-8):
        y = orc.rmsnorm(x, gamma, eps)
        _assert_rel(y, x * gamma / np.sqrt(eps), 1e-9, f"eps-dominated eps={eps}")


def check_rms_of_output(orc):
    """With gamma = 1 the output has mean square ms / (ms + eps) (section 12.3 check:
    rms(y) = 1 for eps -> 0)."""
    g = _rng(14)
    x = np.vstack([c * g.standard_normal(1000) for c in (1e-3, 1.0, 30.0)])
    eps = 1e-5
    y = orc.rmsnorm(x, np.ones(1000), eps)
    for r in range(x.shape[0]):
        xs = [Fraction(v) for v in x[r]]
        ms = float(sum(v * v for v in xs) / len(xs))
        _assert_rel(np.mean(y[r] * y[r]), ms / (ms + eps), 1e-13, f"mean(y^2) row {r}")


def check_against_torch_rms_norm(orc):
    """torch.nn.functional.rms_norm in float64, several shapes and epsilons."""
    g = _rng(15)
    for rows, n in ((3, 5), (4, 6656), (2, 65536), (7, 2)):
        x = g.standard_normal((rows, n)) * 10.0 ** g.uniform(-3, 2, size=(rows, 1))
        gamma = 1.0 + 0.1 * g.standard_normal(n)
        for eps in (1e-5, 1e-6, 1e-8):
            _assert_rel(orc.rmsnorm(x, gamma, eps), _torch_rms(x, gamma, eps), 1e-12,
                        f"torch rms_norm rows={rows} n={n} eps={eps}", floor=1e-300)


def check_layer_norm_identity(orc):
    """Mean-centred rows: RMSNorm == LayerNorm without bias; and in general
    rms = sqrt(sigma^2 + mu^2) (section 12.2, 'A useful identity')."""
    g = _rng(16)
    n = 777
    x = g.standard_normal((4, n)) * 3.0
    gamma = 1.0 + 0.1 * g.standard_normal(n)
    eps = 1e-5
    xc = x - x.mean(axis=1, keepdims=True)
    ln = F.layer_norm(torch.from_numpy(xc), (n,), weight=torch.from_numpy(gamma),
                      bias=None, eps=eps).numpy()
    _assert_rel(orc.rmsnorm(xc, gamma, eps), ln, 1e-12, "layer_norm on centred rows",
                floor=1e-15)
    t = torch.from_numpy(x + 0.7)
    var, mu = torch.var_mean(t, dim=1, unbiased=False, keepdim=True)
    want = (t / torch.sqrt(var + mu * mu + eps) * torch.from_numpy(gamma)).numpy()
    _assert_rel(orc.rmsnorm(x + 0.7, gamma, eps), want, 1e-12, "sigma^2 + mu^2 identity")


def _decimal_inv_rms(row, eps):
    ss = sum(Fraction(v) * Fraction(v) for v in row)
    d = ss / len(row) + Fraction(eps)
    return Decimal(1) / (Decimal(d.numerator) / Decimal(d.denominator)).sqrt()


def check_exact_small(orc):
    """n <= 8: compare with exact rationals and a 50-digit decimal square root."""
    getcontext().prec = 50
    g = _rng(17)
    for n in range(1, 9):
        x = g.standard_normal((3, n))
        res = g.standard_normal((3, n))
        gamma = 1.0 + 0.1 * g.standard_normal(n)
        gamma2 = 1.0 + 0.1 * g.standard_normal(n)
        eps, eps2 = 1e-5, 1e-8
        y = orc.rmsnorm(x, gamma, eps)
        t = orc.rmsnorm_then_add(x, gamma, res, eps)
        s, o = orc.norm_residual_norm(x, res, gamma, gamma2, eps2, eps)
        for r in range(3):
            inv = _decimal_inv_rms(x[r], eps)
            p = [Decimal(x[r, j]) * inv * Decimal(gamma[j]) for j in range(n)]
            want_y = np.array([float(v) for v in p])
            want_t = np.array([float(p[j] + Decimal(res[r, j])) for j in range(n)])
            _assert_rel(y[r], want_y, 4e-15, f"exact rmsnorm n={n}", floor=1e-300)
            scale_t = np.abs(want_y) + np.abs(res[r])
            _assert_close(t[r], want_t, 4e-15 * scale_t, f"exact then-add n={n}")
            inv_post = _decimal_inv_rms(x[r], eps2)
            st = [Decimal(x[r, j]) * inv_post * Decimal(gamma[j]) + Decimal(res[r, j])
                  for j in range(n)]
            want_s = np.array([float(v) for v in st])
            _assert_close(s[r], want_s, 4e-15 * scale_t + 1e-300, f"exact stream n={n}")
            # second norm of the stored stream
            inv_pre = _decimal_inv_rms(s[r], eps)
            want_o = np.array([float(Decimal(s[r, j]) * inv_pre * Decimal(gamma2[j]))
                               for j in range(n)])
            _assert_rel(o[r], want_o, 4e-15, f"exact normed n={n}", floor=1e-300)


def check_row_and_column_permutations(orc):
    """Rows are independent (row permutation permutes outputs bit for bit);
    permuting columns together with gamma permutes the outputs."""
    g = _rng(18)
    x = g.standard_normal((9, 130))
    res = g.standard_normal((9, 130))
    gamma = 1.0 + 0.1 * g.standard_normal(130)
    eps = 1e-5
    pr = g.permutation(9)
    pc = g.permutation(130)
    y = orc.rmsnorm_then_add(x, gamma, res, eps)
    assert np.array_equal(orc.rmsnorm_then_add(x[pr], gamma, res[pr], eps), y[pr]), \
        "row permutation"
    _assert_rel(orc.rmsnorm_then_add(x[:, pc], gamma[pc], res[:, pc], eps), y[:, pc],
                1e-13, "column permutation", floor=1e-15)


# ---------------------------------------------------------------------------
# post-norm then add (Hesper rmsNormThenAddKernel) and the sandwich tail
# ---------------------------------------------------------------------------
def check_then_add_against_torch(orc):
    g = _rng(19)
    for rows, n in ((5, 6656), (3, 7), (64, 128)):
        x = g.standard_normal((rows, n)) * 10.0 ** g.uniform(-2, 2, size=(rows, 1))
        res = g.standard_normal((rows, n))
        gamma = 1.0 + 0.1 * g.standard_normal(n)
        p = _torch_rms(x, gamma, 1e-6)
        got = orc.rmsnorm_then_add(x, gamma, res, 1e-6)
        _assert_close(got, p + res, 1e-12 * (np.abs(p) + np.abs(res)),
                      f"then-add rows={rows} n={n}")
    # zero rows give the residual exactly
    x[1:3] = 0.0
    got = orc.rmsnorm_then_add(x, gamma, res, 1e-6)
    assert np.array_equal(got[1:3], res[1:3]), "zero rows must return the residual"


def _torch_sandwich(b, r, gp, gq, eps_post, eps_pre):
    s = _torch_rms(b, gp, eps_post) + r
    return s, _torch_rms(s, gq, eps_pre)


def check_sandwich_against_torch(orc):
    """Section 12.4.3 as two library norms and an add, in float64."""
    g = _rng(20)
    rows, n = 6, 6656
    b = 2.0 * g.standard_normal((rows, n)) * 10.0 ** g.uniform(-2, 1, size=(rows, 1))
    r = g.standard_normal((rows, n))
    gp = 1.0 + 0.1 * g.standard_normal(n)
    gq = 1.0 + 0.1 * g.standard_normal(n)
    s, o = orc.norm_residual_norm(b, r, gp, gq, 1e-8, 1e-5)
    ts, to = _torch_sandwich(b, r, gp, gq, 1e-8, 1e-5)
    p = _torch_rms(b, gp, 1e-8)
    _assert_close(s, ts, 1e-12 * (np.abs(p) + np.abs(r)), "sandwich stream vs torch")
    _assert_rel(o, _torch_rms(s, gq, 1e-5), 1e-12, "sandwich normed vs torch(stream)",
                floor=1e-300)


def check_sandwich_epsilon_routing(orc):
    """A case where each epsilon is visible: the block output has mean square
    1e-8 (so eps_post = 1e-8 halves the first norm's scale) and the stream is
    small enough (mean square ~1e-6) that eps_pre = 1e-5 dominates the second.
    Swapping the epsilons moves both outputs by more than 10%."""
    g = _rng(21)
    rows, n = 4, 4096
    b = 1e-4 * np.where(g.random((rows, n)) < 0.5, -1.0, 1.0)   # mean square exactly 1e-8
    r = 1e-3 * g.standard_normal((rows, n))
    gp = 1e-3 * (1.0 + 0.1 * g.standard_normal(n))
    gq = 1.0 + 0.1 * g.standard_normal(n)
    s, o = orc.norm_residual_norm(b, r, gp, gq, 1e-8, 1e-5)
    ts, to = _torch_sandwich(b, r, gp, gq, 1e-8, 1e-5)
    _assert_close(s, ts, 1e-12 * (np.abs(ts) + np.abs(r)), "routing case stream")
    _assert_rel(o, _torch_rms(s, gq, 1e-5), 1e-12, "routing case normed", floor=1e-300)
    ws, wo = _torch_sandwich(b, r, gp, gq, 1e-5, 1e-8)       # epsilons swapped
    assert np.max(np.abs(ws - ts)) > 0.1 * np.max(np.abs(ts - r)), "swap invisible (stream)"
    assert np.max(np.abs(wo - to)) > 0.1 * np.max(np.abs(to)), "swap invisible (normed)"


def check_sandwich_closed_form(orc):
    """residual = 0, gamma_post = 1, block_out = +-c with mean square c^2:
    stream_j = b_j / sqrt(c^2 + eps_post), its mean square m = c^2/(c^2 + eps_post),
    normed_j = stream_j / sqrt(m + eps_pre) * gamma_pre_j."""
    g = _rng(22)
    n = 1000
    gq = 1.0 + 0.1 * g.standard_normal(n)
    for c in (1e-4, 1e-2, 5.0):
        b = c * np.where(g.random((3, n)) < 0.5, -1.0, 1.0)
        s, o = orc.norm_residual_norm(b, np.zeros_like(b), np.ones(n), gq, 1e-8, 1e-5)
        want_s = b / np.sqrt(c * c + 1e-8)
        m = c * c / (c * c + 1e-8)
        want_o = want_s / np.sqrt(m + 1e-5) * gq
        _assert_rel(s, want_s, 1e-13, f"closed-form stream c={c}")
        _assert_rel(o, want_o, 1e-13, f"closed-form normed c={c}")


def check_sandwich_degenerate(orc):
    """gamma_post = 0 or block_out = 0 leaves the stream equal to the residual."""
    g = _rng(23)
    b = g.standard_normal((3, 50))
    r = g.standard_normal((3, 50))
    gq = 1.0 + 0.1 * g.standard_normal(50)
    s, o = orc.norm_residual_norm(b, r, np.zeros(50), gq, 1e-8, 1e-5)
    assert np.array_equal(s, r), "gamma_post = 0"
    s, o = orc.norm_residual_norm(np.zeros_like(b), r, gq, gq, 1e-8, 1e-5)
    assert np.array_equal(s, r), "block_out = 0"
    _assert_rel(o, _torch_rms(r, gq, 1e-5), 1e-12, "normed of the bare residual")


def check_add_rmsnorm(orc):
    """Residual add then norm (Hesper residualAddRmsNormKernel): against torch in
    float64, symmetric in its two inputs, b = 0 gives RMSNorm(a), constant rows
    in closed form, and the bf16 sum is the rounded sum re-normed."""
    g = _rng(26)
    rows, n = 5, 1000
    a = g.standard_normal((rows, n)) * 10.0 ** g.uniform(-2, 2, size=(rows, 1))
    b = g.standard_normal((rows, n))
    gamma = 1.0 + 0.1 * g.standard_normal(n)
    s, o = orc.add_rmsnorm(a, b, gamma, 1e-5)
    assert np.array_equal(s, a + b), "residual_out is the plain sum"
    _assert_rel(o, _torch_rms(a + b, gamma, 1e-5), 1e-12, "add+norm vs torch", floor=1e-300)
    s2, o2 = orc.add_rmsnorm(b, a, gamma, 1e-5)
    assert np.array_equal(s2, s) and np.array_equal(o2, o), "symmetric in a and b"
    s3, o3 = orc.add_rmsnorm(a, np.zeros_like(a), gamma, 1e-5)
    assert np.array_equal(s3, a)
    _assert_rel(o3, _torch_rms(a, gamma, 1e-5), 1e-12, "b = 0", floor=1e-300)
    for c, d in ((1.5, -0.25), (1e-4, 2e-4)):
        sc, oc = orc.add_rmsnorm(np.full((2, 7), c), np.full((2, 7), d), gamma[:7], 1e-8)
        _assert_rel(oc, np.broadcast_to((c + d) / np.sqrt((c + d) ** 2 + 1e-8) * gamma[:7],
                                        oc.shape), 1e-13, f"constant rows {c}+{d}")
    sb, ob = orc.add_rmsnorm(a, b, gamma, 1e-5, sum_bf16=True)
    tb = _torch_bf16_bits((a + b).astype(np.float32))
    exact32 = (a + b).astype(np.float32).astype(np.float64) == a + b
    bits = orc.bf16_from_double(sb)
    assert np.array_equal(orc.double_from_bf16(bits), sb), "bf16 sum is representable"
    assert np.array_equal(bits[exact32], tb[exact32]), "bf16 sum is the rounded sum"
    _assert_rel(ob, _torch_rms(sb, gamma, 1e-5), 1e-12, "bf16 sum re-normed", floor=1e-300)


def check_then_add_scale(orc):
    """(RMSNorm(x) gamma + r) * s (Hesper rmsNormThenAddThenBroadcastScaleKernel):
    against torch, s = 1 is the then-add, s = 0 gives zeros, a power of two
    scales exactly."""
    g = _rng(27)
    rows, n = 4, 777
    x = g.standard_normal((rows, n)) * 3.0
    r = g.standard_normal((rows, n))
    gamma = 1.0 + 0.1 * g.standard_normal(n)
    base = orc.rmsnorm_then_add(x, gamma, r, 1e-6)
    assert np.array_equal(orc.rmsnorm_then_add_scale(x, gamma, r, 1.0, 1e-6), base)
    assert np.array_equal(orc.rmsnorm_then_add_scale(x, gamma, r, -2.0, 1e-6), -2.0 * base)
    assert np.all(orc.rmsnorm_then_add_scale(x, gamma, r, 0.0, 1e-6) == 0.0)
    p = _torch_rms(x, gamma, 1e-6)
    got = orc.rmsnorm_then_add_scale(x, gamma, r, 0.37, 1e-6)
    _assert_close(got, (p + r) * 0.37, 1e-12 * 0.37 * (np.abs(p) + np.abs(r)), "vs torch")


def check_q8_round(orc):
    """WGSL round(): nearest integer, ties to even; clamped to int8."""
    cases = {2.5: 2, 3.5: 4, -2.5: -2, -3.5: -4, 0.5: 0, 1.5: 2, 0.49999: 0, -0.51: -1,
             126.5: 126, 127.4: 127, 127.6: 127, 200.0: 127, -127.5: -128, -128.4: -128,
             -128.6: -128, -300.0: -128}
    for v, want in cases.items():
        assert orc.q8_round(v) == want, (v, orc.q8_round(v), want)


def check_rmsnorm_q8_1(orc):
    """RMSNorm + Q8_1 (Hesper fusedRMSNormQ8_1Kernel): d = amax/127 of the torch
    float64 norm per 32-block, q = nearest of x_normed/d, each non-zero block
    reaches |q| = 127 at its amax, dequantisation within d/2, zero blocks give
    d = q = 0."""
    g = _rng(28)
    rows, n = 6, 2560                     # D = 2560 is the page's example width
    x = g.standard_normal((rows, n)) * 10.0 ** g.uniform(-2, 2, size=(rows, 1))
    x[2, 64:96] = 0.0                     # one all-zero block
    gamma = 1.0 + 0.1 * g.standard_normal(n)
    d, qreal, q = orc.rmsnorm_q8_1(x, gamma, 1e-6)
    xn = _torch_rms(x, gamma, 1e-6)
    amax = np.abs(xn).reshape(rows, n // 32, 32).max(axis=2)
    _assert_rel(d, amax / 127.0, 1e-13, "d = amax / 127")
    assert d[2, 2] == 0.0 and np.all(q[2, 64:96] == 0), "zero block"
    blocks = np.abs(q.astype(np.int64)).reshape(rows, n // 32, 32).max(axis=2)
    assert np.all((blocks == 127) | (amax == 0)), "every non-zero block reaches 127"
    dd = np.repeat(d, 32, axis=1)
    nz = dd > 0
    ref = np.where(nz, xn / np.where(nz, dd, 1.0), 0.0)
    _assert_close(qreal, ref, 1e-12 * (1 + np.abs(ref)), "x_normed / d")
    margin = np.abs(np.abs(ref - np.floor(ref)) - 0.5)
    safe = margin > 1e-9
    assert np.array_equal(q[safe], np.clip(np.rint(ref[safe]), -128, 127).astype(np.int8)), \
        "q = nearest integer of x_normed / d"
    _assert_close(q * dd, xn, 0.5 * dd * (1 + 1e-9) + 1e-300, "dequantisation within d/2")


def check_f16_conversions(orc):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    sample = bits[::37]
    got = orc.double_from_f16(sample)
    want = sample.view(np.float16).astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan) and np.array_equal(got[~nan], want[~nan])
    g = _rng(29)
    v = np.concatenate([g.standard_normal(3000) * 10.0 ** g.uniform(-9, 5, 3000),
                        [65504.0, 65519.9, 65520.0, 2.0 ** -24, 3 * 2.0 ** -25, 2.0 ** -25,
                         0.0, -0.0, 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11,
                         # rounding that carries into the next binade, odd and even fields
                         2047.5, -2047.75, 4095.5, 1.0 - 2.0 ** -12, 0.5 - 2.0 ** -13,
                         2.0 ** -14 - 2.0 ** -26]])
    with np.errstate(over="ignore"):
        ref = v.astype(np.float16).view(np.uint16)
    assert np.array_equal(orc.f16_from_double(v), ref), "f16 rounding vs numpy"


# ---------------------------------------------------------------------------
# bf16 conversions
# ---------------------------------------------------------------------------
def _torch_bf16_bits(f32):
    t = torch.from_numpy(np.ascontiguousarray(f32, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def check_bf16_widen_all_patterns(orc):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = orc.double_from_bf16(bits)
    want = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan), "NaN patterns"
    assert np.array_equal(got[~nan], want[~nan]), "bf16 widening"
    back = orc.bf16_from_double(got[~nan])
    assert np.array_equal(back, bits[~nan]), "round trip of every finite/inf pattern"


def check_bf16_round_against_torch(orc):
    g = _rng(24)
    raw = g.integers(0, 2 ** 32, size=200000, dtype=np.uint64).astype(np.uint32)
    f = raw.view(np.float32)
    f = f[~np.isnan(f)]
    assert np.array_equal(orc.bf16_from_double(f.astype(np.float64)), _torch_bf16_bits(f)), \
        "random float32 patterns"
    # exact midpoints between neighbouring bf16 values (representable in f32): ties
    lo = g.integers(0, 0x7F7F, size=50000).astype(np.uint16)
    vlo = orc.double_from_bf16(lo)
    vhi = orc.double_from_bf16(lo + 1)
    mid = ((vlo + vhi) / 2).astype(np.float32)
    assert np.array_equal(mid.astype(np.float64), (vlo + vhi) / 2)
    for sgn in (1.0, -1.0):
        m = sgn * mid
        assert np.array_equal(orc.bf16_from_double(m.astype(np.float64)), _torch_bf16_bits(m)), \
            "ties to even"
    special = np.array([np.inf, -np.inf, 3.4e38, -3.4e38, 0.0, -0.0, 2.0 ** -134,
                        1.5 * 2.0 ** -133], dtype=np.float32)
    assert np.array_equal(orc.bf16_from_double(special.astype(np.float64)),
                          _torch_bf16_bits(special)), "specials"
    assert orc.bf16_from_double([np.nan])[0] & 0x7FFF > 0x7F80, "NaN stays NaN"


def check_bf16_sandwich_stream(orc):
    """stream_bf16: the stored stream is the bf16 rounding of the f64 stream and the
    second norm reads the rounded values (section 12.4.4)."""
    g = _rng(25)
    rows, n = 4, 300
    b = g.standard_normal((rows, n))
    r = g.standard_normal((rows, n))
    gp = 1.0 + 0.1 * g.standard_normal(n)
    gq = 1.0 + 0.1 * g.standard_normal(n)
    s, o = orc.norm_residual_norm(b, r, gp, gq, 1e-8, 1e-5, stream_bf16=True)
    ts, _ = _torch_sandwich(b, r, gp, gq, 1e-8, 1e-5)
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(ts), 2.0 ** -126))) - 7)
    _assert_close(s, ts, 0.5 * ulp * (1 + 1e-9), "stream within half a bf16 ulp")
    bits = orc.bf16_from_double(s)
    assert np.array_equal(orc.double_from_bf16(bits), s), "stream is bf16-representable"
    _assert_rel(o, _torch_rms(s, gq, 1e-5), 1e-12, "normed of the rounded stream",
                floor=1e-300)
    s32, _ = orc.norm_residual_norm(b, r, gp, gq, 1e-8, 1e-5, stream_bf16=False)
    assert not np.array_equal(s32, s), "rounding must change the stream"


# ---------------------------------------------------------------------------
# Split-norm seam (section 12.7): u = T(x * inv), y = T(u * gamma)
# ---------------------------------------------------------------------------
def _nearest_in_format(v: Fraction, frac_bits: int, min_exp: int, max_exp: int) -> Fraction:
    """Exact nearest value (ties to even) of a binary format with `frac_bits`
    fraction bits, normal exponents [min_exp, max_exp] and gradual underflow;
    beyond the largest finite value by half a unit, infinity (as None)."""
    if v == 0:
        return Fraction(0)
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    e = max(e, min_exp)
    quantum = Fraction(2) ** (e - frac_bits)
    k, rem = divmod(a, quantum)
    if rem * 2 > quantum or (rem * 2 == quantum and k % 2 == 1):
        k += 1
    r = k * quantum
    if r >= Fraction(2) ** (max_exp + 1):
        return None
    return r if v > 0 else -r


def _exact_seam(x_row, gamma, eps, frac_bits, min_exp, max_exp):
    """u and y of one row by exact rationals and a 60-digit square root."""
    getcontext().prec = 60
    inv = _decimal_inv_rms(x_row, eps)
    u, y = [], []
    for xj, gj in zip(x_row, gamma):
        p = Fraction(Decimal(xj) * inv)
        uj = _nearest_in_format(p, frac_bits, min_exp, max_exp)
        yj = _nearest_in_format(uj * Fraction(gj), frac_bits, min_exp, max_exp)
        u.append(float(uj))
        y.append(float(yj) if yj is not None else np.copysign(np.inf, float(uj * Fraction(gj))))
    return np.array(u), np.array(y)


F16_FORMAT = (10, -14, 15)
BF16_FORMAT = (7, -126, 127)


def check_seam_worked_example(orc):
    """Section 12.3's row x = [3, 4, 0, 0], eps = 1e-5, with the page's shaped
    gamma [2, 0.5, 1, 1], through the seam.  x * inv = 1.19999904..,
    1.59999872..; binary16 has spacing 2^-10 on [1, 2), so u = 1229/1024 and
    1638/1024 (1228.799.. and 1638.398.. units); bf16 has spacing 2^-7, so
    u = 154/128 and 205/128.  The power-of-two gammas scale u exactly."""
    g = load_golden("rmsnorm_worked_example.txt")
    eps = g["eps"][0][0]
    x = g["x"][0][None, :]
    gamma = g["gamma_shaped"][0]
    u, y = orc.rmsnorm_seam(x, gamma, eps, "f16")
    _assert_close(u[0], [1229 / 1024, 1638 / 1024, 0, 0], 0.0, "f16 seam u")
    _assert_close(y[0], [2 * 1229 / 1024, 0.5 * 1638 / 1024, 0, 0], 0.0, "f16 seam y")
    u, y = orc.rmsnorm_seam(x, gamma, eps, "bf16")
    _assert_close(u[0], [154 / 128, 205 / 128, 0, 0], 0.0, "bf16 seam u")
    _assert_close(y[0], [2 * 154 / 128, 0.5 * 205 / 128, 0, 0], 0.0, "bf16 seam y")


def check_seam_exact_small(orc):
    """n <= 8 rows (f32-valued x, T-valued gamma, some products in the T
    subnormal range and some beyond its largest value) against exact rational
    rounding of the exact norm."""
    g = _rng(41)
    for seam, fmt in (("f16", F16_FORMAT), ("bf16", BF16_FORMAT)):
        for n in range(1, 9):
            x = g.standard_normal((3, n)).astype(np.float32).astype(np.float64)
            x[1] *= 1e-3
            gamma = 1.0 + 0.3 * g.standard_normal(n)
            if seam == "f16":
                gamma[0] = 3e4 if n > 2 else gamma[0]        # may overflow binary16
                gamma[-1] *= 1e-6                             # binary16 subnormal products
                gamma = gamma.astype(np.float16).astype(np.float64)
            else:
                gamma[-1] *= 1e-39
                gamma = orc.double_from_bf16(orc.bf16_from_double(gamma))
            u, y = orc.rmsnorm_seam(x, gamma, 1e-5, seam)
            for r in range(3):
                wu, wy = _exact_seam(x[r], gamma, 1e-5, *fmt)
                assert np.array_equal(u[r], wu), f"{seam} exact u n={n}: {u[r]} vs {wu}"
                assert np.array_equal(y[r], wy), f"{seam} exact y n={n}: {y[r]} vs {wy}"


def check_seam_against_numpy_f16(orc):
    """binary16 seam against torch's float64 rms_norm (gamma = 1) and numpy's
    float64 -> float16 cast, element by element; elements whose x * inv lies
    within 1e-12 of a rounding tie are left to the exact check."""
    g = _rng(42)
    rows, n = 8, 1000
    x = (g.standard_normal((rows, n)) * 10.0 ** g.uniform(-3, 3, size=(rows, 1)))
    x = x.astype(np.float32).astype(np.float64)
    gamma = (1.0 + 0.1 * g.standard_normal(n)).astype(np.float16).astype(np.float64)
    gamma[:50] = (g.standard_normal(50) * 1e-5).astype(np.float16)   # subnormal products
    u, y = orc.rmsnorm_seam(x, gamma, 1e-6, "f16")
    p = _torch_rms(x, np.ones(n), 1e-6)
    wu = p.astype(np.float16).astype(np.float64)
    wy = (wu * gamma).astype(np.float16).astype(np.float64)
    lo = np.nextafter(p.astype(np.float16), np.float16(-np.inf)).astype(np.float64)
    hi = np.nextafter(p.astype(np.float16), np.float16(np.inf)).astype(np.float64)
    mid_gap = np.minimum(np.abs(p - (wu + lo) / 2), np.abs(p - (wu + hi) / 2))
    safe = mid_gap > 1e-12 * np.abs(p)
    assert safe.mean() > 0.99
    assert np.array_equal(u[safe], wu[safe]), "u = float16(x * inv)"
    assert np.array_equal(y[safe], wy[safe]), "y = float16(u * gamma)"


def check_seam_rounding_point(orc):
    """The seam keeps its intermediate rounding: gamma = 1 gives y = u; a
    power-of-two gamma scales u exactly; a general gamma gives results that
    differ from a single rounding of x * inv * gamma for some elements, each
    within two units of the last place of y."""
    g = _rng(43)
    rows, n = 4, 4096
    x = g.standard_normal((rows, n))
    for seam in ("f16", "bf16"):
        u1, y1 = orc.rmsnorm_seam(x, np.ones(n), 1e-5, seam)
        assert np.array_equal(y1, u1), f"{seam}: gamma = 1"
        u4, y4 = orc.rmsnorm_seam(x, np.full(n, 4.0), 1e-5, seam)   # |4u| << max, exact
        assert np.array_equal(u4, u1) and np.array_equal(y4, 4.0 * u1), f"{seam}: gamma = 4"
        gamma = 1.0 + 0.1 * g.standard_normal(n)
        gamma = (gamma.astype(np.float16).astype(np.float64) if seam == "f16"
                 else orc.double_from_bf16(orc.bf16_from_double(gamma)))
        u, y = orc.rmsnorm_seam(x, gamma, 1e-5, seam)
        one = orc.rmsnorm(x, gamma, 1e-5)
        one_t = (one.astype(np.float16).astype(np.float64) if seam == "f16"
                 else orc.double_from_bf16(orc.bf16_from_double(one)))
        assert np.array_equal(u, u1), f"{seam}: u does not depend on gamma"
        assert np.sum(y != one_t) > 0, f"{seam}: the intermediate rounding must show"
        bits = 10 if seam == "f16" else 7
        ulp = 2.0 ** (np.floor(np.log2(np.abs(one_t))) - bits)
        _assert_close(y, one, 2 * ulp, f"{seam}: within two units of one rounding")


ALL_CHECKS = [
    check_worked_example,
    check_constant_rows,
    check_two_element_rows,
    check_scale_law,
    check_eps_dominated,
    check_rms_of_output,
    check_against_torch_rms_norm,
    check_layer_norm_identity,
    check_exact_small,
    check_row_and_column_permutations,
    check_then_add_against_torch,
    check_sandwich_against_torch,
    check_sandwich_epsilon_routing,
    check_sandwich_closed_form,
    check_sandwich_degenerate,
    check_add_rmsnorm,
    check_then_add_scale,
    check_q8_round,
    check_rmsnorm_q8_1,
    check_f16_conversions,
    check_bf16_widen_all_patterns,
    check_bf16_round_against_torch,
    check_bf16_sandwich_stream,
    check_seam_worked_example,
    check_seam_exact_small,
    check_seam_against_numpy_f16,
    check_seam_rounding_point,
]
