"""The parity gate goes red (CPU only, no GPU): the checks that the GPU tests
apply to every output reject planted mistakes in a result array -- an element
2e-5 off, a dropped tail (zeros where the definition is not zero), a nonzero
where it is zero, a bf16 value two units off -- and accept results within the
stated tolerances (1e-5 relative for f32, one bf16 unit, the summands' bound
under cancellation)."""
import numpy as np
import pytest

import gpu_util as gu
import oracle


def _want(seed=3, n=1000):
    return np.random.default_rng(seed).standard_normal(n)


def test_f32_norm_gate():
    want = _want()
    gu.check_f32_norm(want.astype(np.float32), want, "f32 rounding of the definition")
    gu.check_f32_norm(want * (1 + 0.9e-5), want, "0.9e-5 relative")
    off = want.copy()
    off[17] *= 1 + 2e-5
    with pytest.raises(AssertionError):
        gu.check_f32_norm(off, want, "one element 2e-5 off")
    tail = want.copy()
    tail[-3:] = 0.0
    with pytest.raises(AssertionError):
        gu.check_f32_norm(tail, want, "dropped tail")
    w0 = want.copy()
    w0[5] = 0.0
    g0 = w0.copy()
    g0[5] = 1e-30
    with pytest.raises(AssertionError):
        gu.check_f32_norm(g0, w0, "nonzero where the definition is zero")


def test_f32_sum_gate_is_relative_to_the_summands():
    rng = np.random.default_rng(4)
    a = rng.standard_normal(1000)
    b = -a + 1e-9 * rng.standard_normal(1000)    # sums that cancel
    want = a + b
    scale = np.abs(a) + np.abs(b)
    gu.check_f32_sum(want + 0.9e-5 * scale, want, scale, "within 1e-5 of the summands")
    off = want.copy()
    off[9] += 2e-5 * scale[9]
    with pytest.raises(AssertionError):
        gu.check_f32_sum(off, want, scale, "2e-5 of the summands")
    with pytest.raises(AssertionError):
        gu.check_f32_sum(want - b, want, scale, "residual dropped")


def test_bf16_gate():
    want = _want(5)
    bits = oracle.bf16_from_double(want)
    scale = np.abs(want)
    gu.check_bf16(bits, want, scale, "the rounding of the definition")
    up = (bits.astype(np.int64) + 1).astype(np.uint16)       # one unit (same sign, no overflow)
    gu.check_bf16(up, want, scale, "one unit")
    two = bits.copy()
    two[11] = np.uint16(int(bits[11]) + 2)
    with pytest.raises(AssertionError):
        gu.check_bf16(two, want, scale, "two units off")
    tail = bits.copy()
    tail[-2:] = 0
    with pytest.raises(AssertionError):
        gu.check_bf16(tail, want, scale, "dropped tail")


def test_bf16_gate_under_cancellation():
    """A result that is small against its summands may sit a few units from
    the rounding of the definition, within one unit plus 1e-5 of the
    summands; beyond that the gate is red."""
    want = np.array([3.0e-4, -2.0e-4])
    scale = np.array([10.0, 10.0])
    bits = oracle.bf16_from_double(want)
    three = (bits.astype(np.int64) + 3).astype(np.uint16)
    gu.check_bf16(three, want, scale, "3 units under cancellation")
    far = oracle.bf16_from_double(want + 1e-3)
    with pytest.raises(AssertionError):
        gu.check_bf16(far, want, scale, "beyond 1e-5 of the summands")


def _q8_blocks(x, gamma, eps):
    """The oracle's own Q8_1 result laid out as the kernels write it: per block
    f16 d (bytes 0-1), s = 0 (bytes 2-3), 32 int8 codes."""
    d64, qreal, q64 = oracle.rmsnorm_q8_1(x.astype(np.float64), gamma.astype(np.float64),
                                          float(np.float32(eps)))
    rows, n = x.shape
    raw = np.zeros((rows, n // 32, 36), dtype=np.uint8)
    raw[:, :, 0:2] = oracle.f16_from_double(d64).astype(np.uint16)[..., None].view(np.uint8)
    raw[:, :, 4:36] = q64.reshape(rows, n // 32, 32).view(np.uint8)
    return raw, qreal, q64


def test_q8_1_gate():
    g = np.random.default_rng(6)
    rows, n, eps = 64, 2048, 1e-6                            # ~16 codes within the tie margin
    x = g.standard_normal((rows, n)).astype(np.float32)
    x[0, :32] = 0.0                                          # one all-zero block
    gamma = (1 + 0.1 * g.standard_normal(n)).astype(np.float32)
    raw, qreal, q64 = _q8_blocks(x, gamma, eps)
    one_off, near = gu.check_q8_1_blocks(raw, x, gamma, eps, "f32", what="exact")
    assert one_off == 0 and near > 0
    margin = np.abs(np.abs(qreal - np.floor(qreal)) - 0.5)
    inner = np.abs(q64.astype(np.int64)) < 127
    r_near, c_near = np.argwhere((margin < gu.Q8_TIE_MARGIN) & inner)[0]
    r_far, c_far = np.argwhere((margin > 0.1) & inner)[0]

    def code(r, c, delta):
        bad = raw.copy()
        bad[r, c // 32, 4 + c % 32] = np.uint8((int(q64[r, c]) + delta) & 0xFF)
        return bad

    gu.check_q8_1_blocks(code(r_near, c_near, 1), x, gamma, eps, "f32", what="near a tie")
    for bad, what in ((code(r_far, c_far, 1), "one off away from a tie"),
                      (code(r_near, c_near, 2), "two off"),
                      (code(0, 3, 1), "a code in an all-zero block")):
        with pytest.raises(AssertionError):
            gu.check_q8_1_blocks(bad, x, gamma, eps, "f32", what=what)
    s_bad = raw.copy()
    s_bad[2, 1, 2] = 1
    d_bad = raw.copy()
    d_bits = d_bad[3, 2, 0:2].view(np.uint16)
    d_bits += 2
    for bad, what in ((s_bad, "s not 0"), (d_bad, "d two f16 units off")):
        with pytest.raises(AssertionError):
            gu.check_q8_1_blocks(bad, x, gamma, eps, "f32", what=what)


def test_seam_gate():
    from dual_epsilon_sandwich_gb300 import workloads as wl
    d = wl.seam_rows(7, 8, 512, "f32", "f16")
    u, _, alt, _, near = gu.seam_expected(d["x"], d["gamma"], 1e-5, "f32", "f16")
    assert gu.check_seam_bits(u, u, alt, near, "exact") == 0
    assert near.any() and (~near).any()
    gu.check_seam_bits(np.where(near, alt, u), u, alt, near, "the other side of near ties")
    far = np.flatnonzero(~near.ravel())[0]
    bad = u.copy()
    bad.flat[far] = alt.flat[far]
    with pytest.raises(AssertionError):
        gu.check_seam_bits(bad, u, alt, near, "the other neighbour away from a tie")
    two = u.copy()
    two.flat[far] = np.uint16(int(u.flat[far]) + 2)
    with pytest.raises(AssertionError):
        gu.check_seam_bits(two, u, alt, near, "two units off")


def _sandwich_case():
    from dual_epsilon_sandwich_gb300 import workloads as wl
    w = wl.sandwich_decode()
    a = w.arrays
    args = (a["block_out"], a["residual"], a["gamma_post"], a["gamma_pre"], w.eps, w.eps_pre)
    e1, e2 = float(np.float32(w.eps)), float(np.float32(w.eps_pre))
    s, o = oracle.norm_residual_norm(*(a[k].astype(np.float64) for k in
                                       ("block_out", "residual", "gamma_post", "gamma_pre")),
                                     e1, e2)
    return args, s, o


def test_sandwich_strict_gate_on_normed():
    """normed: a 2e-5 relative error on a well-conditioned element is red even
    though the end-to-end (carried) bound would admit it; the same error on an
    element whose stream cancels is admitted by the end-to-end bound and
    counted as excused; the f32 rounding of the definition is green."""
    args, s, o = _sandwich_case()
    got_s, got_o = s.astype(np.float32), o.astype(np.float32)
    _, _, rep = gu.check_sandwich(got_s, got_o, *args, "f32", "rounded definition")
    assert rep["excused"] > 0 and rep["strict"] > 0.9 * o.size and rep["worst"] < 1e-7
    b, r, gp, gq = (np.asarray(v, dtype=np.float64) for v in args[:4])
    e1, e2 = float(np.float32(args[4])), float(np.float32(args[5]))
    scale_s = np.abs(oracle.rmsnorm(b, gp, e1)) + np.abs(r)
    kappa = gu.sandwich_normed_scale(s, gu.F32_TOL * scale_s, gq, e2) / gu.F32_TOL / np.abs(o)
    well = int(np.argmin(kappa))
    cancel = int(np.argmax(np.where(kappa < 1e3, kappa, 0.0)))
    assert kappa.flat[well] <= gu.KAPPA_STRICT < kappa.flat[cancel]
    bad = got_o.astype(np.float64)
    bad.flat[well] *= 1 + 2e-5
    with pytest.raises(AssertionError):
        gu.check_sandwich(got_s, bad, *args, "f32", "2e-5 on a well-conditioned element")
    ok = got_o.astype(np.float64)
    ok.flat[cancel] *= 1 + 2e-5
    _, _, rep2 = gu.check_sandwich(got_s, ok, *args, "f32", "2e-5 where the stream cancels")
    assert rep2["excused"] == rep["excused"]


def test_sandwich_strict_gate_bf16():
    """bf16 normed: two units off on an element whose stream cannot flip is red."""
    from dual_epsilon_sandwich_gb300 import workloads as wl
    w = wl.llama_bf16(rows=4, n=512)
    a = w.arrays
    x, r, g = a["x"], a["residual"], a["gamma"]
    X, R, G = gu.widen(x, "bf16"), gu.widen(r, "bf16"), gu.widen(g, "bf16")
    e1, e2 = float(np.float32(1e-8)), float(np.float32(1e-5))
    raw_s, _ = oracle.norm_residual_norm(X, R, G, G, e1, e2, stream_bf16=False)
    _, want_o = oracle.norm_residual_norm(X, R, G, G, e1, e2, stream_bf16=True)
    got_s, got_o = oracle.bf16_from_double(raw_s), oracle.bf16_from_double(want_o)
    _, _, rep = gu.check_sandwich(got_s, got_o, x, r, g, g, 1e-8, 1e-5, "bf16", "exact")
    assert rep["worst"] == 0 and rep["strict"] > 0.9 * want_o.size
    well = np.flatnonzero((gu.bf16_tie_distance(raw_s) > 1e-3 * np.abs(raw_s)).ravel()
                          & (np.abs(want_o) > 0.5).ravel())[0]
    bad = got_o.copy()
    bad.flat[well] = np.uint16(int(bad.flat[well]) + 2)
    with pytest.raises(AssertionError):
        gu.check_sandwich(got_s, bad, x, r, g, g, 1e-8, 1e-5, "bf16", "two units off")


def test_bf16_tie_distance():
    """Distance to the nearest bf16 rounding boundary: 0 on a midpoint, half a
    unit on a representable value, and monotone between."""
    one = 1.0
    ulp = 2.0 ** -7
    v = np.array([one, one + ulp / 2, one + ulp / 4, -one - ulp / 4, 0.0])
    d = gu.bf16_tie_distance(v)
    np.testing.assert_allclose(d[:4], [ulp / 2, 0.0, ulp / 4, ulp / 4])
    assert d[4] > 0
