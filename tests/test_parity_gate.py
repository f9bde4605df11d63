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
    rows, n, eps = 8, 512, 1e-6
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
