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
