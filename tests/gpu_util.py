"""Helpers for the GPU parity tests: device buffers with guard bands, the
tolerance rules, and calls through the C ABI.

Tolerances (the contract the tests enforce):
* f32 outputs that are plain norms (rmsnorm y, sandwich normed):
  |gpu - oracle| <= 1e-5 * |oracle|, and an exact 0 where the oracle is 0.
* f32 outputs that are sums (then-add out, sandwich out_stream): the relative
  bound is taken against the size of the summands,
  |gpu - oracle| <= 1e-5 * (|x * inv * gamma| + |residual|), because a sum
  that cancels has no meaningful relative error.
* bf16 outputs: at most 1 unit in the last place from the round-to-nearest-even
  bf16 of the f64 oracle value, or |gpu - oracle| <= ulp(oracle) + 1e-5 *
  summands: the f32 accumulation tolerance plus one bf16 rounding.  The
  second clause only differs from the first under cancellation, where the
  result is small against its summands and the f32 error of the summands is
  no longer small against one bf16 ulp of the result.
* normed is checked against the oracle's own sandwich (the oracle never sees
  a GPU value) with its own bound plus the stream's bound carried through the
  second norm; for bf16 the stream may also land one bf16 ulp away from the
  oracle's rounded stream before it is re-normed.  On top of that end-to-end
  bound, every well-conditioned element of normed (condition number at most
  KAPPA_STRICT with respect to the stream) must meet the plain 1e-5 relative
  (f32) or 1 ulp (bf16) bound; the excused elements are counted.
* Q8_1 codes are integers decided in f32: equal to the oracle's, except one
  off where the oracle's quotient lies within Q8_TIE_MARGIN (derived from the
  f32 roundings of the kernels) of a rounding tie.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from dual_epsilon_sandwich_gb300 import mrn

F32_TOL = 1e-5
GUARD_BYTES = 64
SENTINEL = {"f32": 0x7FBADBAD, "bf16": 0x7FBD}   # NaN patterns no kernel produces


def elem_bytes(dtype):
    return 4 if dtype == "f32" else 2


def code(dtype):
    return mrn.MRN_F32 if dtype == "f32" else mrn.MRN_BF16


def to_device(a, dtype) -> torch.Tensor:
    """numpy f32 array or uint16 bf16 bit patterns -> CUDA tensor."""
    if dtype == "f32":
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()
    bits = np.ascontiguousarray(a, dtype=np.uint16).view(np.int16)
    return torch.from_numpy(bits).cuda().view(torch.bfloat16)


def widen(a, dtype) -> np.ndarray:
    """Host array (f32 or bf16 bits) -> exact float64."""
    if dtype == "f32":
        return np.asarray(a, dtype=np.float32).astype(np.float64)
    return oracle.double_from_bf16(a)


def to_host(t: torch.Tensor, dtype) -> np.ndarray:
    """CUDA tensor -> f32 array or uint16 bit patterns."""
    t = t.detach().cpu().contiguous()
    if dtype == "f32":
        return t.numpy()
    return t.view(torch.int16).numpy().view(np.uint16)


class Guarded:
    """An output buffer [rows x n] inside a larger allocation whose guard bands
    (64 bytes before and after) and body are prefilled with a sentinel NaN."""

    def __init__(self, rows, n, dtype, offset_elems=0):
        self.dtype = dtype
        e = elem_bytes(dtype)
        self.guard = GUARD_BYTES // e
        self.off = self.guard + offset_elems
        self.count = rows * n
        total = self.off + self.count + self.guard
        itype = torch.int32 if dtype == "f32" else torch.int16
        sent = SENTINEL[dtype]
        if dtype == "bf16":
            sent = np.int16(np.uint16(sent))
        else:
            sent = np.int32(np.uint32(sent))
        self.raw = torch.full((total,), int(sent), dtype=itype, device="cuda")
        self.sentinel = int(sent)
        ftype = torch.float32 if dtype == "f32" else torch.bfloat16
        self.tensor = self.raw[self.off:self.off + self.count].view(ftype).view(rows, n)

    def ptr(self):
        return self.tensor.data_ptr()

    def check(self, what=""):
        raw = self.raw
        head = raw[:self.off]
        tail = raw[self.off + self.count:]
        assert bool((head == self.sentinel).all()), f"{what}: write before the output"
        assert bool((tail == self.sentinel).all()), f"{what}: write after the output"
        body = raw[self.off:self.off + self.count]
        unwritten = int((body == self.sentinel).sum())
        assert unwritten == 0, f"{what}: {unwritten} outputs never written"

    def host(self):
        return to_host(self.tensor, self.dtype)


# ---------------------------------------------------------------------------
# tolerance checks (return the worst error seen, for reporting)
# ---------------------------------------------------------------------------
def check_f32_norm(got, want, what):
    got = np.asarray(got, dtype=np.float64)
    zero = want == 0
    assert np.all(got[zero] == 0), f"{what}: nonzero output where the oracle is 0"
    err = np.abs(got - want)
    bad = err > F32_TOL * np.abs(want)
    if np.any(bad):
        i = np.flatnonzero(bad.ravel())[:5]
        raise AssertionError(f"{what}: {bad.sum()} elements over 1e-5 relative; e.g. "
                             f"got {got.ravel()[i]} want {want.ravel()[i]}")
    nz = ~zero
    return float(np.max(err[nz] / np.abs(want[nz]))) if np.any(nz) else 0.0


def check_f32_sum(got, want, scale, what):
    got = np.asarray(got, dtype=np.float64)
    err = np.abs(got - want)
    bad = err > F32_TOL * scale
    if np.any(bad):
        i = np.flatnonzero(bad.ravel())[:5]
        raise AssertionError(f"{what}: {bad.sum()} elements over 1e-5 of the summands; e.g. "
                             f"got {got.ravel()[i]} want {want.ravel()[i]} "
                             f"scale {scale.ravel()[i]}")
    pos = scale > 0
    return float(np.max(err[pos] / scale[pos])) if np.any(pos) else 0.0


def _ordered(bits):
    b = bits.astype(np.int64)
    return np.where(b & 0x8000, -(b & 0x7FFF), b & 0x7FFF)


def bf16_ulp(v):
    a = np.maximum(np.abs(v), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(a)) - 7)


def check_bf16(got_bits, want, scale, what):
    """got_bits: uint16; want: f64 oracle; scale: size of the summands (or |want|).

    Pass: at most 1 ulp from the bf16 rounding of the oracle value, or -- where
    the f32 tolerance on the summands is not small against one bf16 ulp of the
    result, i.e. under cancellation -- within one ulp plus that f32 tolerance.
    Returns (max ulp distance, number of elements that needed the second clause)."""
    exp_bits = oracle.bf16_from_double(want)
    dist = np.abs(_ordered(got_bits) - _ordered(exp_bits))
    got = oracle.double_from_bf16(got_bits)
    within_ulp = dist <= 1
    cancel = np.abs(got - want) <= bf16_ulp(want) + F32_TOL * scale
    ok = within_ulp | cancel
    if not np.all(ok):
        i = np.flatnonzero(~ok.ravel())[:5]
        raise AssertionError(f"{what}: {np.sum(~ok)} elements beyond 1 bf16 ulp; e.g. got "
                             f"{got.ravel()[i]} want {want.ravel()[i]} ulps {dist.ravel()[i]}")
    return int(dist.max()), int(np.sum(~within_ulp))


# ---------------------------------------------------------------------------
# C-ABI calls on torch buffers (pointers and sizes only)
# ---------------------------------------------------------------------------
def stream_handle():
    return torch.cuda.current_stream().cuda_stream


def call_rmsnorm(x, g, y, rows, n, eps, dtype):
    return mrn.mrn_rmsnorm(x.data_ptr(), g.data_ptr(), _p(y), rows, n, eps, code(dtype),
                           stream_handle())


def call_then_add(x, g, r, out, rows, n, eps, dtype):
    return mrn.mrn_rmsnorm_then_add(x.data_ptr(), g.data_ptr(), r.data_ptr(), _p(out), rows, n,
                                    eps, code(dtype), stream_handle())


def call_sandwich(b, r, gp, gq, s, o, rows, n, eps_post, eps_pre, dtype):
    return mrn.mrn_norm_residual_norm(b.data_ptr(), r.data_ptr(), gp.data_ptr(), gq.data_ptr(),
                                      _p(s), _p(o), rows, n, eps_post, eps_pre, code(dtype),
                                      stream_handle())


def _p(t):
    return t.ptr() if isinstance(t, Guarded) else t.data_ptr()


# ---------------------------------------------------------------------------
# whole-operation parity: run on the GPU, compare with the oracle
# ---------------------------------------------------------------------------
def parity_rmsnorm(x, gamma, eps, dtype, rows_sample=None, what="rmsnorm"):
    rows, n = x.shape
    dx, dg = to_device(x, dtype), to_device(gamma, dtype)
    y = Guarded(rows, n, dtype)
    st = call_rmsnorm(dx, dg, y, rows, n, eps, dtype)
    assert st == 0, f"{what}: status {mrn.STATUS.get(st)}"
    torch.cuda.synchronize()
    y.check(what)
    got = y.host()
    sel = slice(None) if rows_sample is None else rows_sample
    xs, gs = widen(x[sel], dtype), widen(gamma, dtype)
    want = oracle.rmsnorm(xs, gs, float(np.float32(eps)))
    if dtype == "f32":
        return check_f32_norm(got[sel], want, what)
    return check_bf16(got[sel], want, np.abs(want), what)


def parity_then_add(x, gamma, res, eps, dtype, rows_sample=None, what="then_add"):
    rows, n = x.shape
    dx, dg, dr = to_device(x, dtype), to_device(gamma, dtype), to_device(res, dtype)
    out = Guarded(rows, n, dtype)
    st = call_then_add(dx, dg, dr, out, rows, n, eps, dtype)
    assert st == 0, f"{what}: status {mrn.STATUS.get(st)}"
    torch.cuda.synchronize()
    out.check(what)
    got = out.host()
    sel = slice(None) if rows_sample is None else rows_sample
    xs, gs, rs = widen(x[sel], dtype), widen(gamma, dtype), widen(res[sel], dtype)
    e = float(np.float32(eps))
    want = oracle.rmsnorm_then_add(xs, gs, rs, e)
    scale = np.abs(oracle.rmsnorm(xs, gs, e)) + np.abs(rs)
    if dtype == "f32":
        return check_f32_sum(got[sel], want, scale, what)
    return check_bf16(got[sel], want, scale, what)


def sandwich_normed_scale(want_s, stream_err, gq, eps_pre):
    """Propagated error bound of `normed` per element, from an error bound
    `stream_err` of each stream element (oracle values only):
    normed_j = s_j * inv2 * g_j with inv2 = 1/sqrt(mean(s^2) + eps), so
    |d normed_j| <= inv2 |g_j| (|d s_j| + |s_j| * mean(|s| |d s|) / (mean(s^2) + eps))."""
    ms = np.mean(want_s * want_s, axis=1, keepdims=True)
    inv2 = 1.0 / np.sqrt(ms + eps_pre)
    rel = np.mean(np.abs(want_s) * stream_err, axis=1, keepdims=True) / (ms + eps_pre)
    return inv2 * np.abs(gq) * (stream_err + np.abs(want_s) * rel)


# Strict gate on `normed`: the stated plain "<= 1e-5 relative" (f32) or
# "<= 1 bf16 ulp" (bf16), asserted on every element whose problem is well
# conditioned.  The condition number of normed_j with respect to the stream,
# kappa_j = carried_j / (1e-5 |o_j|) with `carried` the stream's 1e-5-of-the-
# summands bound pushed through the second norm, is >= 2 by construction and
# large only where the stream cancels (|s_j| small against |x inv gamma| +
# |r|).  The kernels' f32 arithmetic perturbs the stream by well under 1e-6
# of its summands (an f32 reduction tree of a few dozen levels at 2^-24 each,
# then a few roundings), so where kappa_j <= KAPPA_STRICT the GPU's normed_j
# lies within ~1e-6 * 10 of the oracle's: inside 1e-5 relative with margin.
KAPPA_STRICT = 10.0


def bf16_tie_distance(v):
    """|v - m| for the rounding boundary m (the midpoint between two bf16
    neighbours) nearest to each f64 value v: a value that far from every
    boundary rounds to the same bf16 under any perturbation smaller than it."""
    v = np.asarray(v, dtype=np.float64)
    bits = oracle.bf16_from_double(v)
    r = oracle.double_from_bf16(bits)
    up = oracle.double_from_bf16(_seam_step(bits, v >= r))
    with np.errstate(invalid="ignore"):
        mid = np.where(np.isfinite(up), (r + np.where(np.isfinite(up), up, 0.0)) / 2, np.inf)
    return np.abs(v - mid)


def check_sandwich(got_s, got_o, b, res, gp, gq, eps_post, eps_pre, dtype, what="sandwich"):
    """Both sandwich outputs (host arrays of the selected rows) against the
    oracle's own sandwich of the same inputs (the oracle never sees a GPU value).

    out_stream: the sum rule.  normed, end to end: its own relative bound plus
    the stream's bound carried through the second norm (for bf16 the stream
    may also land one bf16 ulp away from the oracle's rounded stream before it
    is re-normed).  normed, strict: 1e-5 relative (f32) / 1 ulp (bf16) on the
    well-conditioned elements (KAPPA_STRICT); the excused rest is counted.
    Returns (stream result, normed result, strict report dict)."""
    bs, rs = widen(b, dtype), widen(res, dtype)
    gps, gqs = widen(gp, dtype), widen(gq, dtype)
    e1, e2 = float(np.float32(eps_post)), float(np.float32(eps_pre))
    scale_s = np.abs(oracle.rmsnorm(bs, gps, e1)) + np.abs(rs)
    if dtype == "f32":
        want_s, want_o = oracle.norm_residual_norm(bs, rs, gps, gqs, e1, e2)
        es = check_f32_sum(got_s, want_s, scale_s, what + " out_stream")
        carried = sandwich_normed_scale(want_s, F32_TOL * scale_s, gqs, e2) / F32_TOL
        eo = check_f32_sum(got_o, want_o, np.abs(want_o) + carried, what + " normed")
        strict = carried <= KAPPA_STRICT * np.abs(want_o)
        worst = check_f32_norm(np.asarray(got_o)[strict], want_o[strict],
                               what + " normed (strict 1e-5 relative, kappa <= 10)")
    else:
        # bf16: the oracle rounds its own stream before the second norm
        raw_s, _ = oracle.norm_residual_norm(bs, rs, gps, gqs, e1, e2, stream_bf16=False)
        want_s, want_o = oracle.norm_residual_norm(bs, rs, gps, gqs, e1, e2, stream_bf16=True)
        es = check_bf16(got_s, raw_s, scale_s, what + " out_stream")
        stream_err = bf16_ulp(raw_s) + F32_TOL * scale_s
        carried = sandwich_normed_scale(want_s, stream_err, gqs, e2)
        eo = check_bf16(got_o, want_o, np.abs(want_o) + carried / F32_TOL, what + " normed")
        # strict: a stream element can round to the other bf16 neighbour only
        # where its exact value lies within the f32 stream error of a rounding
        # boundary; elsewhere the GPU stores the oracle's rounded stream.  Where
        # the remaining error (own f32 error plus what the stream carries) is
        # under one ulp of o, the two roundings are at most one unit apart.
        f32_err = F32_TOL * scale_s
        may_flip = bf16_tie_distance(raw_s) <= f32_err
        carried_strict = sandwich_normed_scale(want_s, f32_err + may_flip * bf16_ulp(raw_s),
                                               gqs, e2)
        strict = carried_strict + F32_TOL * np.abs(want_o) < bf16_ulp(want_o)
        exp_bits = oracle.bf16_from_double(want_o[strict])
        dist = np.abs(_ordered(np.asarray(got_o)[strict]) - _ordered(exp_bits))
        if dist.size and dist.max() > 1:
            i = np.flatnonzero(dist > 1)[:5]
            raise AssertionError(f"{what} normed (strict 1 ulp): {int(np.sum(dist > 1))} "
                                 f"elements beyond one bf16 ulp; ulps {dist[i]}")
        worst = int(dist.max()) if dist.size else 0
    report = {"strict": int(strict.sum()), "excused": int(strict.size - strict.sum()),
              "worst": worst}
    print(f"{what}: normed strict on {report['strict']} of {strict.size} elements "
          f"({report['excused']} excused, stream near cancellation), worst "
          f"{'relative error' if dtype == 'f32' else 'ulps'} {worst:.3g}")
    return es, eo, report


def parity_sandwich(b, res, gp, gq, eps_post, eps_pre, dtype, rows_sample=None,
                    what="sandwich", inplace=None, report=None):
    """inplace: None, "residual" (out_stream == residual) or "block_out".

    Runs the fused tail on the GPU and applies check_sandwich to the selected
    rows; returns (stream result, normed result) and fills `report` (a dict)
    with the strict gate's counts when given."""
    rows, n = b.shape
    db, dr = to_device(b, dtype), to_device(res, dtype)
    dgp, dgq = to_device(gp, dtype), to_device(gq, dtype)
    o = Guarded(rows, n, dtype)
    if inplace == "residual":
        s_t = dr
    elif inplace == "block_out":
        s_t = db
    else:
        s_t = Guarded(rows, n, dtype)
    st = call_sandwich(db, dr, dgp, dgq, s_t, o, rows, n, eps_post, eps_pre, dtype)
    assert st == 0, f"{what}: status {mrn.STATUS.get(st)}"
    torch.cuda.synchronize()
    o.check(what + " normed")
    if isinstance(s_t, Guarded):
        s_t.check(what + " out_stream")
        got_s = s_t.host()
    else:
        got_s = to_host(s_t, dtype)
    got_o = o.host()
    sel = slice(None) if rows_sample is None else rows_sample
    es, eo, rep = check_sandwich(got_s[sel], got_o[sel], b[sel], res[sel], gp, gq, eps_post,
                                 eps_pre, dtype, what)
    if report is not None:
        report.update(rep)
    return es, eo


def call_add_rmsnorm(a, b, g, s, o, rows, n, eps, dtype):
    return mrn.mrn_add_rmsnorm(a.data_ptr(), b.data_ptr(), g.data_ptr(), _p(s), _p(o), rows, n,
                               eps, code(dtype), stream_handle())


def call_then_add_scale(x, g, r, sc, out, rows, n, eps, dtype):
    return mrn.mrn_rmsnorm_then_add_scale(x.data_ptr(), g.data_ptr(), r.data_ptr(),
                                          sc.data_ptr(), _p(out), rows, n, eps, code(dtype),
                                          stream_handle())


def parity_add_rmsnorm(a, b, gamma, eps, dtype, rows_sample=None, what="add_rmsnorm",
                       inplace=None):
    """inplace: None, "a" or "b" (residual_out == that input)."""
    rows, n = a.shape
    da, db, dg = to_device(a, dtype), to_device(b, dtype), to_device(gamma, dtype)
    o = Guarded(rows, n, dtype)
    s_t = {"a": da, "b": db}.get(inplace) if inplace else Guarded(rows, n, dtype)
    st = call_add_rmsnorm(da, db, dg, s_t, o, rows, n, eps, dtype)
    assert st == 0, f"{what}: status {mrn.STATUS.get(st)}"
    torch.cuda.synchronize()
    o.check(what + " normed")
    if isinstance(s_t, Guarded):
        s_t.check(what + " residual_out")
        got_s = s_t.host()
    else:
        got_s = to_host(s_t, dtype)
    got_o = o.host()
    sel = slice(None) if rows_sample is None else rows_sample
    as_, bs, gs = widen(a[sel], dtype), widen(b[sel], dtype), widen(gamma, dtype)
    e = float(np.float32(eps))
    if dtype == "f32":
        want_s, want_o = oracle.add_rmsnorm(as_, bs, gs, e)
        # the f32 sum of two f32 values is correctly rounded: bit-exact
        assert np.array_equal(got_s[sel], want_s.astype(np.float32)), what + " residual_out"
        return check_f32_norm(got_o[sel], want_o, what + " normed")
    raw_s, _ = oracle.add_rmsnorm(as_, bs, gs, e, sum_bf16=False)
    want_s, want_o = oracle.add_rmsnorm(as_, bs, gs, e, sum_bf16=True)
    check_bf16(got_s[sel], raw_s, np.abs(as_) + np.abs(bs), what + " residual_out")
    carried = sandwich_normed_scale(want_s, bf16_ulp(raw_s), gs, e)
    return check_bf16(got_o[sel], want_o, np.abs(want_o) + carried / F32_TOL, what + " normed")


def parity_then_add_scale(x, gamma, res, scale, eps, dtype, rows_sample=None,
                          what="then_add_scale"):
    rows, n = x.shape
    dx, dg, dr = to_device(x, dtype), to_device(gamma, dtype), to_device(res, dtype)
    sc_host = np.array([scale], dtype=np.float32)
    if dtype == "bf16":
        sc_host = oracle.bf16_from_double(sc_host.astype(np.float64))
    dsc = to_device(sc_host, dtype)
    out = Guarded(rows, n, dtype)
    st = call_then_add_scale(dx, dg, dr, dsc, out, rows, n, eps, dtype)
    assert st == 0, f"{what}: status {mrn.STATUS.get(st)}"
    torch.cuda.synchronize()
    out.check(what)
    got = out.host()
    sel = slice(None) if rows_sample is None else rows_sample
    xs, gs, rs = widen(x[sel], dtype), widen(gamma, dtype), widen(res[sel], dtype)
    s64 = float(widen(sc_host, dtype)[0])
    e = float(np.float32(eps))
    want = oracle.rmsnorm_then_add_scale(xs, gs, rs, s64, e)
    scale_t = (np.abs(oracle.rmsnorm(xs, gs, e)) + np.abs(rs)) * abs(s64)
    if dtype == "f32":
        return check_f32_sum(got[sel], want, scale_t, what)
    return check_bf16(got[sel], want, scale_t, what)


# How far the GPU's f32 quotient x_normed * 127 / amax can sit from the
# oracle's exact one.  x_normed_j = fl(fl(x_j gamma_j) * inv) and amax is the
# largest |x_normed| of the block, so the row's inv (and its f32 error)
# cancels from the ratio x_normed_j / amax; what is left is two roundings on
# x_normed_j and two on amax (the x * gamma product is exact for bf16; one
# rounding for f32), the block reciprocal 127 / amax by the approximate
# divide (at most 2 ulp = 4 units of 2^-24 relative), and the fma that adds
# 1.5 * 2^23, whose single rounding is the integer rounding itself.  The
# exact path (x_normed / fl(amax / 127)) has fewer.  So the quotient moves by
# at most 8 * 2^-24 relative, and |quotient| <= 127.
Q8_TIE_MARGIN = 127 * 8 * 2.0 ** -24   # ~6.06e-5: codes this close to a tie may differ by one


def decode_q8_1(raw):
    """uint8 [rows, n/32, 36] -> (d f16 bits [rows, n/32], s bits, q int8 [rows, n])."""
    raw = np.ascontiguousarray(raw)
    d_bits = raw[:, :, 0:2].copy().view(np.uint16)[:, :, 0]
    s_bits = raw[:, :, 2:4].copy().view(np.uint16)[:, :, 0]
    q = raw[:, :, 4:36].copy().view(np.int8).reshape(raw.shape[0], -1)
    return d_bits, s_bits, q


def f16_ulps(a_bits, b_bits):
    def ordered(b):
        b = b.astype(np.int64)
        return np.where(b & 0x8000, -(b & 0x7FFF), b & 0x7FFF)
    return np.abs(ordered(a_bits) - ordered(b_bits))


def parity_q8_1(x, gamma, eps, dtype, rows_sample=None, what="q8_1", x_offset=0, y_offset=0):
    """RMSNorm + Q8_1 against the oracle: header s == 0, d within one f16 ulp
    of the oracle's d, codes equal except within Q8_TIE_MARGIN of a tie (one
    off allowed there: the GPU's f32 norm may land on the other side of a
    tie), zero blocks exactly zero.  64-byte guard bands around the blocks,
    which start y_offset bytes past a 16-byte boundary."""
    rows, n = x.shape
    if x_offset:
        base = to_device(np.concatenate([np.zeros(x_offset, x.dtype), x.ravel()]), dtype)
        dx = base[x_offset:].view(rows, n)
    else:
        dx = to_device(x, dtype)
    dg = to_device(gamma, dtype)
    nb = n // 32
    guard = 64
    raw = torch.full((rows * nb * 36 + 2 * guard + y_offset,), 0xA5, dtype=torch.uint8,
                     device="cuda")
    lo = guard + y_offset
    blocks = raw[lo:lo + rows * nb * 36]
    assert blocks.data_ptr() % 16 == y_offset % 16
    st = mrn.mrn_rmsnorm_q8_1(dx.data_ptr(), dg.data_ptr(), blocks.data_ptr(), rows, n, eps,
                              code(dtype), stream_handle())
    assert st == 0, f"{what}: status {mrn.STATUS.get(st)}"
    torch.cuda.synchronize()
    host = raw.cpu().numpy()
    assert np.all(host[:lo] == 0xA5) and np.all(host[-guard:] == 0xA5), what + ": guard bands"
    return check_q8_1_blocks(host[lo:-guard], x, gamma, eps, dtype, rows_sample, what)


def check_q8_1_blocks(host_blocks, x, gamma, eps, dtype, rows_sample=None, what="q8_1"):
    """The checks of parity_q8_1 on the blocks as bytes on the host (rows x n/32
    blocks of 36 bytes): s == 0, d within one f16 ulp of the oracle's, zero
    blocks zero, codes equal except one off within Q8_TIE_MARGIN of a tie.
    Returns (codes one off, elements near a tie)."""
    rows, n = x.shape
    nb = n // 32
    d_bits, s_bits, q = decode_q8_1(np.asarray(host_blocks).reshape(rows, nb, 36))
    sel = slice(None) if rows_sample is None else rows_sample
    d64, qreal, q64 = oracle.rmsnorm_q8_1(widen(x[sel], dtype), widen(gamma, dtype),
                                          float(np.float32(eps)))
    assert np.all(s_bits[sel] == 0), what + ": s must be 0"
    ulps = f16_ulps(d_bits[sel], oracle.f16_from_double(d64))
    assert ulps.max() <= 1, f"{what}: d off by {ulps.max()} f16 ulps"
    zero = np.repeat(d64 == 0, 32, axis=1)
    assert np.all(q[sel][zero] == 0), what + ": zero blocks"
    margin = np.abs(np.abs(qreal - np.floor(qreal)) - 0.5)
    diff = np.abs(q[sel].astype(np.int64) - q64.astype(np.int64))
    near_tie = margin < Q8_TIE_MARGIN
    bad = (diff > 1) | ((diff == 1) & ~near_tie)
    if np.any(bad):
        i = np.flatnonzero(bad.ravel())[:5]
        raise AssertionError(f"{what}: {bad.sum()} codes differ; got {q[sel].ravel()[i]} "
                             f"want {q64.ravel()[i]} qreal {qreal.ravel()[i]}")
    one_off, near = int(np.sum(diff == 1)), int(near_tie.sum())
    print(f"{what}: {one_off} codes one off, {near} of {diff.size} within "
          f"{Q8_TIE_MARGIN:.2e} of a tie")
    return one_off, near


def sample_rows(rows, count, seed, must=()):
    g = np.random.Generator(np.random.PCG64(seed))
    pick = set(int(v) for v in g.choice(rows, size=min(rows, count), replace=False))
    pick.update(int(v) for v in must)
    pick.update({0, rows - 1})
    return np.array(sorted(pick))


# ---------------------------------------------------------------------------
# Split-norm seam: u = S(x * inv), y = S(u * gamma), S = binary16 or bf16
# ---------------------------------------------------------------------------
SEAM_TIE_MARGIN = 2e-5     # relative distance of x * inv to an S rounding tie


def seam_code(seam):
    return mrn.MRN_F16 if seam == "f16" else mrn.MRN_BF16


def seam_bits_from_double(v, seam):
    return oracle.f16_from_double(v) if seam == "f16" else oracle.bf16_from_double(v)


def seam_double_from_bits(bits, seam):
    return oracle.double_from_f16(bits) if seam == "f16" else oracle.double_from_bf16(bits)


def _seam_step(bits, up):
    """The neighbouring S pattern above (up) or below; signed-magnitude order."""
    o = _ordered(bits) + np.where(up, 1, -1)
    return np.where(o >= 0, o, 0x8000 | (-o)).astype(np.uint16)


def seam_expected(x, gamma_bits, eps, dtype, seam, rows_sample=None):
    """Oracle bit patterns of u and y, the other admissible pair (u', y') for
    elements whose x * inv lies within SEAM_TIE_MARGIN of a tie between u and
    its neighbour (the GPU's f32 norm may round to either side there), and
    the near-tie mask."""
    sel = slice(None) if rows_sample is None else rows_sample
    x64 = widen(x[sel], dtype)
    g64 = seam_double_from_bits(gamma_bits, seam)
    e = float(np.float32(eps))
    u, y = oracle.rmsnorm_seam(x64, g64, e, seam)
    p = oracle.rmsnorm(x64, np.ones(x64.shape[1]), e)          # x * inv in f64
    u_bits = seam_bits_from_double(u, seam)
    y_bits = seam_bits_from_double(y, seam)
    alt_bits = _seam_step(u_bits, p > u)
    alt = seam_double_from_bits(alt_bits, seam)
    finite = np.isfinite(alt) & np.isfinite(u)
    mid = np.where(finite, (u + np.where(finite, alt, 0.0)) / 2, np.inf)
    near = np.abs(p - mid) <= SEAM_TIE_MARGIN * np.abs(p)
    y_alt_bits = seam_bits_from_double(np.where(finite, alt, 0.0) * g64, seam)
    return u_bits, y_bits, alt_bits, y_alt_bits, near


def check_seam_bits(got, want, alt, near, what):
    """got == want, or got == alt where near."""
    got = np.asarray(got, dtype=np.uint16)
    ok = (got == want) | (near & (got == alt))
    if not np.all(ok):
        i = np.flatnonzero(~ok.ravel())[:5]
        raise AssertionError(f"{what}: {int((~ok).sum())} of {ok.size} differ; got "
                             f"{[hex(v) for v in got.ravel()[i]]} want "
                             f"{[hex(v) for v in np.asarray(want).ravel()[i]]}")
    return int(np.sum(near & (got == alt) & (got != want)))


def _guarded_16(rows, n):
    raw = torch.full((rows * n * 2 + 2 * GUARD_BYTES,), 0xA5, dtype=torch.uint8, device="cuda")
    return raw, raw[GUARD_BYTES:GUARD_BYTES + rows * n * 2].view(torch.int16)


def _unguard_16(raw, rows, n, what):
    host = raw.cpu().numpy()
    assert np.all(host[:GUARD_BYTES] == 0xA5) and np.all(host[-GUARD_BYTES:] == 0xA5), \
        what + ": guard bands"
    return host[GUARD_BYTES:-GUARD_BYTES].copy().view(np.uint16).reshape(rows, n)


def run_seam(x, gamma_bits, eps, dtype, seam, x_offset=0):
    """(u, y_split, y_fused) bit patterns from the GPU: the weightless norm, the
    split route's scale of it, and the fused kernel, each in guarded buffers."""
    rows, n = x.shape
    if x_offset:
        base = to_device(np.concatenate([np.zeros(x_offset, x.dtype), x.ravel()]), dtype)
        dx = base[x_offset:].view(rows, n)
    else:
        dx = to_device(x, dtype)
    dg = torch.from_numpy(np.ascontiguousarray(gamma_bits).view(np.int16)).cuda()
    ru, du = _guarded_16(rows, n)
    rs, ds = _guarded_16(rows, n)
    rf, df = _guarded_16(rows, n)
    sh, sc = stream_handle(), seam_code(seam)
    st = mrn.mrn_rmsnorm_unweighted(dx.data_ptr(), du.data_ptr(), rows, n, eps, code(dtype), sc, sh)
    assert st == 0, f"unweighted: status {mrn.STATUS.get(st)}"
    st = mrn.mrn_seam_scale(du.data_ptr(), dg.data_ptr(), ds.data_ptr(), rows, n, sc, sh)
    assert st == 0, f"seam_scale: status {mrn.STATUS.get(st)}"
    st = mrn.mrn_rmsnorm_seam(dx.data_ptr(), dg.data_ptr(), df.data_ptr(), rows, n, eps,
                              code(dtype), sc, sh)
    assert st == 0, f"seam: status {mrn.STATUS.get(st)}"
    torch.cuda.synchronize()
    return (_unguard_16(ru, rows, n, "u"), _unguard_16(rs, rows, n, "split y"),
            _unguard_16(rf, rows, n, "fused y"))


def parity_seam(x, gamma_bits, eps, dtype, seam, rows_sample=None, what="seam", x_offset=0):
    """All three seam calls against the oracle (u and y, near-tie alternatives
    admitted), and the fused y bit-identical to the split route's y."""
    u, ys, yf = run_seam(x, gamma_bits, eps, dtype, seam, x_offset)
    assert np.array_equal(yf, ys), f"{what}: fused differs from split in " \
                                   f"{int(np.sum(yf != ys))} elements"
    sel = slice(None) if rows_sample is None else rows_sample
    ub, yb, ab, yab, near = seam_expected(x, gamma_bits, eps, dtype, seam, rows_sample)
    flips = check_seam_bits(u[sel], ub, ab, near, what + " u")
    check_seam_bits(yf[sel], yb, yab, near, what + " y")
    return flips, int(near.sum())
