"""The oracle's pins have power: every planted mistake fails at least one pin.

Each mutant is the oracle's own C source with one plausible error edited in (a
dropped term, a wrong sign, index or epsilon, a transposed operand, a rounding
slip).  It is compiled on the CPU into a temporary library and run through
every pin of ``oracle_pins``.  A mutant that passes them all means the pins
could not tell that mistake from the definition.
"""
import os

import pytest

import oracle
import oracle_pins

MUTANTS = [
    ("eps dropped", "return 1.0 / sqrt(mean_sq + eps);", "return 1.0 / sqrt(mean_sq);"),
    ("eps added to the sum, not the mean",
     "double mean_sq = sum_sq / (double)n;\n    return 1.0 / sqrt(mean_sq + eps);",
     "double mean_sq = (sum_sq + eps) / (double)n;\n    return 1.0 / sqrt(mean_sq);"),
    ("divide by n - 1", "sum_sq / (double)n", "sum_sq / (double)(n - 1)"),
    ("rms instead of its reciprocal", "return 1.0 / sqrt(", "return sqrt("),
    ("sum of |x| instead of x^2", "sum_sq += row[j] * row[j];", "sum_sq += fabs(row[j]);"),
    ("first element skipped", "for (int64_t j = 0; j < n; ++j)\n        sum_sq",
     "for (int64_t j = 1; j < n; ++j)\n        sum_sq"),
    ("gamma dropped", "yr[j] = xr[j] * inv_rms * gamma[j];", "yr[j] = xr[j] * inv_rms;"),
    ("gamma reversed", "yr[j] = xr[j] * inv_rms * gamma[j];",
     "yr[j] = xr[j] * inv_rms * gamma[n - 1 - j];"),
    ("then-add residual subtracted", "outr[j] = xr[j] * inv_rms * gamma[j] + rr[j];",
     "outr[j] = xr[j] * inv_rms * gamma[j] - rr[j];"),
    ("then-add residual dropped", "outr[j] = xr[j] * inv_rms * gamma[j] + rr[j];",
     "outr[j] = xr[j] * inv_rms * gamma[j];"),
    ("then-add residual row offset lost", "const double *rr = residual + r * n;\n        double *outr",
     "const double *rr = residual;\n        double *outr"),
    ("sandwich eps_post used for both", "row_inv_rms(sr, n, eps_pre)", "row_inv_rms(sr, n, eps_post)"),
    ("sandwich eps_pre used for both", "row_inv_rms(br, n, eps_post)", "row_inv_rms(br, n, eps_pre)"),
    ("sandwich second norm over block_out", "row_inv_rms(sr, n, eps_pre)", "row_inv_rms(br, n, eps_pre)"),
    ("sandwich gammas transposed (post)", "br[j] * inv_post * gamma_post[j] + rr[j]",
     "br[j] * inv_post * gamma_pre[j] + rr[j]"),
    ("sandwich gammas transposed (pre)", "sr[j] * inv_pre * gamma_pre[j]",
     "sr[j] * inv_pre * gamma_post[j]"),
    ("sandwich residual dropped", "br[j] * inv_post * gamma_post[j] + rr[j]",
     "br[j] * inv_post * gamma_post[j]"),
    ("sandwich residual row offset lost", "const double *rr = residual + r * n;\n        double *sr",
     "const double *rr = residual;\n        double *sr"),
    ("bf16 stream rounding skipped", "if (stream_bf16)", "if (0)"),
    ("add-norm: b dropped", "double s = ar[j] + br[j];", "double s = ar[j];"),
    ("add-norm: b subtracted", "double s = ar[j] + br[j];", "double s = ar[j] - br[j];"),
    ("add-norm: norm of a, not the sum", "double inv_rms = row_inv_rms(sr, n, eps);\n        for (int64_t j = 0; j < n; ++j)\n            nr[j]",
     "double inv_rms = row_inv_rms(ar, n, eps);\n        for (int64_t j = 0; j < n; ++j)\n            nr[j]"),
    ("add-norm: bf16 sum rounding skipped", "if (sum_bf16)", "if (0)"),
    ("add-norm: normed from a", "nr[j] = sr[j] * inv_rms * gamma[j];", "nr[j] = ar[j] * inv_rms * gamma[j];"),
    ("then-add-scale: scale dropped", "+ rr[j]) * out_scale;", "+ rr[j]);"),
    ("then-add-scale: scale on the norm only", "outr[j] = (xr[j] * inv_rms * gamma[j] + rr[j]) * out_scale;",
     "outr[j] = xr[j] * inv_rms * gamma[j] * out_scale + rr[j];"),
    ("q8: ties away from zero", "double r = nearbyint(qreal);", "double r = round(qreal);"),
    ("q8: truncation", "double r = nearbyint(qreal);", "double r = trunc(qreal);"),
    ("q8: clamp at 128", "if (r > 127.0)\n        r = 127.0;", "if (r > 128.0)\n        r = 128.0;"),
    ("q8: d = amax / 128", "double scale = amax / 127.0;", "double scale = amax / 128.0;"),
    ("q8: signed max", "if (fabs(normed[l]) > amax)\n                    amax = fabs(normed[l]);",
     "if (normed[l] > amax)\n                    amax = normed[l];"),
    ("q8: gamma dropped", "normed[l] = xr[j] * gamma[j] * inv_rms;", "normed[l] = xr[j] * inv_rms;"),
    ("q8: zero block divides by zero", "qreal[j] = (scale == 0.0) ? 0.0 : normed[l] / scale;",
     "qreal[j] = normed[l] / scale;"),
    ("f16: no carry", "if (q == 2048) {", "if (0) {"),
    ("f16: subnormal quantum", "(lead < -14) ? -24 : lead - 10", "(lead < -14) ? -25 : lead - 10"),
    ("f16: widening bias", "field - 15 - 10", "field - 15 - 11"),
    ("bf16 ties away from zero", "(frac == 0.5 && (q & 1u))", "(frac == 0.5)"),
    ("bf16 truncation", "if (frac > 0.5 || (frac == 0.5 && (q & 1u)))", "if (0)"),
    ("bf16 subnormal quantum", "(lead < -126) ? -133 : lead - 7", "(lead < -126) ? -134 : lead - 7"),
    ("bf16 no carry into next binade", "if (q == 256) {", "if (0) {"),
    ("bf16 widening exponent bias", "field - 127 - 7", "field - 127 - 8"),
    ("bf16 NaN as infinity", "v = frac ? NAN : INFINITY;", "v = INFINITY;"),
    ("seam: intermediate rounding skipped", "ur[j] = round_to_seam(xr[j] * inv_rms, seam_bf16);",
     "ur[j] = xr[j] * inv_rms;"),
    ("seam: second rounding skipped", "yr[j] = round_to_seam(ur[j] * gamma[j], seam_bf16);",
     "yr[j] = ur[j] * gamma[j];"),
    ("seam: gamma dropped", "yr[j] = round_to_seam(ur[j] * gamma[j], seam_bf16);",
     "yr[j] = round_to_seam(ur[j], seam_bf16);"),
    ("seam: weight on the unrounded product", "yr[j] = round_to_seam(ur[j] * gamma[j], seam_bf16);",
     "yr[j] = round_to_seam(xr[j] * inv_rms * gamma[j], seam_bf16);"),
    ("seam: formats swapped", "    if (seam_bf16)\n        return oracle_double_from_bf16",
     "    if (!seam_bf16)\n        return oracle_double_from_bf16"),
    ("seam: u row offset lost", "double *ur = u + r * n;", "double *ur = u;"),
    ("seam: eps dropped in the seam's norm", "double inv_rms = row_inv_rms(xr, n, eps);\n        /* first operation",
     "double inv_rms = row_inv_rms(xr, n, 0.0);\n        /* first operation"),
]


@pytest.fixture(scope="module")
def source():
    with open(oracle.SOURCE) as fh:
        return fh.read()


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, source, name, old, new):
    assert source.count(old) >= 1, f"mutation site for '{name}' no longer in oracle.c"
    src = tmp_path / "oracle.c"
    src.write_text(source.replace(old, new, 1))
    lib = oracle.compile_library(str(src), str(tmp_path / "libmutant.so"))
    mutant = oracle.Oracle(lib)
    failures = []
    for check in oracle_pins.ALL_CHECKS:
        try:
            check(mutant)
        except AssertionError as exc:
            failures.append(f"{check.__name__}: {str(exc)[:80]}")
    assert failures, f"no pin catches the mutant '{name}'"


def test_unmutated_copy_passes_every_pin(tmp_path, source):
    """Control: compiling the same source through the same route passes."""
    src = tmp_path / "oracle.c"
    src.write_text(source)
    mutant = oracle.Oracle(oracle.compile_library(str(src), str(tmp_path / "libcopy.so")))
    for check in oracle_pins.ALL_CHECKS:
        check(mutant)
