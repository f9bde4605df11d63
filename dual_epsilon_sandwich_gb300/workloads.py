"""Seeded synthetic inputs for the RMSNorm / then-add / sandwich-tail workloads.

This module only draws random numbers and lays them out; it holds none of the
normalisation arithmetic.  Both the CUDA path and the CPU oracle receive the
arrays it returns (the oracle after an exact widening to float64).

Recipes (the pages name no dataset; every input is synthetic):

* ``plain_decode_rows``   rows=4,  n=6656, f32: x ~ N(0,1); gamma = 1 + 0.1 N(0,1);
  eps = 1e-5.  n = 6656 is the stream width of the model in "Chapter 12 --
  RMSNorm and the dual-epsilon sandwich", section 12.1.
* ``sandwich_decode``     rows=1,  n=6656, f32: block_out ~ N(0, 4) (variance 4,
  i.e. standard deviation 2), residual ~ N(0,1), gamma_post and gamma_pre =
  1 + 0.1 N(0,1); eps_post = 1e-8, eps_pre = 1e-5 (section 12.2, "The two
  epsilons, precisely").
* ``sandwich_prefill``    rows=4096, n=6656, f32: as above, and each block_out row
  is rescaled so that its mean of squares equals 10^U(-4, 2) (log-uniform over
  1e-4 .. 1e2) before rounding to f32.
* ``llama_bf16``          rows=16384, n=4096, bf16 I/O: x = N(0,1) * 10^U(-2, 2) per
  row; gamma = 1 + 0.1 N(0,1); residual ~ N(0,1); all rounded to bf16 (round to
  nearest even, via torch); eps = 1e-6.
* ``sweep``               f32, n in {2, 7, 768, 2048, 5120, 6656, 8192, 16384, 65536}
  x rows in {1, 64, 4096, 65536} (shapes above 4 GiB per operand skipped):
  x ~ N(0,1) and residual ~ N(0,1) drawn directly in float32; round(0.01 * rows)
  rows of x set to zero, picked by a seeded permutation.

Generation is numpy ``Generator(PCG64)``; f32 data of the small cases is drawn
in float64 and rounded once.  Seeds: 20261202 + the workload's index (1..5), and
``SeedSequence([20261202, 5, n, rows])`` for each sweep shape.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

SEED_BASE = 20261202
STREAM_WIDTH = 6656          # hidden width of the pages' model

SWEEP_N = (2, 7, 768, 2048, 5120, 6656, 8192, 16384, 65536)
SWEEP_ROWS = (1, 64, 4096, 65536)
SWEEP_EPS = (1e-5, 1e-8)
SWEEP_MAX_BYTES = 4 << 30    # per f32 operand


def rng(seed) -> np.random.Generator:
    if isinstance(seed, np.random.SeedSequence):
        return np.random.Generator(np.random.PCG64(seed))
    return np.random.Generator(np.random.PCG64(int(seed)))


def to_f32(a) -> np.ndarray:
    """IEEE round-to-nearest-even from float64 to float32 (numpy cast)."""
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64).astype(np.float32))


def to_bf16_bits(a) -> np.ndarray:
    """Round to bf16 through torch's float32 -> bfloat16 conversion; uint16 bits."""
    import torch
    f = torch.from_numpy(np.ascontiguousarray(np.asarray(a, dtype=np.float32)))
    return f.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def to_f16_bits(a) -> np.ndarray:
    """Round to IEEE binary16 through numpy's float64 -> float16 cast; uint16 bits."""
    with np.errstate(over="ignore"):
        return np.asarray(a, dtype=np.float64).astype(np.float16).view(np.uint16).copy()


def to_seam_bits(a, seam: str) -> np.ndarray:
    """16-bit patterns of the seam format "f16" or "bf16"."""
    return to_f16_bits(a) if seam == "f16" else to_bf16_bits(a)


def seam_rows(seed, rows: int, n: int, dtype: str = "f32", seam: str = "f16",
              scale: float = 1.0):
    """Rows for the split-norm seam: x ~ N(0, scale^2) in dtype, gamma =
    1 + 0.1 N(0,1) rounded to the seam format."""
    g = rng(seed)
    x = scale * g.standard_normal((rows, n))
    gamma = gamma_like(g, n)
    conv = to_f32 if dtype == "f32" else to_bf16_bits
    return {"x": conv(x), "gamma": to_seam_bits(gamma, seam)}


def gamma_like(g: np.random.Generator, n: int) -> np.ndarray:
    """gamma = 1 + 0.1 N(0,1) in float64 (rounded by the caller)."""
    return 1.0 + 0.1 * g.standard_normal(n)


@dataclass
class Workload:
    """One synthetic problem.  Row operands are [rows x n] row-major arrays;
    f32 data is float32, bf16 data is uint16 bit patterns."""
    name: str
    op: str                     # "rmsnorm" | "then_add" | "sandwich"
    dtype: str                  # "f32" | "bf16"
    rows: int
    n: int
    eps: float                  # the only epsilon (plain, then-add) or eps_post
    eps_pre: float | None = None
    arrays: dict = field(default_factory=dict)
    seed: object = None
    zero_rows: np.ndarray | None = None

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2


def plain_decode_rows(rows: int = 4, n: int = STREAM_WIDTH) -> Workload:
    seed = SEED_BASE + 1
    g = rng(seed)
    x = to_f32(g.standard_normal((rows, n)))
    gamma = to_f32(gamma_like(g, n))
    return Workload("rmsnorm_f32_rows4_n6656", "rmsnorm", "f32", rows, n, 1e-5,
                    arrays={"x": x, "gamma": gamma}, seed=seed)


def _sandwich_arrays(g: np.random.Generator, rows: int, n: int, rescale: bool):
    z = 2.0 * g.standard_normal((rows, n))              # N(0, 4)
    if rescale:
        target = 10.0 ** g.uniform(-4.0, 2.0, size=rows)
        have = np.mean(z * z, axis=1)
        z = z * np.sqrt(target / have)[:, None]
    residual = g.standard_normal((rows, n))
    gamma_post = gamma_like(g, n)
    gamma_pre = gamma_like(g, n)
    return {"block_out": to_f32(z), "residual": to_f32(residual),
            "gamma_post": to_f32(gamma_post), "gamma_pre": to_f32(gamma_pre)}


def sandwich_decode(n: int = STREAM_WIDTH) -> Workload:
    seed = SEED_BASE + 2
    arrays = _sandwich_arrays(rng(seed), 1, n, rescale=False)
    return Workload("sandwich_f32_rows1_n6656", "sandwich", "f32", 1, n, 1e-8, 1e-5,
                    arrays=arrays, seed=seed)


def sandwich_prefill(rows: int = 4096, n: int = STREAM_WIDTH) -> Workload:
    seed = SEED_BASE + 3
    arrays = _sandwich_arrays(rng(seed), rows, n, rescale=True)
    return Workload(f"sandwich_f32_rows{rows}_n{n}", "sandwich", "f32", rows, n, 1e-8,
                    1e-5, arrays=arrays, seed=seed)


def llama_bf16(rows: int = 16384, n: int = 4096) -> Workload:
    seed = SEED_BASE + 4
    g = rng(seed)
    scale = 10.0 ** g.uniform(-2.0, 2.0, size=rows)
    x = g.standard_normal((rows, n)) * scale[:, None]
    gamma = gamma_like(g, n)
    residual = g.standard_normal((rows, n))
    return Workload(f"rmsnorm_then_add_bf16_rows{rows}_n{n}", "then_add", "bf16", rows, n,
                    1e-6, arrays={"x": to_bf16_bits(x), "gamma": to_bf16_bits(gamma),
                                  "residual": to_bf16_bits(residual)}, seed=seed)


def sweep_shapes():
    """(n, rows) pairs of the f32 shape sweep, skipping operands above 4 GiB."""
    return [(n, r) for n in SWEEP_N for r in SWEEP_ROWS if r * n * 4 <= SWEEP_MAX_BYTES]


def sweep(n: int, rows: int, zero_fraction: float = 0.01) -> Workload:
    seed = np.random.SeedSequence([SEED_BASE, 5, n, rows])
    g = rng(seed)
    x = g.standard_normal((rows, n), dtype=np.float32)
    residual = g.standard_normal((rows, n), dtype=np.float32)
    gamma = to_f32(gamma_like(g, n))
    k = int(round(zero_fraction * rows))
    zero_rows = np.sort(g.permutation(rows)[:k])
    x[zero_rows, :] = 0.0
    return Workload(f"sweep_f32_rows{rows}_n{n}", "then_add", "f32", rows, n, 1e-5,
                    arrays={"x": x, "gamma": gamma, "residual": residual}, seed=seed,
                    zero_rows=zero_rows)


def random_rows(seed, rows: int, n: int, dtype: str = "f32", scale: float = 1.0):
    """Generic N(0, scale^2) rows, gamma = 1 + 0.1 N(0,1) and a residual ~ N(0,1)."""
    g = rng(seed)
    x = scale * g.standard_normal((rows, n))
    residual = g.standard_normal((rows, n))
    gamma = gamma_like(g, n)
    gamma2 = gamma_like(g, n)
    conv = to_f32 if dtype == "f32" else to_bf16_bits
    return {"x": conv(x), "residual": conv(residual), "gamma": conv(gamma),
            "gamma2": conv(gamma2)}
