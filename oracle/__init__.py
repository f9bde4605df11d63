"""Scalar f64 CPU oracle for RMSNorm, post-norm-then-add and the dual-epsilon
sandwich tail.

TEST INFRASTRUCTURE ONLY.  This package is the reference that the CUDA path is
checked against.  Only the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import it; the product package never does, and
the two share no code.

The arithmetic lives in ``oracle.c`` (plain C, double precision, sequential
sums, compiled without fast-math or FMA contraction).  This module compiles it
with the host C compiler and marshals numpy arrays through ctypes.  Every
function cites the passage it follows in ``oracle.c`` / ``oracle.h``:
"Chapter 12 -- RMSNorm and the dual-epsilon sandwich" (sections 12.1, 12.3,
12.4.3, 12.4.4) and the Hesper "RMSNorm Layer" API page (rmsNormThenAddKernel,
rmsNormThenAddThenBroadcastScaleKernel, residualAddRmsNormKernel,
fusedRMSNormQ8_1Kernel), and section 12.7's cross-vendor seam (the weightless
norm stored in F16, the weight applied as a second F16 operation).

ctypes releases the GIL during a foreign call, so callers may run disjoint row
blocks on several threads (the oracle itself stays single-threaded code).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "oracle.c")
HEADER = os.path.join(HERE, "oracle.h")
LIBRARY = os.path.join(HERE, "liboracle.so")

# Plain C, no fast-math, no FMA contraction: identical results on x86_64 and
# aarch64 hosts.
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
          "-fno-fast-math", "-Wall", "-Wextra"]

_lock = threading.Lock()
_default = None


def compile_library(source: str = SOURCE, output: str = LIBRARY) -> str:
    """Compile ``source`` into the shared library ``output`` with gcc."""
    cmd = ["gcc", *CFLAGS, "-I", HERE, "-o", output, source, "-lm"]
    subprocess.run(cmd, check=True)
    return output


def build(force: bool = False) -> str:
    """Build liboracle.so next to its source if it is missing or stale."""
    with _lock:
        stale = (not os.path.exists(LIBRARY)
                 or os.path.getmtime(LIBRARY) < max(os.path.getmtime(SOURCE),
                                                    os.path.getmtime(HEADER)))
        if force or stale:
            compile_library()
    return LIBRARY


_f64p = ctypes.POINTER(ctypes.c_double)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_i64 = ctypes.c_int64


def _as_f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a: np.ndarray, typ=_f64p):
    return a.ctypes.data_as(typ)


class Oracle:
    """ctypes view of one compiled oracle library (the real one or a test mutant)."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        lib.oracle_rmsnorm.argtypes = [_f64p, _f64p, _f64p, _i64, _i64, ctypes.c_double]
        lib.oracle_rmsnorm.restype = None
        lib.oracle_rmsnorm_then_add.argtypes = [_f64p, _f64p, _f64p, _f64p, _i64, _i64,
                                                ctypes.c_double]
        lib.oracle_rmsnorm_then_add.restype = None
        lib.oracle_norm_residual_norm.argtypes = [_f64p, _f64p, _f64p, _f64p, _f64p, _f64p,
                                                  _i64, _i64, ctypes.c_double,
                                                  ctypes.c_double, ctypes.c_int]
        lib.oracle_norm_residual_norm.restype = None
        lib.oracle_add_rmsnorm.argtypes = [_f64p, _f64p, _f64p, _f64p, _f64p, _i64, _i64,
                                           ctypes.c_double, ctypes.c_int]
        lib.oracle_add_rmsnorm.restype = None
        lib.oracle_rmsnorm_then_add_scale.argtypes = [_f64p, _f64p, _f64p, ctypes.c_double,
                                                      _f64p, _i64, _i64, ctypes.c_double]
        lib.oracle_rmsnorm_then_add_scale.restype = None
        lib.oracle_rmsnorm_q8_1.argtypes = [_f64p, _f64p, _i64, _i64, ctypes.c_double, _f64p,
                                            _f64p, ctypes.POINTER(ctypes.c_int8)]
        lib.oracle_rmsnorm_q8_1.restype = None
        lib.oracle_rmsnorm_seam.argtypes = [_f64p, _f64p, _f64p, _f64p, _i64, _i64,
                                             ctypes.c_double, ctypes.c_int]
        lib.oracle_rmsnorm_seam.restype = None
        lib.oracle_q8_round.argtypes = [ctypes.c_double]
        lib.oracle_q8_round.restype = ctypes.c_int
        lib.oracle_f16_from_double.argtypes = [ctypes.c_double]
        lib.oracle_f16_from_double.restype = ctypes.c_uint16
        lib.oracle_double_from_f16.argtypes = [ctypes.c_uint16]
        lib.oracle_double_from_f16.restype = ctypes.c_double
        lib.oracle_bf16_from_double.argtypes = [ctypes.c_double]
        lib.oracle_bf16_from_double.restype = ctypes.c_uint16
        lib.oracle_double_from_bf16.argtypes = [ctypes.c_uint16]
        lib.oracle_double_from_bf16.restype = ctypes.c_double
        lib.oracle_bf16_round_array.argtypes = [_f64p, _u16p, _i64]
        lib.oracle_bf16_round_array.restype = None
        lib.oracle_bf16_widen_array.argtypes = [_u16p, _f64p, _i64]
        lib.oracle_bf16_widen_array.restype = None
        self.lib = lib
        self.path = path

    # -- the three operations -------------------------------------------------
    def rmsnorm(self, x, gamma, eps: float) -> np.ndarray:
        """RMSNorm of every row of x [rows x n] (Chapter 12, section 12.1)."""
        x = _as_f64(x)
        g = _as_f64(gamma)
        rows, n = _shape2(x)
        assert g.shape == (n,)
        y = np.empty((rows, n), dtype=np.float64)
        self.lib.oracle_rmsnorm(_ptr(x), _ptr(g), _ptr(y), rows, n, float(eps))
        return y.reshape(x.shape)

    def rmsnorm_then_add(self, x, gamma, residual, eps: float) -> np.ndarray:
        """RMSNorm(x)*gamma + residual per row (Hesper rmsNormThenAddKernel)."""
        x = _as_f64(x)
        g = _as_f64(gamma)
        r = _as_f64(residual)
        rows, n = _shape2(x)
        assert g.shape == (n,) and r.size == x.size
        out = np.empty((rows, n), dtype=np.float64)
        self.lib.oracle_rmsnorm_then_add(_ptr(x), _ptr(g), _ptr(r), _ptr(out), rows, n,
                                         float(eps))
        return out.reshape(x.shape)

    def norm_residual_norm(self, block_out, residual, gamma_post, gamma_pre,
                           eps_post: float, eps_pre: float, stream_bf16: bool = False):
        """Dual-epsilon sandwich tail (Chapter 12, section 12.4.3).

        Returns (out_stream, normed) as float64 arrays.  With ``stream_bf16``
        the stream is rounded to bf16 before it is stored and re-normed
        (section 12.4.4, the split route's publication boundary).
        """
        b = _as_f64(block_out)
        r = _as_f64(residual)
        gp = _as_f64(gamma_post)
        gq = _as_f64(gamma_pre)
        rows, n = _shape2(b)
        assert r.size == b.size and gp.shape == (n,) and gq.shape == (n,)
        s = np.empty((rows, n), dtype=np.float64)
        o = np.empty((rows, n), dtype=np.float64)
        self.lib.oracle_norm_residual_norm(_ptr(b), _ptr(r), _ptr(gp), _ptr(gq), _ptr(s),
                                           _ptr(o), rows, n, float(eps_post),
                                           float(eps_pre), 1 if stream_bf16 else 0)
        return s.reshape(b.shape), o.reshape(b.shape)

    def add_rmsnorm(self, a, b, gamma, eps: float, sum_bf16: bool = False):
        """(a + b, RMSNorm(a + b) * gamma) per row (Hesper residualAddRmsNormKernel)."""
        a = _as_f64(a)
        b = _as_f64(b)
        g = _as_f64(gamma)
        rows, n = _shape2(a)
        assert b.size == a.size and g.shape == (n,)
        s = np.empty((rows, n), dtype=np.float64)
        o = np.empty((rows, n), dtype=np.float64)
        self.lib.oracle_add_rmsnorm(_ptr(a), _ptr(b), _ptr(g), _ptr(s), _ptr(o), rows, n,
                                    float(eps), 1 if sum_bf16 else 0)
        return s.reshape(a.shape), o.reshape(a.shape)

    def rmsnorm_then_add_scale(self, x, gamma, residual, out_scale: float, eps: float):
        """(RMSNorm(x) * gamma + residual) * out_scale per row
        (Hesper rmsNormThenAddThenBroadcastScaleKernel)."""
        x = _as_f64(x)
        g = _as_f64(gamma)
        r = _as_f64(residual)
        rows, n = _shape2(x)
        assert g.shape == (n,) and r.size == x.size
        out = np.empty((rows, n), dtype=np.float64)
        self.lib.oracle_rmsnorm_then_add_scale(_ptr(x), _ptr(g), _ptr(r), float(out_scale),
                                               _ptr(out), rows, n, float(eps))
        return out.reshape(x.shape)

    def rmsnorm_q8_1(self, x, gamma, eps: float):
        """RMSNorm then Q8_1 block quantisation (Hesper fusedRMSNormQ8_1Kernel).
        Returns (d [rows x n/32], qreal [rows x n], q [rows x n] int8)."""
        x = _as_f64(x)
        g = _as_f64(gamma)
        rows, n = _shape2(x)
        assert g.shape == (n,) and n % 32 == 0
        d = np.empty((rows, n // 32), dtype=np.float64)
        qreal = np.empty((rows, n), dtype=np.float64)
        q = np.empty((rows, n), dtype=np.int8)
        self.lib.oracle_rmsnorm_q8_1(_ptr(x), _ptr(g), rows, n, float(eps), _ptr(d),
                                     _ptr(qreal), q.ctypes.data_as(ctypes.POINTER(ctypes.c_int8)))
        return d, qreal, q

    def rmsnorm_seam(self, x, gamma, eps: float, seam: str = "f16"):
        """Split-norm seam (Chapter 12, section 12.7): u = T(x * inv_rms),
        y = T(u * gamma), T = binary16 ("f16") or bf16 ("bf16"); gamma holds
        values of T.  Returns (u, y), exact values of T patterns, as f64."""
        assert seam in ("f16", "bf16")
        x = _as_f64(x)
        g = _as_f64(gamma)
        rows, n = _shape2(x)
        assert g.shape == (n,)
        u = np.empty((rows, n), dtype=np.float64)
        y = np.empty((rows, n), dtype=np.float64)
        self.lib.oracle_rmsnorm_seam(_ptr(x), _ptr(g), _ptr(u), _ptr(y), rows, n, float(eps),
                                     1 if seam == "bf16" else 0)
        return u, y

    def q8_round(self, qreal: float) -> int:
        return self.lib.oracle_q8_round(float(qreal))

    def f16_from_double(self, v) -> np.ndarray:
        v = _as_f64(v)
        return np.array([self.lib.oracle_f16_from_double(float(t)) for t in v.ravel()],
                        dtype=np.uint16).reshape(v.shape)

    def double_from_f16(self, bits) -> np.ndarray:
        b = np.asarray(bits, dtype=np.uint16)
        return np.array([self.lib.oracle_double_from_f16(int(t)) for t in b.ravel()],
                        dtype=np.float64).reshape(b.shape)

    # -- bf16 conversions -----------------------------------------------------
    def bf16_from_double(self, v) -> np.ndarray:
        """Round to nearest bf16, ties to even; returns uint16 bit patterns."""
        v = _as_f64(v)
        bits = np.empty(v.shape, dtype=np.uint16)
        self.lib.oracle_bf16_round_array(_ptr(v), _ptr(bits, _u16p), v.size)
        return bits

    def double_from_bf16(self, bits) -> np.ndarray:
        """Exact double value of bf16 bit patterns (uint16)."""
        b = np.ascontiguousarray(np.asarray(bits, dtype=np.uint16))
        v = np.empty(b.shape, dtype=np.float64)
        self.lib.oracle_bf16_widen_array(_ptr(b, _u16p), _ptr(v), b.size)
        return v


def _shape2(a: np.ndarray):
    if a.ndim == 1:
        return 1, a.shape[0]
    assert a.ndim == 2, "row operands are [rows x n]"
    return a.shape[0], a.shape[1]


def default() -> Oracle:
    """The oracle built from this package's own source."""
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default


def rmsnorm(x, gamma, eps):
    return default().rmsnorm(x, gamma, eps)


def rmsnorm_then_add(x, gamma, residual, eps):
    return default().rmsnorm_then_add(x, gamma, residual, eps)


def norm_residual_norm(block_out, residual, gamma_post, gamma_pre, eps_post, eps_pre,
                       stream_bf16=False):
    return default().norm_residual_norm(block_out, residual, gamma_post, gamma_pre,
                                        eps_post, eps_pre, stream_bf16)


def add_rmsnorm(a, b, gamma, eps, sum_bf16=False):
    return default().add_rmsnorm(a, b, gamma, eps, sum_bf16)


def rmsnorm_then_add_scale(x, gamma, residual, out_scale, eps):
    return default().rmsnorm_then_add_scale(x, gamma, residual, out_scale, eps)


def rmsnorm_q8_1(x, gamma, eps):
    return default().rmsnorm_q8_1(x, gamma, eps)


def rmsnorm_seam(x, gamma, eps, seam="f16"):
    return default().rmsnorm_seam(x, gamma, eps, seam)


def f16_from_double(v):
    return default().f16_from_double(v)


def double_from_f16(bits):
    return default().double_from_f16(bits)


def bf16_from_double(v):
    return default().bf16_from_double(v)


def double_from_bf16(bits):
    return default().double_from_bf16(bits)
