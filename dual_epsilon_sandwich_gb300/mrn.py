"""Python binding of libmrn (``include/mrn.h``): argument marshalling only.

The functions named ``mrn_*`` mirror the C ABI one to one: pointers are plain
integers (device addresses), sizes are ints, the stream is a ``cudaStream_t``
handle as an int (0 = legacy default stream), and each returns the
``mrn_status`` code.  ``rmsnorm``, ``rmsnorm_then_add`` and
``norm_residual_norm`` are conveniences for torch CUDA tensors: they read
pointers, sizes, dtype and the current stream off the tensors, call the C ABI
and raise ``MrnError`` on a non-zero status.  Every step of the computation
runs in the library's CUDA kernels; there is no other code path.  If
``libmrn.so`` has not been built, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIBRARY = os.path.join(PKG, "libmrn.so")

MRN_F32 = 0
MRN_BF16 = 1
MRN_F16 = 2      # only as the seam's 16-bit publication format

MRN_OP_RMSNORM = 0
MRN_OP_THEN_ADD = 1
MRN_OP_SANDWICH = 2
MRN_OP_ADD_RMSNORM = 3
MRN_OP_THEN_ADD_SCALE = 4
MRN_OP_RMSNORM_Q8_1 = 5
MRN_OP_RMSNORM_SEAM = 6
MRN_OP_RMSNORM_UNWEIGHTED = 7
Q8_1_BLOCK_BYTES = 36

MRN_GEOM_AUTO = 0
MRN_GEOM_ROWS_PER_WARP = 1
MRN_GEOM_CTA = 2
MRN_GEOM_STREAM = 3
MRN_GEOM_TMA = 4
MRN_GEOM_Q8_BLOCKS = 5

MRN_LAUNCH_PDL = 1
MRN_LAUNCH_TEST_WAIT_TIMEOUT = 0x80000000   # test hook (see include/mrn.h)

STATUS = {
    0: "MRN_OK",
    1: "MRN_ERR_NULL_POINTER",
    2: "MRN_ERR_INVALID_SIZE",
    3: "MRN_ERR_INVALID_EPS",
    4: "MRN_ERR_UNSUPPORTED_DTYPE",
    5: "MRN_ERR_ALIASING",
    6: "MRN_ERR_MISALIGNED",
    7: "MRN_ERR_CUDA",
    8: "MRN_ERR_INVALID_GEOMETRY",
}
for _code, _name in STATUS.items():
    globals()[_name] = _code

EXPORTS = ("mrn_rmsnorm", "mrn_rmsnorm_then_add", "mrn_norm_residual_norm",
           "mrn_add_rmsnorm", "mrn_rmsnorm_then_add_scale", "mrn_rmsnorm_q8_1",
           "mrn_status_string", "mrn_last_cuda_error", "mrn_query_geometry",
           "mrn_force_geometry", "mrn_launch_count", "mrn_wait_timeouts",
           "mrn_set_launch_options", "mrn_launch_options", "mrn_rmsnorm_seam",
           "mrn_rmsnorm_unweighted", "mrn_seam_scale")


class MrnError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        name = STATUS.get(status, str(status))
        detail = mrn_status_string(status)
        if status == 7:
            detail += f" (cudaError {mrn_last_cuda_error()})"
        super().__init__(f"{what}: {name}: {detail}" if what else f"{name}: {detail}")


class MrnGeometry(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("vec", ctypes.c_int32), ("k", ctypes.c_int32),
                ("threads", ctypes.c_int32), ("cluster", ctypes.c_int32),
                ("lanes_per_row", ctypes.c_int32), ("rows_per_cta", ctypes.c_int32),
                ("stages", ctypes.c_int32), ("ctas", ctypes.c_int32),
                ("groups", ctypes.c_int32), ("edge", ctypes.c_int32)]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


_lock = threading.Lock()
_lib = None

_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_f = ctypes.c_float
_i = ctypes.c_int


def lib() -> ctypes.CDLL:
    """The loaded libmrn.so.  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIBRARY):
                raise RuntimeError(
                    f"{LIBRARY} is not built; run dual_epsilon_sandwich_gb300._build.build() "
                    "(or __graft_entry__.build()) first")
            L = ctypes.CDLL(LIBRARY)
            L.mrn_rmsnorm.argtypes = [_vp, _vp, _vp, _i64, _i64, _f, _i, _vp]
            L.mrn_rmsnorm_then_add.argtypes = [_vp, _vp, _vp, _vp, _i64, _i64, _f, _i, _vp]
            L.mrn_norm_residual_norm.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64,
                                                 _f, _f, _i, _vp]
            L.mrn_add_rmsnorm.argtypes = [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _f, _i, _vp]
            L.mrn_rmsnorm_then_add_scale.argtypes = [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _f,
                                                     _i, _vp]
            L.mrn_rmsnorm_q8_1.argtypes = [_vp, _vp, _vp, _i64, _i64, _f, _i, _vp]
            L.mrn_rmsnorm_seam.argtypes = [_vp, _vp, _vp, _i64, _i64, _f, _i, _i, _vp]
            L.mrn_rmsnorm_unweighted.argtypes = [_vp, _vp, _i64, _i64, _f, _i, _i, _vp]
            L.mrn_seam_scale.argtypes = [_vp, _vp, _vp, _i64, _i64, _i, _vp]
            for fn in (L.mrn_rmsnorm, L.mrn_rmsnorm_then_add, L.mrn_norm_residual_norm,
                       L.mrn_add_rmsnorm, L.mrn_rmsnorm_then_add_scale, L.mrn_rmsnorm_q8_1,
                       L.mrn_rmsnorm_seam, L.mrn_rmsnorm_unweighted, L.mrn_seam_scale):
                fn.restype = _i
            L.mrn_status_string.argtypes = [_i]
            L.mrn_status_string.restype = ctypes.c_char_p
            L.mrn_last_cuda_error.argtypes = []
            L.mrn_last_cuda_error.restype = _i
            L.mrn_query_geometry.argtypes = [_i, _i64, _i64, _i, ctypes.c_int32, ctypes.c_int32,
                                             ctypes.POINTER(MrnGeometry)]
            L.mrn_query_geometry.restype = _i
            L.mrn_force_geometry.argtypes = [ctypes.POINTER(MrnGeometry)]
            L.mrn_force_geometry.restype = _i
            L.mrn_launch_count.argtypes = []
            L.mrn_launch_count.restype = ctypes.c_uint64
            L.mrn_wait_timeouts.argtypes = []
            L.mrn_wait_timeouts.restype = _i
            L.mrn_set_launch_options.argtypes = [ctypes.c_uint32]
            L.mrn_set_launch_options.restype = _i
            L.mrn_launch_options.argtypes = []
            L.mrn_launch_options.restype = ctypes.c_uint32
            _lib = L
    return _lib


# ---------------------------------------------------------------------------
# The C ABI, one to one
# ---------------------------------------------------------------------------
def mrn_rmsnorm(x, gamma, y, rows, n, eps, dtype, stream=0) -> int:
    return lib().mrn_rmsnorm(x, gamma, y, rows, n, eps, dtype, stream)


def mrn_rmsnorm_then_add(x, gamma, residual, out, rows, n, eps, dtype, stream=0) -> int:
    return lib().mrn_rmsnorm_then_add(x, gamma, residual, out, rows, n, eps, dtype, stream)


def mrn_norm_residual_norm(block_out, residual, gamma_post, gamma_pre, out_stream, normed,
                           rows, n, eps_post, eps_pre, dtype, stream=0) -> int:
    return lib().mrn_norm_residual_norm(block_out, residual, gamma_post, gamma_pre, out_stream,
                                        normed, rows, n, eps_post, eps_pre, dtype, stream)


def mrn_add_rmsnorm(a, b, gamma, residual_out, normed, rows, n, eps, dtype, stream=0) -> int:
    return lib().mrn_add_rmsnorm(a, b, gamma, residual_out, normed, rows, n, eps, dtype, stream)


def mrn_rmsnorm_then_add_scale(x, gamma, residual, out_scale, out, rows, n, eps, dtype,
                               stream=0) -> int:
    return lib().mrn_rmsnorm_then_add_scale(x, gamma, residual, out_scale, out, rows, n, eps,
                                            dtype, stream)


def mrn_rmsnorm_q8_1(x, gamma, blocks, rows, n, eps, dtype, stream=0) -> int:
    return lib().mrn_rmsnorm_q8_1(x, gamma, blocks, rows, n, eps, dtype, stream)


def mrn_rmsnorm_seam(x, gamma, y, rows, n, eps, dtype, seam, stream=0) -> int:
    return lib().mrn_rmsnorm_seam(x, gamma, y, rows, n, eps, dtype, seam, stream)


def mrn_rmsnorm_unweighted(x, u, rows, n, eps, dtype, seam, stream=0) -> int:
    return lib().mrn_rmsnorm_unweighted(x, u, rows, n, eps, dtype, seam, stream)


def mrn_seam_scale(u, gamma, y, rows, n, seam, stream=0) -> int:
    return lib().mrn_seam_scale(u, gamma, y, rows, n, seam, stream)


def mrn_status_string(status: int) -> str:
    return lib().mrn_status_string(status).decode()


def mrn_last_cuda_error() -> int:
    return lib().mrn_last_cuda_error()


def mrn_query_geometry(op, rows, n, dtype, aligned16=True, sm_count=0) -> dict:
    """aligned16: True / 1 (all pointers 16-byte aligned), 2 (the row operands at
    one offset within 16 bytes) or False / 0."""
    g = MrnGeometry()
    code = aligned16 if isinstance(aligned16, int) and not isinstance(aligned16, bool) \
        else (1 if aligned16 else 0)
    st = lib().mrn_query_geometry(op, rows, n, dtype, code, sm_count, ctypes.byref(g))
    if st != 0:
        raise MrnError(st, "mrn_query_geometry")
    return g.as_dict()


def mrn_force_geometry(geometry: dict | None) -> int:
    """Force the calling thread's geometry (None restores the automatic choice)."""
    if geometry is None:
        return lib().mrn_force_geometry(None)
    g = MrnGeometry(**{k: int(v) for k, v in geometry.items() if k != "rows_per_cta"})
    return lib().mrn_force_geometry(ctypes.byref(g))


def mrn_launch_count() -> int:
    return lib().mrn_launch_count()


def mrn_set_launch_options(options: int) -> int:
    """Launch options of the calling thread (MRN_LAUNCH_PDL or 0; MRN_LAUNCH_TEST_WAIT_TIMEOUT
    is a test hook)."""
    return lib().mrn_set_launch_options(options)


def mrn_launch_options() -> int:
    return lib().mrn_launch_options()


def mrn_wait_timeouts() -> int:
    """Bounded waits that ran out since the last call (synchronises the device)."""
    return lib().mrn_wait_timeouts()


# ---------------------------------------------------------------------------
# torch tensor conveniences (marshalling only)
# ---------------------------------------------------------------------------
def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return MRN_F32
    if t.dtype == torch.bfloat16:
        return MRN_BF16
    raise TypeError(f"unsupported dtype {t.dtype}; expected float32 or bfloat16")


def _check(t, name, dtype, shape=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _rows_n(x):
    n = x.shape[-1]
    rows = x.numel() // n if n else 0
    return rows, n


def _stream(t):
    import torch
    return torch.cuda.current_stream(t.device).cuda_stream


def rmsnorm(x, gamma, eps: float, out=None):
    """y = RMSNorm(x) * gamma over the last dimension; out may be x."""
    import torch
    dt = _dtype_code(x)
    _check(x, "x", x.dtype)
    rows, n = _rows_n(x)
    _check(gamma, "gamma", x.dtype, (n,))
    out = torch.empty_like(x) if out is None else out
    _check(out, "out", x.dtype, x.shape)
    st = mrn_rmsnorm(x.data_ptr(), gamma.data_ptr(), out.data_ptr(), rows, n, eps, dt,
                     _stream(x))
    if st != 0:
        raise MrnError(st, "mrn_rmsnorm")
    return out


def rmsnorm_then_add(x, gamma, residual, eps: float, out=None):
    """out = RMSNorm(x) * gamma + residual; out may be x or residual."""
    import torch
    dt = _dtype_code(x)
    _check(x, "x", x.dtype)
    rows, n = _rows_n(x)
    _check(gamma, "gamma", x.dtype, (n,))
    _check(residual, "residual", x.dtype, x.shape)
    out = torch.empty_like(x) if out is None else out
    _check(out, "out", x.dtype, x.shape)
    st = mrn_rmsnorm_then_add(x.data_ptr(), gamma.data_ptr(), residual.data_ptr(),
                              out.data_ptr(), rows, n, eps, dt, _stream(x))
    if st != 0:
        raise MrnError(st, "mrn_rmsnorm_then_add")
    return out


def norm_residual_norm(block_out, residual, gamma_post, gamma_pre, eps_post: float = 1e-8,
                       eps_pre: float = 1e-5, out_stream=None, normed=None):
    """(out_stream, normed) of the dual-epsilon sandwich tail; out_stream may be
    residual (in-place update)."""
    import torch
    dt = _dtype_code(block_out)
    _check(block_out, "block_out", block_out.dtype)
    rows, n = _rows_n(block_out)
    _check(residual, "residual", block_out.dtype, block_out.shape)
    _check(gamma_post, "gamma_post", block_out.dtype, (n,))
    _check(gamma_pre, "gamma_pre", block_out.dtype, (n,))
    out_stream = torch.empty_like(block_out) if out_stream is None else out_stream
    normed = torch.empty_like(block_out) if normed is None else normed
    _check(out_stream, "out_stream", block_out.dtype, block_out.shape)
    _check(normed, "normed", block_out.dtype, block_out.shape)
    st = mrn_norm_residual_norm(block_out.data_ptr(), residual.data_ptr(), gamma_post.data_ptr(),
                                gamma_pre.data_ptr(), out_stream.data_ptr(), normed.data_ptr(),
                                rows, n, eps_post, eps_pre, dt, _stream(block_out))
    if st != 0:
        raise MrnError(st, "mrn_norm_residual_norm")
    return out_stream, normed


def add_rmsnorm(a, b, gamma, eps: float, residual_out=None, normed=None):
    """(a + b, RMSNorm(a + b) * gamma); residual_out may be a or b (in place)."""
    import torch
    dt = _dtype_code(a)
    _check(a, "a", a.dtype)
    rows, n = _rows_n(a)
    _check(b, "b", a.dtype, a.shape)
    _check(gamma, "gamma", a.dtype, (n,))
    residual_out = torch.empty_like(a) if residual_out is None else residual_out
    normed = torch.empty_like(a) if normed is None else normed
    _check(residual_out, "residual_out", a.dtype, a.shape)
    _check(normed, "normed", a.dtype, a.shape)
    st = mrn_add_rmsnorm(a.data_ptr(), b.data_ptr(), gamma.data_ptr(), residual_out.data_ptr(),
                         normed.data_ptr(), rows, n, eps, dt, _stream(a))
    if st != 0:
        raise MrnError(st, "mrn_add_rmsnorm")
    return residual_out, normed


def rmsnorm_then_add_scale(x, gamma, residual, out_scale, eps: float, out=None):
    """(RMSNorm(x) * gamma + residual) * out_scale[0]; out_scale is a one-element
    device tensor of x's dtype."""
    import torch
    dt = _dtype_code(x)
    _check(x, "x", x.dtype)
    rows, n = _rows_n(x)
    _check(gamma, "gamma", x.dtype, (n,))
    _check(residual, "residual", x.dtype, x.shape)
    _check(out_scale, "out_scale", x.dtype, (1,))
    out = torch.empty_like(x) if out is None else out
    _check(out, "out", x.dtype, x.shape)
    st = mrn_rmsnorm_then_add_scale(x.data_ptr(), gamma.data_ptr(), residual.data_ptr(),
                                    out_scale.data_ptr(), out.data_ptr(), rows, n, eps, dt,
                                    _stream(x))
    if st != 0:
        raise MrnError(st, "mrn_rmsnorm_then_add_scale")
    return out


def rmsnorm_q8_1(x, gamma, eps: float, blocks=None):
    """RMSNorm then Q8_1 blocks: returns a uint8 tensor [rows, n/32, 36] (f16 d,
    f16 s = 0, int8 q[32] per block)."""
    import torch
    dt = _dtype_code(x)
    _check(x, "x", x.dtype)
    rows, n = _rows_n(x)
    _check(gamma, "gamma", x.dtype, (n,))
    if n % 32:
        raise ValueError("n must be a multiple of 32")
    if blocks is None:
        blocks = torch.empty((rows, n // 32, Q8_1_BLOCK_BYTES), dtype=torch.uint8,
                             device=x.device)
    _check(blocks, "blocks", torch.uint8, (rows, n // 32, Q8_1_BLOCK_BYTES))
    st = mrn_rmsnorm_q8_1(x.data_ptr(), gamma.data_ptr(), blocks.data_ptr(), rows, n, eps, dt,
                          _stream(x))
    if st != 0:
        raise MrnError(st, "mrn_rmsnorm_q8_1")
    return blocks


def _seam_code(t) -> int:
    import torch
    if t.dtype == torch.float16:
        return MRN_F16
    if t.dtype == torch.bfloat16:
        return MRN_BF16
    raise TypeError(f"seam tensors hold float16 or bfloat16, not {t.dtype}")


def rmsnorm_seam(x, gamma, eps: float, out=None):
    """Split-norm seam in one kernel: S(S(x * inv_rms) * gamma), S = gamma's
    dtype (float16 or bfloat16); x is float32 or bfloat16.  out may be x when
    x is bfloat16."""
    import torch
    dt = _dtype_code(x)
    _check(x, "x", x.dtype)
    rows, n = _rows_n(x)
    seam = _seam_code(gamma)
    _check(gamma, "gamma", gamma.dtype, (n,))
    out = torch.empty(x.shape, dtype=gamma.dtype, device=x.device) if out is None else out
    _check(out, "out", gamma.dtype, x.shape)
    st = mrn_rmsnorm_seam(x.data_ptr(), gamma.data_ptr(), out.data_ptr(), rows, n, eps, dt, seam,
                          _stream(x))
    if st != 0:
        raise MrnError(st, "mrn_rmsnorm_seam")
    return out


def rmsnorm_unweighted(x, eps: float, seam_dtype, out=None):
    """The seam's first operation: S(x * inv_rms) in seam_dtype (torch.float16
    or torch.bfloat16)."""
    import torch
    dt = _dtype_code(x)
    _check(x, "x", x.dtype)
    rows, n = _rows_n(x)
    out = torch.empty(x.shape, dtype=seam_dtype, device=x.device) if out is None else out
    seam = _seam_code(out)
    _check(out, "out", seam_dtype, x.shape)
    st = mrn_rmsnorm_unweighted(x.data_ptr(), out.data_ptr(), rows, n, eps, dt, seam, _stream(x))
    if st != 0:
        raise MrnError(st, "mrn_rmsnorm_unweighted")
    return out


def seam_scale(u, gamma, out=None):
    """The seam's second operation: S(u * gamma), u and gamma of one 16-bit
    dtype; out may be u."""
    import torch
    seam = _seam_code(u)
    _check(u, "u", u.dtype)
    rows, n = _rows_n(u)
    _check(gamma, "gamma", u.dtype, (n,))
    out = torch.empty_like(u) if out is None else out
    _check(out, "out", u.dtype, u.shape)
    st = mrn_seam_scale(u.data_ptr(), gamma.data_ptr(), out.data_ptr(), rows, n, seam, _stream(u))
    if st != 0:
        raise MrnError(st, "mrn_seam_scale")
    return out
