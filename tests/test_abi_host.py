"""Host-only checks of the C ABI (no GPU, no kernel launch).

Every call here fails validation before anything is enqueued, so the pointers
are fake addresses that are never dereferenced.
"""
import os
import re
import subprocess
import sys

import pytest

from dual_epsilon_sandwich_gb300 import _build, mrn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mrn.h")

A = 0x7F0000000000        # fake, 256-byte aligned device addresses
B = 0x7F0100000000
G = 0x7F0200000000
H = 0x7F0300000000
Y = 0x7F0400000000
Z = 0x7F0500000000


@pytest.fixture(scope="module", autouse=True)
def library():
    _build.build()
    return mrn.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mrn_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(library):
    names = declared_functions()
    assert set(names) == set(mrn.EXPORTS), names
    for name in names:
        assert hasattr(library, name), f"libmrn.so does not export {name}"
    nm = subprocess.run(["nm", "-D", "--defined-only", mrn.LIBRARY], capture_output=True,
                        text=True, check=True).stdout
    for name in names:
        assert re.search(rf"\bT {name}$", nm, flags=re.M), name


def header_constants():
    """Every enum value and #define of the header: name -> integer."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    found = {}
    for name, value in re.findall(r"\b(MRN_[A-Z0-9_]+)\s*=\s*(0x[0-9A-Fa-f]+|\d+)", text):
        found[name] = int(value, 0)
    for name, value in re.findall(r"#define\s+(MRN_[A-Z0-9_]+)\s+(0x[0-9A-Fa-f]+|\d+)u?", text):
        found[name] = int(value, 0)
    return found


def test_binding_constants_match_the_header():
    """The binding restates the header's constants; they must agree, and every
    enum value and option bit of the header must be there."""
    consts = header_constants()
    statuses = {v: k for k, v in consts.items() if k == "MRN_OK" or k.startswith("MRN_ERR_")}
    assert mrn.STATUS == statuses
    for name, value in consts.items():
        if name == "MRN_OK" or name.startswith("MRN_ERR_"):
            continue
        assert getattr(mrn, name) == value, name


def test_status_strings():
    for code in range(9):
        assert mrn.mrn_status_string(code)
        assert "unknown" not in mrn.mrn_status_string(code)
    assert "unknown" in mrn.mrn_status_string(99)
    assert mrn.mrn_last_cuda_error() == 0


def test_a_wait_timeout_is_not_a_call_status():
    """The contract: a kernel's bounded wait that runs out is reported only by
    mrn_wait_timeouts(), never as the status of a call (the call returned at
    enqueue time).  No status value stands for it, and the header says so
    (the GPU side of the contract: tests/test_gpu_wait_timeouts.py checks that
    every call whose kernel timed out returned MRN_OK)."""
    consts = header_constants()
    assert not any("TIMEOUT" in k for k in consts if k.startswith("MRN_ERR_")), consts
    assert max(mrn.STATUS) == mrn.MRN_ERR_INVALID_GEOMETRY
    assert "unknown" in mrn.mrn_status_string(mrn.MRN_ERR_INVALID_GEOMETRY + 1)
    text = open(HEADER).read()
    assert "reported only by\n *            mrn_wait_timeouts()" in text
    assert "never as the status of the call" in text


def rms(x=A, g=G, y=Y, rows=4, n=64, eps=1e-5, dt=mrn.MRN_F32):
    return mrn.mrn_rmsnorm(x, g, y, rows, n, eps, dt, 0)


def tadd(x=A, g=G, r=B, o=Y, rows=4, n=64, eps=1e-5, dt=mrn.MRN_F32):
    return mrn.mrn_rmsnorm_then_add(x, g, r, o, rows, n, eps, dt, 0)


def sand(b=A, r=B, gp=G, gq=H, s=Y, o=Z, rows=4, n=64, e1=1e-8, e2=1e-5, dt=mrn.MRN_F32):
    return mrn.mrn_norm_residual_norm(b, r, gp, gq, s, o, rows, n, e1, e2, dt, 0)


def addn(a=A, b=B, g=G, s=Y, o=Z, rows=4, n=64, eps=1e-5, dt=mrn.MRN_F32):
    return mrn.mrn_add_rmsnorm(a, b, g, s, o, rows, n, eps, dt, 0)


def tscale(x=A, g=G, r=B, sc=H, o=Y, rows=4, n=64, eps=1e-5, dt=mrn.MRN_F32):
    return mrn.mrn_rmsnorm_then_add_scale(x, g, r, sc, o, rows, n, eps, dt, 0)


def test_more_ops_validation():
    assert addn(n=0) == mrn.MRN_ERR_INVALID_SIZE
    assert tscale(eps=0.0) == mrn.MRN_ERR_INVALID_EPS
    assert addn(dt=5) == mrn.MRN_ERR_UNSUPPORTED_DTYPE
    assert addn(a=None, b=None, g=None, s=None, o=None, rows=0) == mrn.MRN_OK
    for kw in ("a", "b", "g", "s", "o"):
        assert addn(**{kw: None}) == mrn.MRN_ERR_NULL_POINTER, kw
    for kw in ("x", "g", "r", "sc", "o"):
        assert tscale(**{kw: None}) == mrn.MRN_ERR_NULL_POINTER, kw
    assert tscale(sc=H + 2) == mrn.MRN_ERR_MISALIGNED
    assert addn(o=Y) == mrn.MRN_ERR_ALIASING                 # normed == residual_out
    assert addn(s=A + 8) == mrn.MRN_ERR_ALIASING             # partial over a
    assert addn(o=G) == mrn.MRN_ERR_ALIASING                 # normed over gamma
    assert tscale(sc=Y + 4) == mrn.MRN_ERR_ALIASING          # out over the scale
    assert tscale(o=B + 4) == mrn.MRN_ERR_ALIASING           # partial over residual
    assert mrn.mrn_launch_count() == 0


def test_q8_1_validation():
    q8 = mrn.mrn_rmsnorm_q8_1
    assert q8(A, G, Y, 4, 100, 1e-5, mrn.MRN_F32, 0) == mrn.MRN_ERR_INVALID_SIZE   # n % 32
    assert q8(A, G, Y + 2, 4, 64, 1e-5, mrn.MRN_F32, 0) == mrn.MRN_ERR_MISALIGNED
    assert q8(A, G, A + 64, 4, 64, 1e-5, mrn.MRN_F32, 0) == mrn.MRN_ERR_ALIASING
    assert q8(A, G, G, 4, 64, 1e-5, mrn.MRN_BF16, 0) == mrn.MRN_ERR_ALIASING
    assert q8(None, None, None, 0, 64, 1e-5, mrn.MRN_F32, 0) == mrn.MRN_OK
    assert q8(A, None, Y, 4, 64, 1e-5, mrn.MRN_F32, 0) == mrn.MRN_ERR_NULL_POINTER
    assert mrn.mrn_launch_count() == 0


def seam(x=A, g=G, y=Y, rows=4, n=64, eps=1e-5, dt=mrn.MRN_F32, s=mrn.MRN_F16):
    return mrn.mrn_rmsnorm_seam(x, g, y, rows, n, eps, dt, s, 0)


def unw(x=A, y=Y, rows=4, n=64, eps=1e-5, dt=mrn.MRN_F32, s=mrn.MRN_F16):
    return mrn.mrn_rmsnorm_unweighted(x, y, rows, n, eps, dt, s, 0)


def scl(u=A, g=G, y=Y, rows=4, n=64, s=mrn.MRN_F16):
    return mrn.mrn_seam_scale(u, g, y, rows, n, s, 0)


def test_seam_validation():
    for f in (seam, unw):
        assert f(s=mrn.MRN_F32) == mrn.MRN_ERR_UNSUPPORTED_DTYPE      # S is 16-bit
        assert f(s=3) == mrn.MRN_ERR_UNSUPPORTED_DTYPE
        assert f(dt=mrn.MRN_F16) == mrn.MRN_ERR_UNSUPPORTED_DTYPE     # x is f32 or bf16
        assert f(n=0) == mrn.MRN_ERR_INVALID_SIZE
        assert f(eps=0.0) == mrn.MRN_ERR_INVALID_EPS
        assert f(x=None, y=None, rows=0) == mrn.MRN_OK
        assert f(x=None) == mrn.MRN_ERR_NULL_POINTER
        assert f(y=Y + 1) == mrn.MRN_ERR_MISALIGNED
        assert f(y=A) == mrn.MRN_ERR_ALIASING                 # f32 x: 16-bit y cannot share it
        assert f(y=A + 2, dt=mrn.MRN_BF16) == mrn.MRN_ERR_ALIASING   # partial over bf16 x
    assert seam(g=None) == mrn.MRN_ERR_NULL_POINTER
    assert seam(g=G + 1) == mrn.MRN_ERR_MISALIGNED
    assert seam(y=G - 8) == mrn.MRN_ERR_ALIASING              # output over gamma
    assert scl(s=mrn.MRN_F32) == mrn.MRN_ERR_UNSUPPORTED_DTYPE
    assert scl(n=0) == mrn.MRN_ERR_INVALID_SIZE
    assert scl(rows=2 ** 62) == mrn.MRN_ERR_INVALID_SIZE
    assert scl(u=None, g=None, y=None, rows=0) == mrn.MRN_OK
    for kw in ("u", "g", "y"):
        assert scl(**{kw: None}) == mrn.MRN_ERR_NULL_POINTER, kw
    assert scl(u=A + 1) == mrn.MRN_ERR_MISALIGNED
    assert scl(y=A + 2) == mrn.MRN_ERR_ALIASING               # partial over u
    assert scl(y=G) == mrn.MRN_ERR_ALIASING                   # over gamma
    assert mrn.mrn_launch_count() == 0


def test_seam_geometry():
    for op in (mrn.MRN_OP_RMSNORM_SEAM, mrn.MRN_OP_RMSNORM_UNWEIGHTED):
        got = mrn.mrn_query_geometry(op, 1216, 6656, mrn.MRN_F32, True, 152)
        assert (got["kind"], got["stages"], got["groups"]) == (4, 4, 2)   # staged, 4 stages
        got = mrn.mrn_query_geometry(op, 4096, 6656, mrn.MRN_F32, True, 152)
        assert (got["kind"], got["threads"], got["k"]) == (2, 224, 8)     # register batch
        got = mrn.mrn_query_geometry(op, 2048, 4096, mrn.MRN_BF16, True, 152)
        assert (got["kind"], got["stages"], got["groups"]) == (4, 2, 2)
        got = mrn.mrn_query_geometry(op, 16384, 4096, mrn.MRN_BF16, True, 152)
        assert (got["kind"], got["threads"], got["k"]) == (2, 128, 4)   # register batch
        assert mrn.mrn_query_geometry(op, 4096, 6656, mrn.MRN_F32, False, 152)["kind"] == 2
        assert mrn.mrn_query_geometry(op, 4096, 128, mrn.MRN_BF16, True, 152)["kind"] == 1
        # staged: one row operand per stage, no gamma in shared memory (read through L1)
        assert mrn.mrn_force_geometry({"kind": 4, "k": 4, "threads": 416, "stages": 4}) == 0
        got = mrn.mrn_query_geometry(op, 4096, 6656, mrn.MRN_F32, True, 152)
        assert (got["kind"], got["stages"]) == (4, 4)
        assert mrn.mrn_force_geometry(None) == 0
    with pytest.raises(mrn.MrnError):
        mrn.mrn_query_geometry(8, 4, 64, mrn.MRN_F32, True, 152)


# (op, rows, n, dtype) -> (kind, threads, k) of the automatic choice for batches:
# the register kernel where the sweeps measured it faster, else the staged
# kernel (kind 4) or rows per warp (kind 1); threads and k only for kind 2.
BATCH_CHOICES = [
    (mrn.MRN_OP_RMSNORM, 16384, 4096, mrn.MRN_BF16, (2, 128, 4)),
    (mrn.MRN_OP_THEN_ADD, 16384, 4096, mrn.MRN_BF16, (2, 128, 4)),
    (mrn.MRN_OP_THEN_ADD_SCALE, 16384, 4096, mrn.MRN_BF16, (2, 128, 4)),
    (mrn.MRN_OP_SANDWICH, 16384, 4096, mrn.MRN_BF16, (2, 256, 2)),
    (mrn.MRN_OP_SANDWICH, 4096, 8192, mrn.MRN_BF16, (4,)),
    (mrn.MRN_OP_SANDWICH, 4096, 6656, mrn.MRN_F32, (2, 256, 7)),
    (mrn.MRN_OP_SANDWICH, 1216, 6656, mrn.MRN_F32, (4,)),
    (mrn.MRN_OP_SANDWICH, 1216, 2048, mrn.MRN_F32, (2, 128, 4)),
    (mrn.MRN_OP_RMSNORM, 65536, 2048, mrn.MRN_BF16, (2, 64, 4)),    # was rows per warp
    (mrn.MRN_OP_THEN_ADD, 65536, 2048, mrn.MRN_BF16, (2, 64, 4)),
    (mrn.MRN_OP_RMSNORM, 65536, 512, mrn.MRN_F32, (1,)),            # 128 loads: rows per warp
    (mrn.MRN_OP_RMSNORM, 163840, 128, mrn.MRN_BF16, (1,)),          # per-head QK-norm
    (mrn.MRN_OP_RMSNORM, 4096, 6656, mrn.MRN_F32, (2, 224, 8)),     # eight slots, 3 CTAs/SM
    (mrn.MRN_OP_RMSNORM, 65536, 8192, mrn.MRN_F32, (2, 256, 8)),
    (mrn.MRN_OP_THEN_ADD, 4096, 6656, mrn.MRN_F32, (2, 416, 4)),
    (mrn.MRN_OP_THEN_ADD, 65536, 8192, mrn.MRN_F32, (4,)),
    (mrn.MRN_OP_THEN_ADD_SCALE, 4096, 6656, mrn.MRN_F32, (4,)),
    (mrn.MRN_OP_THEN_ADD_SCALE, 65536, 5120, mrn.MRN_F32, (2, 256, 5)),
    (mrn.MRN_OP_THEN_ADD_SCALE, 4096, 6656, mrn.MRN_BF16, (2, 224, 4)),
    (mrn.MRN_OP_RMSNORM, 65536, 5120, mrn.MRN_F32, (2, 160, 8)),
    (mrn.MRN_OP_RMSNORM, 1216, 4096, mrn.MRN_F32, (4,)),            # rows < 2048, 1024 loads
    (mrn.MRN_OP_RMSNORM, 1216, 2048, mrn.MRN_F32, (2, 128, 4)),
    (mrn.MRN_OP_RMSNORM, 4096, 6656, mrn.MRN_BF16, (2, 224, 4)),
    (mrn.MRN_OP_RMSNORM, 16384, 8192, mrn.MRN_BF16, (4,)),
    (mrn.MRN_OP_THEN_ADD, 16384, 8192, mrn.MRN_BF16, (2, 256, 4)),
    (mrn.MRN_OP_ADD_RMSNORM, 4096, 6656, mrn.MRN_F32, (2, 256, 7)),
    (mrn.MRN_OP_RMSNORM, 100, 4096, mrn.MRN_BF16, (2,)),            # fewer rows than SMs
]


# The same choice on both sides of each threshold of the rule (loads per row,
# rows): (op, rows, n, dtype) -> kind.
BATCH_THRESHOLDS = [
    ((0, 2048, 2048, mrn.MRN_F32), 2), ((0, 2047, 2052, mrn.MRN_F32), 4),
    ((0, 2048, 2052, mrn.MRN_F32), 2), ((0, 2048, 8192, mrn.MRN_F32), 2),
    ((1, 2048, 6656, mrn.MRN_F32), 2), ((1, 2048, 6660, mrn.MRN_F32), 4),
    ((4, 2048, 5120, mrn.MRN_F32), 2), ((4, 2048, 5124, mrn.MRN_F32), 4),
    ((4, 2048, 13312, mrn.MRN_BF16), 2), ((4, 2048, 13320, mrn.MRN_BF16), 4),
    ((0, 2048, 7168, mrn.MRN_BF16), 2), ((0, 2048, 7176, mrn.MRN_BF16), 4),
    ((6, 4095, 4096, mrn.MRN_BF16), 4), ((6, 4096, 4096, mrn.MRN_BF16), 2),
    ((6, 2047, 8192, mrn.MRN_F32), 4), ((6, 2048, 8192, mrn.MRN_F32), 2),
    ((2, 2048, 4096, mrn.MRN_BF16), 2), ((2, 2048, 4104, mrn.MRN_BF16), 4),
    ((2, 2047, 6656, mrn.MRN_F32), 4), ((2, 2048, 6656, mrn.MRN_F32), 2),
]


@pytest.mark.parametrize("call,kind", BATCH_THRESHOLDS, ids=[str(c) for c, _ in BATCH_THRESHOLDS])
def test_register_batch_thresholds(call, kind):
    op, rows, n, dt = call
    assert mrn.mrn_query_geometry(op, rows, n, dt, True, 152)["kind"] == kind


@pytest.mark.parametrize("op,rows,n,dt,want", BATCH_CHOICES,
                         ids=[f"{c[0]}-{c[1]}x{c[2]}-{c[3]}" for c in BATCH_CHOICES])
def test_register_batch_choice(op, rows, n, dt, want):
    got = mrn.mrn_query_geometry(op, rows, n, dt, True, 152)
    assert (got["kind"], got["threads"], got["k"])[:len(want)] == want, got


def test_size_validation():
    assert rms(n=0) == mrn.MRN_ERR_INVALID_SIZE
    assert rms(n=-3) == mrn.MRN_ERR_INVALID_SIZE
    assert rms(rows=-1) == mrn.MRN_ERR_INVALID_SIZE
    assert tadd(rows=2 ** 40, n=2 ** 30) == mrn.MRN_ERR_INVALID_SIZE     # bytes overflow int64
    assert sand(n=2 ** 62) == mrn.MRN_ERR_INVALID_SIZE


def test_rows_zero_is_a_no_op_without_pointers():
    assert rms(x=None, g=None, y=None, rows=0) == mrn.MRN_OK
    assert tadd(x=None, g=None, r=None, o=None, rows=0) == mrn.MRN_OK
    assert sand(b=None, r=None, gp=None, gq=None, s=None, o=None, rows=0) == mrn.MRN_OK
    assert mrn.mrn_launch_count() == 0


@pytest.mark.parametrize("eps", [0.0, -1e-5, float("nan"), float("inf"), -0.0])
def test_eps_validation(eps):
    assert rms(eps=eps) == mrn.MRN_ERR_INVALID_EPS
    assert tadd(eps=eps) == mrn.MRN_ERR_INVALID_EPS
    assert sand(e1=eps) == mrn.MRN_ERR_INVALID_EPS
    assert sand(e2=eps) == mrn.MRN_ERR_INVALID_EPS


def test_dtype_validation():
    assert rms(dt=2) == mrn.MRN_ERR_UNSUPPORTED_DTYPE
    assert tadd(dt=-1) == mrn.MRN_ERR_UNSUPPORTED_DTYPE
    assert sand(dt=7) == mrn.MRN_ERR_UNSUPPORTED_DTYPE


def test_null_pointers():
    assert rms(x=None) == mrn.MRN_ERR_NULL_POINTER
    assert rms(g=None) == mrn.MRN_ERR_NULL_POINTER
    assert tadd(r=None) == mrn.MRN_ERR_NULL_POINTER
    for kw in ("b", "r", "gp", "gq", "s", "o"):
        assert sand(**{kw: None}) == mrn.MRN_ERR_NULL_POINTER, kw


def test_misaligned_pointers():
    assert rms(x=A + 2) == mrn.MRN_ERR_MISALIGNED                 # f32 needs 4 bytes
    assert rms(x=A + 1, dt=mrn.MRN_BF16) == mrn.MRN_ERR_MISALIGNED
    assert tadd(r=B + 1) == mrn.MRN_ERR_MISALIGNED
    assert sand(gq=H + 3) == mrn.MRN_ERR_MISALIGNED


def test_forbidden_aliasing():
    rb = 4 * 64 * 4
    assert rms(y=A + 4) == mrn.MRN_ERR_ALIASING                    # partial overlap
    assert rms(y=G - 8) == mrn.MRN_ERR_ALIASING                    # output over gamma
    assert tadd(o=B + rb - 4) == mrn.MRN_ERR_ALIASING              # tail overlaps residual
    assert sand(o=Y) == mrn.MRN_ERR_ALIASING                       # normed == out_stream
    assert sand(o=Y + 64) == mrn.MRN_ERR_ALIASING                  # outputs overlap
    assert sand(s=G) == mrn.MRN_ERR_ALIASING                       # stream over gamma_post
    assert sand(o=H - 16) == mrn.MRN_ERR_ALIASING                  # normed over gamma_pre
    assert sand(s=A + 256) == mrn.MRN_ERR_ALIASING                 # partial over block_out
    assert mrn.mrn_launch_count() == 0


def test_geometry_covers_every_row_width():
    for dt, e in ((mrn.MRN_F32, 4), (mrn.MRN_BF16, 2)):
        for n in [1, 2, 3, 7, 8, 31, 33, 100, 127, 128, 129, 255, 256, 257, 768, 1000, 2048,
                  4096, 5120, 6656, 6657, 8192, 16384, 32768, 65536, 131072, 262144, 1 << 20]:
            for rows in (1, 4, 64, 4096, 65536):
                for a16 in (True, False):
                    for op in (0, 1, 2, 3, 4, 5, 6, 7):
                        if op == 5 and n % 32:
                            continue
                        g = mrn.mrn_query_geometry(op, rows, n, dt, a16, 152)
                        vec = g["vec"]
                        if g["edge"]:
                            # rows not 16-byte aligned, every row operand at one offset
                            # (aligned buffers with a pitch that is not a multiple of 16)
                            assert a16 and (n * e) % 16 != 0 and op in (0, 1, 2, 4)
                            assert g["kind"] == mrn.MRN_GEOM_TMA and g["groups"] == 2
                            assert vec == 16 // e and rows >= 152 and n > 256
                            gran = (n * e + 15) // 16 + 1
                            assert g["threads"] // 2 * g["k"] >= gran and g["cluster"] == 1
                            assert g["threads"] // 2 % 32 == 0
                            stage = gran * 16
                            four = (op, e) == (0, 4) and stage * 5 <= 232448 - 1024
                            assert g["stages"] == (4 if four else 2)
                            ng = 2 if op == 2 else 1
                            nin = 1 if op == 0 else 2
                            assert stage * (ng + g["stages"] * nin) <= 232448 - 1024
                            continue
                        assert vec == (16 // e if a16 and (n * e) % 16 == 0 else 1)
                        nvec = -(-n // vec)
                        if g["kind"] == mrn.MRN_GEOM_ROWS_PER_WARP:
                            assert g["lanes_per_row"] * g["k"] >= nvec
                            if op == 5:
                                assert g["lanes_per_row"] >= 32 // vec
                            assert g["threads"] == 128 and 32 % g["lanes_per_row"] == 0
                        elif g["kind"] == mrn.MRN_GEOM_CTA:
                            assert g["cluster"] * g["threads"] * g["k"] >= nvec
                            assert g["threads"] % 32 == 0 and 1 <= g["cluster"] <= 16
                            cap = 1024 if g["k"] <= 2 else (512 if g["k"] <= 4 else 256)
                            assert g["threads"] <= cap
                        elif g["kind"] == mrn.MRN_GEOM_Q8_BLOCKS:
                            assert op == 5 and a16 and rows >= 152 and g["k"] in (1, 2)
                            if g["stages"]:                    # staged, two groups
                                per = g["threads"] // g["groups"]
                                assert per * g["k"] * 32 >= n and per <= 256 and per % 32 == 0
                                assert g["stages"] % g["groups"] == 0
                                assert (n * e * (1 + g["stages"]) +
                                        g["groups"] * ((n // 32 * 36 + 15) // 16 * 16)) <= 232448 - 1024
                            else:
                                assert g["threads"] * g["k"] * 32 >= n and g["threads"] <= 512
                                assert g["threads"] % 32 == 0
                        elif g["kind"] == mrn.MRN_GEOM_TMA:
                            assert a16 and rows >= 152
                            cl = g["cluster"]
                            per_group = g["threads"] // g["groups"]
                            assert per_group * g["k"] * cl >= nvec and per_group % 32 == 0
                            assert 2 <= g["stages"] <= 4 and g["ctas"] == 0
                            assert g["groups"] in (1, 2) and g["stages"] % g["groups"] == 0
                            assert cl == 1 or (g["groups"] == 1 and op in (0, 1, 2, 4) and
                                               (n * e) % (16 * cl) == 0)
                            ng = 2 if op == 2 else (0 if op in (6, 7) else 1)
                            ns = 1 if op in (0, 5, 6, 7) else 2
                            assert (ng + g["stages"] * ns) * n * e // cl <= 232448 - 1024
                        else:
                            assert g["kind"] == mrn.MRN_GEOM_STREAM
                            assert g["cluster"] == (8 if rows >= 32 else 16)
                            assert nvec > 16 * 2048


# (op, rows, n, dtype) -> (cluster, stages, threads, k) of the cluster-staged kernel,
# as measured best on GB300: slices of at most 2048 loads; plain 3 stages at C = 2,
# else 2; then-add (and -scale) 3 stages from C = 8; the sandwich doubles C from 8.
CLUSTER_STAGED = [
    ((0, 1024, 16384, 0), (2, 3, 256, 8)),   # (plain f32 from 2048 rows: the register kernel)
    ((1, 4096, 16384, 0), (2, 2, 256, 8)),
    ((2, 16384, 16384, 0), (2, 2, 256, 8)),
    ((0, 1024, 32768, 0), (4, 2, 256, 8)),
    ((1, 8192, 32768, 0), (4, 2, 256, 8)),
    ((0, 1024, 65536, 0), (8, 2, 256, 8)),
    ((0, 4096, 65536, 0), (8, 2, 256, 8)),   # (past 8 x 1024 loads plain f32 stays staged)
    ((1, 4096, 65536, 0), (8, 3, 256, 8)),
    ((4, 4096, 65536, 0), (8, 3, 256, 8)),
    ((2, 4096, 65536, 0), (16, 2, 256, 4)),
    ((0, 8192, 32768, 1), (2, 3, 256, 8)),
    ((2, 8192, 32768, 1), (2, 2, 256, 8)),
    ((0, 4096, 131072, 0), (16, 2, 256, 8)),
]


# Plain f32 batches of 2048 rows or more with rows of 2049 .. 8 x 1024 loads: the
# register kernel at eight slots per thread in clusters of ceil(loads / 1024) CTAs.
REGISTER_CLUSTER = [((4096, 16384), (4, 128)), ((65536, 16384), (4, 128)),
                    ((4096, 32768), (8, 128)), ((4096, 10240), (3, 128)),
                    ((2048, 8196), (3, 96))]


@pytest.mark.parametrize("shape,want", REGISTER_CLUSTER, ids=[str(c) for c, _ in REGISTER_CLUSTER])
def test_plain_f32_wide_batches_use_the_register_cluster_kernel(shape, want):
    g = mrn.mrn_query_geometry(0, shape[0], shape[1], mrn.MRN_F32, True, 152)
    assert (g["kind"], g["cluster"], g["threads"], g["k"]) == (mrn.MRN_GEOM_CTA, *want, 8)
    assert g["threads"] * g["k"] * g["cluster"] >= shape[1] // 4


@pytest.mark.parametrize("call,want", CLUSTER_STAGED, ids=[str(c) for c, _ in CLUSTER_STAGED])
def test_cluster_staged_geometry_choice(call, want):
    op, rows, n, dt = call
    g = mrn.mrn_query_geometry(op, rows, n, dt, True, 152)
    assert g["kind"] == mrn.MRN_GEOM_TMA and g["groups"] == 1
    assert (g["cluster"], g["stages"], g["threads"], g["k"]) == want


def test_cluster_staged_kernel_is_not_chosen_outside_its_range():
    # fewer rows than SMs, slices that are not 16-byte multiples, too wide, or an
    # operation it does not serve: other kernels
    for op, rows, n, dt in ((0, 100, 65536, 0), (1, 4096, 16388, 0), (0, 4096, 262144, 0),
                            (3, 4096, 16384, 0), (6, 4096, 16384, 0)):
        g = mrn.mrn_query_geometry(op, rows, n, dt, True, 152)
        assert not (g["kind"] == mrn.MRN_GEOM_TMA and g["cluster"] > 1), (op, rows, n, g)


def test_force_geometry_validation():
    bad = [
        {"kind": 1, "lanes_per_row": 3, "k": 1},
        {"kind": 1, "lanes_per_row": 64, "k": 1},
        {"kind": 2, "k": 9, "threads": 128, "cluster": 1},
        {"kind": 2, "k": 8, "threads": 512, "cluster": 1},     # above the k=8 launch bound
        {"kind": 2, "k": 1, "threads": 100, "cluster": 1},
        {"kind": 2, "k": 1, "threads": 128, "cluster": 17},
        {"kind": 3, "threads": 1024},
        {"kind": 4, "k": 4, "threads": 416, "stages": 0},
        {"kind": 4, "k": 4, "threads": 416, "stages": 9},
        {"kind": 4, "k": 8, "threads": 512, "stages": 2},
        {"kind": 4, "k": 2, "threads": 96, "stages": 2, "ctas": -1},
        {"kind": 4, "k": 4, "threads": 832, "stages": 3, "groups": 3},
        {"kind": 4, "k": 4, "threads": 832, "stages": 1, "groups": 2},     # a stage per group
        {"kind": 4, "k": 7, "threads": 512, "stages": 3, "groups": 2},     # stages % groups
        {"kind": 4, "k": 4, "threads": 800, "stages": 2, "groups": 2},     # 400 not a warp multiple
        {"kind": 4, "k": 8, "threads": 1024, "stages": 2, "groups": 2},    # 512 > 256 per group
        {"kind": 9},
        {"kind": 5, "k": 3, "threads": 128},
        {"kind": 5, "k": 1, "threads": 1024},
        {"kind": 5, "k": 1, "threads": 100},
        {"kind": 5, "k": 1, "threads": 1024, "stages": 2, "groups": 2},    # 512 > 256 per group
        {"kind": 5, "k": 1, "threads": 256, "stages": 3, "groups": 2},     # stages % groups
        {"kind": 5, "k": 1, "threads": 96, "stages": 2, "groups": 2},      # 48 per group
    ]
    for g in bad:
        assert mrn.mrn_force_geometry(g) == mrn.MRN_ERR_INVALID_GEOMETRY, g
    assert mrn.mrn_force_geometry({"kind": 2, "k": 2, "threads": 64, "cluster": 2}) == 0
    got = mrn.mrn_query_geometry(0, 8, 1024, mrn.MRN_F32, True, 152)
    assert (got["kind"], got["k"], got["threads"], got["cluster"]) == (2, 2, 64, 2)
    with pytest.raises(mrn.MrnError):          # 2*64*2 = 256 loads cannot cover n = 4096
        mrn.mrn_query_geometry(0, 8, 4096, mrn.MRN_F32, True, 152)
    assert mrn.mrn_force_geometry(None) == 0
    assert mrn.mrn_query_geometry(0, 8, 4096, mrn.MRN_F32, True, 152)["kind"] == 2
    # staged kernel: needs aligned rows and shared memory for the stages
    assert mrn.mrn_force_geometry({"kind": 4, "k": 4, "threads": 416, "stages": 3}) == 0
    got = mrn.mrn_query_geometry(2, 4096, 6656, mrn.MRN_F32, True, 152)
    assert (got["kind"], got["k"], got["threads"], got["stages"]) == (4, 4, 416, 3)
    with pytest.raises(mrn.MrnError):          # misaligned rows cannot be bulk-copied
        mrn.mrn_query_geometry(2, 4096, 6656, mrn.MRN_F32, False, 152)
    assert mrn.mrn_force_geometry({"kind": 4, "k": 4, "threads": 416, "stages": 4}) == 0
    with pytest.raises(mrn.MrnError):          # (2 + 4*2) rows of 26 KB exceed 227 KB
        mrn.mrn_query_geometry(2, 4096, 6656, mrn.MRN_F32, True, 152)
    assert mrn.mrn_force_geometry(None) == 0
    # automatic: the f32 sandwich batch in the register kernel (one reduction per row),
    # the bf16 one staged; decode over a cluster of 16 (f32) or 4 (bf16, 832 loads)
    got = mrn.mrn_query_geometry(2, 4096, 6656, mrn.MRN_F32, True, 152)
    assert (got["kind"], got["k"], got["threads"], got["cluster"]) == (2, 7, 256, 1)
    assert mrn.mrn_query_geometry(2, 4096, 6656, mrn.MRN_BF16, True, 152)["kind"] == 4
    got = mrn.mrn_query_geometry(2, 1, 6656, mrn.MRN_F32, True, 152)
    assert (got["kind"], got["threads"], got["cluster"]) == (2, 128, 16)
    assert mrn.mrn_query_geometry(2, 1, 6656, mrn.MRN_BF16, True, 152)["cluster"] == 4


def test_launch_options():
    assert mrn.mrn_launch_options() == mrn.MRN_LAUNCH_PDL          # the default
    assert mrn.mrn_set_launch_options(2) == mrn.MRN_ERR_INVALID_GEOMETRY
    assert mrn.mrn_set_launch_options(0) == 0 and mrn.mrn_launch_options() == 0
    assert mrn.mrn_set_launch_options(mrn.MRN_LAUNCH_PDL) == 0
    both = mrn.MRN_LAUNCH_PDL | mrn.MRN_LAUNCH_TEST_WAIT_TIMEOUT   # the test hook is a known bit
    assert mrn.mrn_set_launch_options(both) == 0 and mrn.mrn_launch_options() == both
    assert mrn.mrn_set_launch_options(mrn.MRN_LAUNCH_PDL) == 0
    assert mrn.mrn_launch_options() == mrn.MRN_LAUNCH_PDL


def test_binding_fails_loudly_without_the_library(tmp_path):
    code = ("import dual_epsilon_sandwich_gb300.mrn as m; m.LIBRARY = '/nonexistent/libmrn.so'\n"
            "try:\n    m.mrn_status_string(0)\nexcept RuntimeError as e:\n"
            "    print('raised', e)\nelse:\n    raise SystemExit('no error')\n")
    res = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True)
    assert res.returncode == 0 and "raised" in res.stdout, res.stderr


def test_unaligned_rows_query_and_force():
    """Row operands at one offset within 16 bytes (aligned16 = 2) take the
    edge-staged kernel for batches of the four operations it serves; the
    others, few rows and short rows move element-wise; a forced edge geometry
    must be a two-group staged one."""
    g = mrn.mrn_query_geometry(mrn.MRN_OP_SANDWICH, 4096, 6656, mrn.MRN_F32, 2, 152)
    assert g["edge"] == 1 and g["kind"] == mrn.MRN_GEOM_TMA and g["vec"] == 4
    g = mrn.mrn_query_geometry(mrn.MRN_OP_RMSNORM, 4096, 6655, mrn.MRN_F32, True, 152)
    assert g["edge"] == 1 and g["threads"] // 2 * g["k"] >= 6655 * 4 // 16 + 2
    for op in (mrn.MRN_OP_ADD_RMSNORM, mrn.MRN_OP_RMSNORM_SEAM):
        g = mrn.mrn_query_geometry(op, 4096, 6655, mrn.MRN_F32, 2, 152)
        assert g["edge"] == 0 and g["vec"] == 1
    g = mrn.mrn_query_geometry(mrn.MRN_OP_THEN_ADD, 64, 6655, mrn.MRN_F32, 2, 152)
    assert g["edge"] == 0 and g["vec"] == 1 and g["kind"] == mrn.MRN_GEOM_CTA
    g = mrn.mrn_query_geometry(mrn.MRN_OP_RMSNORM, 4096, 7, mrn.MRN_F32, 2, 152)
    assert g["edge"] == 0 and g["kind"] == mrn.MRN_GEOM_ROWS_PER_WARP
    g = mrn.mrn_query_geometry(mrn.MRN_OP_RMSNORM, 4096, 5121, mrn.MRN_BF16, 0, 152)
    assert g["edge"] == 0 and g["vec"] == 1
    bad = [{"kind": 2, "k": 4, "threads": 256, "cluster": 1, "edge": 1},
           {"kind": 4, "k": 4, "threads": 416, "stages": 2, "groups": 1, "edge": 1},
           {"kind": 4, "k": 4, "threads": 256, "stages": 1, "groups": 1, "cluster": 2, "edge": 1}]
    for geo in bad:
        full = {"vec": 0, "lanes_per_row": 0, "stages": 0, "ctas": 0, "groups": 0, "cluster": 1}
        full.update(geo)
        assert mrn.mrn_force_geometry(full) == mrn.MRN_ERR_INVALID_GEOMETRY, geo
    ok = {"kind": 4, "vec": 0, "k": 8, "threads": 448, "cluster": 1, "lanes_per_row": 0,
          "stages": 2, "ctas": 0, "groups": 2, "edge": 1}
    assert mrn.mrn_force_geometry(ok) == 0
    try:
        g = mrn.mrn_query_geometry(mrn.MRN_OP_SANDWICH, 4096, 6655, mrn.MRN_F32, 2, 152)
        assert g["edge"] == 1 and g["threads"] == 448
        with pytest.raises(mrn.MrnError):      # add + norm has no edge-staged form
            mrn.mrn_query_geometry(mrn.MRN_OP_ADD_RMSNORM, 4096, 6655, mrn.MRN_F32, 2, 152)
        with pytest.raises(mrn.MrnError):      # 224 x 8 loads per group: 1792 < 1801 granules
            mrn.mrn_query_geometry(mrn.MRN_OP_SANDWICH, 4096, 7200, mrn.MRN_F32, 2, 152)
    finally:
        mrn.mrn_force_geometry(None)
