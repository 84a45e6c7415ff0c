"""CPU tier: the C-ABI library loads, exports every entry point that
include/rmsnorm.h declares, and rejects bad arguments on the host before any
CUDA call (no GPU needed). The argument checks pass made-up addresses, and
the calls that pass the checks are expected to fail only for want of a
device: on a machine with a GPU they would launch kernels on those
addresses, so every test that calls the library is skipped there."""
import ctypes
import os
import re

import pytest

from rmsnorm_fwd_bwd_02_gb300 import rmsnorm as rn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "rmsnorm.h")

OK, NULLPTR, BAD_SHAPE, BAD_DTYPE, BAD_EPS, MISALIGNED, WORKSPACE, \
    UNSUPPORTED, CUDA, ALIAS = 0, -1, -2, -3, -4, -5, -6, -7, -8, -9
F32, BF16, F16 = 0, 1, 2
BAD_STRIDE = -12
NAN = float("nan")


@pytest.fixture(scope="module")
def lib():
    import torch
    if torch.cuda.is_available():
        pytest.skip("calls the library with made-up addresses: host-only (no GPU) tier")
    if not os.path.exists(rn.LIB_PATH):
        from rmsnorm_fwd_bwd_02_gb300 import build
        build.build()
    return rn.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(rmsnorm_\w+)\s*\(", text)))


def test_header_declares_the_four_entry_points():
    names = declared_functions()
    for n in ("rmsnorm_fwd", "rmsnorm_bwd", "rmsnorm_residual_fwd",
              "rmsnorm_residual_bwd"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in rmsnorm.h but not exported"
        assert n in rn.SIGNATURES, f"{n} has no ctypes signature in the binding"


def test_static_scratch_limit_matches_header():
    """The binding's copies of the built-in scratch size and of its refusal
    code are the header's."""
    text = open(HEADER).read()
    m = re.search(r"#define\s+RMSNORM_STATIC_SCRATCH_BYTES\s+\(\(size_t\)(\d+)\s*<<\s*(\d+)\)",
                  text)
    assert m is not None
    assert int(m.group(1)) << int(m.group(2)) == rn.STATIC_SCRATCH_BYTES
    m = re.search(r"RMSNORM_ERR_SCRATCH_LIMIT\s*=\s*(-\d+)", text)
    assert m is not None and int(m.group(1)) == rn.ERR_SCRATCH_LIMIT


def test_status_strings(lib):
    for code in (OK, NULLPTR, BAD_SHAPE, BAD_DTYPE, BAD_EPS, MISALIGNED,
                 WORKSPACE, UNSUPPORTED, CUDA, ALIAS, BAD_STRIDE):
        s = lib.rmsnorm_status_string(code).decode()
        assert s and s != "unknown status"
    assert lib.rmsnorm_status_string(12345).decode() == "unknown status"


# Fake device addresses: the checks below all fail on the host, before the
# library touches CUDA, so nothing is dereferenced.
A = 0x7f0000000000
B = 0x7f0100000000
C = 0x7f0200000000
D = 0x7f0300000000


def fwd(lib, x=A, w=B, y=C, rstd=D, M=4, H=8, eps=1e-6, dtype=BF16):
    return lib.rmsnorm_fwd(x, w, y, rstd, M, H, eps, dtype, None)


def test_fwd_argument_checks(lib):
    assert fwd(lib, dtype=7) == BAD_DTYPE
    assert fwd(lib, M=-1) == BAD_SHAPE
    assert fwd(lib, H=0) == BAD_SHAPE
    assert fwd(lib, H=16385) == UNSUPPORTED
    assert fwd(lib, M=2 ** 62) == BAD_SHAPE
    for e in (NAN, -1e-6, float("inf")):
        assert fwd(lib, eps=e) == BAD_EPS
    assert fwd(lib, x=None) == NULLPTR
    assert fwd(lib, w=None) == NULLPTR
    assert fwd(lib, y=None) == NULLPTR
    assert fwd(lib, x=A + 1) == MISALIGNED           # bf16 needs 2-byte
    assert fwd(lib, x=A + 2, dtype=F32) == MISALIGNED
    assert fwd(lib, rstd=D + 2) == MISALIGNED
    # y overlapping x partially (not the same buffer) is rejected ...
    assert fwd(lib, y=A + 2) == ALIAS
    # ... rstd inside y too
    assert fwd(lib, rstd=C + 4) == ALIAS
    # nothing to do for M == 0, even with NULL pointers
    assert fwd(lib, x=None, w=None, y=None, rstd=None, M=0) == OK


def test_fp16_is_a_dtype(lib):
    # fp16 passes the dtype check and is checked as a 2-byte type
    assert fwd(lib, x=A + 1, dtype=F16) == MISALIGNED
    assert fwd(lib, dtype=3) == BAD_DTYPE
    assert fwd(lib, x=None, w=None, y=None, rstd=None, M=0, dtype=F16) == OK


def no_gpu():
    import torch
    return not torch.cuda.is_available()


def fwd_s(lib, x=A, ldx=256, r=None, ldr=256, w=B, y=C, ldy=256, h=None,
          ldh=256, rstd=D, M=4, H=128, dtype=BF16):
    return lib.rmsnorm_fwd_strided(x, ldx, r, ldr, w, y, ldy, h, ldh, rstd, M,
                                   H, 1e-6, dtype, None)


def test_fwd_strided_argument_checks(lib):
    assert fwd_s(lib, ldx=127) == BAD_STRIDE
    assert fwd_s(lib, ldy=0) == BAD_STRIDE
    assert fwd_s(lib, ldx=2 ** 31) == BAD_STRIDE
    assert fwd_s(lib, M=2 ** 40, ldx=2 ** 30) == BAD_STRIDE   # past 2^63 bytes
    assert fwd_s(lib, r=0x7f0400000000) == NULLPTR            # r without h
    assert fwd_s(lib, h=0x7f0400000000) == NULLPTR            # h without r
    # y at the same start as x but another stride: not the same tensor
    assert fwd_s(lib, y=A, ldy=128) == ALIAS
    # y's columns start 127 elements into x's rows: they meet x's window
    assert fwd_s(lib, y=A + 254) == ALIAS
    # rstd in the gap between x's rows still counts as inside x's range
    assert fwd_s(lib, rstd=A + 256) == ALIAS


@pytest.mark.skipif("not no_gpu()")
def test_fwd_strided_allowed_layouts_reach_the_device(lib):
    """Layouts the alias rule allows pass every host check; without a GPU
    the first CUDA call then fails (status CUDA), which shows it."""
    # y in the other half of x's 256-wide rows: disjoint windows
    assert fwd_s(lib, y=A + 256) == CUDA
    # in place: same start and stride
    assert fwd_s(lib, y=A) == CUDA
    # one row: the stride does not matter
    assert fwd_s(lib, y=A, ldy=128, M=1) == CUDA
    # residual, h in place of r, everything interleaved in one buffer
    assert fwd_s(lib, x=A, r=A + 256, h=A + 256, y=A + 512, ldx=384, ldr=384,
                 ldh=384, ldy=384) == CUDA
    assert fwd_s(lib, dtype=F16) == CUDA


def bwd_s(lib, dy=A, lddy=256, dh=None, lddh=256, x=B, ldx=256, w=C, rstd=D,
          dx=0x7f0400000000, lddx=256, dw=0x7f0500000000, ws=0x7f0600000000,
          wsb=1 << 24, M=4, H=128, flags=0, dtype=BF16):
    return lib.rmsnorm_bwd_strided(dy, lddy, dh, lddh, x, ldx, w, rstd, dx,
                                   lddx, dw, ws, wsb, M, H, 1e-6, dtype,
                                   flags, None)


def test_bwd_strided_argument_checks(lib):
    assert bwd_s(lib, lddy=100) == BAD_STRIDE
    assert bwd_s(lib, ldx=100) == BAD_STRIDE
    assert bwd_s(lib, lddx=2 ** 31) == BAD_STRIDE
    assert bwd_s(lib, dh=0x7f0700000000, lddh=1) == BAD_STRIDE
    assert bwd_s(lib, flags=4) == -11
    assert bwd_s(lib, dx=A + 2) == ALIAS          # dx partially over dy
    assert bwd_s(lib, dx=B + 2) == ALIAS          # dx over x's columns
    assert bwd_s(lib, dw=B + 256) == ALIAS        # dw between x's rows (in its range)


@pytest.mark.skipif("not no_gpu()")
def test_bwd_strided_allowed_layouts_reach_the_device(lib):
    assert bwd_s(lib, dx=A) == CUDA               # in place over dy
    assert bwd_s(lib, dx=A + 256) == CUDA         # other half of dy's rows
    assert bwd_s(lib, dx=B + 256) == CUDA         # other half of x's rows
    assert bwd_s(lib, dtype=F16) == CUDA


def test_gemv_argument_checks(lib):
    f = lib.rmsnorm_gemv_fwd
    E = 0x7f0400000000
    # x r w A out h y rstd M H N
    args = dict(x=A, r=None, w=B, A=C, out=D, h=None, y=None, rstd=None, M=1,
                H=896, N=64, dtype=BF16)

    def call(flags=0, **kw):
        a = dict(args, **kw)
        return f(a["x"], a["r"], a["w"], a["A"], a["out"], a["h"], a["y"],
                 a["rstd"], a["M"], a["H"], a["N"], 1e-6, a["dtype"], flags, None)
    assert call(flags=4) == -11
    assert call(M=65) == UNSUPPORTED
    assert call(H=900) == UNSUPPORTED
    assert call(M=64, H=16384) == UNSUPPORTED
    # wider rows that only a tcgen05 kernel holds pass the checks (and then
    # fail on the missing device): the K-split kernel up to 3584 at 64 rows,
    # the persistent one with K split over up to 8 CTAs up to 7168 at 64
    # rows, 11264 at 48, all of RMSNORM_MAX_H at 32; none above 8 rows
    assert call(M=64, H=3584) == CUDA
    assert call(M=64, H=7168) == CUDA
    assert call(M=64, H=7200) == UNSUPPORTED
    assert call(M=48, H=11264, r=E) == CUDA
    assert call(M=48, H=11296, r=E) == UNSUPPORTED
    assert call(M=32, H=16384, r=E) == CUDA
    assert call(M=8, H=6752) == UNSUPPORTED
    assert call(dtype=F32) == UNSUPPORTED
    assert call(N=0) == BAD_SHAPE
    assert call(h=E) == NULLPTR
    assert call(A=None) == NULLPTR
    assert call(A=C + 8) == MISALIGNED
    assert call(out=A) == ALIAS
    assert call(r=E, h=A) == ALIAS
    assert call(y=C) == ALIAS
    assert call(M=0, x=None, w=None, A=None, out=None) == OK


def test_residual_fwd_argument_checks(lib):
    f = lib.rmsnorm_residual_fwd
    E = 0x7f0400000000
    F = 0x7f0500000000
    assert f(A, B, C, D, E, F, 4, 8, 1e-6, BF16 + 5, None) == BAD_DTYPE
    assert f(A, None, C, D, E, F, 4, 8, 1e-6, BF16, None) == NULLPTR
    # y may not alias anything, h may not partially overlap x
    assert f(A, B, C, D, A, F, 4, 8, 1e-6, BF16, None) == ALIAS
    assert f(A, B, C, A + 2, E, F, 4, 8, 1e-6, BF16, None) == ALIAS
    assert f(A, B, C, D, E, F + 1, 4, 8, 1e-6, BF16, None) == MISALIGNED


def test_bwd_argument_checks(lib):
    f = lib.rmsnorm_bwd
    E = 0x7f0400000000
    W = 0x7f0500000000
    # dy x w rstd dx dw ws
    assert f(A, B, C, D, E, None, W, 1 << 20, 4, 8, 1e-6, BF16, None) == NULLPTR
    assert f(None, B, C, D, E, 0x7f0600000000, W, 1 << 20, 4, 8, 1e-6, BF16,
             None) == NULLPTR
    assert f(A, B, C, D, E, 0x7f0600000000, W + 8, 1 << 20, 4, 8, 1e-6, BF16,
             None) == MISALIGNED    # workspace must be 16-byte aligned
    assert f(A, B, C, D, E, 0x7f0600000002, W, 1 << 20, 4, 8, 1e-6, BF16,
             None) == MISALIGNED    # dw is fp32
    assert f(A, B, C, D, E, 0x7f0600000000, W, 1 << 20, 4, 8, -1.0, BF16,
             None) == BAD_EPS
    assert f(A, B, C, D, E, 0x7f0600000000, W, 1 << 20, -4, 8, 1e-6, BF16,
             None) == BAD_SHAPE


def test_bwd_ex_rejects_unknown_flags(lib):
    f = lib.rmsnorm_bwd_ex
    E = 0x7f0400000000
    W = 0x7f0500000000
    assert f(A, None, B, C, D, E, 0x7f0600000000, W, 1 << 20, 4, 8, 1e-6, BF16,
             2, None) == -11
    assert lib.rmsnorm_status_string(-11).decode() != "unknown status"


def test_workspace_query_without_device(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; covered by the GPU tests")
    assert lib.rmsnorm_bwd_workspace_bytes(1024, 4096, BF16) == 0
    assert lib.rmsnorm_bwd_workspace_bytes(-1, 4096, BF16) == 0


def test_path_override_roundtrip(lib):
    lib.rmsnorm_set_path_override(2)
    lib.rmsnorm_set_path_override(99)     # out of range: back to automatic
    lib.rmsnorm_set_path_override(0)
    assert lib.rmsnorm_last_path() in (0, 1, 2, 3)
    assert lib.rmsnorm_last_cuda_error() >= 0


def test_binding_refuses_cpu_tensors(lib):
    import torch
    x = torch.zeros(2, 8, dtype=torch.bfloat16)
    w = torch.ones(8, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        rn.rmsnorm_fwd(x, w)


def test_product_path_has_no_oracle_dependency():
    """The CUDA path never imports, links, loads or calls the oracle."""
    pkg = os.path.join(ROOT, "rmsnorm_fwd_bwd_02_gb300")
    pat = re.compile(r"\b(import|from)\s+oracle\b|liboracle|oracle_\w+\s*\(|"
                     r"oracle\.c\b|oracle/")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, fn), encoding="utf-8").read()
                m = pat.search(text)
                assert m is None, f"{fn} refers to the oracle: {m.group(0)!r}"


def test_ctypes_loads_standalone():
    # a fresh handle to the same file loads too (no hidden state needed)
    l2 = ctypes.CDLL(rn.LIB_PATH)
    assert hasattr(l2, "rmsnorm_fwd")
