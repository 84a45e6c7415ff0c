"""Python access to the fp64 CPU oracle (oracle.c) through ctypes.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` use this module; the CUDA product path
(``rmsnorm_fwd_bwd_02_gb300``) never imports it and the oracle never imports
the product. What the oracle computes, and which passage of the pages each
function follows, is documented in oracle.c.

Inputs are torch CPU tensors (float32, bfloat16, float16 or float64), contiguous,
row-major ``[M, H]`` with a ``[H]`` weight. Outputs are float64 tensors, except
the residual sum ``h``, which is stored in the input dtype as the method does.
"""
import ctypes
import os

import torch

from . import build as _build

F32, BF16, F64, F16 = 0, 1, 2, 3
_CODES = {torch.float32: F32, torch.bfloat16: BF16, torch.float64: F64,
          torch.float16: F16}

_i64 = ctypes.c_int64
_vp = ctypes.c_void_p
_dbl = ctypes.c_double


def _declare(lib):
    lib.oracle_rmsnorm_fwd.argtypes = [_i64, _i64, _vp, _vp, ctypes.c_int,
                                       _dbl, _vp, _vp]
    lib.oracle_rmsnorm_fwd.restype = None
    lib.oracle_rmsnorm_bwd.argtypes = [_i64, _i64, _vp, _vp, _vp, ctypes.c_int,
                                       _dbl, _vp, _vp, _vp, _vp]
    lib.oracle_rmsnorm_bwd.restype = None
    lib.oracle_residual_fwd.argtypes = [_i64, _i64, _vp, _vp, _vp, ctypes.c_int,
                                        _dbl, _vp, _vp, _vp]
    lib.oracle_residual_fwd.restype = None
    lib.oracle_residual_bwd.argtypes = [_i64, _i64, _vp, _vp, _vp, _vp,
                                        ctypes.c_int, _dbl, _vp, _vp, _vp, _vp]
    lib.oracle_residual_bwd.restype = None
    lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_double.restype = _dbl
    lib.oracle_bf16_from_double.argtypes = [_dbl]
    lib.oracle_bf16_from_double.restype = ctypes.c_uint16
    lib.oracle_rmsnorm_bwd_bwd.argtypes = [_i64, _i64, _vp, _vp, _vp, _vp, _vp,
                                           ctypes.c_int, _dbl, _vp, _vp, _vp, _vp,
                                           _vp, _vp]
    lib.oracle_rmsnorm_bwd_bwd.restype = None
    lib.oracle_rmsnorm_gemv.argtypes = [_i64, _i64, _i64, _vp, _vp, _vp, _vp,
                                        ctypes.c_int, _dbl, _vp, _vp, _vp, _vp,
                                        _vp]
    lib.oracle_rmsnorm_gemv.restype = ctypes.c_int
    lib.oracle_f16_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_f16_to_double.restype = _dbl
    lib.oracle_f16_from_double.argtypes = [_dbl]
    lib.oracle_f16_from_double.restype = ctypes.c_uint16
    return lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check_rows(name, t, dtype, M, H):
    if t.device.type != "cpu" or not t.is_contiguous():
        raise ValueError(f"oracle: {name} must be a contiguous CPU tensor")
    if t.dtype != dtype or t.numel() != M * H:
        raise ValueError(f"oracle: {name} must be {dtype} with {M}x{H} elements")


class Oracle:
    """One loaded copy of the oracle library (the tests also load mutated
    copies of it, to show that the pins catch planted mistakes)."""

    def __init__(self, path=None):
        path = path or _build.build()
        self.path = path
        self.lib = _declare(ctypes.CDLL(path))

    # -- formats
    def bf16_to_double(self, bits: int) -> float:
        return self.lib.oracle_bf16_to_double(bits & 0xFFFF)

    def bf16_from_double(self, v: float) -> int:
        return self.lib.oracle_bf16_from_double(float(v))

    def f16_to_double(self, bits: int) -> float:
        return self.lib.oracle_f16_to_double(bits & 0xFFFF)

    def f16_from_double(self, v: float) -> int:
        return self.lib.oracle_f16_from_double(float(v))

    # -- forward
    def fwd(self, x, w, eps):
        """y, rstd of the RMSNorm forward (float64 results)."""
        M, H = x.shape
        code = _CODES[x.dtype]
        _check_rows("x", x, x.dtype, M, H)
        _check_rows("w", w, x.dtype, 1, H)
        y = torch.empty(M, H, dtype=torch.float64)
        rstd = torch.empty(M, dtype=torch.float64)
        self.lib.oracle_rmsnorm_fwd(M, H, _ptr(x), _ptr(w), code, float(eps),
                                    _ptr(y), _ptr(rstd))
        return y, rstd

    # -- backward
    def bwd(self, dy, x, w, eps, want_dx=True, want_terms=False):
        """dx [M,H] (or None), dw [H]; with want_terms also the error scales
        tdx [M,H] (or None) and tdw [H]."""
        M, H = x.shape
        code = _CODES[x.dtype]
        for name, t in (("dy", dy), ("x", x)):
            _check_rows(name, t, x.dtype, M, H)
        _check_rows("w", w, x.dtype, 1, H)
        dx = torch.empty(M, H, dtype=torch.float64) if want_dx else None
        dw = torch.empty(H, dtype=torch.float64)
        tdx = (torch.empty(M, H, dtype=torch.float64)
               if (want_terms and want_dx) else None)
        tdw = torch.empty(H, dtype=torch.float64) if want_terms else None
        self.lib.oracle_rmsnorm_bwd(M, H, _ptr(dy), _ptr(x), _ptr(w), code,
                                    float(eps), _ptr(dx), _ptr(dw), _ptr(tdx),
                                    _ptr(tdw))
        if want_terms:
            return dx, dw, tdx, tdw
        return dx, dw

    # -- residual variant
    def residual_fwd(self, x, r, w, eps):
        """h (input dtype, rounded once), y, rstd (float64)."""
        M, H = x.shape
        code = _CODES[x.dtype]
        for name, t in (("x", x), ("r", r)):
            _check_rows(name, t, x.dtype, M, H)
        _check_rows("w", w, x.dtype, 1, H)
        h = torch.empty(M, H, dtype=x.dtype)
        y = torch.empty(M, H, dtype=torch.float64)
        rstd = torch.empty(M, dtype=torch.float64)
        self.lib.oracle_residual_fwd(M, H, _ptr(x), _ptr(r), _ptr(w), code,
                                     float(eps), _ptr(h), _ptr(y), _ptr(rstd))
        return h, y, rstd

    def residual_bwd(self, dy, dh_out, h, w, eps, want_dx=True,
                     want_terms=False):
        """dx (= gradient of both x and r) and dw; dh_out may be None."""
        M, H = h.shape
        code = _CODES[h.dtype]
        for name, t in (("dy", dy), ("h", h)):
            _check_rows(name, t, h.dtype, M, H)
        if dh_out is not None:
            _check_rows("dh_out", dh_out, h.dtype, M, H)
        _check_rows("w", w, h.dtype, 1, H)
        dx = torch.empty(M, H, dtype=torch.float64) if want_dx else None
        dw = torch.empty(H, dtype=torch.float64)
        tdx = (torch.empty(M, H, dtype=torch.float64)
               if (want_terms and want_dx) else None)
        tdw = torch.empty(H, dtype=torch.float64) if want_terms else None
        self.lib.oracle_residual_bwd(M, H, _ptr(dy), _ptr(dh_out), _ptr(h),
                                     _ptr(w), code, float(eps), _ptr(dx),
                                     _ptr(dw), _ptr(tdx), _ptr(tdw))
        if want_terms:
            return dx, dw, tdx, tdw
        return dx, dw

    # -- double backward
    def bwd_bwd(self, dy, x, w, gx, gw, eps, want_terms=False):
        """Gradients of sum(gx * dx) + sum(gw * dw) with respect to dy, x and
        w (float64); gx [M,H] in the input dtype or None, gw [H] (any float
        dtype, read as float64) or None. Returns (ddy, dx2, dw2) and with
        want_terms also their error scales."""
        M, H = x.shape
        code = _CODES[x.dtype]
        for name, t in (("dy", dy), ("x", x)):
            _check_rows(name, t, x.dtype, M, H)
        _check_rows("w", w, x.dtype, 1, H)
        if gx is not None:
            _check_rows("gx", gx, x.dtype, M, H)
        gw64 = None if gw is None else gw.detach().to(torch.float64).contiguous()
        ddy = torch.empty(M, H, dtype=torch.float64)
        dx2 = torch.empty(M, H, dtype=torch.float64)
        dw2 = torch.empty(H, dtype=torch.float64)
        t = [torch.empty(M, H, dtype=torch.float64), torch.empty(M, H, dtype=torch.float64),
             torch.empty(H, dtype=torch.float64)] if want_terms else [None] * 3
        self.lib.oracle_rmsnorm_bwd_bwd(M, H, _ptr(dy), _ptr(x), _ptr(w), _ptr(gx),
                                        _ptr(gw64), code, float(eps), _ptr(ddy),
                                        _ptr(dx2), _ptr(dw2), _ptr(t[0]), _ptr(t[1]),
                                        _ptr(t[2]))
        if want_terms:
            return ddy, dx2, dw2, t[0], t[1], t[2]
        return ddy, dx2, dw2

    # -- norm followed by the projection GEMV (decode chain)
    def rmsnorm_gemv(self, x, w, A, eps, r=None):
        """dict with out [M,N] (float64, unrounded), y (the stored norm
        output, input dtype), h (residual variant, else None), rstd and the
        error scale tout [M,N]."""
        M, H = x.shape
        N = A.shape[0]
        code = _CODES[x.dtype]
        _check_rows("x", x, x.dtype, M, H)
        _check_rows("w", w, x.dtype, 1, H)
        _check_rows("A", A, x.dtype, N, H)
        if r is not None:
            _check_rows("r", r, x.dtype, M, H)
        h = torch.empty(M, H, dtype=x.dtype) if r is not None else None
        y = torch.empty(M, H, dtype=x.dtype)
        out = torch.empty(M, N, dtype=torch.float64)
        rstd = torch.empty(M, dtype=torch.float64)
        tout = torch.empty(M, N, dtype=torch.float64)
        st = self.lib.oracle_rmsnorm_gemv(M, H, N, _ptr(x), _ptr(r), _ptr(w),
                                          _ptr(A), code, float(eps), _ptr(h),
                                          _ptr(y), _ptr(out), _ptr(rstd),
                                          _ptr(tout))
        if st != 0:
            raise MemoryError("oracle_rmsnorm_gemv: out of memory")
        return {"out": out, "y": y, "h": h, "rstd": rstd, "tout": tout}


_default = None


def get() -> Oracle:
    """The oracle built from oracle.c (compiled on first use)."""
    global _default
    if _default is None:
        _default = Oracle()
    return _default


def lib_path() -> str:
    return os.path.join(os.path.dirname(os.path.abspath(__file__)),
                        "liboracle.so")
