"""Thin ctypes binding over librmsnorm.so (C ABI in include/rmsnorm.h).

Same entry-point names as the C ABI. Argument marshalling only: tensors are
checked (CUDA, contiguous or row-strided, dtype, shape), outputs that the
caller did not pass are allocated with torch, and raw device pointers, row
strides and the current torch CUDA stream are handed to the library. Every arithmetic step runs in the
CUDA kernels. If the library has not been built this module raises at load
time; there is no fallback.
"""
import ctypes
import os

import torch

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "librmsnorm.so")

RMSNORM_F32, RMSNORM_BF16, RMSNORM_F16 = 0, 1, 2
DTYPES = {torch.float32: RMSNORM_F32, torch.bfloat16: RMSNORM_BF16,
          torch.float16: RMSNORM_F16}
MAX_H = 16384
PATH_AUTO, PATH_ROWS, PATH_SPLIT, PATH_SCALAR, PATH_STREAM = 0, 1, 2, 3, 4
PATH_GEMV = 5            # reported by last_path() after rmsnorm_gemv_fwd: the
PATH_GEMV_TMA = 6        # weight in registers (5), fed by bulk copies (6), or
PATH_GEMV_UMMA = 7       # the product on tcgen05 (7); 6 and 7 also force it
PATH_GEMV_TC = 8         # persistent tcgen05 kernel, y held per CTA (8; forces it)

# Entry points of include/rmsnorm.h with their ctypes signatures.
_i64, _vp, _sz, _int, _f = (ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t,
                            ctypes.c_int, ctypes.c_float)
SIGNATURES = {
    "rmsnorm_fwd": (_int, [_vp, _vp, _vp, _vp, _i64, _i64, _f, _int, _vp]),
    "rmsnorm_bwd": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _i64, _i64,
                           _f, _int, _vp]),
    "rmsnorm_residual_fwd": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64,
                                    _f, _int, _vp]),
    "rmsnorm_residual_bwd": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                    _sz, _i64, _i64, _f, _int, _vp]),
    "rmsnorm_bwd_workspace_bytes": (_sz, [_i64, _i64, _int]),
    "rmsnorm_status_string": (ctypes.c_char_p, [_int]),
    "rmsnorm_last_cuda_error": (_int, []),
    "rmsnorm_set_path_override": (None, [_int]),
    "rmsnorm_last_path": (_int, []),
    "rmsnorm_bwd_static_scratch": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _i64,
                                          _i64, _f, _int, _vp]),
    "rmsnorm_set_static_scratch_test_limit": (None, [_sz]),
    "rmsnorm_wait_timeouts": (_int, [ctypes.POINTER(ctypes.c_uint), _int]),
    "rmsnorm_set_stream_test_fault": (None, [ctypes.c_uint, ctypes.c_uint]),
    "rmsnorm_set_gemv_cluster_test": (None, [_int]),
    "rmsnorm_bwd_ex": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _i64,
                              _i64, _f, _int, _int, _vp]),
    "rmsnorm_fwd_strided": (_int, [_vp, _i64, _vp, _i64, _vp, _vp, _i64, _vp,
                                   _i64, _vp, _i64, _i64, _f, _int, _vp]),
    "rmsnorm_bwd_strided": (_int, [_vp, _i64, _vp, _i64, _vp, _i64, _vp, _vp,
                                   _vp, _i64, _vp, _vp, _sz, _i64, _i64, _f,
                                   _int, _int, _vp]),
    "rmsnorm_bwd_bwd": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                               _sz, _i64, _i64, _f, _int, _vp]),
    "rmsnorm_gemv_fwd": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64,
                                _i64, _i64, _f, _int, _int, _vp]),
}

BWD_ACCUMULATE_DW = 1


class RmsNormError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        msg = lib().rmsnorm_status_string(status).decode()
        if status == -8:
            msg += f" (cudaError {lib().rmsnorm_last_cuda_error()})"
        super().__init__(f"{where}: status {status}: {msg}")


_lib = None


def lib():
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'` "
                "(there is no CPU fallback)")
        l = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(l, name)
            fn.restype = res
            fn.argtypes = args
        _lib = l
    return _lib


def _check(status, where):
    if status != 0:
        raise RmsNormError(status, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _rows(name, t, H, dtype=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if t.shape[-1] != H:
        raise ValueError(f"{name} last dim must be {H}")
    return t.numel() // H if H else 0


def _strided(name, t, H, dtype=None):
    """(M, ld) of a 2-D [M, H] CUDA tensor with unit column stride; ld is its
    row stride in elements (H for one row)."""
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dim() != 2 or t.shape[1] != H:
        raise ValueError(f"{name} must be 2-D [M, {H}]")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    M = t.shape[0]
    if H > 1 and t.stride(1) != 1:
        raise ValueError(f"{name} must have unit column stride")
    ld = t.stride(0) if M > 1 else H
    return M, ld


def as_rows(t, H):
    """t viewed as [M, H] rows without a copy when its strides allow it
    (any row stride, unit column stride), else a contiguous copy."""
    if t.shape[-1] == H and (H == 1 or t.stride(-1) == 1):
        try:
            return t.view(-1, H)
        except RuntimeError:
            pass
    return t.contiguous().view(-1, H)


def _dtype_code(t):
    if t.dtype not in DTYPES:
        raise ValueError(f"unsupported dtype {t.dtype}")
    return DTYPES[t.dtype]


def set_path_override(path: int):
    lib().rmsnorm_set_path_override(int(path))


def last_path() -> int:
    return lib().rmsnorm_last_path()


def wait_timeouts(reset: bool = False) -> int:
    """Streamed-kernel waits that ran out on the current device (0 when all
    is well); synchronous diagnostic."""
    c = ctypes.c_uint(0)
    _check(lib().rmsnorm_wait_timeouts(ctypes.byref(c), int(reset)),
           "rmsnorm_wait_timeouts")
    return int(c.value)


def set_stream_test_fault(extra_tx_bytes: int, wait_limit_us: int):
    """Test hook: make the streamed kernels' waits run out (see rmsnorm.h)."""
    lib().rmsnorm_set_stream_test_fault(int(extra_tx_bytes), int(wait_limit_us))


def set_gemv_cluster_test(cluster_size: int):
    """Test hook: force the persistent projection kernel's cluster size (0:
    the plan's choice; see rmsnorm.h)."""
    lib().rmsnorm_set_gemv_cluster_test(int(cluster_size))


def bwd_workspace_bytes(M: int, H: int, dtype: torch.dtype) -> int:
    return lib().rmsnorm_bwd_workspace_bytes(int(M), int(H), DTYPES[dtype])


def rmsnorm_fwd(x, w, y=None, rstd=None, eps=1e-6, want_rstd=True, stream=None):
    """y = RMSNorm(x) * w over the last dim; returns (y, rstd or None)."""
    H = w.numel()
    M = _rows("x", x, H)
    _rows("w", w.view(-1), H, x.dtype)
    if y is None:
        y = torch.empty_like(x)
    _rows("y", y, H, x.dtype)
    if rstd is None and want_rstd:
        rstd = torch.empty(x.shape[:-1], device=x.device, dtype=torch.float32)
    if rstd is not None and rstd.dtype != torch.float32:
        raise ValueError("rstd must be float32")
    _check(lib().rmsnorm_fwd(_ptr(x), _ptr(w), _ptr(y), _ptr(rstd), M, H,
                             float(eps), _dtype_code(x), _stream(stream)),
           "rmsnorm_fwd")
    return y, rstd


def rmsnorm_bwd(dy, x, w, rstd=None, dx=None, dw=None, workspace=None,
                eps=1e-6, stream=None):
    """(dx, dw) of the RMSNorm; rstd=None recomputes it from x."""
    H = w.numel()
    M = _rows("x", x, H)
    _rows("dy", dy, H, x.dtype)
    if dx is None:
        dx = torch.empty_like(x)
    if dw is None:
        dw = torch.empty(H, device=x.device, dtype=torch.float32)
    need = bwd_workspace_bytes(M, H, x.dtype)
    if workspace is None:
        workspace = torch.empty(max(need, 16), device=x.device, dtype=torch.uint8)
    _check(lib().rmsnorm_bwd(_ptr(dy), _ptr(x), _ptr(w), _ptr(rstd), _ptr(dx),
                             _ptr(dw), _ptr(workspace), workspace.numel()
                             * workspace.element_size(), M, H, float(eps),
                             _dtype_code(x), _stream(stream)), "rmsnorm_bwd")
    return dx, dw


def rmsnorm_residual_fwd(x, r, w, h=None, y=None, rstd=None, eps=1e-6,
                         want_rstd=True, stream=None):
    """h = x + r (rounded to the dtype), y = RMSNorm(h) * w; returns
    (h, y, rstd or None)."""
    H = w.numel()
    M = _rows("x", x, H)
    _rows("r", r, H, x.dtype)
    if h is None:
        h = torch.empty_like(x)
    if y is None:
        y = torch.empty_like(x)
    if rstd is None and want_rstd:
        rstd = torch.empty(x.shape[:-1], device=x.device, dtype=torch.float32)
    _check(lib().rmsnorm_residual_fwd(_ptr(x), _ptr(r), _ptr(w), _ptr(h),
                                      _ptr(y), _ptr(rstd), M, H, float(eps),
                                      _dtype_code(x), _stream(stream)),
           "rmsnorm_residual_fwd")
    return h, y, rstd


def rmsnorm_residual_bwd(dy, dh_out, h, w, rstd=None, dx=None, dw=None,
                         workspace=None, eps=1e-6, stream=None):
    """(dx, dw): dx is the gradient of both the input and the residual."""
    H = w.numel()
    M = _rows("h", h, H)
    _rows("dy", dy, H, h.dtype)
    if dh_out is not None:
        _rows("dh_out", dh_out, H, h.dtype)
    if dx is None:
        dx = torch.empty_like(h)
    if dw is None:
        dw = torch.empty(H, device=h.device, dtype=torch.float32)
    need = bwd_workspace_bytes(M, H, h.dtype)
    if workspace is None:
        workspace = torch.empty(max(need, 16), device=h.device, dtype=torch.uint8)
    _check(lib().rmsnorm_residual_bwd(
        _ptr(dy), _ptr(dh_out), _ptr(h), _ptr(w), _ptr(rstd), _ptr(dx),
        _ptr(dw), _ptr(workspace), workspace.numel() * workspace.element_size(),
        M, H, float(eps), _dtype_code(h), _stream(stream)),
        "rmsnorm_residual_bwd")
    return dx, dw


def rmsnorm_bwd_ex(dy, x, w, rstd=None, dh_out=None, dx=None, dw=None,
                   workspace=None, eps=1e-6, accumulate_dw=False, stream=None):
    """(dx, dw) of the plain (dh_out None) or residual backward; with
    accumulate_dw the call adds its dw into the given dw buffer."""
    H = w.numel()
    M = _rows("x", x, H)
    _rows("dy", dy, H, x.dtype)
    if dh_out is not None:
        _rows("dh_out", dh_out, H, x.dtype)
    if dx is None:
        dx = torch.empty_like(x)
    if dw is None:
        if accumulate_dw:
            raise ValueError("accumulate_dw needs the dw buffer to add into")
        dw = torch.empty(H, device=x.device, dtype=torch.float32)
    need = bwd_workspace_bytes(M, H, x.dtype)
    if workspace is None:
        workspace = torch.empty(max(need, 16), device=x.device, dtype=torch.uint8)
    _check(lib().rmsnorm_bwd_ex(
        _ptr(dy), _ptr(dh_out), _ptr(x), _ptr(w), _ptr(rstd), _ptr(dx), _ptr(dw),
        _ptr(workspace), workspace.numel() * workspace.element_size(), M, H,
        float(eps), _dtype_code(x), BWD_ACCUMULATE_DW if accumulate_dw else 0,
        _stream(stream)), "rmsnorm_bwd_ex")
    return dx, dw


def rmsnorm_fwd_strided(x, w, y=None, r=None, h=None, rstd=None, eps=1e-6,
                        want_rstd=True, stream=None):
    """Forward on row-strided 2-D tensors (each with its own row stride).
    Without r: returns (y, rstd); with r (residual variant): (h, y, rstd).
    Outputs the caller does not pass are allocated dense."""
    H = w.numel()
    M, ldx = _strided("x", x, H)
    _rows("w", w.view(-1), H, x.dtype)
    if y is None:
        y = torch.empty(M, H, device=x.device, dtype=x.dtype)
    _, ldy = _strided("y", y, H, x.dtype)
    ldr = ldh = H
    if r is not None:
        _, ldr = _strided("r", r, H, x.dtype)
        if h is None:
            h = torch.empty(M, H, device=x.device, dtype=x.dtype)
        _, ldh = _strided("h", h, H, x.dtype)
    elif h is not None:
        raise ValueError("h is the residual variant's output: pass r too")
    if rstd is None and want_rstd:
        rstd = torch.empty(M, device=x.device, dtype=torch.float32)
    _check(lib().rmsnorm_fwd_strided(
        _ptr(x), ldx, _ptr(r), ldr, _ptr(w), _ptr(y), ldy, _ptr(h), ldh,
        _ptr(rstd), M, H, float(eps), _dtype_code(x), _stream(stream)),
        "rmsnorm_fwd_strided")
    return (y, rstd) if r is None else (h, y, rstd)


def rmsnorm_bwd_strided(dy, x, w, rstd=None, dh_out=None, dx=None, dw=None,
                        workspace=None, eps=1e-6, accumulate_dw=False,
                        stream=None):
    """(dx, dw) of the plain (dh_out None) or residual backward on row-strided
    2-D tensors; dx is allocated dense unless given."""
    H = w.numel()
    M, ldx = _strided("x", x, H)
    _, lddy = _strided("dy", dy, H, x.dtype)
    lddh = H
    if dh_out is not None:
        _, lddh = _strided("dh_out", dh_out, H, x.dtype)
    if dx is None:
        dx = torch.empty(M, H, device=x.device, dtype=x.dtype)
    _, lddx = _strided("dx", dx, H, x.dtype)
    if dw is None:
        if accumulate_dw:
            raise ValueError("accumulate_dw needs the dw buffer to add into")
        dw = torch.empty(H, device=x.device, dtype=torch.float32)
    need = bwd_workspace_bytes(M, H, x.dtype)
    if workspace is None:
        workspace = torch.empty(max(need, 16), device=x.device, dtype=torch.uint8)
    _check(lib().rmsnorm_bwd_strided(
        _ptr(dy), lddy, _ptr(dh_out), lddh, _ptr(x), ldx, _ptr(w), _ptr(rstd),
        _ptr(dx), lddx, _ptr(dw), _ptr(workspace),
        workspace.numel() * workspace.element_size(), M, H, float(eps),
        _dtype_code(x), BWD_ACCUMULATE_DW if accumulate_dw else 0,
        _stream(stream)), "rmsnorm_bwd_strided")
    return dx, dw


def rmsnorm_bwd_bwd(dy, x, w, rstd=None, gdx=None, gdw=None, ddy=None, dx2=None,
                    dw2=None, workspace=None, eps=1e-6, stream=None):
    """(ddy, dx2, dw2): gradients of sum(gdx * dx) + sum(gdw * dw) with
    respect to the backward's dy, x and w (see rmsnorm.h). gdx in x's dtype
    or None, gdw float32 or None; dw2 is float32."""
    H = w.numel()
    M = _rows("x", x, H)
    _rows("dy", dy, H, x.dtype)
    if gdx is not None:
        _rows("gdx", gdx, H, x.dtype)
    if gdw is not None and (gdw.dtype != torch.float32 or not gdw.is_contiguous()):
        raise ValueError("gdw must be a contiguous float32 tensor")
    if ddy is None:
        ddy = torch.empty_like(x)
    if dx2 is None:
        dx2 = torch.empty_like(x)
    if dw2 is None:
        dw2 = torch.empty(H, device=x.device, dtype=torch.float32)
    need = bwd_workspace_bytes(M, H, x.dtype)
    if workspace is None:
        workspace = torch.empty(max(need, 16), device=x.device, dtype=torch.uint8)
    _check(lib().rmsnorm_bwd_bwd(
        _ptr(dy), _ptr(x), _ptr(w), _ptr(rstd), _ptr(gdx), _ptr(gdw), _ptr(ddy),
        _ptr(dx2), _ptr(dw2), _ptr(workspace),
        workspace.numel() * workspace.element_size(), M, H, float(eps),
        _dtype_code(x), _stream(stream)), "rmsnorm_bwd_bwd")
    return ddy, dx2, dw2


GEMV_STATIC_WEIGHTS = 1


def rmsnorm_gemv_fwd(x, w, A, r=None, out=None, h=None, want_h=True, y=None,
                     rstd=None, eps=1e-6, static_weights=False, stream=None):
    """out = round(RMSNorm(x [+ r]) * w) @ A^T for decode-sized x [M, H]
    (M <= 64) and a row-major weight A [N, H]. Returns (out, h or None,
    rstd or None); y (the norm's output) is written only into a given
    buffer. With r, h (the residual sum) is allocated unless want_h is
    False. static_weights: nothing in flight on the stream writes w or A
    (see RMSNORM_GEMV_STATIC_WEIGHTS)."""
    H = w.numel()
    M = _rows("x", x, H)
    _rows("w", w.view(-1), H, x.dtype)
    if A.dim() != 2:
        raise ValueError("A must be 2-D [N, H]")
    N = _rows("A", A, H, x.dtype)
    if r is not None:
        _rows("r", r, H, x.dtype)
        if h is None and want_h:
            h = torch.empty_like(x)
    elif h is not None:
        raise ValueError("h is the residual variant's output: pass r too")
    if out is None:
        out = torch.empty(x.shape[:-1] + (N,), device=x.device, dtype=x.dtype)
    _rows("out", out, N, x.dtype)
    if y is not None:
        _rows("y", y, H, x.dtype)
    _check(lib().rmsnorm_gemv_fwd(
        _ptr(x), _ptr(r), _ptr(w), _ptr(A), _ptr(out), _ptr(h), _ptr(y),
        _ptr(rstd), M, H, N, float(eps), _dtype_code(x),
        GEMV_STATIC_WEIGHTS if static_weights else 0, _stream(stream)),
        "rmsnorm_gemv_fwd")
    return out, h, rstd


STATIC_SCRATCH_BYTES = 16 << 20     # RMSNORM_STATIC_SCRATCH_BYTES
ERR_SCRATCH_LIMIT = -10             # RMSNORM_ERR_SCRATCH_LIMIT


def rmsnorm_bwd_static_scratch(dy, x, w, rstd=None, dx=None, dw=None, eps=1e-6,
                               stream=None):
    """(dx, dw) like rmsnorm_bwd, but the library keeps the dw partial rows
    in its own fixed device array instead of a workspace, so the call itself
    allocates nothing (outputs the caller does not pass are still allocated
    here by torch). For callers that cannot allocate device memory; calls
    that overlap on the GPU share that array and race (see rmsnorm.h)."""
    H = w.numel()
    M = _rows("x", x, H)
    _rows("dy", dy, H, x.dtype)
    if dx is None:
        dx = torch.empty_like(x)
    if dw is None:
        dw = torch.empty(H, device=x.device, dtype=torch.float32)
    _check(lib().rmsnorm_bwd_static_scratch(
        _ptr(dy), _ptr(x), _ptr(w), _ptr(rstd), _ptr(dx), _ptr(dw), M, H,
        float(eps), _dtype_code(x), _stream(stream)),
        "rmsnorm_bwd_static_scratch")
    return dx, dw


def set_static_scratch_test_limit(nbytes):
    """Test hook: rmsnorm_bwd_static_scratch treats its array as holding only
    nbytes (0: the full RMSNORM_STATIC_SCRATCH_BYTES)."""
    lib().rmsnorm_set_static_scratch_test_limit(int(nbytes))
