"""Tolerances for comparing the CUDA path with the fp64 oracle.

Contract bounds (fixed for this method's workloads):
  * bf16 outputs y, dx:   |gpu - o| <= 1e-2 + 1.6e-2 |o|
  * fp32 rstd:            |gpu - o| <= 1e-3 o
  * fp32 dw:              |gpu - o| <= 1e-3 T_dw,  T_dw = sum_i |dy x r|
  * fp32 y, dx (the fp32 tiny case): |gpu - o| <= 1e-3 T, with T the sum of
    absolute values of the terms that make up the result (T_y = |o|,
    T_dx from the oracle)
  * h (residual sum): bit-exact.

Strict bounds, checked as well, derived from the arithmetic: the kernels
compute in fp32 (unit roundoff 2^-24, rsqrtf within 2 ulp, sums over at most
16384 terms) and round once to bf16 (half an ulp = 2^-9 relative). So a bf16
result is within 2^-8 |o| of the oracle plus the fp32 error of its terms,
bounded generously by 1e-3 T (y has a single term, T = |o|). These catch
errors the contract's 1e-2 absolute floor would hide when the values are
small (dy ~ N(0, 1e-2) makes dx ~ 1e-2).

fp16 outputs (no contract figure is fixed for fp16; derived the same way):
one rounding to binary16 costs at most half an ulp, 2^-11 relative for
normal results and 2^-25 absolute below 2^-14 (subnormal spacing 2^-24), on
top of the fp32 error of the terms. Contract: 2^-10 |o| + 1e-3 T + 2^-24;
strict: 2^-10 |o| + 1e-4 T + 2^-25. Results beyond 65504 must be infinite
with the oracle's sign (checked separately where a test provokes them).
"""
import torch

F64 = torch.float64


def _report(name, err, bound, got, want):
    bad = err > bound
    if bool(bad.any()):
        idx = int(torch.argmax((err - bound).flatten()))
        raise AssertionError(
            f"{name}: {int(bad.sum())} of {err.numel()} outside tolerance; worst "
            f"flat index {idx}: got {float(got.flatten()[idx])!r}, want "
            f"{float(want.flatten()[idx])!r}, |err| {float(err.flatten()[idx]):.3e} "
            f"> {float(bound.flatten()[idx]):.3e}")


def _as64(t):
    return t.detach().to("cpu").to(F64)


def check_rows(name, got, want, dtype, terms=None):
    """y or dx against the oracle (float64 ``want``); ``terms`` = error scale
    T (None means a single-product result, T = |want|)."""
    g = _as64(got).reshape(want.shape)
    err = (g - want).abs()
    T = want.abs() if terms is None else terms.reshape(want.shape)
    if dtype == torch.bfloat16:
        _report(name + " (contract)", err, 1e-2 + 1.6e-2 * want.abs(), g, want)
        _report(name + " (strict)", err, 2.0 ** -8 * want.abs() + 1e-3 * T + 1e-30,
                g, want)
    elif dtype == torch.float16:
        _report(name + " (contract)", err,
                2.0 ** -10 * want.abs() + 1e-3 * T + 2.0 ** -24, g, want)
        _report(name + " (strict)", err,
                2.0 ** -10 * want.abs() + 1e-4 * T + 2.0 ** -25, g, want)
    else:
        _report(name + " (contract)", err, 1e-3 * T + 1e-30, g, want)
        _report(name + " (strict)", err, 2e-5 * T + 1e-30, g, want)


def check_rstd(name, got, want):
    g = _as64(got).reshape(want.shape)
    err = (g - want).abs()
    _report(name + " (contract)", err, 1e-3 * want, g, want)
    _report(name + " (strict)", err, 2e-5 * want, g, want)


def check_dw(name, got, want, tdw):
    g = _as64(got).reshape(want.shape)
    err = (g - want).abs()
    _report(name + " (contract)", err, 1e-3 * tdw + 1e-30, g, want)
    _report(name + " (strict)", err, 1e-4 * tdw + 1e-30, g, want)


def check_bits(name, got, want):
    a = got.detach().cpu().contiguous()
    b = want.detach().cpu().contiguous()
    if a.dtype in (torch.bfloat16, torch.float16):
        a, b = a.view(torch.int16), b.view(torch.int16)
    elif a.dtype == torch.float32:
        a, b = a.view(torch.int32), b.view(torch.int32)
    ne = a != b.reshape(a.shape)
    if bool(ne.any()):
        i = int(torch.nonzero(ne.flatten())[0])
        raise AssertionError(f"{name}: {int(ne.sum())} elements differ; first at "
                             f"flat index {i}")
