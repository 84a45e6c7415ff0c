"""PyTorch autograd functions and modules over the C ABI.

[P1] "训推加速 Qwen3 实战：从“调包”到手写 Triton Kernel（含 backward）" §5.5 wraps
its kernels in a torch.autograd.Function (saving x and the weight, returning
(dx, dw, None)) and exposes an nn.Module; §5.6 lists the backward gotchas:
make dy contiguous, save tensors with save_for_backward, return one gradient
per forward input (None for eps), take eps as a float, and raise on double
backward unless it is implemented. These wrappers follow that shape over the
CUDA kernels of librmsnorm.so, and implement double backward: the backward
is itself an autograd function of (dy, x, w) whose backward runs the double
backward kernel (rmsnorm_bwd_bwd), so torch.autograd.grad(...,
create_graph=True) followed by a second backward works; a third derivative
raises. The forward also saves rstd, so the backward does not recompute it. Inputs and incoming gradients whose rows are evenly
strided (a column window of a wider buffer, a slice along the leading dims)
go to the kernels as they are, through the strided entry points; only
layouts that no row stride describes are copied first. Every arithmetic step
runs in the CUDA kernels; there is no CPU fallback (CPU tensors raise).
"""
import torch
from torch.autograd.function import once_differentiable

from . import rmsnorm as _rn


def _rows2d(t, H):
    """t as [M, H] rows: a view with its own row stride when t's layout has
    one, else a contiguous copy."""
    if not t.is_cuda:
        raise ValueError("RMSNorm: tensors must be on a CUDA device")
    return _rn.as_rows(t, H)


class RMSNormBackward(torch.autograd.Function):
    """(dx, dw) of RMSNormFunction as a differentiable function of (dy, x,
    w); its own backward is the double backward."""

    @staticmethod
    def forward(ctx, dy2, x2, weight, rstd, eps: float):
        dx, dw = _rn.rmsnorm_bwd_strided(dy2, x2, weight, rstd, eps=eps)
        ctx.save_for_backward(dy2, x2, weight, rstd)
        ctx.eps = eps
        return dx, dw

    @staticmethod
    @once_differentiable
    def backward(ctx, gdx, gdw):
        dy2, x2, weight, rstd = ctx.saved_tensors
        gx = None if gdx is None else gdx.contiguous()
        gw = None if gdw is None else gdw.float().contiguous()
        ddy, dx2, dw2 = _rn.rmsnorm_bwd_bwd(dy2.contiguous(), x2.contiguous(), weight,
                                            rstd, gx, gw, eps=ctx.eps)
        return ddy, dx2, dw2.to(weight.dtype), None, None


class RMSNormFunction(torch.autograd.Function):
    """y = w * x / sqrt(mean(x^2) + eps) over the last dimension."""

    @staticmethod
    def forward(ctx, x, weight, eps: float = 1e-6):
        H = weight.numel()
        y, rstd = _rn.rmsnorm_fwd_strided(_rows2d(x, H), weight, eps=float(eps))
        # the input itself is saved (a view made here would carry no autograd
        # history, and the double backward must reach x through it)
        ctx.save_for_backward(x, weight, rstd)
        ctx.eps = float(eps)
        ctx.shape = x.shape
        return y.view(x.shape)

    @staticmethod
    def backward(ctx, dy):
        x, weight, rstd = ctx.saved_tensors
        H = weight.numel()
        dx, dw = RMSNormBackward.apply(_rows2d(dy, H), _rows2d(x, H), weight, rstd, ctx.eps)
        dx = dx.view(ctx.shape) if ctx.needs_input_grad[0] else None
        dw = dw.to(weight.dtype) if ctx.needs_input_grad[1] else None
        return dx, dw, None


class ResidualRMSNormBackward(torch.autograd.Function):
    """(dx, dw) of ResidualRMSNormFunction as a differentiable function of
    (dy, dh, h, w); its own backward is the double backward at h, and the
    gradient on dh is the incoming gradient on dx itself."""

    @staticmethod
    def forward(ctx, dy2, dh2, h, weight, rstd, eps: float):
        dx, dw = _rn.rmsnorm_bwd_strided(dy2, h, weight, rstd, dh_out=dh2, eps=eps)
        ctx.save_for_backward(dy2, h, weight, rstd)
        ctx.has_dh = dh2 is not None
        ctx.eps = eps
        return dx, dw

    @staticmethod
    @once_differentiable
    def backward(ctx, gdx, gdw):
        dy2, h, weight, rstd = ctx.saved_tensors
        gx = None if gdx is None else gdx.contiguous()
        gw = None if gdw is None else gdw.float().contiguous()
        ddy, dh2, dw2 = _rn.rmsnorm_bwd_bwd(dy2.contiguous(), h.contiguous(), weight, rstd,
                                            gx, gw, eps=ctx.eps)
        g_dh = gdx if ctx.has_dh else None
        return ddy, g_dh, dh2, dw2.to(weight.dtype), None, None


class ResidualRMSNormFunction(torch.autograd.Function):
    """h = x + r (rounded to the dtype), y = RMSNorm(h); returns (y, h). The
    gradient of x and of r is the same tensor: the norm's backward at h
    plus the gradient arriving on h."""

    @staticmethod
    def forward(ctx, x, residual, weight, eps: float = 1e-6):
        H = weight.numel()
        x2, r2 = _rows2d(x, H), _rows2d(residual, H)
        h, y, rstd = _rn.rmsnorm_fwd_strided(x2, weight, r=r2, eps=float(eps))
        hv = h.view(x.shape)
        # the returned h itself is saved, so that a double backward reaches it
        ctx.save_for_backward(hv, weight, rstd)
        ctx.eps = float(eps)
        ctx.shape = x.shape
        return y.view(x.shape), hv

    @staticmethod
    def backward(ctx, dy, dh):
        hv, weight, rstd = ctx.saved_tensors
        H = weight.numel()
        h = _rows2d(hv, H)
        if dy is None:
            dy = torch.zeros_like(h)
        dh2 = None if dh is None else _rows2d(dh, H)
        dx, dw = ResidualRMSNormBackward.apply(_rows2d(dy, H), dh2, h, weight, rstd,
                                               ctx.eps)
        dx = dx.view(ctx.shape)
        dw = dw.to(weight.dtype) if ctx.needs_input_grad[2] else None
        gx = dx if ctx.needs_input_grad[0] else None
        gr = dx if ctx.needs_input_grad[1] else None
        return gx, gr, dw, None


def rms_norm(x, weight, eps: float = 1e-6):
    return RMSNormFunction.apply(x, weight, eps)


def residual_rms_norm(x, residual, weight, eps: float = 1e-6):
    return ResidualRMSNormFunction.apply(x, residual, weight, eps)


class RMSNorm(torch.nn.Module):
    """Qwen3-style RMSNorm over the last dimension (weight initialised to 1)."""

    def __init__(self, hidden_size: int, eps: float = 1e-6, device=None,
                 dtype=torch.bfloat16):
        super().__init__()
        self.weight = torch.nn.Parameter(
            torch.ones(hidden_size, device=device, dtype=dtype))
        self.eps = float(eps)

    def forward(self, x):
        return RMSNormFunction.apply(x, self.weight, self.eps)

    def extra_repr(self):
        return f"{self.weight.numel()}, eps={self.eps}"


class ResidualRMSNorm(torch.nn.Module):
    """The residual add fused with the norm: forward(x, residual) returns
    (RMSNorm(x + residual), x + residual)."""

    def __init__(self, hidden_size: int, eps: float = 1e-6, device=None,
                 dtype=torch.bfloat16):
        super().__init__()
        self.weight = torch.nn.Parameter(
            torch.ones(hidden_size, device=device, dtype=dtype))
        self.eps = float(eps)

    def forward(self, x, residual):
        return ResidualRMSNormFunction.apply(x, residual, self.weight, self.eps)

    def extra_repr(self):
        return f"{self.weight.numel()}, eps={self.eps}"
