"""The autograd wrappers (RMSNormFunction / RMSNorm and the residual variant)
against the fp64 oracle, and their gotcha-table behaviour ([P1]
"训推加速 Qwen3 实战：从“调包”到手写 Triton Kernel（含 backward）" §5.5-5.6):
non-contiguous dy, one gradient per input, eps as a float, the double
backward (against the oracle) and a third derivative raising."""
import pytest
import torch

import oracle
from rmsnorm_fwd_bwd_02_gb300 import autograd as A
from rmsnorm_fwd_bwd_02_gb300 import workloads as W
from tests.tolerances import check_bits, check_dw, check_rows, check_rstd  # noqa: F401

DEV = torch.device("cuda:0")


def test_cpu_tensors_raise():
    """No CPU fallback: the wrappers refuse CPU tensors."""
    x = torch.randn(4, 16, dtype=torch.bfloat16)
    w = torch.ones(16, dtype=torch.bfloat16)
    with pytest.raises((ValueError, RuntimeError)):
        A.rms_norm(x, w)


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


@pytest.mark.gpu
@pytest.mark.parametrize("shape", [(4, 257, 4096), (1031, 128), (3, 5, 896)])
def test_module_grads_match_oracle(orc, shape):
    H = shape[-1]
    g = torch.Generator().manual_seed(H)
    x = torch.randn(*shape, generator=g).to(torch.bfloat16)
    dy = (torch.randn(*shape, generator=g) * 1e-2).to(torch.bfloat16)
    w = (1 + 0.1 * torch.randn(H, generator=g)).to(torch.bfloat16)
    mod = A.RMSNorm(H, eps=1e-6, device=DEV)
    with torch.no_grad():
        mod.weight.copy_(w.to(DEV))
    xd = x.to(DEV).requires_grad_()
    y = mod(xd)
    assert y.shape == x.shape and y.dtype == torch.bfloat16
    y.backward(dy.to(DEV))
    torch.cuda.synchronize()
    x2, dy2 = x.reshape(-1, H).contiguous(), dy.reshape(-1, H).contiguous()
    oy, _ = orc.fwd(x2, w, 1e-6)
    odx, odw, tdx, tdw = orc.bwd(dy2, x2, w, 1e-6, want_terms=True)
    check_rows("module y", y.detach().reshape(-1, H), oy, torch.bfloat16)
    check_rows("module dx", xd.grad.reshape(-1, H), odx, torch.bfloat16, tdx)
    # dw comes back in the weight's dtype (bf16): its rounding on top of the
    # fp32 sum's tolerance
    got = mod.weight.grad.double().cpu()
    err = (got - odw).abs()
    assert bool((err <= 1e-3 * tdw + 2.0 ** -8 * odw.abs() + 1e-30).all())


@pytest.mark.gpu
def test_noncontiguous_dy_and_input():
    H = 4096
    base = torch.randn(8, H, 6, device=DEV, dtype=torch.bfloat16)
    x = base.transpose(1, 2)                     # (8, 6, H), not contiguous
    assert not x.is_contiguous()
    w = torch.ones(H, device=DEV, dtype=torch.bfloat16, requires_grad=True)
    xr = x.detach().requires_grad_()
    y = A.rms_norm(xr, w)
    dy = torch.randn(8, H, 6, device=DEV, dtype=torch.bfloat16).transpose(1, 2)
    y.backward(dy)
    xc = x.detach().contiguous().requires_grad_()
    wc = w.detach().clone().requires_grad_()
    yc = A.rms_norm(xc, wc)
    yc.backward(dy.contiguous())
    torch.cuda.synchronize()
    assert torch.equal(y, yc)
    assert torch.equal(xr.grad, xc.grad)
    assert torch.equal(w.grad, wc.grad)


@pytest.mark.gpu
def test_residual_module_grads(orc):
    M, H = 517, 5120
    wl = W.WORKLOADS["residual-14b"].with_rows(M)
    inp = W.make_inputs(wl)
    mod = A.ResidualRMSNorm(H, device=DEV)
    with torch.no_grad():
        mod.weight.copy_(inp["w"].to(DEV))
    x = inp["x"].to(DEV).requires_grad_()
    r = inp["r"].to(DEV).requires_grad_()
    y, h = mod(x, r)
    torch.autograd.backward([y, h], [inp["dy"].to(DEV), inp["dh"].to(DEV)])
    torch.cuda.synchronize()
    oh, oy, _ = orc.residual_fwd(inp["x"], inp["r"], inp["w"], 1e-6)
    odx, odw, tdx, tdw = orc.residual_bwd(inp["dy"], inp["dh"], oh, inp["w"], 1e-6,
                                          want_terms=True)
    assert torch.equal(h.detach().cpu().view(torch.int16), oh.view(torch.int16))
    check_rows("residual y", y.detach(), oy, torch.bfloat16)
    check_rows("residual dx", x.grad, odx, torch.bfloat16, tdx)
    check_rows("residual dr", r.grad, odx, torch.bfloat16, tdx)
    got = mod.weight.grad.double().cpu()
    assert bool(((got - odw).abs() <= 1e-3 * tdw + 2.0 ** -8 * odw.abs()).all())
    # only y used downstream: dh is None
    x.grad = r.grad = mod.weight.grad = None
    y, h = mod(x, r)
    y.backward(inp["dy"].to(DEV))
    torch.cuda.synchronize()
    odx2, _ = orc.residual_bwd(inp["dy"], None, oh, inp["w"], 1e-6)
    check_rows("residual dx, dh None", x.grad, odx2, torch.bfloat16)


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_double_backward_matches_oracle(orc, dtype):
    """grad of (sum(ga * dL/dx) + sum(gb * dL/dw)) with respect to x, w and dy,
    through autograd with create_graph, against the oracle's double
    backward; a third derivative raises."""
    M, H = 67, 896
    g = torch.Generator().manual_seed(21)
    x = (torch.randn(M, H, generator=g) * 2).to(dtype)
    w = (1 + 0.1 * torch.randn(H, generator=g)).to(dtype)
    dy = torch.randn(M, H, generator=g).to(dtype)
    ga = torch.randn(M, H, generator=g).to(dtype)
    gb = torch.randn(H, generator=g).to(dtype)
    xd = x.to(DEV).requires_grad_()
    wd = w.to(DEV).requires_grad_()
    dyd = dy.to(DEV).requires_grad_()
    y = A.rms_norm(xd, wd)
    gx_, gw_ = torch.autograd.grad(y, (xd, wd), dyd, create_graph=True)
    l2 = (gx_.float() * ga.to(DEV).float()).sum() + (gw_.float() * gb.to(DEV).float()).sum()
    d_x, d_w, d_dy = torch.autograd.grad(l2, (xd, wd, dyd), create_graph=True)
    torch.cuda.synchronize()
    ddy, dx2, dw2, tddy, tdx2, tdw2 = orc.bwd_bwd(dy, x, w, ga, gb.float(), 1e-6,
                                                  want_terms=True)
    check_rows("autograd d(dy)", d_dy, ddy, dtype, tddy)
    check_rows("autograd d(x)", d_x, dx2, dtype, tdx2)
    got = d_w.double().cpu()
    ulp = 2.0 ** -8 if dtype == torch.bfloat16 else 2.0 ** -23
    assert bool(((got - dw2).abs() <= 1e-3 * tdw2 + ulp * dw2.abs() + 1e-30).all())
    with pytest.raises(RuntimeError):
        d_x.float().sum().backward()


@pytest.mark.gpu
def test_residual_double_backward(orc):
    """The residual module: the second derivative through h and dh_out."""
    M, H = 33, 896
    g = torch.Generator().manual_seed(22)
    x = torch.randn(M, H, generator=g).to(torch.bfloat16)
    r = torch.randn(M, H, generator=g).to(torch.bfloat16)
    w = (1 + 0.1 * torch.randn(H, generator=g)).to(torch.bfloat16)
    dy = torch.randn(M, H, generator=g).to(torch.bfloat16)
    dh = torch.randn(M, H, generator=g).to(torch.bfloat16)
    ga = torch.randn(M, H, generator=g).to(torch.bfloat16)
    xd, rd, wd = (t.to(DEV).requires_grad_() for t in (x, r, w))
    dyd, dhd = dy.to(DEV).requires_grad_(), dh.to(DEV).requires_grad_()
    y, h = A.residual_rms_norm(xd, rd, wd)
    gx_, = torch.autograd.grad((y, h), (xd,), (dyd, dhd), create_graph=True)
    l2 = (gx_.float() * ga.to(DEV).float()).sum()
    d_dy, d_dh, d_x, d_r = torch.autograd.grad(l2, (dyd, dhd, xd, rd))
    torch.cuda.synchronize()
    oh, _, _ = orc.residual_fwd(x, r, w, 1e-6)
    ddy, dh2, _, tddy, tdh2, _ = orc.bwd_bwd(dy, oh, w, ga, None, 1e-6, want_terms=True)
    check_rows("residual d(dy)", d_dy, ddy, torch.bfloat16, tddy)
    check_bits("residual d(dh_out) = ga", d_dh, ga)
    check_rows("residual d(x)", d_x, dh2, torch.bfloat16, tdh2)
    check_rows("residual d(r)", d_r, dh2, torch.bfloat16, tdh2)


@pytest.mark.gpu
def test_training_step_in_a_cuda_graph():
    """Forward + backward of the module captured once and replayed: same
    bits as eager (static buffers, no allocation in the replay)."""
    H, M = 4096, 512
    mod = A.RMSNorm(H, device=DEV)
    x = torch.randn(M, H, device=DEV, dtype=torch.bfloat16, requires_grad=True)
    dy = torch.randn(M, H, device=DEV, dtype=torch.bfloat16)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(3):                         # warm up
            x.grad = mod.weight.grad = None
            mod(x).backward(dy)
    torch.cuda.current_stream().wait_stream(s)
    ref_dx, ref_dw = x.grad.clone(), mod.weight.grad.clone()
    x.grad = mod.weight.grad = None
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        y = mod(x)
        y.backward(dy)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(x.grad, ref_dx)
    assert torch.equal(mod.weight.grad, ref_dw)


@pytest.mark.gpu
def test_fp16_module_grads_match_oracle(orc):
    M, H = 515, 4096
    g = torch.Generator().manual_seed(5)
    x = torch.randn(M, H, generator=g).to(torch.float16)
    dy = (torch.randn(M, H, generator=g) * 1e-2).to(torch.float16)
    w = (1 + 0.1 * torch.randn(H, generator=g)).to(torch.float16)
    mod = A.RMSNorm(H, device=DEV, dtype=torch.float16)
    with torch.no_grad():
        mod.weight.copy_(w.to(DEV))
    xd = x.to(DEV).requires_grad_()
    y = mod(xd)
    assert y.dtype == torch.float16
    y.backward(dy.to(DEV))
    torch.cuda.synchronize()
    oy, _ = orc.fwd(x, w, 1e-6)
    odx, odw, tdx, tdw = orc.bwd(dy, x, w, 1e-6, want_terms=True)
    check_rows("f16 module y", y.detach(), oy, torch.float16)
    check_rows("f16 module dx", xd.grad, odx, torch.float16, tdx)
    got = mod.weight.grad.double().cpu()
    assert bool(((got - odw).abs() <= 1e-3 * tdw + 2.0 ** -10 * odw.abs()
                 + 2.0 ** -24).all())


@pytest.mark.gpu
def test_column_window_input_is_not_copied():
    """x = the first H columns of a (B, T, ld) buffer: the rows go to the
    kernels in place (a view with row stride ld), with the same bits as a
    contiguous copy."""
    from rmsnorm_fwd_bwd_02_gb300 import rmsnorm as rn
    B, T, H, ld = 3, 70, 4096, 4096 + 512
    buf = torch.randn(B, T, ld, device=DEV, dtype=torch.bfloat16)
    x = buf[:, :, :H]
    rows = rn.as_rows(x, H)
    assert rows.data_ptr() == x.data_ptr() and rows.stride() == (ld, 1)
    w = (1 + 0.1 * torch.randn(H, device=DEV)).to(torch.bfloat16).requires_grad_()
    xr = x.detach().requires_grad_()
    y = A.rms_norm(xr, w)
    dy = torch.randn(B, T, ld, device=DEV, dtype=torch.bfloat16)[:, :, :H]
    y.backward(dy)
    wc = w.detach().clone().requires_grad_()
    xc = x.detach().contiguous().requires_grad_()
    yc = A.rms_norm(xc, wc)
    yc.backward(dy.contiguous())
    torch.cuda.synchronize()
    assert torch.equal(y, yc)
    assert torch.equal(xr.grad, xc.grad)
    assert torch.equal(w.grad, wc.grad)
