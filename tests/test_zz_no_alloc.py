"""GPU tier: the backward entry point that allocates nothing.

rmsnorm_bwd_static_scratch serves callers that cannot call cudaMalloc (a
plug-in whose host runtime owns all device memory, a latency-critical loop
that cannot afford an allocation's synchronisation). It keeps the dw
partial rows in a fixed device array inside the library instead of a
caller workspace.

The test calls it through the C ABI on several problems back to back (bf16
at 4096 and 5120 features, fp16, the 128-wide QK-norm rows), twice on each
in a row, so every call runs over the previous call's leftovers in the shared
array. Each result is compared with the fp64 oracle within the parity
tolerances, and with the workspace entry point rmsnorm_bwd bit for bit (same
kernel, same grid, same fixed reduction order, so one stale partial row
would show). A problem too large for the array must be refused before
anything runs, leaving the outputs untouched. The file is collected last and
needs no state from the other tests.
"""
import pytest
import torch

import oracle
from rmsnorm_fwd_bwd_02_gb300 import rmsnorm as rn
from rmsnorm_fwd_bwd_02_gb300 import workloads as W
from tests.tolerances import check_bits, check_dw, check_rows

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.fail("the gpu tier needs a CUDA device")
    rn.lib()
    rn.set_path_override(rn.PATH_AUTO)
    yield
    rn.set_path_override(rn.PATH_AUTO)


def _problem(name, M, H=None):
    wl = W.WORKLOADS[name].with_rows(M)
    if H is not None:
        wl = wl.with_features(H)
    inp = W.make_inputs(wl)
    g = {k: v.to(DEV) for k, v in inp.items()}
    _, rstd = rn.rmsnorm_fwd(g["x"], g["w"], eps=wl.eps)
    return wl, inp, g, rstd


@pytest.mark.parametrize("rstd_given", [True, False])
def test_static_scratch_against_oracle(rstd_given):
    orc = oracle.get()
    problems = (("qwen3-8b-train", 1037, None), ("qwen3-qknorm", 4099, None),
                ("qwen3-8b-train-fp16", 517, None), ("qwen3-8b-train", 301, 5120))
    for name, M, H in problems:
        wl, inp, g, rstd = _problem(name, M, H)
        r = rstd if rstd_given else None
        assert rn.bwd_workspace_bytes(M, wl.H, wl.dtype) <= rn.STATIC_SCRATCH_BYTES
        odx, odw, tdx, tdw = orc.bwd(inp["dy"], inp["x"], inp["w"], wl.eps, want_terms=True)
        dx_r, dw_r = rn.rmsnorm_bwd(g["dy"], g["x"], g["w"], r, eps=wl.eps)
        path_r = rn.last_path()
        for call in (1, 2):      # the second call finds the first one's rows in the array
            dx_s, dw_s = rn.rmsnorm_bwd_static_scratch(g["dy"], g["x"], g["w"], r,
                                                       eps=wl.eps)
            assert rn.last_path() == path_r
            torch.cuda.synchronize()
            tag = f"{name} H={wl.H} M={M} call {call}"
            check_rows(f"{tag} dx (static scratch) vs oracle", dx_s, odx, wl.dtype, tdx)
            check_dw(f"{tag} dw (static scratch) vs oracle", dw_s, odw, tdw)
            check_bits(f"{tag} dx static vs workspace", dx_s, dx_r)
            check_bits(f"{tag} dw static vs workspace", dw_s, dw_r)


def test_static_scratch_refuses_oversized_problem():
    """A problem that needs more scratch than the array holds is refused with
    RMSNORM_ERR_SCRATCH_LIMIT before anything runs, and writes nothing. On a
    152-SM GB300 no problem within RMSNORM_MAX_H needs the full array, so the
    test hook lowers the usable size below this problem's need."""
    wl, inp, g, rstd = _problem("qwen3-8b-train", 1037)
    need = rn.bwd_workspace_bytes(wl.M, wl.H, wl.dtype)
    assert 0 < need <= rn.STATIC_SCRATCH_BYTES
    dx = torch.full((wl.M, wl.H), 7.0, device=DEV, dtype=wl.dtype)
    dw = torch.full((wl.H,), 7.0, device=DEV)
    torch.cuda.synchronize()
    rn.set_static_scratch_test_limit(need - 16)
    try:
        with pytest.raises(rn.RmsNormError) as ei:
            rn.rmsnorm_bwd_static_scratch(g["dy"], g["x"], g["w"], rstd, dx=dx, dw=dw,
                                          eps=wl.eps)
        assert ei.value.status == rn.ERR_SCRATCH_LIMIT
        torch.cuda.synchronize()
        assert bool((dx == 7.0).all()) and bool((dw == 7.0).all())
        # exactly the need fits
        rn.set_static_scratch_test_limit(need)
        dx_s, dw_s = rn.rmsnorm_bwd_static_scratch(g["dy"], g["x"], g["w"], rstd, dx=dx,
                                                   dw=dw, eps=wl.eps)
    finally:
        rn.set_static_scratch_test_limit(0)
    dx_r, dw_r = rn.rmsnorm_bwd(g["dy"], g["x"], g["w"], rstd, eps=wl.eps)
    torch.cuda.synchronize()
    check_bits("at the limit dx", dx_s, dx_r)
    check_bits("at the limit dw", dw_s, dw_r)
