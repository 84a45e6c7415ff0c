"""GPU tier: the backward entry point that allocates nothing.

rmsnorm_bwd_static_scratch serves callers that cannot call cudaMalloc (a
plug-in whose host runtime owns all device memory, a latency-critical loop
that cannot afford an allocation's synchronisation). It keeps the dw
partial rows in a fixed device array inside the library instead of a
caller workspace. This test calls it through the C ABI twice in a row, on
two different problems (so the second call runs over the first one's
leftovers in the shared array), and checks each result against the regular
rmsnorm_bwd entry point on the same inputs within the parity tolerances.
It sits in its own file, collected last, and needs no state from the other
tests.
"""
import pytest
import torch

import oracle
from rmsnorm_fwd_bwd_02_gb300 import rmsnorm as rn
from rmsnorm_fwd_bwd_02_gb300 import workloads as W
from tests.tolerances import check_dw, check_rows

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


def _problem(name, M):
    wl = W.WORKLOADS[name].with_rows(M)
    inp = W.make_inputs(wl)
    g = {k: v.to(DEV) for k, v in inp.items()}
    _, rstd = rn.rmsnorm_fwd(g["x"], g["w"], eps=wl.eps)
    return wl, inp, g, rstd


def test_static_scratch_matches_workspace_entry_point():
    if not torch.cuda.is_available():
        pytest.fail("the gpu tier needs a CUDA device")
    orc = oracle.get()
    rn.set_path_override(rn.PATH_AUTO)
    # two different problems, back to back through the same scratch array
    for name, M in (("qwen3-8b-train", 1037), ("qwen3-qknorm", 4099)):
        wl, inp, g, rstd = _problem(name, M)
        assert rn.bwd_workspace_bytes(M, wl.H, wl.dtype) <= rn.STATIC_SCRATCH_BYTES
        dx_s, dw_s = rn.rmsnorm_bwd_static_scratch(g["dy"], g["x"], g["w"], rstd,
                                                   eps=wl.eps)
        dx_r, dw_r = rn.rmsnorm_bwd(g["dy"], g["x"], g["w"], rstd, eps=wl.eps)
        torch.cuda.synchronize()
        _, _, _, tdw = orc.bwd(inp["dy"], inp["x"], inp["w"], wl.eps,
                               want_dx=False, want_terms=True)
        check_rows(f"{name} dx static vs workspace", dx_s,
                   dx_r.double().cpu(), wl.dtype, (dx_r.double().cpu().abs()
                                                   + 1e-30))
        check_dw(f"{name} dw static vs workspace", dw_s, dw_r.double().cpu(), tdw)
