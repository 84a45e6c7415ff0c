"""GPU tier: the double backward (rmsnorm_bwd_bwd) against the fp64 oracle.

[P1] "训推加速 Qwen3 实战：从“调包”到手写 Triton Kernel（含 backward）" §5.6: an
autograd wrapper implements double backward or refuses it. The kernel gives
the gradients of sum(gdx * dx) + sum(gdw * dw) with respect to dy, x and w;
compared element by element (ddy, dx2) and on all of dw2, over dtypes,
feature counts (vectorised, masked and scalar layouts), row counts with a
ragged tail, with either incoming gradient absent, rstd given or recomputed,
and at the Qwen3-8B training shape on sampled rows.
"""
import pytest
import torch

import oracle
from rmsnorm_fwd_bwd_02_gb300 import rmsnorm as rn
from rmsnorm_fwd_bwd_02_gb300 import workloads as W
from tests.chunked import chunk_rows, for_row_chunks, rows_of
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


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


def synth(M, H, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    d = {"x": torch.randn(M, H, generator=g) * 2.0,
         "w": 1.0 + 0.1 * torch.randn(H, generator=g),
         "dy": torch.randn(M, H, generator=g),
         "gx": torch.randn(M, H, generator=g)}
    if M > 1:
        d["x"] *= torch.logspace(-2, 2, M).unsqueeze(1)
    out = {k: v.to(dtype).contiguous() for k, v in d.items()}
    out["gw"] = torch.randn(H, generator=g, dtype=torch.float32)
    return out


def run(inp, use_gx, use_gw, with_rstd, eps=1e-6):
    g = {k: v.to(DEV) for k, v in inp.items()}
    rstd = None
    if with_rstd:
        _, rstd = rn.rmsnorm_fwd(g["x"], g["w"], eps=eps)
    out = rn.rmsnorm_bwd_bwd(g["dy"], g["x"], g["w"], rstd,
                             g["gx"] if use_gx else None, g["gw"] if use_gw else None,
                             eps=eps)
    path = rn.last_path()
    torch.cuda.synchronize()
    return out, path


def compare(name, got, o, dtype):
    ddy, dx2, dw2 = got
    check_rows(f"{name} ddy", ddy, o[0], dtype, o[3])
    check_rows(f"{name} dx2", dx2, o[1], dtype, o[4])
    check_dw(f"{name} dw2", dw2, o[2], o[5])


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32],
                         ids=["bf16", "f16", "f32"])
@pytest.mark.parametrize("H", [7, 128, 896, 1000, 4096, 5120, 16384])
@pytest.mark.parametrize("M", [1, 67, 300])
def test_bwd_bwd_matches_oracle(orc, dtype, H, M):
    if M * H > 300 * 5120:
        M = max(1, (300 * 5120) // H)
    inp = synth(M, H, dtype, seed=H + 3 * M)
    for use_gx, use_gw in ((True, True), (True, False), (False, True)):
        o = orc.bwd_bwd(inp["dy"], inp["x"], inp["w"], inp["gx"] if use_gx else None,
                        inp["gw"] if use_gw else None, 1e-6, want_terms=True)
        for with_rstd in (True, False):
            got, _ = run(inp, use_gx, use_gw, with_rstd)
            compare(f"{dtype} M={M} H={H} gx={use_gx} gw={use_gw} rstd={with_rstd}",
                    got, o, dtype)


def test_no_incoming_gradients_give_zeros():
    inp = synth(65, 896, torch.bfloat16, seed=1)
    (ddy, dx2, dw2), _ = run(inp, False, False, True)
    assert not bool(ddy.any()) and not bool(dx2.any()) and not bool(dw2.any())


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_scalar_path(orc, dtype):
    """Rows that are not 16-byte aligned, and the scalar path forced."""
    M, H = 129, 1000
    inp = synth(M, H, dtype, seed=7)
    o = orc.bwd_bwd(inp["dy"], inp["x"], inp["w"], inp["gx"], inp["gw"], 1e-6,
                    want_terms=True)
    rn.set_path_override(rn.PATH_SCALAR)
    try:
        got, path = run(inp, True, True, True)
    finally:
        rn.set_path_override(rn.PATH_AUTO)
    assert path == rn.PATH_SCALAR
    compare(f"scalar {dtype}", got, o, dtype)
    # odd H: not 16-byte aligned rows
    inp = synth(M, 999, dtype, seed=8)
    o = orc.bwd_bwd(inp["dy"], inp["x"], inp["w"], inp["gx"], inp["gw"], 1e-6,
                    want_terms=True)
    got, path = run(inp, True, True, False)
    assert path == rn.PATH_SCALAR
    compare(f"odd H {dtype}", got, o, dtype)


def test_full_size_all_elements(orc):
    """The Qwen3-8B training shape: every element of ddy and dx2 against the
    oracle (row chunks on host threads), dw2 over all rows, same bits run
    to run."""
    wl = W.WORKLOADS["qwen3-8b-train"]
    inp = W.make_inputs(wl)
    g = torch.Generator().manual_seed(99)
    inp["gx"] = (torch.randn(wl.M, wl.H, generator=g) * 1e-2).to(wl.dtype)
    inp["gw"] = torch.randn(wl.H, generator=g, dtype=torch.float32) * 1e-3
    got, _ = run(inp, True, True, True, eps=wl.eps)
    again, _ = run(inp, True, True, True, eps=wl.eps)
    for a, b, nm in zip(got, again, ("ddy", "dx2", "dw2")):
        check_bits(f"full size {nm} run-to-run", a, b)
    _, _, dw2, _, _, tdw2 = orc.bwd_bwd(inp["dy"], inp["x"], inp["w"], inp["gx"],
                                         inp["gw"], wl.eps, want_terms=True)
    check_dw("full size dw2 (all rows)", got[2], dw2, tdw2)
    ddy, dx2 = got[0].cpu(), got[1].cpu()

    def work(a, b):
        sub = rows_of(inp, a, b)
        o = orc.bwd_bwd(sub["dy"], sub["x"], sub["w"], sub["gx"], sub["gw"], wl.eps,
                        want_terms=True)
        check_rows(f"full size ddy rows {a}:{b}", ddy[a:b], o[0], wl.dtype, o[3])
        check_rows(f"full size dx2 rows {a}:{b}", dx2[a:b], o[1], wl.dtype, o[4])

    for_row_chunks(wl.M, work, chunk_rows(wl.H))


def test_error_returns():
    lib = rn.lib()
    s = torch.cuda.current_stream().cuda_stream
    M, H = 8, 128
    t = lambda: torch.randn(M, H, device=DEV, dtype=torch.bfloat16)  # noqa: E731
    dy, x, gx, ddy, dx2 = t(), t(), t(), t(), t()
    w = torch.ones(H, device=DEV, dtype=torch.bfloat16)
    gw = torch.zeros(H + 8, device=DEV)
    dw2 = torch.empty(H, device=DEV)
    ws = torch.empty(1 << 20, device=DEV, dtype=torch.uint8)
    P = lambda v: v if isinstance(v, int) or v is None else v.data_ptr()  # noqa: E731

    def call(ddy=ddy, dx2=dx2, dw2=dw2, gw=gw, gx=gx):
        return lib.rmsnorm_bwd_bwd(P(dy), P(x), P(w), None, P(gx), P(gw), P(ddy), P(dx2),
                                   P(dw2), P(ws), ws.numel(), M, H, 1e-6,
                                   rn.RMSNORM_BF16, s)
    assert call(dw2=None) == -1
    assert call(ddy=dy) == -9                 # an output over an input
    assert call(dx2=ddy) == -9                # two outputs overlapping
    assert call(gw=gw.data_ptr() + 4) == -5   # gw must be 16-byte aligned
    assert call() == 0
    torch.cuda.synchronize()


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16], ids=["bf16", "f16"])
@pytest.mark.parametrize("H", [4096, 5120])
@pytest.mark.parametrize("M", [1, 7, 1037])
def test_streamed_and_row_wise_agree_with_oracle(orc, dtype, H, M):
    """Rows of 4096 and 5120 take the streamed kernel automatically; both it
    and the row-wise kernel (forced) against the oracle, with gx or gw
    absent and rstd recomputed too."""
    inp = synth(M, H, dtype, seed=M + H)
    for use_gx, use_gw, with_rstd in ((True, True, True), (False, True, False),
                                      (True, False, True)):
        o = orc.bwd_bwd(inp["dy"], inp["x"], inp["w"], inp["gx"] if use_gx else None,
                        inp["gw"] if use_gw else None, 1e-6, want_terms=True)
        for path, expect in ((rn.PATH_AUTO, rn.PATH_STREAM), (rn.PATH_ROWS, rn.PATH_ROWS)):
            rn.set_path_override(path)
            try:
                got, used = run(inp, use_gx, use_gw, with_rstd)
            finally:
                rn.set_path_override(rn.PATH_AUTO)
            assert used == expect, (path, used)
            compare(f"{dtype} H={H} M={M} path={path} gx={use_gx} gw={use_gw} "
                    f"rstd={with_rstd}", got, o, dtype)


def test_streamed_wait_runs_out_and_context_survives(orc):
    """Every streamed wait of the double backward runs out (16 bytes that no
    copy delivers, 20 ms limit): counted, drained, and the next call is
    right."""
    inp = synth(300, 4096, torch.bfloat16, seed=3)
    rn.wait_timeouts(reset=True)
    rn.set_stream_test_fault(16, 20000)
    try:
        run(inp, True, True, True)            # results incomplete by design
        torch.cuda.synchronize()
    finally:
        rn.set_stream_test_fault(0, 0)
    assert rn.wait_timeouts(reset=True) > 0
    o = orc.bwd_bwd(inp["dy"], inp["x"], inp["w"], inp["gx"], inp["gw"], 1e-6,
                    want_terms=True)
    got, used = run(inp, True, True, True)
    assert used == rn.PATH_STREAM
    compare("after timeouts", got, o, torch.bfloat16)
    assert rn.wait_timeouts() == 0
