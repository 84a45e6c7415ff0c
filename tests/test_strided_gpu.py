"""GPU tier: row-strided tensors through rmsnorm_fwd_strided and
rmsnorm_bwd_strided, against the fp64 oracle.

The forward kernel printed in [P1] "训推加速 Qwen3 实战：从“调包”到手写
Triton Kernel（含 backward）" §4.2 takes a row stride for its input and its
output; here every [M, H] tensor has its own. Inputs sit in the first H
columns of wider buffers whose other columns hold NaN, so a read outside the
rows poisons the results; outputs sit in buffers whose other columns hold a
guard pattern that must survive. Wherever a strided call runs the same
kernel family as the dense call on the same values, the results must agree
bit for bit (the strides change no arithmetic).
"""
import pytest
import torch

import oracle
from rmsnorm_fwd_bwd_02_gb300 import rmsnorm as rn
from rmsnorm_fwd_bwd_02_gb300 import workloads as W
from tests.chunked import chunk_rows, for_row_chunks, rows_of
from tests.tolerances import check_bits, check_dw, check_rows, check_rstd

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
GUARD = {torch.bfloat16: 0x7FA5, torch.float16: 0x7E5A, torch.float32: 0x7FA5A5A5}
INT = {torch.bfloat16: torch.int16, torch.float16: torch.int16,
       torch.float32: torch.int32}


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


class forced_path:
    def __init__(self, path):
        self.path = path

    def __enter__(self):
        rn.set_path_override(self.path)

    def __exit__(self, *a):
        rn.set_path_override(rn.PATH_AUTO)


def synth(M, H, dtype, seed, residual):
    g = torch.Generator().manual_seed(seed)
    d = {"x": torch.randn(M, H, generator=g) * 2.0,
         "w": 1.0 + 0.1 * torch.randn(H, generator=g),
         "dy": torch.randn(M, H, generator=g)}
    if residual:
        d["r"] = torch.randn(M, H, generator=g)
        d["dh"] = torch.randn(M, H, generator=g)
    if M > 1:
        d["x"] *= torch.logspace(-2, 2, M).unsqueeze(1)
    return {k: v.to(dtype).contiguous() for k, v in d.items()}


def in_rows(t, ld):
    """Input rows: t's values in the first H columns of an [M, ld] buffer
    filled with NaN."""
    return W.in_strided(t.to(DEV), ld, float("nan"))


def out_rows(M, H, ld, dtype):
    """Output rows: the first H columns of an [M, ld] buffer whose bits are
    all the guard pattern; returns (buffer, view)."""
    buf = torch.empty(M, ld, device=DEV, dtype=dtype)
    buf.view(INT[dtype]).fill_(GUARD[dtype])
    return buf, buf[:, :H]


def gaps_intact(buf, H, name):
    gap = buf[:, H:]
    if gap.numel():
        ok = bool((gap.contiguous().view(INT[buf.dtype]) == GUARD[buf.dtype]).all())
        assert ok, f"{name}: a write landed between the rows"


def oracle_all(orc, inp, eps, residual, dh=True):
    o = {}
    if residual:
        o["h"], o["y"], o["rstd"] = orc.residual_fwd(inp["x"], inp["r"], inp["w"], eps)
        o["dx"], o["dw"], o["tdx"], o["tdw"] = orc.residual_bwd(
            inp["dy"], inp["dh"] if dh else None, o["h"], inp["w"], eps,
            want_terms=True)
    else:
        o["y"], o["rstd"] = orc.fwd(inp["x"], inp["w"], eps)
        o["dx"], o["dw"], o["tdx"], o["tdw"] = orc.bwd(
            inp["dy"], inp["x"], inp["w"], eps, want_terms=True)
    return o


def run_strided(inp, ld_in, ld_out, residual, dh=True, eps=1e-6):
    """Forward and backward with inputs at row stride ld_in and outputs at
    ld_out; returns the outputs (views) and their buffers."""
    M, H = inp["x"].shape
    dt = inp["x"].dtype
    x = in_rows(inp["x"], ld_in)
    dy = in_rows(inp["dy"], ld_in)
    w = inp["w"].to(DEV)
    yb, y = out_rows(M, H, ld_out, dt)
    dxb, dx = out_rows(M, H, ld_out, dt)
    bufs = {"y": yb, "dx": dxb}
    if residual:
        r = in_rows(inp["r"], ld_in)
        dhv = in_rows(inp["dh"], ld_in) if dh else None
        hb, h = out_rows(M, H, ld_out, dt)
        bufs["h"] = hb
        h, y, rstd = rn.rmsnorm_fwd_strided(x, w, y=y, r=r, h=h, eps=eps)
        path_f = rn.last_path()
        dx, dw = rn.rmsnorm_bwd_strided(dy, h, w, rstd, dh_out=dhv, dx=dx, eps=eps)
        out = {"h": h, "y": y, "rstd": rstd, "dx": dx, "dw": dw}
    else:
        y, rstd = rn.rmsnorm_fwd_strided(x, w, y=y, eps=eps)
        path_f = rn.last_path()
        dx, dw = rn.rmsnorm_bwd_strided(dy, x, w, rstd, dx=dx, eps=eps)
        out = {"y": y, "rstd": rstd, "dx": dx, "dw": dw}
    path_b = rn.last_path()
    torch.cuda.synchronize()
    return out, bufs, (path_f, path_b)


def run_dense(inp, residual, dh=True, eps=1e-6):
    g = {k: v.to(DEV) for k, v in inp.items()}
    if residual:
        h, y, rstd = rn.rmsnorm_residual_fwd(g["x"], g["r"], g["w"], eps=eps)
        path_f = rn.last_path()
        dx, dw = rn.rmsnorm_residual_bwd(g["dy"], g["dh"] if dh else None, h,
                                         g["w"], rstd, eps=eps)
        out = {"h": h, "y": y, "rstd": rstd, "dx": dx, "dw": dw}
    else:
        y, rstd = rn.rmsnorm_fwd(g["x"], g["w"], eps=eps)
        path_f = rn.last_path()
        dx, dw = rn.rmsnorm_bwd(g["dy"], g["x"], g["w"], rstd, eps=eps)
        out = {"y": y, "rstd": rstd, "dx": dx, "dw": dw}
    path_b = rn.last_path()
    torch.cuda.synchronize()
    return out, (path_f, path_b)


def same_bits_where_same_family(name, got, used, dense, dense_used):
    """Strided and dense results agree bit for bit in each direction whose
    calls ran the same kernel family (the strides change no arithmetic)."""
    keys = {0: ("h", "y", "rstd"), 1: ("dx", "dw")}
    for d in (0, 1):
        if used[d] == dense_used[d]:
            for k in keys[d]:
                if k in got:
                    check_bits(f"{name} {k} vs dense", got[k], dense[k])


def compare(name, got, o, dtype):
    if "h" in o:
        check_bits(f"{name} h", got["h"], o["h"])
    check_rows(f"{name} y", got["y"], o["y"], dtype)
    check_rstd(f"{name} rstd", got["rstd"], o["rstd"])
    check_rows(f"{name} dx", got["dx"], o["dx"], dtype, o["tdx"])
    check_dw(f"{name} dw", got["dw"], o["dw"], o["tdw"])


DTYPES = [torch.bfloat16, torch.float16, torch.float32]


@pytest.mark.parametrize("dtype", DTYPES, ids=["bf16", "f16", "f32"])
@pytest.mark.parametrize("H", [7, 128, 896, 1000, 4096, 5120])
@pytest.mark.parametrize("path", [rn.PATH_AUTO, rn.PATH_ROWS, rn.PATH_SPLIT,
                                  rn.PATH_SCALAR, rn.PATH_STREAM])
def test_strided_matches_oracle_and_dense(orc, dtype, H, path):
    es = torch.empty(0, dtype=dtype).element_size()
    pad16 = 32 // es            # keeps rows 32-byte aligned
    for M, residual in ((5, False), (300, True), (300, False)):
        inp = synth(M, H, dtype, seed=H + M, residual=residual)
        o = oracle_all(orc, inp, 1e-6, residual)
        with forced_path(path):
            dense, dense_used = run_dense(inp, residual)
            for ld_in, ld_out in ((H + pad16, H + 2 * pad16), (H + 3, H),
                                  (H, H + pad16)):
                got, bufs, used = run_strided(inp, ld_in, ld_out, residual)
                name = f"{dtype} H={H} M={M} res={residual} path={path} " \
                       f"ld={ld_in}/{ld_out}"
                for k, b in bufs.items():
                    gaps_intact(b, H, f"{name} {k}")
                compare(name, got, o, dtype)
                vec = (H * es) % 16 == 0 and (ld_in * es) % 16 == 0 and \
                    (ld_out * es) % 16 == 0
                if not vec or path == rn.PATH_SCALAR:
                    assert used[1] == rn.PATH_SCALAR, (name, used)
                if vec:
                    same_bits_where_same_family(name, got, used, dense, dense_used)


def test_streamed_backward_takes_strides(orc):
    """Rows of 4096 and 5120 at a padded stride stay on the streamed
    backward; 128-wide rows (block copies of consecutive rows) leave it."""
    for H, expect in ((4096, rn.PATH_STREAM), (5120, rn.PATH_STREAM),
                      (128, rn.PATH_ROWS)):
        for dt in (torch.bfloat16, torch.float16):
            inp = synth(1031, H, dt, seed=H, residual=False)
            o = oracle_all(orc, inp, 1e-6, False)
            got, bufs, used = run_strided(inp, H + 64, H + 128, False)
            assert used[1] == expect, (H, dt, used)
            for k, b in bufs.items():
                gaps_intact(b, H, f"H={H} {k}")
            compare(f"stream-strided H={H} {dt}", got, o, dt)


def test_residual_dh_none_strided(orc):
    inp = synth(517, 5120, torch.bfloat16, seed=3, residual=True)
    o = oracle_all(orc, inp, 1e-6, True, dh=False)
    got, bufs, _ = run_strided(inp, 5120 + 256, 5120 + 64, True, dh=False)
    compare("resid dh=None strided", got, o, torch.bfloat16)


def test_interleaved_column_windows(orc):
    """x and y as two column windows of one [M, 2H] buffer, dy and dx as two
    windows of another: the alias rule lets them share memory, and nothing
    bleeds between the windows."""
    M, H, dt = 700, 4096, torch.bfloat16
    inp = synth(M, H, dt, seed=11, residual=False)
    o = oracle_all(orc, inp, 1e-6, False)
    for path in (rn.PATH_AUTO, rn.PATH_ROWS, rn.PATH_SCALAR):
        a = torch.empty(M, 2 * H, device=DEV, dtype=dt)
        b = torch.empty(M, 2 * H, device=DEV, dtype=dt)
        x, y = a[:, :H], a[:, H:]
        dy, dx = b[:, H:], b[:, :H]
        x.copy_(inp["x"].to(DEV))
        dy.copy_(inp["dy"].to(DEV))
        w = inp["w"].to(DEV)
        with forced_path(path):
            y, rstd = rn.rmsnorm_fwd_strided(x, w, y=y)
            dx, dw = rn.rmsnorm_bwd_strided(dy, x, w, rstd, dx=dx)
        torch.cuda.synchronize()
        check_bits(f"interleaved x untouched path={path}", x, inp["x"])
        check_bits(f"interleaved dy untouched path={path}", dy, inp["dy"])
        compare(f"interleaved path={path}", {"y": y, "rstd": rstd, "dx": dx,
                                             "dw": dw}, o, dt)


def test_strided_in_place(orc):
    """y over x and dx over dy, both strided (same view)."""
    M, H, dt = 300, 4096, torch.float16
    inp = synth(M, H, dt, seed=12, residual=False)
    o = oracle_all(orc, inp, 1e-6, False)
    x = in_rows(inp["x"], H + 512)
    w = inp["w"].to(DEV)
    xs = in_rows(inp["x"], H + 512)
    y, rstd = rn.rmsnorm_fwd_strided(x, w, y=x)
    dy = in_rows(inp["dy"], H + 256)
    dx, dw = rn.rmsnorm_bwd_strided(dy, xs, w, rstd, dx=dy)
    torch.cuda.synchronize()
    assert y.data_ptr() == x.data_ptr() and dx.data_ptr() == dy.data_ptr()
    compare("strided in place", {"y": y, "rstd": rstd, "dx": dx, "dw": dw}, o, dt)


def test_strided_rejects_bad_strides():
    x = torch.randn(8, 256, device=DEV, dtype=torch.bfloat16)
    w = torch.ones(128, device=DEV, dtype=torch.bfloat16)
    # a view whose stride cannot be expressed (columns not unit-stride)
    with pytest.raises(ValueError):
        rn.rmsnorm_fwd_strided(x[:, ::2], w)
    # the C ABI refuses a stride below H
    lib = rn.lib()
    st = lib.rmsnorm_fwd_strided(x.data_ptr(), 64, None, 0, w.data_ptr(),
                                 x.data_ptr(), 256, None, 0, None, 8, 128, 1e-6,
                                 rn.RMSNORM_BF16,
                                 torch.cuda.current_stream().cuda_stream)
    assert st == -12


def test_full_size_strided_workload_all_elements(orc):
    """The strided benchmark workload at full size, in the layout the
    benchmark times: every element against the oracle (row chunks on host
    threads), dw over all rows, and the same bits as the dense call."""
    wl = W.WORKLOADS["qwen3-8b-train-strided"]
    inp = W.make_inputs(wl)
    got, bufs, used = run_strided(inp, wl.ld, wl.ld, False, eps=wl.eps)
    for k, b in bufs.items():
        gaps_intact(b, wl.H, f"full strided {k}")
    _, dw, _, tdw = orc.bwd(inp["dy"], inp["x"], inp["w"], wl.eps, want_dx=False,
                            want_terms=True)
    check_dw("full strided dw (all rows)", got["dw"], dw, tdw)
    host = {k: got[k].cpu() for k in ("y", "rstd", "dx")}

    def work(a, b):
        o = oracle_all(orc, rows_of(inp, a, b), wl.eps, False)
        check_rows(f"full strided y rows {a}:{b}", host["y"][a:b], o["y"], wl.dtype)
        check_rstd(f"full strided rstd rows {a}:{b}", host["rstd"][a:b], o["rstd"])
        check_rows(f"full strided dx rows {a}:{b}", host["dx"][a:b], o["dx"], wl.dtype,
                   o["tdx"])

    for_row_chunks(wl.M, work, chunk_rows(wl.H))
    dense, dense_used = run_dense(inp, False, eps=wl.eps)
    assert used == dense_used, (used, dense_used)
    same_bits_where_same_family("full strided", got, used, dense, dense_used)
