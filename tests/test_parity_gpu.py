"""GPU tier: the CUDA path (through the C ABI) against the fp64 oracle.

* every workload at a reduced row count that spans several tiles and ends in
  a ragged tail, compared element by element;
* the three large workloads (and fp16 storage) at full size in the launch
  configuration the benchmark times, every element of y, rstd, dx, h and dw
  (the oracle runs over row chunks on host threads, tests/chunked.py);
* edge shapes and dtypes, misaligned and odd rows (scalar kernels), in-place
  calls, saved vs recomputed rstd, split-row vs row-wise, determinism,
  guard words around every output, M == 0, error returns, CUDA-graph replay.
Tolerances: tests/tolerances.py.
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


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.fail("the gpu tier needs a CUDA device")
    rn.lib()          # raises if the library has not been built
    rn.set_path_override(rn.PATH_AUTO)
    yield
    rn.set_path_override(rn.PATH_AUTO)


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


def to_dev(d):
    return {k: v.to(DEV) for k, v in d.items()}


class forced_path:
    def __init__(self, path):
        self.path = path

    def __enter__(self):
        rn.set_path_override(self.path)

    def __exit__(self, *a):
        rn.set_path_override(rn.PATH_AUTO)


def gpu_fwd_bwd(wl, g, dh=True, with_rstd=True):
    """Run the workload's forward and backward on the GPU."""
    out = {}
    if wl.residual:
        h, y, rstd = rn.rmsnorm_residual_fwd(g["x"], g["r"], g["w"], eps=wl.eps)
        out.update(h=h, y=y, rstd=rstd)
        if wl.backward:
            dx, dw = rn.rmsnorm_residual_bwd(g["dy"], g["dh"] if dh else None, h,
                                             g["w"], rstd if with_rstd else None,
                                             eps=wl.eps)
            out.update(dx=dx, dw=dw)
    else:
        y, rstd = rn.rmsnorm_fwd(g["x"], g["w"], eps=wl.eps)
        out.update(y=y, rstd=rstd)
        if wl.backward:
            dx, dw = rn.rmsnorm_bwd(g["dy"], g["x"], g["w"],
                                    rstd if with_rstd else None, eps=wl.eps)
            out.update(dx=dx, dw=dw)
    torch.cuda.synchronize()
    return out


def oracle_all(orc, wl, inp, dh=True):
    o = {}
    if wl.residual:
        o["h"], o["y"], o["rstd"] = orc.residual_fwd(inp["x"], inp["r"], inp["w"], wl.eps)
        if wl.backward:
            o["dx"], o["dw"], o["tdx"], o["tdw"] = orc.residual_bwd(
                inp["dy"], inp["dh"] if dh else None, o["h"], inp["w"], wl.eps,
                want_terms=True)
    else:
        o["y"], o["rstd"] = orc.fwd(inp["x"], inp["w"], wl.eps)
        if wl.backward:
            o["dx"], o["dw"], o["tdx"], o["tdw"] = orc.bwd(
                inp["dy"], inp["x"], inp["w"], wl.eps, want_terms=True)
    return o


def compare_all(name, wl, got, o):
    if "h" in o:
        check_bits(f"{name} h", got["h"], o["h"])
    check_rows(f"{name} y", got["y"], o["y"], wl.dtype)
    check_rstd(f"{name} rstd", got["rstd"], o["rstd"])
    if "dx" in o:
        check_rows(f"{name} dx", got["dx"], o["dx"], wl.dtype, o["tdx"])
        check_dw(f"{name} dw", got["dw"], o["dw"], o["tdw"])


# --------------------------------------------------------------- workloads
REDUCED = {
    "tiny-fp32": 64, "decode-m1": 1, "decode-m8": 8, "decode-m64": 64,
    "qwen3-8b-train": 1037, "qwen3-qknorm": 4099, "residual-14b": 517,
    "qwen3-8b-train-fp16": 1037,
}


@pytest.mark.parametrize("name", list(REDUCED))
def test_workload_reduced_all_elements(orc, name):
    wl = W.WORKLOADS[name]
    if REDUCED[name] != wl.M:
        wl = wl.with_rows(REDUCED[name])
    inp = W.make_inputs(wl)
    o = oracle_all(orc, wl, inp)
    got = gpu_fwd_bwd(wl, to_dev(inp))
    compare_all(name, wl, got, o)
    if wl.residual:      # and without the incoming residual gradient
        o2 = oracle_all(orc, wl, inp, dh=False)
        got2 = gpu_fwd_bwd(wl, to_dev(inp), dh=False)
        compare_all(name + " dh=None", wl, got2, o2)


def check_full_size(orc, wl, inp, got, tag):
    """Every element of the GPU results `got` (host tensors) against the
    oracle, over row chunks: y, rstd, dx and (residual) h bit-exact; then dw
    over all rows (for the residual variant, from the oracle's own h)."""
    oh_full = torch.empty_like(inp["x"]) if wl.residual else None

    def work(a, b):
        o = oracle_all(orc, wl.with_rows(b - a), rows_of(inp, a, b))
        t = f"{tag} rows {a}:{b}"
        if wl.residual:
            check_bits(f"{t} h", got["h"][a:b], o["h"])
            oh_full[a:b] = o["h"]
        check_rows(f"{t} y", got["y"][a:b], o["y"], wl.dtype)
        check_rstd(f"{t} rstd", got["rstd"][a:b], o["rstd"])
        check_rows(f"{t} dx", got["dx"][a:b], o["dx"], wl.dtype, o["tdx"])

    for_row_chunks(wl.M, work, chunk_rows(wl.H))
    if wl.residual:
        _, dw, _, tdw = orc.residual_bwd(inp["dy"], inp["dh"], oh_full, inp["w"], wl.eps,
                                         want_dx=False, want_terms=True)
    else:
        _, dw, _, tdw = orc.bwd(inp["dy"], inp["x"], inp["w"], wl.eps, want_dx=False,
                                want_terms=True)
    check_dw(f"{tag} dw (all rows)", got["dw"], dw, tdw)


@pytest.mark.parametrize("name", ["qwen3-8b-train", "qwen3-qknorm", "residual-14b",
                                  "qwen3-8b-train-fp16"])
def test_workload_full_size_all_elements(orc, name):
    """The large workloads at full size, as the benchmark runs them (automatic
    kernel choice, dh_out given), every output element against the oracle."""
    wl = W.WORKLOADS[name]
    inp = W.make_inputs(wl)
    got = {k: v.cpu() for k, v in gpu_fwd_bwd(wl, to_dev(inp)).items()}
    check_full_size(orc, wl, inp, got, name)


# ------------------------------------------------------------ edge shapes
def synth(M, H, dtype, seed=0, residual=False):
    g = torch.Generator().manual_seed(seed)
    d = {"x": torch.randn(M, H, generator=g) * 2.0,
         "w": 1.0 + 0.1 * torch.randn(H, generator=g),
         "dy": torch.randn(M, H, generator=g)}
    if residual:
        d["r"] = torch.randn(M, H, generator=g)
        d["dh"] = torch.randn(M, H, generator=g)
    # rows with very different scales catch row mix-ups
    d["x"] *= torch.logspace(-2, 2, M).unsqueeze(1) if M > 1 else 1.0
    return {k: v.to(dtype).contiguous() for k, v in d.items()}


EDGE_H = [1, 2, 7, 8, 9, 64, 127, 128, 129, 512, 895, 896, 1000, 1024, 2048,
          4095, 4096, 4104, 5120, 8192, 16384]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32, torch.float16],
                         ids=["bf16", "f32", "f16"])
@pytest.mark.parametrize("H", EDGE_H)
@pytest.mark.parametrize("M", [1, 67, 300])
def test_edge_shapes(orc, M, H, dtype):
    if M * H > 300 * 4104:
        M = max(1, (300 * 4104) // H)
    for residual in (False, True):
        wl = W.Workload(f"edge-{M}x{H}", M, H, dtype, residual=residual)
        inp = synth(M, H, dtype, seed=H + M, residual=residual)
        o = oracle_all(orc, wl, inp)
        got = gpu_fwd_bwd(wl, to_dev(inp))
        compare_all(f"M={M} H={H} {dtype} res={residual}", wl, got, o)


STREAM_H = (128, 4096, 5120)     # 16-bit feature counts with a streamed layout
HALF = (torch.bfloat16, torch.float16)


@pytest.mark.parametrize("path", [rn.PATH_ROWS, rn.PATH_SPLIT, rn.PATH_SCALAR,
                                  rn.PATH_STREAM])
@pytest.mark.parametrize("H", [1, 7, 128, 896, 4096, 5120, 16384])
def test_forced_paths_agree_with_oracle(orc, path, H):
    M = 5
    for dtype in (torch.bfloat16, torch.float32, torch.float16):
        for residual in (False, True):
            wl = W.Workload(f"forced-{path}", M, H, dtype, residual=residual)
            inp = synth(M, H, dtype, seed=3, residual=residual)
            o = oracle_all(orc, wl, inp)
            with forced_path(path):
                got = gpu_fwd_bwd(wl, to_dev(inp))
                used = rn.last_path()
            vec_ok = (H * inp["x"].element_size()) % 16 == 0
            if path == rn.PATH_SCALAR or not vec_ok:
                assert used == rn.PATH_SCALAR
            elif path == rn.PATH_STREAM and dtype in HALF and H in STREAM_H:
                assert used == rn.PATH_STREAM
            else:
                assert used == rn.PATH_ROWS   # the backward reports last
            compare_all(f"path={path} H={H} {dtype} res={residual}", wl, got, o)


@pytest.mark.parametrize("name,M", [("qwen3-8b-train", 1), ("qwen3-8b-train", 7),
                                    ("qwen3-8b-train", 1037), ("residual-14b", 3),
                                    ("residual-14b", 517), ("qwen3-qknorm", 1),
                                    ("qwen3-qknorm", 7), ("qwen3-qknorm", 33),
                                    ("qwen3-qknorm", 40961)])
def test_stream_path_ragged(orc, name, M):
    """Streamed kernels: every variant (residual, dh_out given or not, rstd
    given or recomputed) on row counts that leave groups idle or uneven."""
    wl = W.WORKLOADS[name].with_rows(M)
    inp = W.make_inputs(wl)
    g = to_dev(inp)
    variants = [(wl, inp, g)]
    if name == "qwen3-qknorm":       # the residual variant on short rows too
        rw = W.Workload("qk-res", M, 128, torch.bfloat16, residual=True, dy_std=1e-2)
        ri = synth(M, 128, torch.bfloat16, seed=M, residual=True)
        variants.append((rw, ri, to_dev(ri)))
    for wl, inp, g in variants:
        for dh in ((True, False) if wl.residual else (True,)):
            for with_rstd in (True, False):
                o = oracle_all(orc, wl, inp, dh=dh)
                with forced_path(rn.PATH_STREAM):
                    got = gpu_fwd_bwd(wl, g, dh=dh, with_rstd=with_rstd)
                    assert rn.last_path() == rn.PATH_STREAM
                compare_all(f"stream {wl.name} M={M} dh={dh} rstd={with_rstd}",
                            wl, got, o)


@pytest.mark.parametrize("name", ["qwen3-8b-train", "residual-14b", "qwen3-qknorm"])
def test_stream_path_full_size_all_elements(orc, name):
    """The streamed kernels forced for both directions at full size: every
    element against the oracle, and the same bits run to run."""
    wl = W.WORKLOADS[name]
    inp = W.make_inputs(wl)
    with forced_path(rn.PATH_STREAM):
        got = gpu_fwd_bwd(wl, to_dev(inp))
        assert rn.last_path() == rn.PATH_STREAM
    host = {k: v.cpu() for k, v in got.items()}
    check_full_size(orc, wl, inp, host, f"stream {name}")
    with forced_path(rn.PATH_STREAM):
        again = gpu_fwd_bwd(wl, to_dev(inp))
    for k in got:
        check_bits(f"stream {name} {k} run-to-run", again[k], got[k])


@pytest.mark.parametrize("H,M", [(128, 1), (128, 33), (128, 4099), (4096, 7),
                                 (4096, 1037), (5120, 3), (5120, 517)])
def test_stream_path_fp16(orc, H, M):
    """The streamed kernels with fp16 storage: plain and residual, dh_out
    given or not, rstd given or recomputed, ragged row counts."""
    for residual in (False, True):
        wl = W.Workload("stream-f16", M, H, torch.float16, residual=residual,
                        dy_std=1e-2)
        inp = synth(M, H, torch.float16, seed=M + H, residual=residual)
        g = to_dev(inp)
        for dh in ((True, False) if residual else (True,)):
            for with_rstd in (True, False):
                o = oracle_all(orc, wl, inp, dh=dh)
                with forced_path(rn.PATH_STREAM):
                    got = gpu_fwd_bwd(wl, g, dh=dh, with_rstd=with_rstd)
                    assert rn.last_path() == rn.PATH_STREAM
                compare_all(f"stream f16 H={H} M={M} res={residual} dh={dh} "
                            f"rstd={with_rstd}", wl, got, o)


def test_fp16_overflow_and_subnormal_results(orc):
    """fp16 results beyond 65504 are infinite with the right sign; tiny
    results land on the subnormal grid as the one-step rounding puts them."""
    H = 4
    # a spike row: x r = +-sqrt(H) = +-2 at the spike, y = 2 w there
    x = torch.tensor([[3.0, 0, 0, 0], [0, -5.0, 0, 0]], dtype=torch.float16)
    w = torch.tensor([60000.0, 40000.0, 1.0, 1.0], dtype=torch.float16)
    y, rstd = rn.rmsnorm_fwd(x.to(DEV), w.to(DEV), eps=0.0)
    torch.cuda.synchronize()
    oy, _ = orc.fwd(x, w, 0.0)
    yc = y.cpu().double()
    assert yc[0, 0] == float("inf") and oy[0, 0] > 65520
    assert yc[1, 1] == float("-inf") and oy[1, 1] < -65520
    # tiny weights: results in the fp16 subnormal range
    M, H = 300, 1024
    inp = synth(M, H, torch.float16, seed=9)
    inp["w"] = (inp["w"].float() * 1e-6).to(torch.float16)
    wl = W.Workload("f16-tiny", M, H, torch.float16)
    o = oracle_all(orc, wl, inp)
    got = gpu_fwd_bwd(wl, to_dev(inp))
    assert bool((o["y"].abs() < 2.0 ** -14).any())
    compare_all("f16 subnormal y", wl, got, o)


def test_auto_path_choice():
    x = torch.randn(64, 896, device=DEV, dtype=torch.bfloat16)
    w = torch.ones(896, device=DEV, dtype=torch.bfloat16)
    rn.rmsnorm_fwd(x, w)
    assert rn.last_path() == rn.PATH_SPLIT
    x = torch.randn(65, 896, device=DEV, dtype=torch.bfloat16)
    rn.rmsnorm_fwd(x, w)
    assert rn.last_path() == rn.PATH_ROWS
    x = torch.randn(65, 895, device=DEV, dtype=torch.bfloat16)
    rn.rmsnorm_fwd(x, torch.ones(895, device=DEV, dtype=torch.bfloat16))
    assert rn.last_path() == rn.PATH_SCALAR
    # 16-bit rows of 128 / 4096 / 5120: the forward row-wise, the backward
    # streamed
    for dt in HALF:
        for H in STREAM_H:
            x = torch.randn(100, H, device=DEV, dtype=dt)
            w = torch.ones(H, device=DEV, dtype=dt)
            _, rstd = rn.rmsnorm_fwd(x, w)
            assert rn.last_path() == rn.PATH_ROWS
            rn.rmsnorm_bwd(x, x, w, rstd)
            assert rn.last_path() == rn.PATH_STREAM
    torch.cuda.synchronize()


def test_misaligned_rows_take_scalar_path(orc):
    """Row pointers offset by one element (not 16-byte aligned); M > 64 so
    the row-wise kernels run (M <= 64 takes the split-row kernel)."""
    M, H = 337, 4096
    for dtype in (torch.bfloat16, torch.float32, torch.float16):
        inp = synth(M, H, dtype, seed=5)
        o = oracle_all(orc, W.Workload("mis", M, H, dtype), inp)
        bx = torch.empty(M * H + 1, device=DEV, dtype=dtype)
        bdy = torch.empty(M * H + 1, device=DEV, dtype=dtype)
        x = bx[1:].view(M, H); x.copy_(inp["x"].to(DEV))
        dy = bdy[1:].view(M, H); dy.copy_(inp["dy"].to(DEV))
        w = inp["w"].to(DEV)
        y, rstd = rn.rmsnorm_fwd(x, w)
        assert rn.last_path() == rn.PATH_SCALAR
        dx, dw = rn.rmsnorm_bwd(dy, x, w, rstd)
        assert rn.last_path() == rn.PATH_SCALAR
        torch.cuda.synchronize()
        compare_all(f"misaligned {dtype}", W.Workload("mis", M, H, dtype),
                    {"y": y, "rstd": rstd, "dx": dx, "dw": dw}, o)


@pytest.mark.parametrize("H", [128, 4096, 5120])
def test_rows_16_byte_aligned_only(orc, H):
    """Row starts on a 16-byte but not a 32-byte boundary: the forward cannot
    use its 32-byte packs and falls back to 16-byte ones, with the same
    results."""
    M, dt = 301, torch.bfloat16
    for residual in (False, True):
        wl = W.Workload("a16", M, H, dt, residual=residual)
        inp = synth(M, H, dt, seed=H, residual=residual)
        o = oracle_all(orc, wl, inp)
        g = {}
        for k, v in inp.items():
            b = torch.empty(v.numel() + 8, device=DEV, dtype=dt)
            t = b[8:].view(v.shape)            # 16 bytes past a 256-byte boundary
            t.copy_(v.to(DEV))
            g[k] = t
        got = gpu_fwd_bwd(wl, g)
        compare_all(f"16B-aligned H={H} res={residual}", wl, got, o)


def test_in_place(orc):
    M, H, dt = 300, 4096, torch.bfloat16
    inp = synth(M, H, dt, seed=7, residual=True)
    wl = W.Workload("inplace", M, H, dt)
    o = oracle_all(orc, wl, inp)
    g = to_dev(inp)
    x = g["x"].clone()
    _, rstd = rn.rmsnorm_fwd(x, g["w"], y=x)            # y == x
    torch.cuda.synchronize()
    check_rows("in-place y", x, o["y"], dt)
    dy = g["dy"].clone()
    dx, dw = rn.rmsnorm_bwd(dy, g["x"], g["w"], rstd, dx=dy)   # dx == dy
    torch.cuda.synchronize()
    check_rows("in-place dx", dx, o["dx"], dt, o["tdx"])
    check_dw("in-place dw", dw, o["dw"], o["tdw"])
    # residual: h written over x
    wl = W.Workload("inplace-res", M, H, dt, residual=True)
    o = oracle_all(orc, wl, inp)
    x2 = g["x"].clone()
    h, y, rstd = rn.rmsnorm_residual_fwd(x2, g["r"], g["w"], h=x2)
    dh = g["dh"].clone()
    dx, dw = rn.rmsnorm_residual_bwd(g["dy"], dh, h, g["w"], rstd, dx=dh)
    torch.cuda.synchronize()
    check_bits("in-place h", x2, o["h"])
    check_rows("in-place resid y", y, o["y"], dt)
    check_rows("in-place resid dx", dx, o["dx"], dt, o["tdx"])


@pytest.mark.parametrize("name", ["qwen3-8b-train", "qwen3-qknorm", "residual-14b"])
def test_bwd_ex_accumulates_dw_over_chunks(orc, name):
    """dw accumulated over chunks of rows equals the dw of all rows (within
    the dw tolerance), dx of each chunk is right, and flags = 0 gives the
    bits of the plain entry point."""
    wl = W.WORKLOADS[name].with_rows(2051)
    inp = W.make_inputs(wl)
    g = to_dev(inp)
    o = oracle_all(orc, wl, inp)
    xk = "x"
    if wl.residual:
        h, _, rstd = rn.rmsnorm_residual_fwd(g["x"], g["r"], g["w"], eps=wl.eps)
        g["h"] = h
        xk = "h"
    else:
        _, rstd = rn.rmsnorm_fwd(g["x"], g["w"], eps=wl.eps)
    dh = g.get("dh")
    dw = torch.full((wl.H,), float("nan"), device=DEV)
    dx = torch.empty_like(g[xk])
    bounds = [0, 1, 700, 1500, 2051]          # uneven chunks, one of one row
    for i, (a, b) in enumerate(zip(bounds[:-1], bounds[1:])):
        rn.rmsnorm_bwd_ex(g["dy"][a:b], g[xk][a:b], g["w"], rstd[a:b],
                          dh_out=None if dh is None else dh[a:b], dx=dx[a:b], dw=dw,
                          eps=wl.eps, accumulate_dw=i > 0)
    torch.cuda.synchronize()
    check_rows(f"{name} chunked dx", dx, o["dx"], wl.dtype, o["tdx"])
    check_dw(f"{name} accumulated dw", dw, o["dw"], o["tdw"])
    # M == 0 with accumulation leaves dw as it is
    before = dw.clone()
    rn.rmsnorm_bwd_ex(g["dy"][:0], g[xk][:0], g["w"], rstd[:0], dw=dw,
                      accumulate_dw=True)
    torch.cuda.synchronize()
    check_bits(f"{name} M=0 accumulate", dw, before)
    # flags = 0: same bits as the plain entry points
    dx1, dw1 = rn.rmsnorm_bwd_ex(g["dy"], g[xk], g["w"], rstd, dh_out=dh, eps=wl.eps)
    if wl.residual:
        dx2, dw2 = rn.rmsnorm_residual_bwd(g["dy"], dh, g[xk], g["w"], rstd, eps=wl.eps)
    else:
        dx2, dw2 = rn.rmsnorm_bwd(g["dy"], g[xk], g["w"], rstd, eps=wl.eps)
    torch.cuda.synchronize()
    check_bits(f"{name} bwd_ex dx", dx1, dx2)
    check_bits(f"{name} bwd_ex dw", dw1, dw2)


def test_rstd_recompute_matches_saved(orc):
    wl = W.WORKLOADS["qwen3-8b-train"].with_rows(513)
    inp = W.make_inputs(wl)
    g = to_dev(inp)
    saved = gpu_fwd_bwd(wl, g, with_rstd=True)
    recomputed = gpu_fwd_bwd(wl, g, with_rstd=False)
    o = oracle_all(orc, wl, inp)
    check_rows("recompute dx", recomputed["dx"], o["dx"], wl.dtype, o["tdx"])
    check_dw("recompute dw", recomputed["dw"], o["dw"], o["tdw"])
    check_rows("saved dx", saved["dx"], o["dx"], wl.dtype, o["tdx"])


def test_split_row_matches_row_wise(orc):
    for M in (1, 8, 64):
        wl = W.WORKLOADS[f"decode-m{M}"]
        inp = W.make_inputs(wl)
        g = to_dev(inp)
        with forced_path(rn.PATH_SPLIT):
            ys, rs = rn.rmsnorm_fwd(g["x"], g["w"])
        with forced_path(rn.PATH_ROWS):
            yr, rr = rn.rmsnorm_fwd(g["x"], g["w"])
        torch.cuda.synchronize()
        o = oracle_all(orc, wl, inp)
        check_rows(f"split M={M}", ys, o["y"], wl.dtype)
        check_rows(f"rows M={M}", yr, o["y"], wl.dtype)
        check_rstd(f"split rstd M={M}", rs, o["rstd"])
        # both round fp32 values that differ only in summation order
        a = ys.view(torch.int16).to(torch.int32).cpu()
        b = yr.view(torch.int16).to(torch.int32).cpu()
        assert int((a - b).abs().max()) <= 1, f"split vs rows M={M}: > 1 ulp apart"


@pytest.mark.parametrize("name", ["qwen3-8b-train", "qwen3-qknorm", "residual-14b",
                                  "decode-m64", "tiny-fp32"])
def test_deterministic(name):
    wl = W.WORKLOADS[name]
    if wl.M > 8192:
        wl = wl.with_rows(8192 + 37)
    g = to_dev(W.make_inputs(wl))
    a = gpu_fwd_bwd(wl, g)
    b = gpu_fwd_bwd(wl, g)
    for k in a:
        check_bits(f"{name} {k} run-to-run", a[k], b[k])


def test_guard_words_untouched(orc):
    """Every output sits between guard regions that must keep their bits."""
    M, H, dt = 257, 896, torch.bfloat16
    G = 64
    inp = synth(M, H, dt, seed=9, residual=True)
    g = to_dev(inp)

    def guarded(n, dtype):
        b = torch.empty(n + 2 * G, device=DEV, dtype=dtype)
        if dtype == torch.bfloat16:
            b.view(torch.int16).fill_(0x7FA5)
        else:
            b.view(torch.int32).fill_(0x7FA5A5A5)
        return b, b[G:G + n]

    def intact(b, n, name):
        head, tail = b[:G], b[G + n:]
        if b.dtype == torch.bfloat16:
            ok = bool((head.view(torch.int16) == 0x7FA5).all()) and \
                bool((tail.view(torch.int16) == 0x7FA5).all())
        else:
            ok = bool((head.view(torch.int32) == 0x7FA5A5A5).all()) and \
                bool((tail.view(torch.int32) == 0x7FA5A5A5).all())
        assert ok, f"{name}: guard words overwritten"

    for path in (rn.PATH_AUTO, rn.PATH_SPLIT, rn.PATH_SCALAR):
        by, y = guarded(M * H, dt)
        bh, h = guarded(M * H, dt)
        br, rstd = guarded(M, torch.float32)
        bdx, dx = guarded(M * H, dt)
        bdw, dw = guarded(H, torch.float32)
        with forced_path(path):
            rn.rmsnorm_residual_fwd(g["x"], g["r"], g["w"], h=h.view(M, H),
                                    y=y.view(M, H), rstd=rstd)
            rn.rmsnorm_residual_bwd(g["dy"], g["dh"], h.view(M, H), g["w"], rstd,
                                    dx=dx.view(M, H), dw=dw)
        torch.cuda.synchronize()
        for b, n, nm in ((by, M * H, "y"), (bh, M * H, "h"), (br, M, "rstd"),
                         (bdx, M * H, "dx"), (bdw, H, "dw")):
            intact(b, n, f"path {path} {nm}")
        o = oracle_all(orc, W.Workload("g", M, H, dt, residual=True), inp)
        compare_all(f"guarded path {path}", W.Workload("g", M, H, dt, residual=True),
                    {"h": h.view(M, H), "y": y.view(M, H), "rstd": rstd,
                     "dx": dx.view(M, H), "dw": dw}, o)


def test_m_zero():
    H, dt = 4096, torch.bfloat16
    x = torch.empty(0, H, device=DEV, dtype=dt)
    w = torch.ones(H, device=DEV, dtype=dt)
    y, rstd = rn.rmsnorm_fwd(x, w)
    dw = torch.full((H,), 7.0, device=DEV)
    dx, dw = rn.rmsnorm_bwd(x, x, w, rstd, dw=dw)
    torch.cuda.synchronize()
    assert y.numel() == 0 and dx.numel() == 0
    assert bool((dw == 0).all())


def test_error_returns():
    M, H, dt = 128, 4096, torch.bfloat16
    x = torch.randn(M, H, device=DEV, dtype=dt)
    w = torch.ones(H, device=DEV, dtype=dt)
    need = rn.bwd_workspace_bytes(M, H, dt)
    # the query covers every kernel variant: whole fp32 rows, more than one
    assert need > H * 4 and need % (H * 4) == 0
    small = torch.empty(H * 4, device=DEV, dtype=torch.uint8)   # one row
    with pytest.raises(rn.RmsNormError) as e:
        rn.rmsnorm_bwd(x, x, w, None, workspace=small)
    assert e.value.status == -6
    wbig = torch.ones(16385, device=DEV, dtype=dt)
    with pytest.raises(rn.RmsNormError) as e:
        rn.rmsnorm_fwd(torch.randn(2, 16385, device=DEV, dtype=dt), wbig)
    assert e.value.status == -7


def test_zero_row_with_eps_zero_does_not_crash():
    """A zero row with eps = 0 has no defined result (0/0); the call must
    still complete and leave the other rows right."""
    M, H = 70, 512
    x = torch.randn(M, H, device=DEV, dtype=torch.bfloat16)
    x[3].zero_()
    w = torch.ones(H, device=DEV, dtype=torch.bfloat16)
    y, rstd = rn.rmsnorm_fwd(x, w, eps=0.0)
    torch.cuda.synchronize()
    assert torch.isinf(rstd[3]).item()
    keep = torch.ones(M, dtype=torch.bool)
    keep[3] = False
    assert bool(torch.isfinite(y[keep.to(DEV)]).all())


def test_cuda_graph_replay_matches_eager():
    """All four entry points allocate and synchronise nothing, so they can be
    captured in a CUDA graph; the replay gives the eager bits."""
    wl = W.WORKLOADS["residual-14b"].with_rows(1024)
    g = to_dev(W.make_inputs(wl))
    w8 = W.WORKLOADS["qwen3-8b-train"].with_rows(1024)
    g8 = to_dev(W.make_inputs(w8))
    M, H = 1024, 5120
    bufs = {k: torch.empty(M, H, device=DEV, dtype=torch.bfloat16)
            for k in ("h", "y", "dx")}
    b8 = {k: torch.empty(1024, 4096, device=DEV, dtype=torch.bfloat16)
          for k in ("y", "dx")}
    rstd = torch.empty(M, device=DEV)
    rstd8 = torch.empty(1024, device=DEV)
    dw = torch.empty(H, device=DEV)
    dw8 = torch.empty(4096, device=DEV)
    ws = torch.empty(max(rn.bwd_workspace_bytes(M, H, torch.bfloat16),
                         rn.bwd_workspace_bytes(1024, 4096, torch.bfloat16)),
                     device=DEV, dtype=torch.uint8)

    def step():
        rn.rmsnorm_residual_fwd(g["x"], g["r"], g["w"], h=bufs["h"], y=bufs["y"], rstd=rstd)
        rn.rmsnorm_residual_bwd(g["dy"], g["dh"], bufs["h"], g["w"], rstd,
                                dx=bufs["dx"], dw=dw, workspace=ws)
        rn.rmsnorm_fwd(g8["x"], g8["w"], y=b8["y"], rstd=rstd8)
        rn.rmsnorm_bwd(g8["dy"], g8["x"], g8["w"], rstd8, dx=b8["dx"], dw=dw8,
                       workspace=ws)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.synchronize()
    eager = [t.clone() for t in (bufs["h"], bufs["y"], bufs["dx"], rstd, dw,
                                 b8["y"], b8["dx"], rstd8, dw8)]
    for t in (bufs["h"], bufs["y"], bufs["dx"], rstd, dw, b8["y"], b8["dx"], rstd8, dw8):
        t.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        step()
    graph.replay()
    torch.cuda.synchronize()
    for a, b in zip(eager, (bufs["h"], bufs["y"], bufs["dx"], rstd, dw, b8["y"],
                            b8["dx"], rstd8, dw8)):
        check_bits("graph replay", b, a)


def test_side_stream():
    wl = W.WORKLOADS["qwen3-8b-train"].with_rows(777)
    g = to_dev(W.make_inputs(wl))
    ref = gpu_fwd_bwd(wl, g)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        y, rstd = rn.rmsnorm_fwd(g["x"], g["w"], stream=s)
        dx, dw = rn.rmsnorm_bwd(g["dy"], g["x"], g["w"], rstd, stream=s)
    s.synchronize()
    for k, v in (("y", y), ("rstd", rstd), ("dx", dx), ("dw", dw)):
        check_bits(f"side stream {k}", v, ref[k])


@pytest.mark.parametrize("name,M", [("qwen3-8b-train", 257), ("residual-14b", 129),
                                    ("qwen3-qknorm", 1000)])
def test_stream_wait_runs_out_and_context_survives(orc, name, M):
    """Make every streamed wait run out (each stage expects 16 bytes that no
    copy delivers, 20 ms limit): the kernels record it, drain their copies,
    end, and the next normal calls are right."""
    wl = W.WORKLOADS[name].with_rows(M)
    inp = W.make_inputs(wl)
    g = to_dev(inp)
    before = rn.wait_timeouts(reset=True)
    assert before == 0
    rn.set_stream_test_fault(16, 20000)
    try:
        with forced_path(rn.PATH_STREAM):
            gpu_fwd_bwd(wl, g)          # results incomplete by design
        torch.cuda.synchronize()
    finally:
        rn.set_stream_test_fault(0, 0)
    assert rn.wait_timeouts(reset=True) > 0
    with forced_path(rn.PATH_STREAM):
        got = gpu_fwd_bwd(wl, g)
    compare_all(f"after timeouts {name}", wl, got, oracle_all(orc, wl, inp))
    assert rn.wait_timeouts() == 0


@pytest.mark.parametrize("name", ["decode-m1", "decode-m64"])
def test_split_wait_runs_out_and_context_survives(orc, name):
    """Make the split-row forward's wait for its peers' sums run out (each
    CTA expects 16 bytes more than its peers store, 20 ms limit): every CTA
    counts it and ends, and the next normal calls are right."""
    wl = W.WORKLOADS[name]
    inp = W.make_inputs(wl)
    g = to_dev(inp)
    assert rn.wait_timeouts(reset=True) == 0
    rn.set_stream_test_fault(16, 20000)
    try:
        with forced_path(rn.PATH_SPLIT):
            rn.rmsnorm_fwd(g["x"], g["w"], eps=wl.eps)     # results wrong by design
            assert rn.last_path() == rn.PATH_SPLIT
        torch.cuda.synchronize()
    finally:
        rn.set_stream_test_fault(0, 0)
    # every CTA of every row's cluster (at least two per row) gave up once
    assert rn.wait_timeouts(reset=True) >= 2 * wl.M
    with forced_path(rn.PATH_SPLIT):
        got = gpu_fwd_bwd(wl, g)
    compare_all(f"after timeouts {name}", wl, got, oracle_all(orc, wl, inp))
    assert rn.wait_timeouts() == 0


def test_no_stream_wait_ran_out():
    """Every bounded wait in the streamed kernels completed during this module."""
    assert rn.wait_timeouts() == 0


def test_tensors_beyond_2_31_elements(orc):
    """M x H above 2^31 elements in every row tensor (524291 x 4096 bf16,
    4.3 GB each): the forward and the (streamed) backward index rows with 64
    bits. Sampled rows across the whole range, the last ones included,
    against the oracle; dw over all rows."""
    M, H = (1 << 31) // 4096 + 3, 4096
    wl = W.Workload("big", M, H, torch.bfloat16, seed=6, dy_std=1e-2)
    g = torch.Generator(device=DEV).manual_seed(6)
    x = torch.randn(M, H, device=DEV, dtype=torch.bfloat16, generator=g)
    dy = (torch.randn(M, H, device=DEV, generator=g) * 1e-2).to(torch.bfloat16)
    w = (1 + 0.1 * torch.randn(H, device=DEV, generator=g)).to(torch.bfloat16)
    y, rstd = rn.rmsnorm_fwd(x, w)
    dx, dw = rn.rmsnorm_bwd(dy, x, w, rstd)
    assert rn.last_path() == rn.PATH_STREAM
    torch.cuda.synchronize()
    rows = sorted(set(W.random_rows(M, 24, seed=1)) | {M - 2, (1 << 31) // H - 1,
                                                        (1 << 31) // H})
    xs, dys, ws = x[rows].cpu(), dy[rows].cpu(), w.cpu()
    oy, orstd = orc.fwd(xs, ws, 1e-6)
    odx, _, tdx, _ = orc.bwd(dys, xs, ws, 1e-6, want_terms=True)
    check_rows("big y", y[rows], oy, torch.bfloat16)
    check_rstd("big rstd", rstd[rows], orstd)
    check_rows("big dx", dx[rows], odx, torch.bfloat16, tdx)
    del y, dx
    # dw over all rows, by a property that holds at any size: it equals the
    # dw accumulated over chunks of rows below 2^31 elements (the chunked
    # accumulation is pinned to the oracle at smaller sizes). Tolerance:
    # 1e-4 of sum_i |dy x r| per column (fp32 on the GPU, a scale only).
    dwc = torch.empty(H, device=DEV)
    bounds = [0, M // 3, 2 * M // 3, M]
    for i, (a, b) in enumerate(zip(bounds[:-1], bounds[1:])):
        rn.rmsnorm_bwd_ex(dy[a:b], x[a:b], w, rstd[a:b], dx=torch.empty_like(dy[a:b]),
                          dw=dwc, accumulate_dw=i > 0)
    scale = torch.zeros(H, device=DEV, dtype=torch.float64)
    for a in range(0, M, 65536):
        b = min(M, a + 65536)
        scale += (dy[a:b].float() * x[a:b].float() * rstd[a:b, None]).abs().sum(0).double()
    torch.cuda.synchronize()
    err = (dw.double() - dwc.double()).abs()
    assert bool((err <= 1e-4 * scale).all()), float((err / scale).max())
