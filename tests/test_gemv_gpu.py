"""GPU tier: RMSNorm fused with the projection GEMV (rmsnorm_gemv_fwd)
against the fp64 oracle.

The decode chain of the 0.8B Qwen decode article (trdm.cn news/483216,
§2.1 and §3.1: rms_norm, then the q/k/v or gate/up projections of a
[1, 896] hidden state; §6: fuse them) in one call: out = round(y) A^T with
y the norm's output as the separate norm would store it. Compared element
by element on every output (out, h, y, rstd) over dtypes, row counts that
fill one to four 16-row MMA tiles (and leave them ragged), feature counts,
output counts that leave the last 8-row tile of A ragged, with and without
the residual add, for the four kernels: the weight in registers (gemv.cuh,
forced with the row-wise path override), the weight fed by bulk copies
(gemv_tma.cuh), the product on tcgen05 with K split over a cluster
(gemv_umma.cuh) and the persistent product on tcgen05 with y held whole
per CTA (gemv_tc.cuh), each forced with its own override; a kernel whose
shared memory does not fit the call falls back to the next, and rows only
the K-split tcgen05 kernel holds are refused when a warp-level kernel is
forced. The automatic choice (bulk copies up to 8 rows; above them the
persistent tcgen05 kernel on wide rows with more tiles than SMs where y fits
one CTA, else the K-split one) is checked too, and so are projections with more 128-feature tiles than SMs
(each CTA of the persistent kernel takes several).
"""
import pytest
import torch

import oracle
from rmsnorm_fwd_bwd_02_gb300 import rmsnorm as rn
from rmsnorm_fwd_bwd_02_gb300 import workloads as W
from tests.tolerances import check_bits, check_rows, check_rstd

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
KERNELS = {"regs": rn.PATH_ROWS, "tma": rn.PATH_GEMV_TMA, "umma": rn.PATH_GEMV_UMMA,
           "tc": rn.PATH_GEMV_TC}


def umma_layout_bytes(T, H, KS, res):
    """Shared memory of one CTA of the tcgen05 kernel for T tokens, H
    features, K split over KS CTAs: its atoms (64 columns) of y, r (with the
    residual) and A (128 rows), the partial products received (over r when
    they fit there), w, 3 + atoms mbarriers, 16 bytes of words, the partial
    sums and rstd of T tokens, 1023 bytes of alignment."""
    na = (H + 63) // 64
    apc = (na + KS - 1) // KS
    rs = ((T // 4 + KS - 1) // KS) | 1
    y = apc * T * 128
    r = y if res else 0
    a = apc * 16384
    xchg = KS * 128 * rs * 16
    total = y + r + a + (0 if r >= xchg else xchg)
    return total + apc * 128 + 8 * (apc + 3) + 16 + 8 * T + 1023


def umma_fits(M, H, res=True):
    """Whether the tcgen05 kernel takes the call: at most 64 tokens, H a
    multiple of 16, and a cluster of at most 8 CTAs (no more than the atoms
    of K) whose shared memory fits in 227 KB."""
    T = (M + 15) // 16 * 16
    na = (H + 63) // 64
    return T <= 64 and H % 16 == 0 and any(
        umma_layout_bytes(T, H, ks, res) <= 227 * 1024 for ks in range(1, min(8, na) + 1))


def tc_layout_bytes(T, H, KS, nst, aps):
    """Shared memory of one CTA of the persistent tcgen05 kernel with K split
    over KS CTAs: its slice of y (atoms of T x 64 columns), the ring of A
    (nst stages of aps 16 KB atoms), its slice of w, with KS > 1 the
    exchange blocks (2 KS blocks of ceil(128 / KS) features x (T + 4) floats),
    2 nst + 14 mbarriers, 32 bytes of words, rstd, the CTA's sums and the
    per-atom partial sums of T tokens, 1023 bytes of alignment."""
    na = (H + 63) // 64
    apc = (na + KS - 1) // KS
    xbytes = 2 * KS * ((128 + KS - 1) // KS) * (T + 4) * 4 if KS > 1 else 0
    return (apc * T * 128 + nst * aps * 16384 + apc * 128 + xbytes + 8 * (2 * nst + 14) + 32
            + 8 * T + 4 * apc * T + 1023)


def tc_fits(M, H):
    """Whether the persistent tcgen05 kernel takes the call: at most 64
    tokens, H a multiple of 16, and for some cluster size (1 to 8, at most
    the atoms of K) a ring of two 16 KB stages in 227 KB."""
    T = (M + 15) // 16 * 16
    na = (H + 63) // 64
    return T <= 64 and H % 16 == 0 and any(
        ks <= na and tc_layout_bytes(T, H, ks, 2, 1) <= 227 * 1024 for ks in range(1, 9))


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.fail("the gpu tier needs a CUDA device")
    rn.lib()
    yield


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


def synth(M, H, N, dtype, seed, residual):
    g = torch.Generator().manual_seed(seed)
    d = {"x": torch.randn(M, H, generator=g) * 2.0,
         "w": 1.0 + 0.1 * torch.randn(H, generator=g),
         "A": torch.randn(N, H, generator=g) * 0.05}
    if residual:
        d["r"] = torch.randn(M, H, generator=g)
    if M > 1:
        d["x"] *= torch.logspace(-2, 2, M).unsqueeze(1)
    return {k: v.to(dtype).contiguous() for k, v in d.items()}


def run(inp, residual, eps=1e-6, want_y=True, static=False, kernel="tma"):
    g = {k: v.to(DEV) for k, v in inp.items()}
    torch.cuda.synchronize()             # the weights are in place before the call
    M, H = g["x"].shape
    y = torch.empty(M, H, device=DEV, dtype=g["x"].dtype) if want_y else None
    rstd = torch.empty(M, device=DEV)
    rn.set_path_override(KERNELS[kernel])
    try:
        out, h, _ = rn.rmsnorm_gemv_fwd(g["x"], g["w"], g["A"],
                                        r=g["r"] if residual else None, y=y,
                                        rstd=rstd, eps=eps, static_weights=static)
        path = rn.last_path()
    finally:
        rn.set_path_override(rn.PATH_AUTO)
    # a forced kernel runs where its shared memory fits; the bulk-copy kernel
    # falls back to the register one, the tcgen05 kernel to the other two
    if kernel == "regs":
        assert path == rn.PATH_GEMV, path
    elif kernel == "tma":
        assert path in (rn.PATH_GEMV, rn.PATH_GEMV_TMA), path
    elif kernel == "tc":
        if tc_fits(M, H):
            assert path == rn.PATH_GEMV_TC, (M, H, path)
        else:
            assert path in (rn.PATH_GEMV, rn.PATH_GEMV_TMA), (M, H, path)
    elif umma_fits(M, H, residual):
        assert path == rn.PATH_GEMV_UMMA, (M, H, path)
    else:
        assert path in (rn.PATH_GEMV, rn.PATH_GEMV_TMA), (M, H, path)
    torch.cuda.synchronize()
    return {"out": out, "h": h, "y": y, "rstd": rstd}


def oracle_all(orc, inp, residual, eps=1e-6):
    """The oracle's fused result plus the norm's unrounded output (the
    stored y is one rounding of it)."""
    r = inp["r"] if residual else None
    o = orc.rmsnorm_gemv(inp["x"], inp["w"], inp["A"], eps, r=r)
    if residual:
        _, o["y_exact"], _ = orc.residual_fwd(inp["x"], r, inp["w"], eps)
    else:
        o["y_exact"], _ = orc.fwd(inp["x"], inp["w"], eps)
    return o


def compare(name, got, o, dtype):
    check_rows(f"{name} out", got["out"], o["out"], dtype, o["tout"])
    check_rstd(f"{name} rstd", got["rstd"], o["rstd"])
    if got.get("y") is not None:
        check_rows(f"{name} y", got["y"], o["y_exact"], dtype)
    if o["h"] is not None:
        check_bits(f"{name} h", got["h"], o["h"])


@pytest.mark.parametrize("kernel", list(KERNELS))
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16], ids=["bf16", "f16"])
@pytest.mark.parametrize("M", [1, 7, 16, 17, 33, 64])
@pytest.mark.parametrize("H,N", [(128, 1), (128, 9), (896, 1024), (896, 2051),
                                 (1024, 13), (1664, 64), (896, 9728)])
def test_gemv_matches_oracle(orc, kernel, dtype, M, H, N):
    for residual in (False, True):
        inp = synth(M, H, N, dtype, seed=M * 7 + H + N, residual=residual)
        o = oracle_all(orc, inp, residual)
        for static in (False, True):
            got = run(inp, residual, static=static, kernel=kernel)
            compare(f"{kernel} {dtype} M={M} H={H} N={N} res={residual} static={static}",
                    got, o, dtype)


@pytest.mark.parametrize("kernel", list(KERNELS))
@pytest.mark.parametrize("H,M", [(4096, 16), (6720, 1), (6720, 16), (3424, 32),
                                 (2272, 48), (1664, 64)])
def test_gemv_largest_shared_memory(orc, kernel, H, M):
    """The largest y tile each row count allows (up to 227 KB of shared
    memory), after smaller calls of the same kernels have run; for the
    bulk-copy kernel, K is then streamed in slices."""
    small = synth(M, 128, 8, torch.bfloat16, seed=1, residual=False)
    run(small, False, kernel=kernel)
    inp = synth(M, H, 200, torch.bfloat16, seed=H, residual=True)
    o = oracle_all(orc, inp, True)
    compare(f"large {kernel} H={H} M={M}", run(inp, True, kernel=kernel), o,
            torch.bfloat16)


@pytest.mark.parametrize("H,M", [(4608, 32), (4096, 48), (3584, 64), (4096, 17)])
def test_gemv_widest_rows_tcgen05_only(orc, H, M):
    """Rows that only the tcgen05 kernels hold, with the residual: right
    through the K-split kernel and the automatic choice (the persistent
    kernel at these widths), and refused when a warp-level MMA kernel is
    forced."""
    inp = synth(M, H, 300, torch.bfloat16, seed=H + M, residual=True)
    assert umma_fits(M, H, True) and tc_fits(M, H)
    o = oracle_all(orc, inp, True)
    compare(f"widest tcgen05 H={H} M={M}", run(inp, True, kernel="umma"), o, torch.bfloat16)
    g = {k: v.to(DEV) for k, v in inp.items()}
    out, _, _ = rn.rmsnorm_gemv_fwd(g["x"], g["w"], g["A"], r=g["r"])
    torch.cuda.synchronize()
    assert rn.last_path() == rn.PATH_GEMV_TC       # the automatic choice at these widths
    check_rows(f"widest tcgen05 automatic H={H} M={M}", out, o["out"], torch.bfloat16, o["tout"])
    for forced in (rn.PATH_GEMV_TMA, rn.PATH_ROWS):
        rn.set_path_override(forced)
        try:
            with pytest.raises(rn.RmsNormError):
                rn.rmsnorm_gemv_fwd(g["x"], g["w"], g["A"], r=g["r"])
        finally:
            rn.set_path_override(rn.PATH_AUTO)


@pytest.mark.parametrize("name", ["decode-qkv-m1", "decode-gateup-m1"])
def test_decode_workloads_full(orc, name):
    wl = W.WORKLOADS[name]
    inp = W.make_inputs(wl)
    o = oracle_all(orc, inp, True, wl.eps)
    for kernel in KERNELS:
        got = run(inp, True, eps=wl.eps, static=True, kernel=kernel)
        compare(f"{name} {kernel}", got, o, wl.dtype)
    # the same at 8 and 64 decode rows
    for M in (8, 64):
        wm = wl.with_rows(M)
        im = W.make_inputs(wm)
        om = oracle_all(orc, im, True, wm.eps)
        for kernel in KERNELS:
            compare(f"{name} M={M} {kernel}", run(im, True, eps=wm.eps, kernel=kernel),
                    om, wm.dtype)


def test_automatic_choice():
    """Up to 8 rows the bulk-copy kernel (wherever its ring fits); above, the
    persistent tcgen05 kernel on rows of at least 2048 features; on narrower
    rows the K-split tcgen05 kernel wherever a cluster of it fits, else the
    persistent one, else the bulk-copy one."""
    for M, H, N in ((1, 896, 2048), (8, 896, 9728), (9, 896, 2048), (64, 896, 2048),
                    (64, 896, 9728), (16, 4096, 6144), (16, 4096, 24576), (9, 4096, 24576),
                    (17, 4096, 24576), (48, 4096, 512), (64, 4096, 512), (1, 6720, 64)):
        inp = synth(M, H, N, torch.bfloat16, seed=2, residual=True)
        g = {k: v.to(DEV) for k, v in inp.items()}
        rn.rmsnorm_gemv_fwd(g["x"], g["w"], g["A"], r=g["r"])
        want = (rn.PATH_GEMV_TC if M > 8 and H >= 2048 and tc_fits(M, H) else
                rn.PATH_GEMV_UMMA if M > 8 and umma_fits(M, H) else
                rn.PATH_GEMV_TC if M > 8 and tc_fits(M, H) else rn.PATH_GEMV_TMA)
        got = rn.last_path()
        if want == rn.PATH_GEMV_TMA and got == rn.PATH_GEMV:
            want = rn.PATH_GEMV          # no ring of the bulk-copy kernel fits either
        assert got == want, (M, H, N, got)
    torch.cuda.synchronize()


@pytest.mark.parametrize("kernel", list(KERNELS))
def test_y_matches_the_unfused_norm(kernel):
    """The fused kernels' y and h equal the residual forward's to within one
    ulp of y (the fp32 sums of squares run in a different order) and
    bit-exactly for h."""
    for dt in (torch.bfloat16, torch.float16):
        inp = synth(64, 896, 16, dt, seed=3, residual=True)
        got = run(inp, True, kernel=kernel)
        g = {k: v.to(DEV) for k, v in inp.items()}
        h, y, rstd = rn.rmsnorm_residual_fwd(g["x"], g["r"], g["w"])
        torch.cuda.synchronize()
        check_bits(f"{dt} h fused vs unfused", got["h"], h)
        a = got["y"].view(torch.int16).to(torch.int32).cpu()
        b = y.view(torch.int16).to(torch.int32).cpu()
        assert int((a - b).abs().max()) <= 1, f"{dt}: fused y > 1 ulp from unfused"


def test_deterministic_and_optional_outputs(orc):
    inp = synth(17, 896, 2048, torch.bfloat16, seed=5, residual=True)
    a = run(inp, True)
    b = run(inp, True)
    c = run(inp, True, static=True)
    for k in ("out", "h", "y", "rstd"):
        check_bits(f"run-to-run {k}", a[k], b[k])
        check_bits(f"static weights {k}", c[k], a[k])
    # the other kernels: the same h bits; y within one ulp (their norms run
    # the fp32 sums in other orders); each deterministic too
    forced = {}
    for other in ("regs", "umma", "tc"):
        d = forced[other] = run(inp, True, kernel=other)
        check_bits(f"{other} vs tma h", d["h"], a["h"])
        ya = a["y"].view(torch.int16).to(torch.int32).cpu()
        yd = d["y"].view(torch.int16).to(torch.int32).cpu()
        assert int((ya - yd).abs().max()) <= 1, f"{other} vs tma y: more than 1 ulp apart"
        e = run(inp, True, kernel=other)
        for k in ("out", "h", "y", "rstd"):
            check_bits(f"{other} run-to-run {k}", e[k], d[k])
    # no y, no h, no rstd: out unchanged (the automatic choice at 17 rows of
    # 896 is the K-split tcgen05 kernel)
    g = {k: v.to(DEV) for k, v in inp.items()}
    out, h, rstd = rn.rmsnorm_gemv_fwd(g["x"], g["w"], g["A"], r=g["r"], want_h=False)
    torch.cuda.synchronize()
    assert rn.last_path() == rn.PATH_GEMV_UMMA
    assert h is None and rstd is None
    check_bits("out without optional outputs", out, forced["umma"]["out"])


def test_guard_words_untouched(orc):
    M, H, N, G = 5, 896, 1003, 64
    inp = synth(M, H, N, torch.float16, seed=8, residual=True)
    g = {k: v.to(DEV) for k, v in inp.items()}

    def guarded(n, dtype):
        b = torch.empty(n + 2 * G, device=DEV, dtype=dtype)
        b.view(torch.int16 if dtype != torch.float32 else torch.int32).fill_(0x7E5A)
        return b, b[G:G + n]

    bo, out = guarded(M * N, torch.float16)
    bh, h = guarded(M * H, torch.float16)
    by, y = guarded(M * H, torch.float16)
    br, rstd = guarded(M, torch.float32)
    rn.rmsnorm_gemv_fwd(g["x"], g["w"], g["A"], r=g["r"], out=out.view(M, N),
                        h=h.view(M, H), y=y.view(M, H), rstd=rstd)
    torch.cuda.synchronize()
    for b, n, nm in ((bo, M * N, "out"), (bh, M * H, "h"), (by, M * H, "y"),
                     (br, M, "rstd")):
        it = torch.int32 if b.dtype == torch.float32 else torch.int16
        head, tail = b[:G].view(it), b[G + n:].view(it)
        assert bool((head == 0x7E5A).all()) and bool((tail == 0x7E5A).all()), \
            f"{nm}: guard words overwritten"
    o = oracle_all(orc, inp, True)
    compare("guarded", {"out": out.view(M, N), "h": h.view(M, H), "y": y.view(M, H),
                        "rstd": rstd}, o, torch.float16)


@pytest.mark.parametrize("rows", [1, 24])
def test_cuda_graph_replay(orc, rows):
    """Captured once and replayed with new activations copied into the
    static inputs (the decode loop of the article's §4): one row (the
    bulk-copy kernel) and 24 rows (the tcgen05 kernel, whose tensor maps
    are captured with the launch)."""
    wl = W.WORKLOADS["decode-qkv-m1"].with_rows(rows)
    inp = W.make_inputs(wl)
    g = {k: v.to(DEV) for k, v in inp.items()}
    out = torch.empty(rows, wl.N, device=DEV, dtype=wl.dtype)
    h = torch.empty_like(g["x"])
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        rn.rmsnorm_gemv_fwd(g["x"], g["w"], g["A"], r=g["r"], out=out, h=h, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        rn.rmsnorm_gemv_fwd(g["x"], g["w"], g["A"], r=g["r"], out=out, h=h,
                            static_weights=True)
    assert rn.last_path() == (rn.PATH_GEMV_TMA if rows == 1 else rn.PATH_GEMV_UMMA)
    for step in range(3):
        x2 = (torch.randn(rows, wl.H, generator=torch.Generator().manual_seed(step))
              ).to(wl.dtype)
        g["x"].copy_(x2.to(DEV))
        graph.replay()
        torch.cuda.synchronize()
        o = orc.rmsnorm_gemv(x2, inp["w"], inp["A"], wl.eps, r=inp["r"])
        check_rows(f"graph step {step} out", out, o["out"], wl.dtype, o["tout"])
        check_bits(f"graph step {step} h", h, o["h"])


def test_error_returns():
    lib = rn.lib()
    s = torch.cuda.current_stream().cuda_stream
    x = torch.randn(65, 896, device=DEV, dtype=torch.bfloat16)
    w = torch.ones(896, device=DEV, dtype=torch.bfloat16)
    A = torch.randn(64, 896, device=DEV, dtype=torch.bfloat16)
    out = torch.empty(65, 64, device=DEV, dtype=torch.bfloat16)
    P = lambda t: None if t is None else t.data_ptr()  # noqa: E731

    def call(x=x, r=None, w=w, A=A, out=out, h=None, y=None, M=1, H=896, N=64,
             dtype=rn.RMSNORM_BF16, flags=0):
        return lib.rmsnorm_gemv_fwd(P(x) if hasattr(x, "data_ptr") else x, P(r),
                                    P(w), P(A) if hasattr(A, "data_ptr") else A,
                                    P(out) if hasattr(out, "data_ptr") else out,
                                    P(h), P(y), None, M, H, N, 1e-6, dtype, flags, s)
    assert call(flags=2) == -11
    assert call(M=65) == -7                  # beyond 64 rows
    assert call(H=900) == -7                 # H not a multiple of 32
    assert call(M=64, H=16384) == -7         # y tile beyond shared memory
    assert call(dtype=rn.RMSNORM_F32) == -7
    assert call(N=0) == -2
    assert call(h=x) == -1                   # h without r
    assert call(A=A.data_ptr() + 2) == -5
    assert call(out=x.data_ptr()) == -9      # out over x
    assert call(r=x, h=x) == -9              # h over x (every CTA reads x)
    assert call(M=0) == 0
    torch.cuda.synchronize()


def test_gemv_wait_runs_out_and_context_survives(orc):
    """Every bulk-copy wait of the weight ring runs out (each stage expects 16
    bytes that no copy delivers, 20 ms limit): the kernel records it, drains
    its copies and ends, and the next normal call is right."""
    inp = synth(3, 896, 1024, torch.bfloat16, seed=4, residual=True)
    rn.wait_timeouts(reset=True)
    rn.set_stream_test_fault(16, 20000)
    try:
        run(inp, True)                   # results incomplete by design
        torch.cuda.synchronize()
    finally:
        rn.set_stream_test_fault(0, 0)
    assert rn.wait_timeouts(reset=True) > 0
    o = oracle_all(orc, inp, True)
    compare("after timeouts", run(inp, True), o, torch.bfloat16)
    assert rn.wait_timeouts() == 0


def test_umma_wait_runs_out_and_context_survives(orc):
    """Every copy of A into the tcgen05 kernel's ring is made to wait for 16
    bytes no copy delivers (20 ms limit): the waits run out, are counted, the
    copies in flight are let land, the tensor memory is freed, and the next
    call is right."""
    inp = synth(40, 896, 1000, torch.bfloat16, seed=11, residual=True)
    rn.wait_timeouts(reset=True)
    rn.set_stream_test_fault(16, 20000)
    try:
        run(inp, True, kernel="umma")             # results incomplete by design
        torch.cuda.synchronize()
    finally:
        rn.set_stream_test_fault(0, 0)
    assert rn.wait_timeouts(reset=True) > 0
    o = oracle_all(orc, inp, True)
    compare("umma after timeouts", run(inp, True, kernel="umma"), o, torch.bfloat16)
    assert rn.wait_timeouts() == 0


@pytest.mark.parametrize("M,H,N", [(16, 4096, 24576), (64, 896, 40000), (33, 896, 20001),
                                   (9, 128, 50000), (1, 896, 38913), (32, 4096, 24576),
                                   (64, 4096, 600), (48, 6720, 300), (16, 16384, 1000),
                                   (24, 2048, 30000), (40, 1024, 3000)])
def test_tc_many_tiles_per_cta(orc, M, H, N):
    """The persistent kernel over shapes that make its planner take each
    cluster size (1 to 8 CTAs splitting K, which exchange partial products
    per tile) and, with more tiles than clusters, several tiles per
    cluster: its weight ring running on across tiles, its four accumulators
    in turn, the exchange's flow control wrapping round; ragged last
    tiles; rows only it holds (64 x 4096, 48 x 6720, 16 x 16384); against
    the oracle, and the same bits run to run."""
    assert tc_fits(M, H)
    for residual in (True, False):
        inp = synth(M, H, N, torch.bfloat16, seed=M + H + N, residual=residual)
        o = oracle_all(orc, inp, residual)
        a = run(inp, residual, static=True, kernel="tc")
        compare(f"tc many tiles M={M} H={H} N={N} res={residual}", a, o, torch.bfloat16)
        b = run(inp, residual, kernel="tc")
        for k in ("out", "h", "y", "rstd"):
            if a[k] is not None:
                check_bits(f"tc run-to-run {k}", b[k], a[k])


def test_tc_wait_runs_out_and_context_survives(orc):
    """Every copy of A into the persistent kernel's ring is made to wait for
    16 bytes no copy delivers (20 ms limit): a wait runs out, every role
    stops, the copies in flight land and the MMAs finish before the tensor
    memory is freed, one timeout per CTA is counted, and the next call is
    right."""
    inp = synth(40, 896, 40000, torch.bfloat16, seed=12, residual=True)
    rn.wait_timeouts(reset=True)
    rn.set_stream_test_fault(16, 20000)
    try:
        run(inp, True, kernel="tc")               # results incomplete by design
        torch.cuda.synchronize()
    finally:
        rn.set_stream_test_fault(0, 0)
    assert rn.wait_timeouts(reset=True) > 0
    o = oracle_all(orc, inp, True)
    compare("tc after timeouts", run(inp, True, kernel="tc"), o, torch.bfloat16)
    assert rn.wait_timeouts() == 0


def test_tc_cluster_wait_runs_out_and_context_survives(orc):
    """The same with K split over a cluster (rows of 4096 features run in
    clusters of 4): the waits on A's copies run out, the CTAs stop their
    exchanges, wait (bounded) for anything still landing in them, meet at
    the final cluster barrier and free their tensor memory; the timeouts are
    counted and the next call is right."""
    inp = synth(16, 4096, 6144, torch.bfloat16, seed=13, residual=True)
    rn.wait_timeouts(reset=True)
    rn.set_stream_test_fault(16, 20000)
    try:
        run(inp, True, kernel="tc")               # results incomplete by design
        torch.cuda.synchronize()
    finally:
        rn.set_stream_test_fault(0, 0)
    assert rn.wait_timeouts(reset=True) > 0
    o = oracle_all(orc, inp, True)
    compare("tc cluster after timeouts", run(inp, True, kernel="tc"), o, torch.bfloat16)
    assert rn.wait_timeouts() == 0


def test_tc_graph_replay(orc):
    """The persistent kernel (forced) captured in a CUDA graph with its tensor
    maps and replayed with new activations copied into the static inputs."""
    wl = W.WORKLOADS["decode-gateup-m1"].with_rows(24)
    inp = W.make_inputs(wl)
    g = {k: v.to(DEV) for k, v in inp.items()}
    out = torch.empty(24, wl.N, device=DEV, dtype=wl.dtype)
    h = torch.empty_like(g["x"])
    rn.set_path_override(rn.PATH_GEMV_TC)
    try:
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            rn.rmsnorm_gemv_fwd(g["x"], g["w"], g["A"], r=g["r"], out=out, h=h, stream=s)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            rn.rmsnorm_gemv_fwd(g["x"], g["w"], g["A"], r=g["r"], out=out, h=h,
                                static_weights=True)
        assert rn.last_path() == rn.PATH_GEMV_TC
    finally:
        rn.set_path_override(rn.PATH_AUTO)
    for step in range(3):
        x2 = (torch.randn(24, wl.H, generator=torch.Generator().manual_seed(step + 9))
              ).to(wl.dtype)
        g["x"].copy_(x2.to(DEV))
        graph.replay()
        torch.cuda.synchronize()
        o = orc.rmsnorm_gemv(x2, inp["w"], inp["A"], wl.eps, r=inp["r"])
        check_rows(f"tc graph step {step} out", out, o["out"], wl.dtype, o["tout"])
        check_bits(f"tc graph step {step} h", h, o["h"])


@pytest.mark.parametrize("ks", [1, 2, 3, 4, 5, 6, 7, 8])
def test_tc_every_cluster_size(orc, ks):
    """The persistent kernel with K split over clusters of every size 1-8
    (forced with the test hook): sizes that do not divide the 128 features
    of a tile leave the last owner fewer; several tiles per cluster, ragged
    N, 16 to 48 tokens, with and without the residual."""
    rn.set_gemv_cluster_test(ks)
    try:
        for M, H, N, residual in ((16, 2048, 3000, True), (33, 4096, 2050, False),
                                  (48, 1024, 5000, True)):
            T = (M + 15) // 16 * 16
            if (H + 63) // 64 < ks or tc_layout_bytes(T, H, ks, 2, 1) > 227 * 1024:
                continue                 # this size does not fit the call
            assert tc_fits(M, H)
            inp = synth(M, H, N, torch.bfloat16, seed=ks * 100 + M, residual=residual)
            got = run(inp, residual, kernel="tc")
            compare(f"tc clusters of {ks} M={M} H={H} N={N}", got, oracle_all(orc, inp, residual),
                    torch.bfloat16)
    finally:
        rn.set_gemv_cluster_test(0)
