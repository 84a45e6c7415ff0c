"""Pins for the fp64 CPU oracle: checks against what the pages and the
mathematics fix, never against the oracle itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError
on a violation. ``tests/test_oracle_pins.py`` runs them on the real oracle;
``tests/test_oracle_mutants.py`` runs them on copies of the oracle with a
planted mistake and requires every mutant to fail at least one pin.

Sources:
  [P1] "训推加速 Qwen3 实战：从“调包”到手写 Triton Kernel（含 backward）"
       §4.1 (definition), §5.3 (backward derivation), §5.6 (gradcheck in
       double on a (2, 32) input with eps 1e-6)
  [P2] article on 21 hand-written Triton kernels for a 0.8B Qwen decoder
       (trdm.cn, news/483216) §2.1, §3.2-3.3 (residual add; split sums)
"""
import math

import torch

F64 = torch.float64


def _close(a, b, rtol, atol=0.0, what=""):
    a = torch.as_tensor(a, dtype=F64)
    b = torch.as_tensor(b, dtype=F64)
    err = (a - b).abs()
    bound = atol + rtol * b.abs()
    if not bool((err <= bound).all()):
        i = int(torch.argmax(err - bound))
        raise AssertionError(
            f"{what}: |a-b| = {float(err.flatten()[i]):.3e} > "
            f"{float(bound.flatten()[i]):.3e} at flat index {i} "
            f"(a={float(a.flatten()[i])!r}, b={float(b.flatten()[i])!r})")


def _gen(seed):
    return torch.Generator().manual_seed(seed)


# ----------------------------------------------------------------- formats

def pin_bf16_decode(o):
    """bfloat16 bit patterns decode to the values the binary32 layout gives
    (sign, 8-bit exponent with bias 127, 7 stored fraction bits)."""
    cases = {
        0x3F80: 1.0, 0xBF80: -1.0, 0x4049: 3.140625, 0xC2F7: -123.5,
        0x0080: 2.0 ** -126, 0x0001: 2.0 ** -133, 0x8000: -0.0,
        0x7F7F: (2.0 - 2.0 ** -7) * 2.0 ** 127, 0x7F80: math.inf,
        0xFF80: -math.inf,
    }
    for bits, want in cases.items():
        got = o.bf16_to_double(bits)
        assert got == want, f"decode {bits:#06x}: {got!r} != {want!r}"
    assert math.isnan(o.bf16_to_double(0x7FC0))


def pin_bf16_round_hand_cases(o):
    """Round-to-nearest-even to bfloat16, on ties and edges worked by hand."""
    one = 1.0
    u = 2.0 ** -7                     # bf16 spacing just above 1.0
    cases = [
        (one + u / 2, 0x3F80),        # tie between 1 and 1+u: even is 1
        (one + 3 * u / 2, 0x3F82),    # tie between 1+u and 1+2u: even is 1+2u
        (one + u / 2 + 2.0 ** -30, 0x3F81),  # just above the tie: up
        (one + u / 2 - 2.0 ** -30, 0x3F80),  # just below the tie: down
        (-(one + u / 2), 0xBF80),
        (2.0 ** -134, 0x0000),        # half the smallest subnormal: tie to 0
        (3 * 2.0 ** -134, 0x0002),    # 1.5 x smallest subnormal: tie to 2
        (2.0 ** -134 + 2.0 ** -160, 0x0001),
        ((2.0 - 2.0 ** -8) * 2.0 ** 127, 0x7F80),   # tie max/2^128: inf
        ((2.0 - 2.0 ** -7) * 2.0 ** 127, 0x7F7F),   # the largest finite
        (1e300, 0x7F80), (-1e300, 0xFF80),
        (0.0, 0x0000),
    ]
    for v, want in cases:
        got = o.bf16_from_double(v)
        assert got == want, f"round({v!r}) = {got:#06x}, want {want:#06x}"


def pin_bf16_round_vs_library(o):
    """On binary32 inputs (where one rounding step is unambiguous) the
    oracle's rounding equals torch's float32 -> bfloat16 conversion, which is
    round-to-nearest-even; covers normals, subnormals and huge values."""
    g = _gen(11)
    parts = [
        torch.randn(4000, generator=g),
        torch.randn(2000, generator=g) * 1e-38,          # bf16 subnormals
        torch.randn(2000, generator=g) * 3e38 / 4,
        (torch.randint(0, 2 ** 16, (3000,), generator=g, dtype=torch.int32)
         .to(torch.int16).view(torch.bfloat16).float()
         + torch.randn(3000, generator=g) * 1e-3),
    ]
    # exact ties in binary32: bf16 value + half its spacing
    base = torch.randn(2000, generator=g).to(torch.bfloat16).float()
    bits = base.view(torch.int32) | 0x8000
    parts.append(bits.view(torch.float32))
    xs = torch.cat(parts)
    xs = xs[torch.isfinite(xs)]
    want = xs.to(torch.bfloat16).view(torch.int16).to(torch.int32) & 0xFFFF
    for v, w in zip(xs.tolist(), want.tolist()):
        got = o.bf16_from_double(v)
        assert got == w, f"round({v!r}) = {got:#06x}, library {w:#06x}"


def pin_f16_decode(o):
    """IEEE binary16 bit patterns decode to the values of their layout (sign,
    5-bit exponent with bias 15, 10 stored fraction bits, subnormals at
    multiples of 2^-24), worked by hand."""
    cases = {
        0x3C00: 1.0, 0xBC00: -1.0, 0x4248: 3.140625, 0xD7B8: -123.5,
        0x0400: 2.0 ** -14, 0x0001: 2.0 ** -24, 0x03FF: 1023 * 2.0 ** -24,
        0x8000: -0.0, 0x7BFF: 65504.0, 0x3555: 1365 * 2.0 ** -12,
        0x7C00: math.inf, 0xFC00: -math.inf,
    }
    for bits, want in cases.items():
        got = o.f16_to_double(bits)
        assert got == want, f"f16 decode {bits:#06x}: {got!r} != {want!r}"
    assert math.copysign(1.0, o.f16_to_double(0x8000)) == -1.0
    assert math.isnan(o.f16_to_double(0x7E00))


def pin_f16_round_hand_cases(o):
    """Round-to-nearest-even to binary16 on ties and edges worked by hand."""
    u = 2.0 ** -10                    # f16 spacing just above 1.0
    cases = [
        (1.0 + u / 2, 0x3C00),        # tie between 1 and 1+u: even is 1
        (1.0 + 3 * u / 2, 0x3C02),    # tie between 1+u and 1+2u: 1+2u
        (1.0 + u / 2 + 2.0 ** -40, 0x3C01),
        (1.0 + u / 2 - 2.0 ** -40, 0x3C00),
        (-(1.0 + 3 * u / 2), 0xBC02),
        (2.0 ** -25, 0x0000),         # half the smallest subnormal: tie to 0
        (3 * 2.0 ** -25, 0x0002),     # 1.5 x smallest subnormal: tie to 2
        (2.0 ** -25 + 2.0 ** -50, 0x0001),
        (1023.5 * 2.0 ** -24, 0x0400),  # largest subnormal + half: to 2^-14
        (65504.0, 0x7BFF), (65519.99, 0x7BFF),
        (65520.0, 0x7C00),            # tie between 65504 and 2^16: inf
        (1e300, 0x7C00), (-1e300, 0xFC00),
        (2049.0, 0x6800),             # tie between 2048 and 2050: 2048
        (2051.0, 0x6802),             # tie between 2050 and 2052: 2052
        (0.0, 0x0000), (-0.0, 0x8000),
    ]
    for v, want in cases:
        got = o.f16_from_double(v)
        assert got == want, f"f16 round({v!r}) = {got:#06x}, want {want:#06x}"


def pin_f16_round_vs_library(o):
    """On binary32 inputs the oracle's binary16 rounding equals torch's
    float32 -> float16 conversion (round-to-nearest-even): normals,
    subnormals, values near the overflow threshold and exact ties."""
    g = _gen(16)
    parts = [
        torch.randn(4000, generator=g),
        torch.randn(2000, generator=g) * 3e-6,           # f16 subnormals
        torch.randn(2000, generator=g) * 6e4,            # near overflow
        (torch.randint(0, 0x7C00, (3000,), generator=g, dtype=torch.int32)
         .to(torch.int16).view(torch.float16).float()
         * (1 + torch.randn(3000, generator=g) * 1e-3)),
    ]
    # exact ties: an f16 value + half its spacing (13 float32 bits below)
    base = (torch.randn(2000, generator=g) * 100).to(torch.float16).float()
    base = base[base.abs() >= 2.0 ** -14]                 # normals only
    bits = base.view(torch.int32) | 0x1000
    parts.append(bits.view(torch.float32))
    xs = torch.cat(parts)
    xs = xs[torch.isfinite(xs)]
    want = xs.to(torch.float16).view(torch.int16).to(torch.int32) & 0xFFFF
    for v, w in zip(xs.tolist(), want.tolist()):
        got = o.f16_from_double(v)
        assert got == w, f"f16 round({v!r}) = {got:#06x}, library {w:#06x}"


def pin_f16_fwd_reads_f16(o):
    """The forward decodes fp16 storage: on fp16 inputs it equals the fp64
    forward applied to the same values widened (exactly) by torch."""
    g = _gen(17)
    x = (torch.randn(5, 96, generator=g) * 3).to(torch.float16)
    x.view(-1)[::31] = torch.tensor(6e-6, dtype=torch.float16)   # subnormals
    w = (1.0 + 0.1 * torch.randn(96, generator=g)).to(torch.float16)
    y, rstd = o.fwd(x, w, 1e-6)
    yd, rd = o.fwd(x.double(), w.double(), 1e-6)
    _close(y, yd, 0.0, what="f16 y")
    _close(rstd, rd, 0.0, what="f16 rstd")
    dy = torch.randn(5, 96, generator=g).to(torch.float16)
    dx, dw = o.bwd(dy, x, w, 1e-6)
    dxd, dwd = o.bwd(dy.double(), x.double(), w.double(), 1e-6)
    _close(dx, dxd, 0.0, what="f16 dx")
    _close(dw, dwd, 0.0, what="f16 dw")


# ----------------------------------------------------------------- forward

def pin_fwd_constant_row(o):
    """Constant row x_j = a: mean(x^2) = a^2, so r = 1/sqrt(a^2 + eps) and
    y_j = w_j * a * r ([P1 §4.1] with the mean worked out by hand)."""
    g = _gen(1)
    for H in (1, 7, 32, 896):
        w = 1.0 + 0.1 * torch.randn(H, generator=g, dtype=F64)
        for a in (-3.0, 0.5, 1e-3, 96.0):
            for eps in (0.0, 1e-6, 0.25):
                x = torch.full((2, H), a, dtype=F64)
                y, rstd = o.fwd(x, w, eps)
                r = 1.0 / math.sqrt(a * a + eps)
                _close(rstd, torch.full((2,), r, dtype=F64), 1e-14,
                       what=f"const rstd H={H} a={a} eps={eps}")
                _close(y, (w * a * r).expand(2, H), 1e-14, 1e-300,
                       what=f"const y H={H} a={a} eps={eps}")
    # in bfloat16 storage (a and w exactly representable)
    H = 896
    w = torch.tensor([1.0 + (j % 5) / 8 for j in range(H)]).to(torch.bfloat16)
    x = torch.full((1, H), -2.5).to(torch.bfloat16)
    y, rstd = o.fwd(x, w, 1e-6)
    r = 1.0 / math.sqrt(6.25 + 1e-6)
    _close(rstd, [r], 1e-14, what="const bf16 rstd")
    _close(y[0], w.double() * -2.5 * r, 1e-14, what="const bf16 y")


def pin_fwd_worked_examples(o):
    """Small rows worked by hand from [P1 §4.1]."""
    # x = (3, 4, 0, 0): mean(x^2) = 25/4, r = 2/5, y = w * x * 2/5
    x = torch.tensor([[3.0, 4.0, 0.0, 0.0]], dtype=F64)
    w = torch.tensor([1.0, 2.0, 3.0, 4.0], dtype=F64)
    y, rstd = o.fwd(x, w, 0.0)
    _close(rstd, [0.4], 1e-15, what="(3,4,0,0) rstd")
    _close(y[0], [1.2, 3.2, 0.0, 0.0], 1e-15, 1e-300, what="(3,4,0,0) y")
    # x = (1, -1, 1, -1): r = 1, y = w * x
    x = torch.tensor([[1.0, -1.0, 1.0, -1.0]], dtype=F64)
    y, rstd = o.fwd(x, w, 0.0)
    _close(y[0], [1.0, -2.0, 3.0, -4.0], 0.0, what="(1,-1,1,-1) y")
    # x = (1, 1), eps = 3: r = 1/sqrt(1 + 3) = 1/2
    x = torch.tensor([[1.0, 1.0]], dtype=F64)
    y, rstd = o.fwd(x, torch.tensor([5.0, -6.0], dtype=F64), 3.0)
    _close(rstd, [0.5], 0.0, what="eps=3 rstd")
    _close(y[0], [2.5, -3.0], 0.0, what="eps=3 y")
    # H = 1: y = w x / sqrt(x^2 + eps)
    x = torch.tensor([[-2.0], [0.75]], dtype=F64)
    y, rstd = o.fwd(x, torch.tensor([3.0], dtype=F64), 0.25)
    _close(y[:, 0], [3.0 * -2.0 / math.sqrt(4.25), 3.0 * 0.75 / math.sqrt(0.8125)],
           1e-15, what="H=1 y")


def pin_fwd_unit_rms(o):
    """With w = 1 and eps = 0 every output row has mean(y^2) = 1; a wrong
    divisor (H-1, a padded block size) or a misplaced square root breaks it."""
    g = _gen(2)
    for H in (1, 5, 128, 896, 1000):
        x = torch.randn(3, H, generator=g, dtype=F64) * 3.0
        y, _ = o.fwd(x, torch.ones(H, dtype=F64), 0.0)
        _close((y * y).mean(dim=1), torch.ones(3, dtype=F64), 1e-13,
               what=f"unit rms H={H}")


def pin_fwd_scale_invariance(o):
    """At eps = 0: y(a x) = sign(a) y(x) and rstd(a x) = rstd(x) / |a|."""
    g = _gen(3)
    H = 96
    x = torch.randn(4, H, generator=g, dtype=F64)
    w = 1.0 + 0.1 * torch.randn(H, generator=g, dtype=F64)
    y0, r0 = o.fwd(x, w, 0.0)
    for a in (2.0 ** -3, 3.0, 1024.0, -2.0):
        y1, r1 = o.fwd(x * a, w, 0.0)
        _close(y1, math.copysign(1.0, a) * y0, 1e-14, 1e-300,
               what=f"scale y a={a}")
        _close(r1, r0 / abs(a), 1e-14, what=f"scale rstd a={a}")


def pin_fwd_rows_independent(o):
    """Each row is normalised on its own: the batch result equals the
    row-by-row results, and rows scaled differently stay distinct."""
    g = _gen(4)
    M, H = 5, 33
    x = torch.randn(M, H, generator=g, dtype=F64) * torch.arange(
        1, M + 1, dtype=F64)[:, None] ** 2
    w = 1.0 + 0.1 * torch.randn(H, generator=g, dtype=F64)
    y, rstd = o.fwd(x, w, 1e-6)
    for i in range(M):
        yi, ri = o.fwd(x[i:i + 1].contiguous(), w, 1e-6)
        _close(y[i], yi[0], 0.0, what=f"row {i} y")
        _close(rstd[i:i + 1], ri, 0.0, what=f"row {i} rstd")
    # weight applies per feature, not per position reversed or shifted
    x1 = torch.zeros(1, H, dtype=F64)
    x1[0, 3] = 1.0
    y1, _ = o.fwd(x1, w, 0.0)
    want = torch.zeros(H, dtype=F64)
    want[3] = w[3] * math.sqrt(H)      # mean(x^2) = 1/H
    _close(y1[0], want, 1e-14, 1e-300, what="one-hot row")


# ---------------------------------------------------------------- backward

def _loss(o, x, w, dy, eps):
    y, _ = o.fwd(x, w, eps)
    return float((dy * y).sum())


def pin_bwd_finite_differences(o):
    """Central differences of L = sum(dy * y) in double, for dx and dw, on the
    page's gradcheck shape (2, 32) and smaller odd shapes ([P1 §5.6])."""
    g = _gen(5)
    for (M, H, eps) in ((2, 32, 1e-6), (3, 7, 1e-6), (2, 2, 0.25),
                        (1, 1, 0.25), (3, 5, 0.25)):
        x = torch.randn(M, H, generator=g, dtype=F64)
        w = 1.0 + 0.3 * torch.randn(H, generator=g, dtype=F64)
        dy = torch.randn(M, H, generator=g, dtype=F64)
        dx, dw = o.bwd(dy, x, w, eps)
        h = 1e-6
        fd = torch.empty(M, H, dtype=F64)
        for i in range(M):
            for j in range(H):
                xp = x.clone(); xp[i, j] += h
                xm = x.clone(); xm[i, j] -= h
                fd[i, j] = (_loss(o, xp, w, dy, eps)
                            - _loss(o, xm, w, dy, eps)) / (2 * h)
        _close(dx, fd, 1e-6, 1e-7, what=f"FD dx M={M} H={H} eps={eps}")
        fdw = torch.empty(H, dtype=F64)
        for j in range(H):
            wp = w.clone(); wp[j] += h
            wm = w.clone(); wm[j] -= h
            fdw[j] = (_loss(o, x, wp, dy, eps) - _loss(o, x, wm, dy, eps)) / (2 * h)
        _close(dw, fdw, 1e-6, 1e-7, what=f"FD dw M={M} H={H} eps={eps}")


def pin_bwd_vs_autograd(o):
    """The backward agrees with torch autograd differentiating the forward
    definition in float64 (an independent derivation of [P1 §5.3])."""
    g = _gen(6)
    for (M, H, eps) in ((4, 64, 1e-6), (2, 9, 0.5)):
        x = torch.randn(M, H, generator=g, dtype=F64, requires_grad=True)
        w = (1.0 + 0.1 * torch.randn(H, generator=g, dtype=F64)).requires_grad_()
        dy = torch.randn(M, H, generator=g, dtype=F64)
        y = w * x * torch.rsqrt((x * x).mean(dim=1, keepdim=True) + eps)
        y.backward(dy)
        dx, dw = o.bwd(dy, x.detach(), w.detach(), eps)
        _close(dx, x.grad, 1e-12, 1e-14, what=f"autograd dx H={H}")
        _close(dw, w.grad, 1e-12, 1e-14, what=f"autograd dw H={H}")


def pin_bwd_orthogonality(o):
    """sum_j x_j dx_j = eps r^3 sum_j w_j dy_j x_j per row (this follows from
    the derivative of r in [P1 §5.3]); at eps = 0, with any w (including the
    all-ones weight), it vanishes."""
    g = _gen(7)
    for H in (7, 896):
        x = torch.randn(3, H, generator=g, dtype=F64)
        w = 1.0 + 0.1 * torch.randn(H, generator=g, dtype=F64)
        dy = torch.randn(3, H, generator=g, dtype=F64)
        for eps in (0.0, 0.3):
            dx, _ = o.bwd(dy, x, w, eps)
            _, r = o.fwd(x, w, eps)
            lhs = (x * dx).sum(dim=1)
            rhs = eps * r ** 3 * (w * dy * x).sum(dim=1)
            scale = (x * dx).abs().sum(dim=1) + rhs.abs()
            _close(lhs - rhs, torch.zeros(3, dtype=F64), 0.0,
                   float(scale.max()) * 1e-13, what=f"x.dx H={H} eps={eps}")
        dx1, _ = o.bwd(dy, x, torch.ones(H, dtype=F64), 0.0)
        s = (x * dx1).sum(dim=1)
        _close(s, torch.zeros(3, dtype=F64), 0.0,
               float((x * dx1).abs().sum(dim=1).max()) * 1e-13,
               what=f"x.dx w=1 H={H}")


def pin_bwd_h1(o):
    """H = 1: y = w x / sqrt(x^2 + eps), so dy/dx = w eps / (x^2 + eps)^(3/2)
    and dL/dw = dy * x / sqrt(x^2 + eps)."""
    x = torch.tensor([[0.5], [-1.5], [2.0]], dtype=F64)
    w = torch.tensor([1.25], dtype=F64)
    dy = torch.tensor([[1.0], [-2.0], [0.5]], dtype=F64)
    eps = 0.3
    dx, dw = o.bwd(dy, x, w, eps)
    xs = x[:, 0]
    want_dx = dy[:, 0] * 1.25 * eps / (xs * xs + eps) ** 1.5
    want_dw = (dy[:, 0] * xs / torch.sqrt(xs * xs + eps)).sum()
    _close(dx[:, 0], want_dx, 1e-14, what="H=1 dx")
    _close(dw, want_dw.reshape(1), 1e-14, what="H=1 dw")


def pin_bwd_dw_structure(o):
    """dw is a sum over rows: splitting the rows adds up, permuting them
    leaves it unchanged, and one row gives dy_j x_j r ([P1 §5.3])."""
    g = _gen(8)
    M, H = 6, 40
    x = torch.randn(M, H, generator=g, dtype=F64)
    w = 1.0 + 0.1 * torch.randn(H, generator=g, dtype=F64)
    dy = torch.randn(M, H, generator=g, dtype=F64)
    _, dw = o.bwd(dy, x, w, 1e-6)
    _, dw_a = o.bwd(dy[:2].contiguous(), x[:2].contiguous(), w, 1e-6)
    _, dw_b = o.bwd(dy[2:].contiguous(), x[2:].contiguous(), w, 1e-6)
    _close(dw, dw_a + dw_b, 1e-13, 1e-15, what="dw split")
    p = torch.randperm(M, generator=g)
    _, dw_p = o.bwd(dy[p].contiguous(), x[p].contiguous(), w, 1e-6)
    _close(dw, dw_p, 1e-13, 1e-15, what="dw permuted")
    _, r = o.fwd(x[:1].contiguous(), w, 1e-6)
    _, dw1 = o.bwd(dy[:1].contiguous(), x[:1].contiguous(), w, 1e-6)
    _close(dw1, dy[0] * x[0] * r[0], 1e-14, 1e-300, what="dw one row")


def pin_bwd_error_scales(o):
    """The error scales bound the results (triangle inequality) and take
    their closed forms on a constant row with w = dy = 1:
    dx = eps r^3, tdx = r + a^2 r^3; with dy = x, tdw = dw = sum_i x^2 r."""
    g = _gen(9)
    M, H = 4, 50
    x = torch.randn(M, H, generator=g, dtype=F64)
    w = 1.0 + 0.1 * torch.randn(H, generator=g, dtype=F64)
    dy = torch.randn(M, H, generator=g, dtype=F64)
    dx, dw, tdx, tdw = o.bwd(dy, x, w, 1e-6, want_terms=True)
    assert bool((dx.abs() <= tdx * (1 + 1e-14)).all()), "tdx < |dx|"
    assert bool((dw.abs() <= tdw * (1 + 1e-14)).all()), "tdw < |dw|"
    a, eps = 1.5, 0.2
    xc = torch.full((1, H), a, dtype=F64)
    ones = torch.ones(H, dtype=F64)
    dxc, _, tdxc, _ = o.bwd(torch.ones(1, H, dtype=F64), xc, ones, eps,
                            want_terms=True)
    r = 1.0 / math.sqrt(a * a + eps)
    _close(dxc[0], torch.full((H,), eps * r ** 3, dtype=F64), 1e-12,
           what="const dx")
    _close(tdxc[0], torch.full((H,), r + a * a * r ** 3, dtype=F64), 1e-14,
           what="const tdx")
    _, dwx, _, tdwx = o.bwd(x.clone(), x, w, 1e-6, want_terms=True)
    _close(tdwx, dwx, 1e-14, what="tdw = dw when dy = x")


# ------------------------------------------------------- residual variant

def pin_residual_h_exact(o):
    """h = round(x + r) in the stored dtype: for bf16 it equals torch's
    float32 add followed by its round-to-nearest-even bf16 conversion (the
    float32 add of two bf16 values cannot round to a different bf16 result);
    the same holds for fp16 (binary32 carries at least 2 x 11 + 2 bits, so
    rounding the float32 sum again to binary16 is the single rounding); for
    float32 it equals torch's float32 add; for float64 it is x + r."""
    g = _gen(12)
    M, H = 8, 200
    for dt in (torch.bfloat16, torch.float16, torch.float32):
        x = torch.randn(M, H, generator=g)
        r = torch.randn(M, H, generator=g)
        x.view(-1)[::97] *= 100.0                  # outliers
        r.view(-1)[5::89] *= -1e-4                 # far-apart magnitudes
        x, r = x.to(dt), r.to(dt)
        w = (1.0 + 0.1 * torch.randn(H, generator=g)).to(dt)
        h, _, _ = o.residual_fwd(x, r, w, 1e-6)
        want = (x.float() + r.float()).to(dt)
        half = dt in (torch.bfloat16, torch.float16)
        assert torch.equal(h.view(torch.int16) if half else h,
                           want.view(torch.int16) if half else want), \
            f"h not exact for {dt}"
    x = torch.randn(2, 9, generator=g, dtype=F64)
    r = torch.randn(2, 9, generator=g, dtype=F64)
    h, _, _ = o.residual_fwd(x, r, torch.ones(9, dtype=F64), 0.0)
    _close(h, x + r, 0.0, what="h f64")


def pin_residual_fwd_on_stored_h(o):
    """The norm of the residual variant acts on the stored (rounded) h."""
    g = _gen(13)
    M, H = 4, 64
    x = torch.randn(M, H, generator=g).to(torch.bfloat16)
    r = torch.randn(M, H, generator=g).to(torch.bfloat16)
    w = (1.0 + 0.1 * torch.randn(H, generator=g)).to(torch.bfloat16)
    h, y, rstd = o.residual_fwd(x, r, w, 1e-6)
    hd = h.double()
    want_r = 1.0 / torch.sqrt((hd * hd).mean(dim=1) + 1e-6)
    _close(rstd, want_r, 1e-14, what="resid rstd")
    _close(y, w.double() * hd * want_r[:, None], 1e-14, 1e-300, what="resid y")


def pin_residual_bwd_finite_differences(o):
    """For L(x, r) = sum(dy * y(x + r)) + sum(dh * (x + r)), central
    differences in x and in r both give the residual backward's dx."""
    g = _gen(14)
    M, H, eps = 2, 6, 0.1
    x = torch.randn(M, H, generator=g, dtype=F64)
    r = torch.randn(M, H, generator=g, dtype=F64)
    w = 1.0 + 0.2 * torch.randn(H, generator=g, dtype=F64)
    dy = torch.randn(M, H, generator=g, dtype=F64)
    for dh in (None, torch.randn(M, H, generator=g, dtype=F64)):
        def loss(xx, rr):
            hh, yy, _ = o.residual_fwd(xx, rr, w, eps)
            val = float((dy * yy).sum())
            if dh is not None:
                val += float((dh * hh).sum())
            return val
        h, _, _ = o.residual_fwd(x, r, w, eps)
        dx, _ = o.residual_bwd(dy, dh, h, w, eps)
        step = 1e-6
        for which in ("x", "r"):
            fd = torch.empty(M, H, dtype=F64)
            for i in range(M):
                for j in range(H):
                    ap, am = x.clone(), x.clone()
                    bp, bm = r.clone(), r.clone()
                    if which == "x":
                        ap[i, j] += step; am[i, j] -= step
                    else:
                        bp[i, j] += step; bm[i, j] -= step
                    fd[i, j] = (loss(ap, bp) - loss(am, bm)) / (2 * step)
            _close(dx, fd, 1e-6, 1e-7,
                   what=f"resid FD d{which} dh={'yes' if dh is not None else 'no'}")


def pin_residual_dh_none_is_zero(o):
    g = _gen(15)
    M, H = 3, 16
    h = torch.randn(M, H, generator=g, dtype=F64)
    w = torch.randn(H, generator=g, dtype=F64)
    dy = torch.randn(M, H, generator=g, dtype=F64)
    a = o.residual_bwd(dy, None, h, w, 1e-6)
    b = o.residual_bwd(dy, torch.zeros(M, H, dtype=F64), h, w, 1e-6)
    _close(a[0], b[0], 0.0, what="dh None dx")
    _close(a[1], b[1], 0.0, what="dh None dw")
    c = o.bwd(dy, h, w, 1e-6)
    _close(a[0], c[0], 0.0, what="resid bwd = bwd on h")


# ------------------------------------------------------- double backward

def _l2(o, dy, x, w, gx, gw, eps):
    dx, dw = o.bwd(dy, x, w, eps)
    return float((gx * dx).sum() + (gw * dw).sum())


def pin_bwd_bwd_finite_differences(o):
    """Central differences of L2 = sum(gx dx) + sum(gw dw), with (dx, dw)
    from the (pinned) backward, in every element of dy, x and w."""
    g = _gen(31)
    M, H, eps = 2, 6, 0.1
    dy = torch.randn(M, H, generator=g, dtype=F64)
    x = torch.randn(M, H, generator=g, dtype=F64)
    w = 1.0 + 0.3 * torch.randn(H, generator=g, dtype=F64)
    gx = torch.randn(M, H, generator=g, dtype=F64)
    gw = torch.randn(H, generator=g, dtype=F64)
    ddy, dx2, dw2 = o.bwd_bwd(dy, x, w, gx, gw, eps)
    step = 1e-6
    for name, t, got in (("dy", dy, ddy), ("x", x, dx2), ("w", w, dw2)):
        fd = torch.empty_like(t)
        flat = t.view(-1)
        for k in range(flat.numel()):
            keep = float(flat[k])
            flat[k] = keep + step
            lp = _l2(o, dy, x, w, gx, gw, eps)
            flat[k] = keep - step
            lm = _l2(o, dy, x, w, gx, gw, eps)
            flat[k] = keep
            fd.view(-1)[k] = (lp - lm) / (2 * step)
        _close(got, fd, 1e-6, 1e-8, what=f"double backward FD d{name}")


def pin_bwd_bwd_vs_autograd(o):
    """torch's float64 double backward of the definition y = w x r (r from
    mean(x^2) + eps), through autograd with create_graph."""
    g = _gen(32)
    M, H, eps = 3, 32, 1e-6
    dy = torch.randn(M, H, generator=g, dtype=F64)
    x = torch.randn(M, H, generator=g, dtype=F64)
    w = 1.0 + 0.1 * torch.randn(H, generator=g, dtype=F64)
    gx = torch.randn(M, H, generator=g, dtype=F64)
    gw = torch.randn(H, generator=g, dtype=F64)
    dyr, xr, wr = (t.clone().requires_grad_() for t in (dy, x, w))
    y = wr * xr / torch.sqrt((xr * xr).mean(dim=1, keepdim=True) + eps)
    dx, dw = torch.autograd.grad(y, (xr, wr), dyr, create_graph=True)
    l2 = (gx * dx).sum() + (gw * dw).sum()
    a_dy, a_x, a_w = torch.autograd.grad(l2, (dyr, xr, wr))
    ddy, dx2, dw2 = o.bwd_bwd(dy, x, w, gx, gw, eps)
    _close(ddy, a_dy, 1e-11, 1e-13, what="double backward ddy vs autograd")
    _close(dx2, a_x, 1e-11, 1e-13, what="double backward dx vs autograd")
    _close(dw2, a_w, 1e-11, 1e-13, what="double backward dw vs autograd")


def pin_bwd_bwd_linear_and_zero(o):
    """The result is linear in (gx, gw) and zero without them; each error
    scale bounds its value."""
    g = _gen(33)
    M, H = 3, 16
    dy = torch.randn(M, H, generator=g, dtype=F64)
    x = torch.randn(M, H, generator=g, dtype=F64)
    w = torch.randn(H, generator=g, dtype=F64)
    gx = torch.randn(M, H, generator=g, dtype=F64)
    gw = torch.randn(H, generator=g, dtype=F64)
    z = o.bwd_bwd(dy, x, w, None, None, 1e-6)
    for t in z:
        _close(t, torch.zeros_like(t), 0.0, what="double backward without gradients")
    a = o.bwd_bwd(dy, x, w, gx, None, 1e-6)
    b = o.bwd_bwd(dy, x, w, None, gw, 1e-6)
    ab = o.bwd_bwd(dy, x, w, gx, gw, 1e-6, want_terms=True)
    for i in range(3):
        _close(ab[i], a[i] + b[i], 1e-12, 1e-15, what=f"double backward linearity {i}")
        assert bool((ab[i].abs() <= ab[3 + i] * (1 + 1e-12) + 1e-300).all()), \
            f"double backward error scale {i} below |value|"


# ------------------------------------------- norm, then projection (decode)

def _round_like(o, v, dtype):
    """v (float64 tensor) rounded element by element to bf16/fp16 with the
    oracle's pinned rounding, returned as float64."""
    f = o.bf16_from_double if dtype == torch.bfloat16 else o.f16_from_double
    d = o.bf16_to_double if dtype == torch.bfloat16 else o.f16_to_double
    return torch.tensor([d(f(x)) for x in v.flatten().tolist()],
                        dtype=F64).reshape(v.shape)


def pin_gemv_closed_form(o):
    """Rows x_i = a_i s_i with s_i in {-1, +1}^H and eps = 0 have rms a_i, so
    y = w s exactly; with small-integer w and A the output is the integer
    product (w s) A^T, computed here with torch int64 ([P2 §3.1] shapes
    shrunk: M = 3 rows, N = 5 outputs, H = 32)."""
    g = _gen(21)
    M, H, N = 3, 32, 5
    s = torch.randint(0, 2, (M, H), generator=g) * 2 - 1
    a = torch.tensor([2.0, 0.5, 8.0])
    x = (a[:, None] * s).to(torch.bfloat16)
    wi = torch.randint(-4, 5, (H,), generator=g)
    Ai = torch.randint(-3, 4, (N, H), generator=g)
    d = o.rmsnorm_gemv(x, wi.to(torch.bfloat16), Ai.to(torch.bfloat16), 0.0)
    want = ((wi[None, :] * s) @ Ai.T).to(F64)
    _close(d["out"], want, 0.0, what="gemv closed form")
    _close(d["y"].double(), (wi[None, :] * s).to(F64), 0.0, what="gemv y")
    _close(d["rstd"], 1.0 / a.double(), 1e-15, what="gemv rstd")


def pin_gemv_vs_library(o):
    """out = round(y) A^T with y the (pinned) forward's output rounded by the
    (pinned) rounding and the product taken by torch in float64; tout =
    |round(y)| |A|^T; the stored y is that rounding; for bf16 and fp16."""
    g = _gen(22)
    M, H, N = 4, 48, 7
    for dt in (torch.bfloat16, torch.float16):
        x = (torch.randn(M, H, generator=g) * 3).to(dt)
        w = (1.0 + 0.1 * torch.randn(H, generator=g)).to(dt)
        A = (torch.randn(N, H, generator=g) * 0.05).to(dt)
        d = o.rmsnorm_gemv(x, w, A, 1e-6)
        y, _ = o.fwd(x, w, 1e-6)
        yq = _round_like(o, y, dt)
        _close(d["y"].double(), yq, 0.0, what=f"gemv stored y {dt}")
        want = yq @ A.double().T
        mag = yq.abs() @ A.double().abs().T
        _close(d["out"], want, 1e-12, 1e-300, what=f"gemv out {dt}")
        _close(d["tout"], mag, 1e-12, what=f"gemv tout {dt}")


def pin_gemv_identity_weight(o):
    """With A = I (N = H) the output is the stored y itself."""
    g = _gen(23)
    H = 40
    x = torch.randn(3, H, generator=g).to(torch.float16)
    w = (1.0 + 0.1 * torch.randn(H, generator=g)).to(torch.float16)
    d = o.rmsnorm_gemv(x, w, torch.eye(H).to(torch.float16), 1e-6)
    _close(d["out"], d["y"].double(), 0.0, what="gemv identity")
    y, _ = o.fwd(x, w, 1e-6)
    _close(d["out"], _round_like(o, y, torch.float16), 0.0,
           what="gemv identity = rounded forward")


def pin_gemv_residual_composes(o):
    """The residual variant writes the residual forward's h and projects
    the norm of that stored h: the same as the plain variant applied to h."""
    g = _gen(24)
    M, H, N = 3, 64, 6
    x = torch.randn(M, H, generator=g).to(torch.bfloat16)
    r = torch.randn(M, H, generator=g).to(torch.bfloat16)
    w = (1.0 + 0.1 * torch.randn(H, generator=g)).to(torch.bfloat16)
    A = torch.randn(N, H, generator=g).to(torch.bfloat16)
    d = o.rmsnorm_gemv(x, w, A, 1e-6, r=r)
    h, _, _ = o.residual_fwd(x, r, w, 1e-6)
    assert torch.equal(d["h"].view(torch.int16), h.view(torch.int16)), "gemv h"
    e = o.rmsnorm_gemv(h, w, A, 1e-6)
    _close(d["out"], e["out"], 0.0, what="gemv residual out")
    _close(d["rstd"], e["rstd"], 0.0, what="gemv residual rstd")


def pin_gemv_permutations(o):
    """Permuting the rows of A permutes the output columns the same way;
    rows of x are independent."""
    g = _gen(25)
    M, H, N = 4, 24, 9
    x = torch.randn(M, H, generator=g).to(torch.bfloat16)
    w = (1.0 + 0.1 * torch.randn(H, generator=g)).to(torch.bfloat16)
    A = torch.randn(N, H, generator=g).to(torch.bfloat16)
    d = o.rmsnorm_gemv(x, w, A, 1e-6)
    p = torch.randperm(N, generator=g)
    e = o.rmsnorm_gemv(x, w, A[p].contiguous(), 1e-6)
    _close(e["out"], d["out"][:, p], 0.0, what="gemv column permutation")
    q = torch.randperm(M, generator=g)
    f = o.rmsnorm_gemv(x[q].contiguous(), w, A, 1e-6)
    _close(f["out"], d["out"][q], 0.0, what="gemv row permutation")


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]


def failing_pins(o):
    """Names of the pins that fail on oracle ``o`` (used by the mutant test)."""
    bad = []
    for p in ALL_PINS:
        try:
            p(o)
        except AssertionError:
            bad.append(p.__name__)
    return bad


__all__ = ["ALL_PINS", "failing_pins"] + [p.__name__ for p in ALL_PINS]
