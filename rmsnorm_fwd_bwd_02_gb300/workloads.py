"""Seeded synthetic inputs for the RMSNorm workloads.

The only module shared by the CUDA path's tests/benchmark and the oracle's
checks. It draws random numbers and nothing else: no normalisation, no
reduction, none of the method's arithmetic.

Shapes and distributions are those of the Qwen3 workloads the RMSNorm pages
work on ("训推加速 Qwen3 实战：从“调包”到手写 Triton Kernel（含 backward）" §4.4
and §6.2: bf16 activations of batch 4-8 x 4096 tokens x hidden 4096; the
decode article on a 0.8B Qwen model, trdm.cn news/483216 §1: hidden 896, one
token at a time). Every tensor is drawn on the CPU from its own
``torch.Generator`` seed, in float32, scaled, then rounded once to the
storage dtype. Outlier entries ("0.1 % of entries x50 / x100") are exactly
``round(0.001 * numel)`` positions drawn without replacement by numpy's
PCG64 generator, scaled in float32 before the rounding.
"""
from dataclasses import dataclass, replace

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    H: int
    dtype: torch.dtype
    eps: float = 1e-6
    seed: int = 0
    dy_std: float = 1.0
    outlier_frac: float = 0.0      # fraction of x (and r) entries scaled
    outlier_scale: float = 1.0
    residual: bool = False         # also draw r (residual) and dh_out
    backward: bool = True          # the workload runs the backward too
    ld: int = 0                    # row stride of every [M, H] tensor (0: H)
    N: int = 0                     # rows of a projection weight A [N, H] that
                                   # the norm feeds (fused norm + GEMV); 0: none
    double_backward: bool = False  # the step is the double backward
    note: str = ""

    def with_rows(self, M: int) -> "Workload":
        return replace(self, M=int(M), name=f"{self.name}[M={M}]")

    def with_features(self, H: int) -> "Workload":
        return replace(self, H=int(H), name=f"{self.name}[H={H}]")

    @property
    def elem_bytes(self) -> int:
        return torch.empty(0, dtype=self.dtype).element_size()

    @property
    def row_stride(self) -> int:
        return self.ld or self.H


WORKLOADS = {
    w.name: w for w in [
        Workload("tiny-fp32", 64, 896, torch.float32, seed=0, dy_std=1.0,
                 note="tiny reference case: x, dy ~ N(0,1), w ~ 1+0.1N(0,1)"),
        Workload("decode-m1", 1, 896, torch.bfloat16, seed=1, outlier_frac=1e-3,
                 outlier_scale=50.0, backward=False,
                 note="decode split-row, one token"),
        Workload("decode-m8", 8, 896, torch.bfloat16, seed=1, outlier_frac=1e-3,
                 outlier_scale=50.0, backward=False,
                 note="decode split-row, 8 tokens"),
        Workload("decode-m64", 64, 896, torch.bfloat16, seed=1,
                 outlier_frac=1e-3, outlier_scale=50.0, backward=False,
                 note="decode split-row, 64 tokens"),
        Workload("qwen3-8b-train", 32768, 4096, torch.bfloat16, seed=2,
                 dy_std=1e-2,
                 note="Qwen3-8B training shape, batch 8 x seq 4096, hidden 4096"),
        Workload("qwen3-qknorm", 524288, 128, torch.bfloat16, seed=3,
                 dy_std=1e-2,
                 note="Qwen3 QK-norm: 4 x 4096 tokens x 32 heads, head_dim 128, "
                      "one shared weight"),
        Workload("residual-14b", 16384, 5120, torch.bfloat16, seed=4,
                 dy_std=1e-2, outlier_frac=1e-3, outlier_scale=100.0,
                 residual=True,
                 note="fused residual-add + RMSNorm at Qwen3-14B width"),
        Workload("qwen3-8b-train-fp16", 32768, 4096, torch.float16, seed=2,
                 dy_std=1e-2,
                 note="the Qwen3-8B training shape with fp16 storage"),
        Workload("qwen3-8b-train-strided", 32768, 4096, torch.bfloat16, seed=2,
                 dy_std=1e-2, ld=4608,
                 note="the Qwen3-8B training shape, every [M, H] tensor the "
                      "first 4096 columns of an [M, 4608] buffer"),
        Workload("qwen3-8b-train-bwd2", 32768, 4096, torch.bfloat16, seed=2,
                 dy_std=1e-2, double_backward=True,
                 note="double backward at the Qwen3-8B training shape: gradients "
                      "gx ~ N(0, 1e-2) on dx and gw ~ N(0, 1e-3) (fp32) on dw"),
        Workload("decode-qkv-m1", 1, 896, torch.bfloat16, seed=5,
                 outlier_frac=1e-3, outlier_scale=50.0, residual=True,
                 backward=False, N=2048,
                 note="one decode token: residual add + RMSNorm + the stacked "
                      "q|k|v projection (1024 + 512 + 512 rows of 896)"),
        Workload("decode-gateup-m1", 1, 896, torch.bfloat16, seed=6,
                 outlier_frac=1e-3, outlier_scale=50.0, residual=True,
                 backward=False, N=9728,
                 note="one decode token: residual add + RMSNorm + the stacked "
                      "gate|up projection (2 x 4864 rows of 896)"),
        Workload("decode-8b-qkv-m16", 16, 4096, torch.bfloat16, seed=7,
                 outlier_frac=1e-3, outlier_scale=50.0, residual=True,
                 backward=False, N=6144,
                 note="16 decode tokens at Qwen3-8B width: residual add + RMSNorm "
                      "+ the stacked q|k|v projection (4096 + 1024 + 1024 rows "
                      "of 4096)"),
        Workload("decode-8b-gateup-m16", 16, 4096, torch.bfloat16, seed=8,
                 outlier_frac=1e-3, outlier_scale=50.0, residual=True,
                 backward=False, N=24576,
                 note="16 decode tokens at Qwen3-8B width: residual add + RMSNorm "
                      "+ the stacked gate|up projection (2 x 12288 rows of 4096)"),
    ]
}


def _normal(shape, seed, std=1.0, mean=0.0):
    g = torch.Generator().manual_seed(int(seed))
    t = torch.randn(shape, generator=g, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    if mean != 0.0:
        t.add_(mean)
    return t


def _outliers(t, seed, frac, scale):
    """Scale exactly round(frac * numel) distinct entries of t (in place)."""
    n = t.numel()
    k = int(round(frac * n))
    if k == 0:
        return t
    idx = np.random.default_rng(int(seed)).choice(n, size=k, replace=False)
    flat = t.view(-1)
    flat[torch.from_numpy(idx.astype(np.int64))] *= scale
    return t


def make_inputs(w: Workload) -> dict:
    """CPU tensors for workload ``w``: x, w (weight), dy, with
    ``w.residual`` also r and dh (the incoming gradient of the residual
    stream), with ``w.N`` the projection weight A [N, H], and with
    ``w.double_backward`` the incoming gradients gx [M, H] (dtype) and gw [H]
    (float32). Same seed, same values, on every machine with the same torch
    random generator."""
    base = 1000 * w.seed
    shape = (w.M, w.H)
    x = _normal(shape, base + 1)
    if w.outlier_frac:
        _outliers(x, base + 11, w.outlier_frac, w.outlier_scale)
    out = {"x": x}
    out["w"] = _normal((w.H,), base + 2, std=0.1, mean=1.0)
    out["dy"] = _normal(shape, base + 3, std=w.dy_std)
    if w.residual:
        r = _normal(shape, base + 4)
        if w.outlier_frac:
            _outliers(r, base + 14, w.outlier_frac, w.outlier_scale)
        out["r"] = r
        out["dh"] = _normal(shape, base + 5, std=w.dy_std)
    if w.N:
        # a projection weight at the usual initialisation scale
        out["A"] = _normal((w.N, w.H), base + 6, std=0.02)
    if w.double_backward:
        out["gx"] = _normal(shape, base + 7, std=w.dy_std)
    res = {k: v.to(w.dtype).contiguous() for k, v in out.items()}
    if w.double_backward:
        res["gw"] = _normal((w.H,), base + 8, std=1e-3)      # fp32, as dw is
    return res


def in_strided(t, ld: int, fill=float("nan")):
    """A copy of the [M, H] tensor t (on t's device) as the first H columns
    of a new [M, ld] buffer whose other columns hold ``fill``; returns the
    [M, H] view (row stride ld)."""
    M, H = t.shape
    buf = torch.full((M, ld), fill, dtype=t.dtype, device=t.device)
    view = buf[:, :H]
    view.copy_(t)
    return view


def random_rows(M: int, k: int, seed: int = 0):
    """k distinct row indices in [0, M) including the first and last rows
    (for sampled parity checks at full size)."""
    k = min(k, M)
    rng = np.random.default_rng(seed)
    pick = set([0, M - 1])
    if M > 2:
        pick.update(rng.choice(M, size=max(0, k - 2), replace=False).tolist())
    return sorted(pick)[:max(k, min(2, M))]
