"""Write tests/golden/oracle_small_cases.json from the fp64 oracle alone.

The inputs are fixed small patterns written out below (no random numbers),
so the file pins the oracle's results across machines and over time: a later
change to the oracle's arithmetic that moves these numbers must regenerate
the file, and its commit names the passage of the pages that justifies it.
Calls nothing but oracle/.

    python tests/golden/make_oracle_golden.py
"""
import json
import os
import sys

import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.dirname(
    os.path.abspath(__file__)))))
import oracle  # noqa: E402

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)),
                   "oracle_small_cases.json")


def pattern_inputs(M, H, dtype):
    """x_ij = ((7i + 3j) mod 11 - 5) / 4, r_ij = ((5i + 2j) mod 9 - 4) / 8,
    dy_ij = ((3i + 5j) mod 13 - 6) / 16, dh_ij = ((i + j) mod 5 - 2) / 32,
    w_j = 1 + (j mod 5) / 8: all exact in bf16, fp32 and fp64."""
    i = torch.arange(M, dtype=torch.float64)[:, None]
    j = torch.arange(H, dtype=torch.float64)[None, :]
    x = (torch.remainder(7 * i + 3 * j, 11) - 5) / 4
    r = (torch.remainder(5 * i + 2 * j, 9) - 4) / 8
    dy = (torch.remainder(3 * i + 5 * j, 13) - 6) / 16
    dh = (torch.remainder(i + j, 5) - 2) / 32
    w = 1 + torch.remainder(torch.arange(H, dtype=torch.float64), 5) / 8
    return [t.to(dtype).contiguous() for t in (x, r, dy, dh, w)]


def cases():
    o = oracle.get()
    out = []
    for name, dtype in (("f64", torch.float64), ("f32", torch.float32),
                        ("bf16", torch.bfloat16)):
        for (M, H, eps) in ((3, 8, 1e-6), (2, 5, 0.5), (1, 1, 1e-6)):
            x, r, dy, dh, w = pattern_inputs(M, H, dtype)
            y, rstd = o.fwd(x, w, eps)
            dx, dw = o.bwd(dy, x, w, eps)
            h, hy, hrstd = o.residual_fwd(x, r, w, eps)
            hdx, hdw = o.residual_bwd(dy, dh, h, w, eps)
            out.append({
                "dtype": name, "M": M, "H": H, "eps": eps,
                "y": y.flatten().tolist(), "rstd": rstd.tolist(),
                "dx": dx.flatten().tolist(), "dw": dw.tolist(),
                "h": h.double().flatten().tolist(),
                "resid_y": hy.flatten().tolist(), "resid_rstd": hrstd.tolist(),
                "resid_dx": hdx.flatten().tolist(), "resid_dw": hdw.tolist(),
            })
    return out


if __name__ == "__main__":
    with open(OUT, "w") as f:
        json.dump({"generator": "tests/golden/make_oracle_golden.py",
                   "cases": cases()}, f, indent=1)
        f.write("\n")
    print(OUT)
