"""CPU tier: the oracle built on this machine reproduces the stored drift pin
tests/golden/oracle_small_cases.json (written by make_oracle_golden.py from
the oracle alone; see tests/golden/README.md)."""
import json
import os

import pytest
import torch

import oracle
from tests.golden.make_oracle_golden import pattern_inputs

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                      "oracle_small_cases.json")
DTYPES = {"f64": torch.float64, "f32": torch.float32, "bf16": torch.bfloat16}


def _cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _cases(),
                         ids=lambda c: f"{c['dtype']}-{c['M']}x{c['H']}")
def test_oracle_matches_golden(case):
    o = oracle.get()
    M, H, eps = case["M"], case["H"], case["eps"]
    x, r, dy, dh, w = pattern_inputs(M, H, DTYPES[case["dtype"]])
    y, rstd = o.fwd(x, w, eps)
    dx, dw = o.bwd(dy, x, w, eps)
    h, hy, hrstd = o.residual_fwd(x, r, w, eps)
    hdx, hdw = o.residual_bwd(dy, dh, h, w, eps)
    got = {"y": y, "rstd": rstd, "dx": dx, "dw": dw, "h": h.double(),
           "resid_y": hy, "resid_rstd": hrstd, "resid_dx": hdx, "resid_dw": hdw}
    for k, v in got.items():
        want = torch.tensor(case[k], dtype=torch.float64)
        torch.testing.assert_close(v.flatten(), want, rtol=1e-15, atol=1e-300,
                                   msg=lambda m, k=k: f"{k}: {m}")
