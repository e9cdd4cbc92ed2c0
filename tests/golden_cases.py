"""Load the hand-derived fixtures in ``tests/golden`` as tensors.

Every fixture is tiny (head_dim 2).  ``pad_d`` embeds it in a wider head by
appending zero columns to q, k and v: the dot products and therefore the
weights do not change, and the extra output columns are exactly 0.  That lets
the same fixtures run through the CUDA library, which serves head_dim 128
and 256.
"""
from __future__ import annotations

import glob
import json
import math
import os

import torch

GOLDEN_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def fixture_names():
    return sorted(os.path.splitext(os.path.basename(p))[0]
                  for p in glob.glob(os.path.join(GOLDEN_DIR, "*.json")))


def _pad(x: torch.Tensor, d: int) -> torch.Tensor:
    if x.shape[-1] == d:
        return x
    pad = torch.zeros(x.shape[:-1] + (d - x.shape[-1],), dtype=x.dtype)
    return torch.cat([x, pad], dim=-1)


def load(name: str, pad_d: int | None = None):
    with open(os.path.join(GOLDEN_DIR, name + ".json")) as f:
        fx = json.load(f)
    d0 = len(fx["q"][0][0][0])
    d = pad_d or d0
    q = _pad(torch.tensor(fx["q"], dtype=torch.float64), d)
    if fx.get("int8"):
        k = _pad(torch.tensor(fx["k"], dtype=torch.int8), d)
        v = _pad(torch.tensor(fx["v"], dtype=torch.int8), d)
        ks = torch.tensor(fx["k_scale"], dtype=torch.float32)
        vs = torch.tensor(fx["v_scale"], dtype=torch.float32)
    else:
        k = _pad(torch.tensor(fx["k"], dtype=torch.float64), d).to(torch.bfloat16)
        v = _pad(torch.tensor(fx["v"], dtype=torch.float64), d).to(torch.bfloat16)
        ks = vs = None
    q16 = q.to(torch.bfloat16)
    assert torch.equal(q16.double(), q), "fixture q must be bf16-exact"
    env = {"e": math.e, "__builtins__": {}}
    exp = torch.tensor([[[[eval(s, env) for s in row] for row in heads]
                         for heads in rows] for rows in fx["expected"]],
                       dtype=torch.float64)
    exp = _pad(exp, d)
    out = dict(fx)
    out.update(q=q16, k=k, v=v, k_scale=ks, v_scale=vs, expected=exp, d=d)
    if "kv_lengths" in fx:
        out["kv_lengths"] = torch.tensor(fx["kv_lengths"], dtype=torch.int32)
    if "idx" in fx:
        out["idx"] = torch.tensor(fx["idx"], dtype=torch.int32)
    return out
