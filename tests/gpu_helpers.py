"""Shared helpers for the GPU parity tests (inputs from datagen, expected values from the oracle)."""
from __future__ import annotations

import numpy as np

import datagen
import oracle
from oracle import rounding
from oracle import tra as otra

# Tolerances ("EinDecomp ... tensor relational algebra" gives none; the bar is
# 1e-5 relative for fp32 CUDA-core semirings and 2e-2 of max|ref| for BF16-input
# tensor-core paths).  Relative to what, per element:
#   sum of products : |g - r| <= 1e-5 * sum|x*y|   (forward-error scale of a sum)
#   squared distance: |g - r| <= 1e-5 * |r|        (all terms are >= 0)
#   logsumexp       : |g - r| <= 1e-5 * max(|r|, 1)
#   max / min       : bit-exact (an fp32 add is exact in double; one rounding)
#   BF16 inputs     : |g - r| <= 2e-2 * max|r|, plus |g - r| <= 1e-4 * sum|x*y|
FP32_REL = 1e-5
BF16_MAX_REL = 2e-2
BF16_SUM_REL = 1e-4


def torch_mod():
    import torch

    return torch


def to_dev(a: np.ndarray):
    torch = torch_mod()
    if a.dtype == np.uint16:
        t = torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(a))
    return t.cuda()


def from_dev(t) -> np.ndarray:
    torch = torch_mod()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def as_f64(a: np.ndarray) -> np.ndarray:
    if a.dtype == np.uint16:
        return rounding.bf16_bits_to_f32(a).astype(np.float64)
    return a.astype(np.float64)


def empty(n, bf16: bool):
    torch = torch_mod()
    return torch.empty(n, dtype=torch.bfloat16 if bf16 else torch.float32, device="cuda")


def gen(shape, seed, tensor, dist="normal", bf16=False, a=None, b=None):
    if dist == "uniform":
        lo, hi = (-1.0 if a is None else a), (1.0 if b is None else b)
        return datagen.uniform_bf16(shape, seed, tensor, lo, hi) if bf16 else datagen.uniform_f32(shape, seed, tensor, lo, hi)
    mu, sig = (0.0 if a is None else a), (1.0 if b is None else b)
    return datagen.normal_bf16(shape, seed, tensor, mu, sig) if bf16 else datagen.normal_f32(shape, seed, tensor, mu, sig)


def relation_on_device(lib, dense: np.ndarray, d):
    """Dense host tensor -> device relation under d (the library's repartition kernel)."""
    src = to_dev(dense).reshape(-1)
    if all(v == 1 for v in d):
        return src
    dst = torch_mod().empty_like(src)
    lib.repartition(src, dst, list(dense.shape), [1] * dense.ndim, list(d))
    return dst


def run_plan(lib, spec, bounds, d, X, Y=None, out_bf16=False, workspace=True):
    """Execute one plan on dense host inputs; returns (plan, dense host output as float64)."""
    torch = torch_mod()
    p = lib.Plan(spec, bounds, d)
    rx = len(p.operands[0])
    xd = relation_on_device(lib, X, d[:rx])
    yd = relation_on_device(lib, Y, d[rx:]) if Y is not None else None
    zshape = p.shape("z")
    z = empty(int(np.prod(zshape)), out_bf16)
    ws = None
    if workspace and p.workspace_bytes:
        ws = torch.empty(p.workspace_bytes, dtype=torch.uint8, device="cuda")
    p.execute(xd, yd, z, ws)
    lib.ein_status()
    zb = from_dev(z)
    return p, as_f64(otra.unblock(zb, zshape, p.dvec("z")))


def check_sum(g, r, S, rel):
    bad = np.abs(g - r) > rel * S + 1e-30
    assert not bad.any(), f"{bad.sum()} outside {rel}*S; worst {np.max(np.abs(g - r) / (S + 1e-30)):.3e}"


def check_rel(g, r, rel, floor=0.0):
    scale = np.maximum(np.abs(r), floor)
    bad = np.abs(g - r) > rel * scale
    assert not bad.any(), f"{bad.sum()} outside {rel}; worst {np.max(np.abs(g - r) / scale):.3e}"


def check_bf16_bar(g, r):
    err = np.abs(g - r).max()
    assert err <= BF16_MAX_REL * np.abs(r).max(), f"max err {err} vs max|ref| {np.abs(r).max()}"


def sample_points(shape, n, seed=0, extra=()):
    rng = np.random.default_rng(seed)
    total = int(np.prod(shape))
    pts = rng.integers(0, total, size=n)
    return np.unique(np.concatenate([pts, np.array([0, total - 1] + list(extra), dtype=np.int64)]))
