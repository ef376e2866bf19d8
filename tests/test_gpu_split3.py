"""split=bf16x3: the squared distance and logsumexp semirings rewritten onto BF16 tensor cores
("EinDecomp ... tensor relational algebra", section 2.1: extended aggregation and join ops),
against the oracle in double.

  sum_j (x - y)^2 = |x|^2 + |y|^2 - 2 x.y            (the closed form the pages' example rests on)
  lse_j (x + y)   = mx + my + log sum_j e^(x - mx) e^(y - my)

The sum of products runs with each fp32 operand split as hi + lo bf16 and the product taken as
hi.hi + hi.lo + lo.hi.  With bf16's unit roundoff 2^-8, |x - hi - lo| <= 2^-16 |x|, so one
product is off by at most 3 * 2^-16 |x y|.  Tolerances:
  squared distance: |g - r| <= 1e-5 |r| + 6 * 2^-16 * sum_j |x_j y_j|     (the -2 x.y term)
  logsumexp:        |g - r| <= 1e-5 max(|r|, 1) + 4 * 2^-16               (a sum of positive terms)
and, at the pages' size and distribution, the fp32 bar alone (1e-5 relative).
"""
import numpy as np
import pytest

import oracle

from gpu_helpers import FP32_REL, as_f64, gen, run_plan, sample_points

pytestmark = pytest.mark.gpu

U = 2.0 ** -16


def _check(eq, X, Y, op, agg, g):
    r = oracle.einsum(eq, as_f64(X), as_f64(Y), op=op, agg=agg)
    if agg == "sum":
        S = oracle.einsum(eq, np.abs(as_f64(X)), np.abs(as_f64(Y)), op="mul", agg="sum")
        bound = FP32_REL * np.abs(r) + 6 * U * S
    else:
        bound = FP32_REL * np.maximum(np.abs(r), 1.0) + 4 * U
    err = np.abs(g - r)
    assert np.all(err <= bound), f"{int((err > bound).sum())} outside; worst ratio {np.max(err / bound):.3f}"
    return r


# Z's last label must be N with a block extent that is a multiple of 32 (the planner refuses
# other outputs); rows, the contracted extent and the padding of the GEMM's tiles are free.
CASES = [
    # eq, bounds, d
    ("ij,jk->ik", [256, 64, 384], [1, 1, 1, 1]),
    ("ij,jk->ik", [300, 96, 192], [2, 1, 1, 3]),      # ragged row tiles, columns padded to 256
    ("ij,jk->ik", [128, 64, 256], [2, 2, 2, 4]),      # contracted label split into keys
    ("ij,kj->ik", [200, 40, 128], [2, 2, 2, 2]),      # Y K-contiguous (a transposed operand)
    ("bij,bjk->bik", [3, 130, 24, 96], [3, 2, 1, 3, 1, 3]),  # batch label, tails, K = 24
]


@pytest.mark.parametrize("eq,bounds,d", CASES)
@pytest.mark.parametrize("op,agg", [("sqdiff", "sum"), ("add", "lse")])
def test_split3_against_oracle(lib, cuda, eq, bounds, d, op, agg):
    xs, ys = eq.split("->")[0].split(",")
    B = dict(zip(dict.fromkeys(xs + ys), bounds))
    X = gen(tuple(B[c] for c in xs), 61, 0)
    Y = gen(tuple(B[c] for c in ys), 61, 1)
    p, g = run_plan(lib, f"{eq}:{op}:{agg}:split=bf16x3", bounds, d, X, Y)
    assert p.kernel == "tc_split3"
    _check(eq, X, Y, op, agg, g)


def test_split3_alpha_and_bf16_output(lib, cuda):
    X = gen((128, 64), 62, 0)
    Y = gen((64, 256), 62, 1)
    p, g = run_plan(lib, "ij,jk->ik:sqdiff:sum:split=bf16x3:alpha=0.5:out=bf16", [128, 64, 256], [1, 1, 1, 1], X, Y,
                    out_bf16=True)
    r = 0.5 * oracle.einsum("ij,jk->ik", as_f64(X), as_f64(Y), op="sqdiff", agg="sum")
    assert np.all(np.abs(g - r) <= 2 ** -8 * np.abs(r) + 1e-3)


def test_split3_lse_underflow_fix_up(lib, cuda):
    # every exp-shifted product of output (0, 0) underflows (row max 0 and column max 0 sit in
    # different j): the epilogue marks it and the fix-up pass recomputes it from the operands
    X = gen((128, 64), 63, 0)
    Y = gen((64, 128), 63, 1)
    X[0, :] = -200.0
    X[0, 0] = 0.0
    Y[:, 0] = -200.0
    Y[1, 0] = 0.0
    p, g = run_plan(lib, "ij,jk->ik:add:lse:split=bf16x3", [128, 64, 128], [1, 1, 1, 1], X, Y)
    _check("ij,jk->ik", X, Y, "add", "lse", g)
    assert np.isfinite(g).all()


@pytest.mark.parametrize("op,agg", [("sqdiff", "sum"), ("add", "lse")])
def test_split3_pages_size_fp32_bar(lib, cuda, op, agg):
    # the semiring pair's workload: X 8192 x 256, Y 256 x 8192 N(0, 1), d = [8, 1, 1, 8];
    # sampled outputs against the oracle, fp32 bar alone
    X = gen((8192, 256), 0, 0)
    Y = gen((256, 8192), 0, 1)
    _, g = run_plan(lib, f"ij,jk->ik:{op}:{agg}:split=bf16x3", [8192, 256, 8192], [8, 1, 1, 8], X, Y)
    pts = sample_points((8192, 8192), 4096, extra=[i * 8192 + j for i in range(64) for j in range(64)])
    r = oracle.einsum_points("ij,jk->ik", as_f64(X), as_f64(Y), pts, op=op, agg=agg)
    gv = g.reshape(-1)[pts]
    scale = np.abs(r) if agg == "sum" else np.maximum(np.abs(r), 1.0)
    worst = np.max(np.abs(gv - r) / scale)
    assert worst <= FP32_REL, f"worst relative error {worst:.3e}"
