"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Element-by-element comparisons on seeded inputs ("EinDecomp ... tensor
relational algebra": section 2.1 EinSum semantics, section 2.2 relations, join,
aggregation and repartition).  Small cases run the oracle in full; the full-size
workloads compare sampled outputs plus one whole output tile region.
"""
import numpy as np
import pytest

import oracle
from oracle import rounding
from oracle import tra as otra

from gpu_helpers import (BF16_SUM_REL, FP32_REL, as_f64, check_bf16_bar, check_rel, check_sum, empty, from_dev,
                         gen, relation_on_device, run_plan, sample_points, to_dev)

pytestmark = pytest.mark.gpu

MM = "ij,jk->ik"


def ref_full(eq, X, Y, op, agg, alpha=1.0):
    r = oracle.einsum(eq, as_f64(X), as_f64(Y) if Y is not None else None, op=op, agg=agg, alpha=alpha)
    S = None
    if agg == "sum" and op == "mul":
        S = oracle.einsum(eq, np.abs(as_f64(X)), np.abs(as_f64(Y)), op="mul", agg="sum") * abs(alpha)
    return r, S


def check(op, agg, g, r, S=None, bf16=False):
    if bf16:
        check_bf16_bar(g, r)
        if S is not None:
            check_sum(g, r, S, BF16_SUM_REL)
        return
    if agg in ("max", "min"):
        np.testing.assert_array_equal(g, rounding.to_f32(r).astype(np.float64))
    elif agg == "sum" and op == "mul":
        check_sum(g, r, S, FP32_REL)
    elif agg == "lse":
        check_rel(g, r, FP32_REL, floor=1.0)
    else:
        check_rel(g, r, FP32_REL)


# ------------------------------------------------------------------ repartition (bit-exact)
@pytest.mark.parametrize("shape,src_d,dst_d,dtype", [
    ((64, 64, 64, 64), [4, 1, 4, 1], [1, 4, 1, 4], "f32"),
    ((6, 10, 12), [3, 2, 4], [1, 5, 6], "f32"),
    ((6, 10, 12), [1, 1, 1], [2, 5, 3], "bf16"),
    ((4096, 32, 128), [1, 1, 1], [1, 32, 1], "bf16"),
    ((256, 8192), [1, 1], [1, 8], "f32"),
    ((7, 9), [7, 3], [1, 9], "f32"),
    ((16, 16), [2, 4], [8, 2], "f64"),
    ((1,), [1], [1], "f32"),
    # the TMA path (at most 4 dimensions of extent > 1, 16-byte rows, boxes of 4-32 KB) for
    # every element size, unit dimensions dropped; and a 5-dimensional case that falls back
    ((64, 128, 256), [2, 1, 4], [4, 2, 1], "u8"),
    ((1, 128, 64, 256), [1, 2, 1, 4], [1, 1, 4, 2], "f32"),
    ((2, 1, 32, 64, 128), [2, 1, 2, 1, 4], [1, 1, 1, 4, 2], "bf16"),
    ((256, 512), [4, 2], [2, 8], "f64"),
    ((4, 4, 8, 16, 64), [2, 2, 2, 2, 2], [1, 4, 1, 8, 1], "f32"),
])
def test_repartition_bit_exact(lib, cuda, shape, src_d, dst_d, dtype):
    import torch

    if dtype == "f64":
        dense = gen(shape, 0, 7).astype(np.float64)
    elif dtype == "u8":
        dense = (gen(shape, 0, 7) * 40).astype(np.int16).astype(np.uint8)
    else:
        dense = gen(shape, 0, 7, bf16=(dtype == "bf16"))
    src_blocked = otra.block(dense, src_d)
    src = to_dev(src_blocked)
    dst = torch.empty_like(src)
    lib.repartition(src, dst, list(shape), src_d, dst_d)
    lib.ein_status()
    np.testing.assert_array_equal(from_dev(dst), otra.block(dense, dst_d))


# ------------------------------------------------------------------ config: matmul 64^3 fp32 under three d
@pytest.mark.parametrize("d", [[4, 1, 1, 4], [1, 4, 4, 1], [2, 2, 2, 2]])
@pytest.mark.parametrize("mode", ["fused", "literal"])
def test_matmul64_partition_vectors(lib, cuda, d, mode):
    X = gen((64, 64), 0, 0, "uniform")
    Y = gen((64, 64), 0, 1, "uniform")
    p, g = run_plan(lib, MM + ":mul:sum:mode=" + mode, [64, 64, 64], d, X, Y)
    r, S = ref_full(MM, X, Y, "mul", "sum")
    check("mul", "sum", g, r, S)
    ref = otra.plan_bruteforce(MM, {"i": 64, "j": 64, "k": 64}, d)
    assert (p.n_tasks, p.n_groups, p.n_agg, p.cost_join, p.cost_agg) == (
        ref["n_tasks"], ref["n_groups"], ref["n_agg"], ref["cost_join"], ref["cost_agg"])
    assert p.keys() == ref["tasks"]


def test_matmul64_results_agree_across_d(lib, cuda):
    X = gen((64, 64), 0, 0, "uniform")
    Y = gen((64, 64), 0, 1, "uniform")
    outs = [run_plan(lib, MM + ":mul:sum", [64, 64, 64], d, X, Y)[1] for d in ([4, 1, 1, 4], [1, 4, 4, 1], [2, 2, 2, 2])]
    S = oracle.einsum(MM, np.abs(X), np.abs(Y))
    for o in outs[1:]:
        check_sum(o, outs[0], S, 2 * FP32_REL)


# ------------------------------------------------------------------ semirings, several tiles + ragged tails
SEMIRINGS = [("mul", "sum"), ("sqdiff", "sum"), ("add", "max"), ("add", "min"), ("add", "lse"), ("sub", "max"),
             ("mul", "max")]


@pytest.mark.parametrize("op,agg", SEMIRINGS)
@pytest.mark.parametrize("d", [[1, 1, 1, 1], [2, 7, 7, 5], [3, 1, 1, 2]])
def test_semiring_ragged(lib, cuda, op, agg, d):
    M, K, N = 300, 77, 260
    X = gen((M, K), 3, 0)
    Y = gen((K, N), 3, 1)
    _, g = run_plan(lib, f"{MM}:{op}:{agg}", [M, K, N], d, X, Y)
    r, S = ref_full(MM, X, Y, op, agg)
    check(op, agg, g, r, S)


# fp32 operands contiguous along K (X) and N (Y) in runs of 4: the cp.async pipelined kernel,
# 9 tiles with ragged M / N tails, and 18 x 18 tiles (more CTAs than fit at once).
@pytest.mark.parametrize("op,agg", SEMIRINGS)
@pytest.mark.parametrize("d", [[1, 1, 1, 1], [2, 2, 2, 2]])
def test_semiring_async_ragged(lib, cuda, op, agg, d):
    M, K, N = 300, 96, 264
    X = gen((M, K), 13, 0)
    Y = gen((K, N), 13, 1)
    _, g = run_plan(lib, f"{MM}:{op}:{agg}", [M, K, N], d, X, Y)
    r, S = ref_full(MM, X, Y, op, agg)
    check(op, agg, g, r, S)


@pytest.mark.parametrize("op,agg", [("mul", "sum"), ("add", "max"), ("sqdiff", "sum")])
def test_semiring_async_many_tiles(lib, cuda, op, agg):
    M, K, N = 2304, 64, 2304
    X = gen((M, K), 14, 0)
    Y = gen((K, N), 14, 1)
    _, g = run_plan(lib, f"{MM}:{op}:{agg}", [M, K, N], [1, 1, 1, 1], X, Y)
    r, S = ref_full(MM, X, Y, op, agg)
    check(op, agg, g, r, S)


@pytest.mark.parametrize("op,agg", [("mul", "sum"), ("add", "max"), ("add", "lse"), ("sqdiff", "sum")])
def test_semiring_literal_mode(lib, cuda, op, agg):
    M, K, N = 96, 60, 70
    X = gen((M, K), 4, 0)
    Y = gen((K, N), 4, 1)
    for d in ([2, 3, 3, 2], [1, 4, 4, 1]):
        _, g = run_plan(lib, f"{MM}:{op}:{agg}:mode=literal", [M, K, N], d, X, Y)
        r, S = ref_full(MM, X, Y, op, agg)
        check(op, agg, g, r, S)


@pytest.mark.parametrize("form", ["expand", "direct"])
@pytest.mark.parametrize("d", [[2, 1, 1, 2], [1, 4, 4, 1]])
def test_sqdiff_forms(lib, cuda, form, d):
    M, K, N = 200, 256, 130
    X = gen((M, K), 5, 0)
    Y = gen((K, N), 5, 1)
    _, g = run_plan(lib, MM + ":sqdiff:sum:sqdiff=" + form, [M, K, N], d, X, Y)
    r, _ = ref_full(MM, X, Y, "sqdiff", "sum")
    check_rel(g, r, FP32_REL)


def test_sqdiff_full_output_pair_workload(lib, cuda):
    # every one of the 8192 x 8192 outputs of the squared-distance workload, both forms
    X = gen((8192, 256), 0, 0)
    Y = gen((256, 8192), 1, 0)
    r = oracle.einsum(MM, X, Y, op="sqdiff", agg="sum")
    for form in ("expand", "direct"):
        _, g = run_plan(lib, MM + ":sqdiff:sum:sqdiff=" + form, [8192, 256, 8192], [8, 1, 1, 8], X, Y)
        check_rel(g, r, FP32_REL)


def test_lse_underflow_fallback(lib, cuda):
    # every exp-shifted product underflows for output (0,0): x row [0,-200], y column [-200,0]
    X = np.array([[0.0, -200.0], [1.0, 2.0]], dtype=np.float32)
    Y = np.array([[-200.0, 0.5], [0.0, -1.0]], dtype=np.float32)
    _, g = run_plan(lib, MM + ":add:lse", [2, 2, 2], [1, 1, 1, 1], X, Y)
    r, _ = ref_full(MM, X, Y, "add", "lse")
    check_rel(g, r, FP32_REL, floor=1.0)


@pytest.mark.parametrize("eq,bounds,d,op,agg", [
    ("abef,cfed->abcd", [8, 6, 4, 10, 5, 12], [2, 1, 2, 5, 5, 5, 2, 3], "mul", "sum"),
    ("shd,thd->hst", [40, 3, 16, 24], [2, 3, 1, 2, 3, 1], "mul", "sum"),
    ("hst,thd->shd", [3, 40, 24, 16], [3, 2, 4, 4, 3, 2], "mul", "sum"),
    ("shd,ahd->sa", [40, 3, 16, 24], [1, 3, 2, 2, 3, 2], "mul", "sum"),
    ("sa,ahd->shd", [40, 24, 3, 16], [2, 1, 1, 3, 2], "mul", "sum"),
    ("ijl,jk->ik", [12, 10, 3, 14], [2, 5, 1, 5, 7], "add", "max"),
    ("ij,jk->ik", [1, 1, 1], [1, 1, 1, 1], "mul", "sum"),
    ("ij,jk->ik", [1, 300, 1], [1, 3, 3, 1], "sqdiff", "sum"),
    # degenerate forms: full contraction to a scalar, rank-1 operands, an outer product
    # (no contracted label), every block 1 x 1, a batch label split into keys with lse
    ("ij,ij->", [12, 20], [3, 4, 3, 4], "mul", "sum"),
    ("ij,ij->", [12, 20], [3, 4, 3, 4], "add", "max"),
    ("i,i->", [300], [3, 3], "add", "lse"),
    ("i,j->ij", [7, 9], [7, 3], "mul", "none"),
    ("ij,jk->ik", [4, 6, 8], [4, 6, 6, 8], "add", "max"),
    ("ij,jk->ik", [4, 6, 8], [4, 6, 6, 8], "mul", "sum"),
    ("bij,bjk->bik", [2, 3, 5, 7], [2, 3, 5, 2, 5, 7], "add", "lse"),
])
def test_general_einsums(lib, cuda, eq, bounds, d, op, agg):
    ins, out = eq.split("->")[0].split(","), eq.split("->")[1]
    order = []
    for c in "".join(ins):
        if c not in order:
            order.append(c)
    B = dict(zip(order, bounds))
    X = gen(tuple(B[c] for c in ins[0]), 6, 0)
    Y = gen(tuple(B[c] for c in ins[1]), 6, 1)
    for bf in ([False, True] if (op, agg) == ("mul", "sum") else [False]):
        Xi = rounding.f32_to_bf16_bits(X) if bf else X
        Yi = rounding.f32_to_bf16_bits(Y) if bf else Y
        spec = f"{eq}:{op}:{agg}" + (":in=bf16" if bf else "")
        _, g = run_plan(lib, spec, bounds, d, Xi, Yi)
        r, S = ref_full(eq, Xi, Yi, op, agg)
        if bf:
            check_sum(g, r, S, FP32_REL)  # identical bf16 inputs: only fp32 summation order differs
        else:
            check(op, agg, g, r, S)


# ------------------------------------------------------------------ unary aggregation and broadcast join
@pytest.mark.parametrize("agg", ["lse", "max", "sum", "min"])
@pytest.mark.parametrize("d", [[1, 1, 1], [4, 2, 1], [2, 1, 3]])
def test_row_reduce(lib, cuda, agg, d):
    S = gen((8, 20, 300), 7, 0, b=5.0)
    _, g = run_plan(lib, "hst->hs::" + agg, [8, 20, 300], d, S)
    r = oracle.einsum("hst->hs", as_f64(S), agg=agg)
    if agg in ("max", "min"):
        np.testing.assert_array_equal(g, r)
    elif agg == "sum":
        check_sum(g, r, oracle.einsum("hst->hs", np.abs(as_f64(S)), agg="sum"), FP32_REL)
    else:
        check_rel(g, r, FP32_REL, floor=1.0)


@pytest.mark.parametrize("agg", ["lse", "max"])
def test_row_reduce_long_rows_with_masked_entries(lib, cuda, agg):
    # rows of 1100: several 512-value rounds per lane group and a ragged last round; -inf
    # entries (masked scores) contribute nothing
    S = gen((4, 6, 1100), 17, 0, b=4.0)
    S[0, 0, ::7] = -np.inf
    S[3, 5, 1:] = -np.inf
    _, g = run_plan(lib, "hst->hs::" + agg, [4, 6, 1100], [1, 1, 1], S)
    r = oracle.einsum("hst->hs", as_f64(S), agg=agg)
    if agg == "max":
        np.testing.assert_array_equal(g, r)
    else:
        check_rel(g, r, FP32_REL, floor=1.0)


def test_broadcast_expsub_long_rows(lib, cuda):
    S = gen((4, 6, 1100), 18, 0, b=3.0)
    L = gen((4, 6), 18, 1, b=3.0)
    _, g = run_plan(lib, "hst,hs->hst:expsub:none:out=bf16", [4, 6, 1100], [1, 1, 1, 1, 1], S, L, out_bf16=True)
    r = oracle.einsum("hst,hs->hst", as_f64(S), as_f64(L), op="expsub", agg="none")
    check_rel(g, rounding.to_bf16(r).astype(np.float64), 2 ** -7)


@pytest.mark.parametrize("d", [[1, 1, 1, 1, 1], [2, 3, 1, 2, 3], [2, 3, 4, 2, 3]])
@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_broadcast_expsub_flat(lib, cuda, d, out):
    # innermost extent a multiple of 8: the flat kernel when the innermost label is unsplit
    S = gen((4, 6, 1024), 19, 0, b=3.0)
    L = gen((4, 6), 19, 1, b=3.0)
    bf = out == "bf16"
    _, g = run_plan(lib, f"hst,hs->hst:expsub:none:out={out}", [4, 6, 1024], d, S, L, out_bf16=bf)
    r = oracle.einsum("hst,hs->hst", as_f64(S), as_f64(L), op="expsub", agg="none")
    if bf:
        check_rel(g, rounding.to_bf16(r).astype(np.float64), 2 ** -7)
    else:
        check_rel(g, r, 1e-5)


@pytest.mark.parametrize("op", ["mul", "add", "sub", "sqdiff"])
def test_same_layout_join_flat(lib, cuda, op):
    X = gen((3, 10, 64), 20, 0)
    Y = gen((3, 10, 64), 20, 1)
    _, g = run_plan(lib, f"hst,hst->hst:{op}:none:alpha=0.5", [3, 10, 64], [3, 2, 1, 3, 2, 1], X, Y)
    r = oracle.einsum("hst,hst->hst", as_f64(X), as_f64(Y), op=op, agg="none", alpha=0.5)
    check_rel(g, r, 1e-6, floor=1e-3)


@pytest.mark.parametrize("d", [[1, 1, 1, 1, 1], [4, 2, 3, 4, 2]])
def test_broadcast_expsub(lib, cuda, d):
    S = gen((8, 20, 300), 8, 0, b=3.0)
    L = gen((8, 20), 8, 1, b=3.0)
    _, g = run_plan(lib, "hst,hs->hst:expsub:none:out=bf16", [8, 20, 300], d, S, L, out_bf16=True)
    r = oracle.einsum("hst,hs->hst", as_f64(S), as_f64(L), op="expsub", agg="none")
    check_rel(g, rounding.to_bf16(r).astype(np.float64), 2 ** -7)


# ------------------------------------------------------------------ full-size workloads (sampled)
def _sampled(lib, spec, bounds, d, X, Y, op, agg, n=4096, tile=(0, 0, 128), bf16=False):
    p, g = run_plan(lib, spec, bounds, d, X, Y)
    M, N = g.shape
    r0, c0, t = tile
    extra = [(r0 + i) * N + c0 + j for i in range(t) for j in range(t)]
    pts = sample_points((M, N), n, extra=extra)
    Xd, Yd = as_f64(X), as_f64(Y)
    r = oracle.einsum_points(MM, Xd, Yd, pts, op=op, agg=agg)
    gv = g.reshape(-1)[pts]
    S = oracle.einsum_points(MM, np.abs(Xd), np.abs(Yd), pts) if (op, agg) == ("mul", "sum") else None
    check(op, agg, gv, r, S, bf16=bf16)
    if bf16:
        check_sum(gv, r, S, BF16_SUM_REL)
    return p


@pytest.mark.parametrize("op,agg", [("sqdiff", "sum"), ("add", "max")])
def test_semiring_pair_full_size(lib, cuda, op, agg):
    X = gen((8192, 256), 0, 0)
    Y = gen((256, 8192), 1, 0)
    p = _sampled(lib, f"{MM}:{op}:{agg}", [8192, 256, 8192], [8, 1, 1, 8], X, Y, op, agg, tile=(1000, 1000, 64))
    assert p.n_tasks == 64 and p.cost_join == 33554432 and p.cost_agg == 0


@pytest.mark.parametrize("d", [[1, 1, 1, 1], [2, 2, 2, 2]])
def test_lse_8192_full_size(lib, cuda, d):
    X = gen((8192, 8192), 0, 0)
    Y = gen((8192, 8192), 0, 1)
    _sampled(lib, MM + ":add:lse", [8192] * 3, d, X, Y, "add", "lse", n=1024, tile=(4000, 4000, 16))


def test_contraction_4d_full_size(lib, cuda):
    A = gen((64, 64, 64, 64), 0, 0, bf16=True)
    B = gen((64, 64, 64, 64), 0, 1, bf16=True)
    eq = "abef,cfed->abcd"
    p, g = run_plan(lib, eq + ":mul:sum:in=bf16", [64] * 6, [4, 1, 1, 1, 4, 1, 1, 1], A, B)
    assert p.n_tasks == 16 and p.cost_join == 134217728
    pts = sample_points(g.shape, 4096, extra=list(range(0, 64 * 64)))
    Ad, Bd = as_f64(A), as_f64(B)
    r = oracle.einsum_points(eq, Ad, Bd, pts)
    S = oracle.einsum_points(eq, np.abs(Ad), np.abs(Bd), pts)
    gv = g.reshape(-1)[pts]
    check_bf16_bar(gv, r)
    check_sum(gv, r, S, BF16_SUM_REL)


@pytest.mark.parametrize("d", [[1, 1, 1, 1], [4, 1, 1, 4], [1, 8, 8, 1], [2, 2, 2, 2], [4, 2, 2, 2]])
def test_large_bf16_matmul(lib, cuda, d):
    n = 16384
    X = gen((n, n), 0, 0, bf16=True)
    Y = gen((n, n), 0, 1, bf16=True)
    _sampled(lib, MM + ":mul:sum:in=bf16", [n] * 3, d, X, Y, "mul", "sum", n=2048, tile=(8100, 8100, 64), bf16=True)


# ---------------------------------------------------------------- empty EinSums
EMPTY_FILL = [
    # a contracted label of extent 0 (binary and unary): each output aggregates the empty set
    ("ij,jk->ik", [64, 0, 32], [4, 2, 2, 2]),
    ("abef,cfed->abcd", [4, 2, 0, 3, 2, 4], [2, 1, 4, 3, 2, 3, 4, 2]),
    ("hst->hs", [2, 8, 0], [2, 2, 1]),
]


@pytest.mark.parametrize("alpha", [1.0, -0.5])
@pytest.mark.parametrize("out", ["f32", "bf16"])
@pytest.mark.parametrize("agg", ["sum", "max", "min", "lse"])
@pytest.mark.parametrize("eq,bounds,d", EMPTY_FILL)
def test_empty_contraction(lib, cuda, eq, bounds, d, agg, out, alpha):
    import torch

    ins = eq.split("->")[0].split(",")
    unary = len(ins) == 1
    op = "" if unary else ("mul" if agg == "sum" else "add")
    p = lib.Plan(f"{eq}:{op}:{agg}:out={out}:alpha={alpha}", bounds, d)
    assert p.kernel == "fill"
    order = []
    for c in "".join(ins):
        if c not in order:
            order.append(c)
    B = dict(zip(order, bounds))
    X = np.zeros(tuple(B[c] for c in ins[0]), np.float32)
    Y = None if unary else np.zeros(tuple(B[c] for c in ins[1]), np.float32)
    z = torch.full((int(np.prod(p.shape("z"))),), 7.0, device="cuda",
                   dtype=torch.bfloat16 if out == "bf16" else torch.float32)
    p.execute(None, None, z)  # nothing is read
    lib.ein_status()
    g = as_f64(from_dev(z))
    r = oracle.einsum(eq, X, Y, op=op or "mul", agg=agg, alpha=alpha).reshape(-1)
    np.testing.assert_array_equal(g, r)  # 0 or an infinity, exactly
    np.testing.assert_array_equal(np.signbit(g), np.signbit(r))


@pytest.mark.parametrize("spec,bounds,d", [
    (MM + ":sqdiff:sum", [300, 96, 264], [2, 2, 2, 2]),
    (MM + ":add:max", [300, 96, 264], [1, 1, 1, 1]),
    ("hst->hs::lse", [4, 96, 200], [2, 3, 1]),
    # tensor cores: the TMA-store epilogue for device memory, warp stores for host memory
    (MM + ":mul:sum:in=bf16", [512, 256, 384], [2, 1, 1, 3]),
    (MM + ":mul:sum:in=bf16:tc=single:out=bf16", [384, 512, 192], [1, 1, 1, 1]),
    (MM + ":mul:sum:in=bf16", [1024, 4096, 1024], [1, 1, 1, 1]),  # K-split tail
    (MM + ":sqdiff:sum:split=bf16x3", [256, 64, 384], [1, 1, 1, 1]),
])
def test_output_in_pinned_host_memory(lib, cuda, spec, bounds, d):
    # the kernels may store their result straight into pinned host memory (unified addressing):
    # bit-identical to the result written to device memory
    import torch

    p = lib.Plan(spec, bounds, d)
    n_in = len(p.operands)
    bf = "in=bf16" in spec
    xs = [to_dev(gen(tuple(p.shape(w)), 15, i, bf16=bf)).reshape(-1) for i, w in enumerate("xy"[:n_in])]
    if n_in == 1:
        xs.append(None)
    nz = int(np.prod(p.shape("z")))
    odt = torch.bfloat16 if "out=bf16" in spec else torch.float32
    zd = torch.empty(nz, device="cuda", dtype=odt)
    zh = torch.full((nz,), 7.0, dtype=odt).pin_memory()
    p.execute(xs[0], xs[1], zd)
    p.execute(xs[0], xs[1], zh)
    torch.cuda.synchronize()
    lib.ein_status()
    assert torch.equal(zh, zd.cpu())
