"""K split of the last wave's tiles on the tensor-core path, against the oracle.

"EinDecomp ... tensor relational algebra", section 2.2: the aggregation over the
contracted keys is a sum, which is commutative and associative, so the K range of an
output tile may be cut into runs whose partial sums are added afterwards.  The
persistent tensor-core kernels do that for the tiles of a last, partly filled wave:
with T tiles on C workers, the T mod C tiles left over are each cut into 2-4 runs on
otherwise idle workers, the partial sums go through the plan's workspace, and they are
added in a fixed order.  A tile cut in two with an fp32 output written through its tensor
map skips the workspace: part 0's worker zeroes the tile at the start of the launch and both
parts add into it with TMA reduce-add (two values added into zero give the same bits in
either order).  Small problems (T < C) are all "last wave".

Checked here: the result against the oracle (the same bars as the unsplit path), the
result of ksplit=off within the fp32 summation bar, bit-identical repeats, and replay
from a CUDA graph bit-identical to eager launches.
"""
import numpy as np
import pytest

import oracle

from gpu_helpers import FP32_REL, BF16_SUM_REL, as_f64, check_bf16_bar, check_sum, empty, from_dev, gen, \
    relation_on_device, run_plan, sample_points
from oracle import tra as otra

pytestmark = pytest.mark.gpu


def labels_of(eq):
    ins, out = eq.split("->")[0].split(","), eq.split("->")[1]
    order = []
    for c in "".join(ins):
        if c not in order:
            order.append(c)
    return ins, out, order


# K of 1024, 1536 and 2048 gives 16, 24 and 32 K steps of 64: 2, 3 and 4 runs of at least 8.
# Two runs into an fp32 output through the TMA-store epilogue add into the zeroed output (TMA
# reduce-add); other splits gather the partial sums in part order.
SPLIT_CASES = [
    ("ij,jk->ik", [256, 2048, 256], [1, 1, 1, 1], ""),                 # one pair tile, 4 runs
    ("ij,jk->ik", [512, 1536, 512], [2, 1, 1, 2], ""),                 # 4 tiles in 4 keys, 3 runs
    ("ij,jk->ik", [256, 1024, 512], [1, 2, 2, 1], ":alpha=0.5"),       # contracted keys, 2 runs
    ("ji,jk->ik", [2048, 256, 256], [1, 1, 1, 1], ":out=bf16"),        # M-major X, bf16 output
    ("ij,kj->ik", [512, 2048, 256], [1, 1, 1, 1], ":tc_n=128"),        # K-major Y, 256 x 128 tiles
    ("bij,bjk->bik", [3, 256, 1536, 256], [3, 1, 1, 3, 1, 1], ""),     # batch keys, 3 tiles
    ("ij,jk->ik", [384, 2048, 256], [1, 1, 1, 1], ":tc=single"),       # one CTA per 128-row tile
    ("abef,cfed->abcd", [2, 128, 8, 128, 2, 128], [2, 1, 1, 1, 2, 1, 1, 1], ""),  # 4-D contraction
]


def _inputs(eq, bounds, seed):
    ins, _, order = labels_of(eq)
    B = dict(zip(order, bounds))
    X = gen(tuple(B[c] for c in ins[0]), seed, 0, bf16=True)
    Y = gen(tuple(B[c] for c in ins[1]), seed, 1, bf16=True)
    return X, Y


@pytest.mark.parametrize("store", [":tc_store=tma", ":tc_store=lsu"])
@pytest.mark.parametrize("eq,bounds,d,opts", SPLIT_CASES)
def test_ksplit_parity(lib, cuda, eq, bounds, d, opts, store):
    spec = f"{eq}:mul:sum:in=bf16{opts}{store}"
    try:
        lib.Plan(spec, bounds, d)
    except lib.TraError as e:
        assert "TRA_ERR_UNSUPPORTED" in str(e)
        pytest.skip("no tiling with this epilogue")
    X, Y = _inputs(eq, bounds, 12)
    out_bf16 = ":out=bf16" in opts
    p, g = run_plan(lib, spec, bounds, d, X, Y, out_bf16=out_bf16)
    assert p.workspace_bytes > 0, "the plan should split the K loop of its tiles here"
    q, g_off = run_plan(lib, spec + ":ksplit=off", bounds, d, X, Y, out_bf16=out_bf16)
    assert q.workspace_bytes == 0
    _, g2 = run_plan(lib, spec, bounds, d, X, Y, out_bf16=out_bf16)
    np.testing.assert_array_equal(g, g2)  # the parts are added in a fixed order
    alpha = float(opts.split("alpha=")[1].split(":")[0]) if "alpha=" in opts else 1.0
    r = oracle.einsum(eq, as_f64(X), as_f64(Y), alpha=alpha)
    S = oracle.einsum(eq, np.abs(as_f64(X)), np.abs(as_f64(Y))) * abs(alpha)
    for out in (g, g_off):
        check_bf16_bar(out, r)
        if out_bf16:
            assert np.all(np.abs(out - r) <= 2.0 ** -8 * np.abs(r) + FP32_REL * S)
        else:
            check_sum(out, r, S, FP32_REL)
    if not out_bf16:
        check_sum(g, g_off, S, 2 * FP32_REL)


def test_ksplit_contraction_4d_full_size(lib, cuda):
    # the 64^6 contraction under d = [4,1,1,1,4,1,1,1]: 256 tiles of 256 x 256, so on a GB300's
    # 76 co-resident pairs 28 tiles are left for the last wave and run in two halves of K
    A = gen((64, 64, 64, 64), 0, 0, bf16=True)
    B = gen((64, 64, 64, 64), 0, 1, bf16=True)
    eq = "abef,cfed->abcd"
    spec = eq + ":mul:sum:in=bf16"
    d = [4, 1, 1, 1, 4, 1, 1, 1]
    p, g = run_plan(lib, spec, [64] * 6, d, A, B)
    _, g_off = run_plan(lib, spec + ":ksplit=off", [64] * 6, d, A, B)
    diff = np.flatnonzero(g.reshape(-1) != g_off.reshape(-1))
    if p.workspace_bytes:
        assert diff.size > 0  # the split tiles sum in another order
    rng = np.random.default_rng(3)
    pick = rng.choice(diff, size=min(2048, diff.size), replace=False) if diff.size else np.zeros(0, np.int64)
    pts = np.unique(np.concatenate([sample_points(g.shape, 2048, seed=4), pick]))
    Ad, Bd = as_f64(A), as_f64(B)
    r = oracle.einsum_points(eq, Ad, Bd, pts)
    S = oracle.einsum_points(eq, np.abs(Ad), np.abs(Bd), pts)
    for out in (g, g_off):
        gv = out.reshape(-1)[pts]
        check_bf16_bar(gv, r)
        check_sum(gv, r, S, BF16_SUM_REL)
    # everywhere: the two summation orders agree to well within the fp32 bar
    assert np.abs(g - g_off).max() <= 1e-5 * np.abs(g_off).max()


@pytest.mark.parametrize("bounds", [[512, 1536, 512], [512, 1024, 512]])
def test_ksplit_graph_replay(lib, cuda, bounds):
    # a CUDA graph freezes the launch's arguments (the flag tag included); the flags of the split
    # tiles are cleared by the last part of each tile, so every replay starts from the same state.
    # K = 1536 splits each tile in three (partial sums gathered in order); K = 1024 in two, whose
    # parts add into the output zeroed by part 0's worker (TMA reduce-add)
    import torch

    eq, d = "ij,jk->ik", [2, 1, 1, 2]
    spec = eq + ":mul:sum:in=bf16"
    p = lib.Plan(spec, bounds, d)
    assert p.workspace_bytes > 0
    ws = torch.empty(p.workspace_bytes, dtype=torch.uint8, device="cuda")
    xs = [_inputs(eq, bounds, s) for s in (20, 21, 22)]
    xd = relation_on_device(lib, xs[0][0], d[:2]).clone()
    yd = relation_on_device(lib, xs[0][1], d[2:]).clone()
    z = empty(int(np.prod(p.shape("z"))), False)
    eager = []
    for X, Y in xs:
        xd.copy_(relation_on_device(lib, X, d[:2]))
        yd.copy_(relation_on_device(lib, Y, d[2:]))
        p.execute(xd, yd, z, ws)
        eager.append(from_dev(z).copy())
    lib.ein_status()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        p.execute(xd, yd, z, ws)
    for i in (0, 1, 2, 1):
        X, Y = xs[i]
        xd.copy_(relation_on_device(lib, X, d[:2]))
        yd.copy_(relation_on_device(lib, Y, d[2:]))
        z.zero_()
        graph.replay()
        torch.cuda.synchronize()
        np.testing.assert_array_equal(from_dev(z), eager[i])
    lib.ein_status()
    X, Y = xs[1]
    r = oracle.einsum(eq, as_f64(X), as_f64(Y))
    S = oracle.einsum(eq, np.abs(as_f64(X)), np.abs(as_f64(Y)))
    g = otra.unblock(eager[1], p.shape("z"), p.dvec("z")).astype(np.float64)
    check_sum(g, r, S, FP32_REL)
