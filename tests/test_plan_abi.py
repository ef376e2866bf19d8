"""C-ABI library without a GPU: symbols, planner facts and error paths.

The planner's key space, task counts and cost terms ("EinDecomp ... tensor
relational algebra", sections 2.2, 3.1, 3.2) must equal the oracle's brute-force
enumeration bit for bit.
"""
import ctypes
import json
import os
import re

import numpy as np
import pytest

from oracle import tra as otra

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLD = os.path.join(ROOT, "tests", "golden")


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "tra.h")).read()
    return sorted(set(re.findall(r"^\s*(?:int|void|const char\*)\s+(ein_\w+)\s*\(", src, re.M)))


def test_library_exports_every_declared_symbol(lib):
    so = ctypes.CDLL(os.path.join(ROOT, "tensor_relational_algebra_gb300", "libtra.so"))
    syms = declared_symbols()
    assert len(syms) >= 9
    for s in syms:
        assert hasattr(so, s), s


CASES = [
    ("ij,jk->ik", {"i": 64, "j": 64, "k": 64}, [4, 1, 1, 4]),
    ("ij,jk->ik", {"i": 64, "j": 64, "k": 64}, [1, 4, 4, 1]),
    ("ij,jk->ik", {"i": 64, "j": 64, "k": 64}, [2, 2, 2, 2]),
    ("ij,jk->ik", {"i": 8192, "j": 256, "k": 8192}, [8, 1, 1, 8]),
    ("abef,cfed->abcd", {c: 64 for c in "abefcd"}, [4, 1, 1, 1, 4, 1, 1, 1]),
    ("abef,cfed->abcd", {c: 8 for c in "abefcd"}, [2, 1, 2, 4, 2, 4, 2, 1]),
    ("ij,jk->ik", {"i": 16384, "j": 16384, "k": 16384}, [4, 2, 2, 2]),
    ("ij,jk->ik", {"i": 16384, "j": 16384, "k": 16384}, [1, 8, 8, 1]),
    ("sa,ahd->shd", {"s": 64, "a": 32, "h": 4, "d": 16}, [2, 2, 2, 4, 1]),
    ("shd,thd->hst", {"s": 64, "h": 4, "d": 16, "t": 32}, [1, 4, 2, 2, 4, 2]),
    ("hst,thd->shd", {"h": 4, "s": 64, "t": 32, "d": 16}, [4, 2, 2, 2, 4, 1]),
    ("shd,ahd->sa", {"s": 64, "h": 4, "d": 16, "a": 32}, [1, 2, 4, 2, 2, 4]),
    ("hst,hs->hst", {"h": 4, "s": 8, "t": 16}, [2, 4, 1, 2, 4]),
    ("ijl,jk->ik", {"i": 4, "j": 6, "l": 2, "k": 4}, [2, 3, 2, 3, 2]),
]


def spec_for(eq):
    if eq == "hst,hs->hst":
        return eq + ":expsub:none"
    return eq + ":mul:sum"


@pytest.mark.parametrize("eq,bounds,d", CASES)
def test_plan_matches_bruteforce(lib, eq, bounds, d):
    p = lib.Plan(spec_for(eq), bounds, d)
    ref = otra.plan_bruteforce(eq, bounds, d)
    for k in ("n_tasks", "n_groups", "n_agg", "cost_join", "cost_agg"):
        assert getattr(p, k) == ref[k], k
    assert p.info.x_sub == ref["x_sub"] and p.info.y_sub == ref["y_sub"] and p.info.z_sub == ref["z_sub"]
    assert p.dvec("z") == ref["dz"]
    if ref["n_tasks"] <= 4096:
        assert p.keys() == ref["tasks"]


EMPTY_CASES = [
    # a contracted label of extent 0: every output aggregates the empty set
    ("ij,jk->ik", {"i": 64, "j": 0, "k": 32}, [4, 2, 2, 2], "fill"),
    ("abef,cfed->abcd", {"a": 4, "b": 2, "e": 0, "f": 3, "c": 2, "d": 4}, [2, 1, 4, 3, 2, 3, 4, 2], "fill"),
    # an output label of extent 0: nothing to compute
    ("ij,jk->ik", {"i": 0, "j": 16, "k": 32}, [2, 4, 4, 2], "empty"),
    ("sa,ahd->shd", {"s": 8, "a": 4, "h": 0, "d": 2}, [2, 2, 2, 1, 1], "empty"),
]


@pytest.mark.parametrize("eq,bounds,d,kernel", EMPTY_CASES)
def test_empty_plan_matches_bruteforce(lib, eq, bounds, d, kernel):
    # the key space and the cost formulas still hold, with sub-tensors of 0 elements
    p = lib.Plan(eq + ":mul:sum", bounds, d)
    assert p.kernel == kernel and p.workspace_bytes == 0
    ref = otra.plan_bruteforce(eq, bounds, d)
    for k in ("n_tasks", "n_groups", "n_agg", "cost_join", "cost_agg"):
        assert getattr(p, k) == ref[k], k
    assert p.info.x_sub == ref["x_sub"] and p.info.y_sub == ref["y_sub"] and p.info.z_sub == ref["z_sub"]
    assert p.keys() == ref["tasks"]
    for agg in ("max", "min", "lse"):
        assert lib.Plan(f"{eq}:add:{agg}", bounds, d).kernel == kernel


def test_empty_output_and_repartition_need_no_buffers(lib):
    # an output of no elements launches nothing (no device needed); nor does a repartition of
    # a tensor with an extent of 0
    p = lib.Plan("ij,jk->ik:mul:sum", [0, 16, 32], [1, 1, 1, 1])
    lib.ein_execute(p.handle, None, None, None, None, 0, 0)
    lib.ein_repartition([0, 4], [1, 1], [1, 2], 4, None, None, 0)
    with pytest.raises(lib.TraError) as e:
        lib.ein_repartition([0, 4], [1, 1], [1, 3], 4, None, None, 0)
    assert "TRA_ERR_DIVISIBILITY" in str(e.value)
    with pytest.raises(lib.TraError) as e:
        lib.ein_execute(lib.Plan("ij,jk->ik:mul:sum", [4, 0, 4], [1, 1, 1, 1]).handle, None, None, None, None, 0, 0)
    assert "TRA_ERR_ARG" in str(e.value)  # a fill needs its output


def test_plan_golden(lib):
    g = json.load(open(os.path.join(GOLD, "cost_terms.json")))
    for c in g["cases"]:
        p = lib.Plan(spec_for(c["eq"]), c["bounds"], c["d"])
        for k in ("n_tasks", "n_groups", "n_agg", "cost_join", "cost_agg"):
            assert getattr(p, k) == c[k], (c["eq"], c["d"], k)


def test_unary_plan(lib):
    p = lib.Plan("hst->hs::lse", {"h": 32, "s": 64, "t": 128}, [4, 2, 1])
    ref = otra.plan_bruteforce("hst->hs", {"h": 32, "s": 64, "t": 128}, [4, 2, 1])
    assert (p.n_tasks, p.n_groups, p.n_agg, p.cost_join, p.cost_agg) == (
        ref["n_tasks"], ref["n_groups"], ref["n_agg"], ref["cost_join"], ref["cost_agg"])
    assert p.kernel == "row_reduce"


def test_kernel_choice(lib):
    assert lib.Plan("ij,jk->ik:sqdiff:sum", [64, 64, 64], [1, 1, 1, 1]).kernel == "semiring_f32"
    # squared distance: expansion (row norms, column norms, one guard word per 128 x 128 tile and
    # the launch's tag word)
    # while K <= 3127, where the guard threshold 3 sqrt(K) 2^-24 / 1e-5 stays below 1
    a = lambda v: (v + 255) // 256 * 256  # noqa: E731
    assert lib.Plan("ij,jk->ik:sqdiff:sum", [300, 3127, 200], [1, 1, 1, 1]).workspace_bytes == a(1200) + a(800) + a(3 * 2 * 4 + 4)
    assert lib.Plan("ij,jk->ik:sqdiff:sum", [300, 3128, 200], [1, 1, 1, 1]).workspace_bytes == 0  # direct
    assert lib.Plan("ij,jk->ik:sqdiff:sum:sqdiff=expand", [300, 3128, 200], [1, 1, 1, 1]).workspace_bytes > 0
    assert lib.Plan("ij,jk->ik:add:lse", [64, 64, 64], [1, 1, 1, 1]).kernel == "lse_factored"
    assert lib.Plan("ij,jk->ik:add:max:mode=literal", [64, 64, 64], [1, 2, 2, 1]).kernel == "literal"
    assert lib.Plan("hst,hs->hst:expsub:none:out=bf16", [2, 4, 8], [1, 1, 1, 1, 1]).kernel == "elementwise"
    p = lib.Plan("ij,jk->ik:add:lse", [64, 32, 16], [2, 1, 1, 2])
    assert p.workspace_bytes >= (64 * 32 + 32 * 16 + 64 + 16) * 4
    assert lib.Plan("ij,jk->ik:mul:sum", [64, 64, 64], [1, 1, 1, 1]).workspace_bytes == 0
    # BF16 sum-of-products: a 256 x 256 tile per CTA pair when rows and columns allow it
    assert lib.Plan("ij,jk->ik:mul:sum:in=bf16", [512, 128, 256], [2, 1, 1, 1]).kernel == "tc_bf16_pair"
    assert lib.Plan("ij,jk->ik:mul:sum:in=bf16:tc=single", [512, 128, 256], [2, 1, 1, 1]).kernel == "tc_bf16"
    assert lib.Plan("ij,jk->ik:mul:sum:in=bf16", [384, 128, 256], [1, 1, 1, 1]).kernel == "tc_bf16"
    assert lib.Plan("ij,jk->ik:mul:sum:in=bf16", [256, 128, 192], [1, 1, 1, 1]).kernel == "tc_bf16"
    assert lib.Plan("ij,jk->ik:mul:sum:in=bf16", [256, 128, 384], [1, 1, 1, 1]).kernel == "tc_bf16_pair"


def test_split3_plans(lib):
    # split=bf16x3: the dense split operands (K tripled, bf16) and one fp32 term per row and column
    a = lambda v: (v + 255) // 256 * 256  # noqa: E731
    p = lib.Plan("ij,jk->ik:sqdiff:sum:split=bf16x3", [8192, 256, 8192], [8, 1, 1, 8])
    assert p.kernel == "tc_split3"
    # + the statistics' partials: 256 row tiles of 32, 8 chunks of the 256 contracted indices at most -> 1
    # + the guard words of the expansion, one per 128 x 128 output tile
    assert p.workspace_bytes == (a(8192 * 768 * 2) + a(8192 * 768 * 2) + a(8192 * 4) + a(8192 * 4) + 256 + a(8192 * 4)
                                 + a(64 * 64 * 4 + 4))
    assert lib.Plan("ij,jk->ik:add:lse:split=bf16x3", [256, 64, 384], [2, 2, 2, 3]).kernel == "tc_split3"
    p = lib.Plan("bij,bjk->bik:sqdiff:sum:split=bf16x3", [3, 130, 24, 96], [3, 2, 1, 3, 1, 3])
    assert p.kernel == "tc_split3"
    # padded to the GEMM's tiles: M 130 -> 256, N 96 -> 128, 3K = 72 -> 128
    assert p.workspace_bytes == (a(3 * 256 * 128 * 2) + a(3 * 128 * 128 * 2) + a(3 * 130 * 4) + a(3 * 96 * 4) + 256
                                 + a(3 * 130 * 4) + a(3 * 2 * 1 * 4 + 4))
    # the cost terms are the plan's own (the split changes how, not what, is computed)
    q = lib.Plan("ij,jk->ik:sqdiff:sum", [8192, 256, 8192], [8, 1, 1, 8])
    p = lib.Plan("ij,jk->ik:sqdiff:sum:split=bf16x3", [8192, 256, 8192], [8, 1, 1, 8])
    assert (p.n_tasks, p.cost_join, p.cost_agg) == (q.n_tasks, q.cost_join, q.cost_agg)
    assert lib.Plan("ij,jk->ik:sqdiff:sum:split=none", [64, 64, 64], [1, 1, 1, 1]).kernel == "semiring_f32"


@pytest.mark.parametrize("spec,bounds,d,code", [
    ("ij,jk->ik:sqdiff:sum:in=bf16:split=bf16x3", [64, 64, 64], [1, 1, 1, 1], "TRA_ERR_UNSUPPORTED"),
    ("ij,jk->ik:mul:sum:split=bf16x3", [64, 64, 64], [1, 1, 1, 1], "TRA_ERR_UNSUPPORTED"),
    ("ij,jk->ik:add:max:split=bf16x3", [64, 64, 64], [1, 1, 1, 1], "TRA_ERR_UNSUPPORTED"),
    ("ij,jk->ik:sqdiff:sum:split=bf16x2", [64, 64, 64], [1, 1, 1, 1], "TRA_ERR_PARSE"),
    ("ij,jk->ik:sqdiff:sum:split=bf16x3", [300, 96, 200], [2, 1, 1, 2], "TRA_ERR_UNSUPPORTED"),  # N blocks of 100
    ("ij,jk->ki:add:lse:split=bf16x3", [64, 64, 64], [1, 1, 1, 1], "TRA_ERR_UNSUPPORTED"),  # Z contiguous along M
    ("ij,jk->ik:add:lse:split=bf16x3:mode=literal", [64, 64, 64], [1, 1, 1, 1], None),
])
def test_split3_plan_errors(lib, spec, bounds, d, code):
    if code is None:  # literal mode takes precedence: the pages' two-phase form
        assert lib.Plan(spec, bounds, d).kernel == "literal"
        return
    with pytest.raises(lib.TraError) as e:
        lib.Plan(spec, bounds, d)
    assert code in str(e.value)


@pytest.mark.parametrize("spec,bounds,d,code", [
    ("ij,jk->ik:mul:sum", [64, 64, 64], [3, 1, 1, 1], "TRA_ERR_DIVISIBILITY"),
    ("ij,jk->ik:mul:sum", [64, 64, 64], [1, 2, 4, 1], "TRA_ERR_SHARED_LABEL_D"),
    ("ij,jk->ik:mul:sum", [64, 64], [1, 1, 1, 1], "TRA_ERR_RANK"),
    ("ij,jk->ik:mul:sum", [64, 64, 64], [1, 1, 1], "TRA_ERR_RANK"),
    ("ij,jk->ik:pow:sum", [64, 64, 64], [1, 1, 1, 1], "TRA_ERR_PARSE"),
    ("ij,jk->ik:mul:avg", [64, 64, 64], [1, 1, 1, 1], "TRA_ERR_PARSE"),
    ("ij,jk:mul:sum", [64, 64, 64], [1, 1, 1, 1], "TRA_ERR_PARSE"),
    ("ii,ik->ik:mul:sum", [64, 64], [1, 1, 1, 1], "TRA_ERR_PARSE"),
    ("ij,jk->iz:mul:sum", [64, 64, 64], [1, 1, 1, 1], "TRA_ERR_PARSE"),
    ("ij,jk->ik:mul:none", [64, 64, 64], [1, 1, 1, 1], "TRA_ERR_PARSE"),
    ("ij,jk->ik:mul:sum:alpha=x", [64, 64, 64], [1, 1, 1, 1], "TRA_ERR_PARSE"),
    ("ij,jk->ik:mul:sum:foo=1", [64, 64, 64], [1, 1, 1, 1], "TRA_ERR_PARSE"),
    ("ij,jk->ik:mul:sum", [64, -1, 64], [1, 1, 1, 1], "TRA_ERR_ARG"),
    ("ij,jk->ik:mul:sum:ksplit=on", [64, 64, 64], [1, 1, 1, 1], "TRA_ERR_PARSE"),
    ("ij,jk->ik:mul:sum:in=bf16:tc=pair", [384, 128, 256], [1, 1, 1, 1], "TRA_ERR_UNSUPPORTED"),
    ("ij,jk->ik:mul:sum:tc=both", [256, 128, 256], [1, 1, 1, 1], "TRA_ERR_PARSE"),
    ("ij,jk->ik:mul:sum:tc_n=64", [256, 128, 256], [1, 1, 1, 1], "TRA_ERR_PARSE"),
    ("ij,jk->ik:mul:sum:in=bf16:tc=pair:tc_n=256", [256, 128, 384], [1, 1, 1, 1], "TRA_ERR_UNSUPPORTED"),
])
def test_plan_errors(lib, spec, bounds, d, code):
    with pytest.raises(lib.TraError) as e:
        lib.Plan(spec, bounds, d)
    assert code in str(e.value)
    assert lib.ein_last_error() != ""


def test_repartition_cost_matches_bruteforce(lib):
    shape = (4, 4, 4, 4)
    ds = [[4, 1, 4, 1], [1, 4, 1, 4], [2, 2, 2, 2], [1, 1, 1, 1], [4, 4, 1, 1], [2, 1, 1, 4]]
    for a in ds:
        for b in ds:
            assert lib.repartition_cost(shape, a, b) == otra.repartition_cost_bruteforce(shape, a, b)
    shape = (6, 4, 10)
    for a, b in [([3, 2, 5], [1, 4, 2]), ([2, 1, 1], [6, 4, 10]), ([1, 2, 5], [3, 1, 1])]:
        assert lib.repartition_cost(shape, a, b) == otra.repartition_cost_bruteforce(shape, a, b)
    # the 4-D contraction's output, 64^4 under [4,1,4,1] -> [1,4,1,4]
    assert lib.repartition_cost((64,) * 4, [4, 1, 4, 1], [1, 4, 1, 4]) == 16777216 - 16 * 16 ** 4
    with pytest.raises(lib.TraError):
        lib.repartition_cost((6, 4), [4, 1], [1, 1])


def test_repartition_cost_scatter_gather_golden(lib):
    # rkmt.cn/news/51250.html: Scatter / Gather move (N-1)/N of the variable (M elements over N
    # nodes); the library's term between the centralized layout (d all ones) and N blocks, both ways
    with open(os.path.join(os.path.dirname(__file__), "golden", "repartition_scatter_gather.json")) as f:
        gold = json.load(f)
    for c in gold["cases"]:
        ones = [1] * len(c["shape"])
        assert lib.repartition_cost(c["shape"], ones, c["d"]) == c["cost"], c
        assert lib.repartition_cost(c["shape"], c["d"], ones) == c["cost"], c


def test_execute_argument_errors(lib):
    p = lib.Plan("ij,jk->ik:add:lse", [64, 64, 64], [1, 1, 1, 1])
    with pytest.raises(lib.TraError) as e:
        lib.ein_execute(p.handle, 0x1000, 0x2000, 0x3000, None, 0, 0)
    assert "TRA_ERR_WORKSPACE" in str(e.value)
    with pytest.raises(lib.TraError) as e:
        lib.ein_execute(p.handle, None, 0x2000, 0x3000, None, 0, 0)
    assert "TRA_ERR_ARG" in str(e.value)
    q = lib.Plan("ij,jk->ik:mul:sum", [64, 64, 64], [1, 1, 1, 1])
    with pytest.raises(lib.TraError) as e:
        lib.ein_execute(q.handle, 0x1000, None, 0x3000, None, 0, 0)
    assert "TRA_ERR_ARG" in str(e.value)
    with pytest.raises(lib.TraError) as e:
        lib.ein_repartition([6, 4], [4, 1], [1, 1], 4, 0x1000, 0x2000, 0)
    assert "TRA_ERR_DIVISIBILITY" in str(e.value)
    with pytest.raises(lib.TraError) as e:
        lib.ein_repartition([6, 4], [1, 1], [2, 1], 3, 0x1000, 0x2000, 0)
    assert "TRA_ERR_ARG" in str(e.value)


def test_attention_function_survives_the_eingraph_import(lib):
    # the attention-EinGraph module is imported beside the package-level attention() call; the
    # import must not rebind the name
    import types

    import tensor_relational_algebra_gb300.eingraph  # noqa: F401

    assert callable(lib.attention) and not isinstance(lib.attention, types.ModuleType)



def test_maximum_sizes(lib):
    # tensors of up to 2^31 - 1 elements plan; one element more is refused, as is a bound past
    # 2^31 - 1; cost terms are 64-bit (n_tasks * (|X_sub| + |Y_sub|) passes 2^31 here)
    big = 2 ** 31 - 1
    p = lib.Plan("ij,jk->ik:add:max", [big, 1, 1], [1, 1, 1, 1])
    assert p.info.x_sub == big and p.info.z_sub == big and p.cost_join == big + 1
    q = lib.Plan("ij,jk->ik:mul:sum", [65536, 16384, 2], [8, 1, 1, 2])
    assert q.n_tasks == 16 and q.cost_join == 16 * (8192 * 16384 + 16384) > 2 ** 31
    for spec, bounds, d, code in [
        ("ij,jk->ik:add:max", [2 ** 31, 1, 1], [1, 1, 1, 1], "TRA_ERR_ARG"),
        ("ij,jk->ik:add:max", [65536, 32768, 1], [1, 1, 1, 1], "TRA_ERR_UNSUPPORTED"),
        ("bij,bjk->bik:add:max", [2, 46341, 46341, 1], [1, 1, 1, 1, 1, 1], "TRA_ERR_UNSUPPORTED"),
    ]:
        with pytest.raises(lib.TraError) as e:
            lib.Plan(spec, bounds, d)
        assert code in str(e.value), (spec, bounds)
    with pytest.raises(lib.TraError) as e:
        lib.ein_repartition([65536, 32768], [1, 1], [2, 1], 4, 0x1000, 0x2000, 0)
    assert "TRA_ERR_UNSUPPORTED" in str(e.value)


def test_back_to_back_detection():
    # the attention EinGraph batches its three projections only when Q, K, V (and the three
    # weight relations) are contiguous views that follow each other in one buffer
    import torch

    from tensor_relational_algebra_gb300.eingraph import AttentionGraph

    buf = torch.zeros(30, dtype=torch.bfloat16)
    assert AttentionGraph.back_to_back(buf[:10], buf[10:20], buf[20:])
    assert not AttentionGraph.back_to_back(buf[:10], buf[20:], buf[10:20])          # out of order
    assert not AttentionGraph.back_to_back(buf[:10], buf[10:20], torch.zeros(10, dtype=torch.bfloat16))
    assert not AttentionGraph.back_to_back(buf[:10], buf[10:19], buf[19:29])        # sizes differ
    assert not AttentionGraph.back_to_back(buf[:10], buf[10:20].float(), buf[20:])  # dtypes differ
    strided = torch.zeros(60, dtype=torch.bfloat16)[::2]
    assert not AttentionGraph.back_to_back(strided[:10], strided[10:20], strided[20:])  # not contiguous


def test_check_build_is_selected_by_the_environment(lib):
    # TRA_CHECK=1 makes the binding load libtra_check.so, whose ein_build_flags reports the
    # bounds-checked kernels; the default library reports none (no GPU needed to ask)
    import subprocess
    import sys

    from tensor_relational_algebra_gb300 import _build

    _build.build(check=True)
    code = ("import tensor_relational_algebra_gb300 as t; l = t.load(); "
            "print(l.ein_build_flags(), t._LIB_PATH.endswith('libtra_check.so'))")
    out = {}
    for flag in ("0", "1"):
        r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True,
                           env=dict(os.environ, TRA_CHECK=flag))
        assert r.returncode == 0, r.stderr
        out[flag] = r.stdout.split()
    assert out["0"] == ["0", "False"]
    assert out["1"] == ["1", "True"]


def test_tensor_maps_merge_contiguous_dimensions(lib):
    """The tensor-core planner describes a relation to TMA as at most five dimensions.  The 4-D
    contraction's output C[a,b,c,d] under d = [4,1,4,1] has six physical dimensions, but the local
    part of a runs on into b and the local part of c into d, both in memory and in their composite
    index, so they merge and the output gets a tensor map (TMA-store epilogue).  With b or d split
    the local parts are no longer contiguous with their neighbours and no map fits."""
    spec = "abef,cfed->abcd:mul:sum:in=bf16"
    assert lib.Plan(spec + ":tc_store=tma", [64] * 6, [4, 1, 1, 1, 4, 1, 1, 1]).kernel == "tc_bf16_pair"
    for d in ([1, 2, 1, 1, 1, 1, 1, 2], [2, 2, 1, 1, 2, 1, 1, 2]):
        with pytest.raises(lib.TraError) as e:
            lib.Plan(spec + ":tc_store=tma", [64] * 6, d)
        assert "TRA_ERR_UNSUPPORTED" in str(e.value)
