"""Tensor-core (tcgen05) BF16 sum-of-products path against the oracle, and the bounded-wait hook.

"EinDecomp ... tensor relational algebra", section 2.2: the join of key-matched
BF16 sub-tensors through multiply and the sum aggregation over contracted keys.
Shapes here are small but span several tiles, both operand majors (K innermost
or M / N innermost), split contracted keys, batch labels, alpha and bf16 output.
"""
import numpy as np
import pytest

import oracle
from oracle import rounding

from gpu_helpers import BF16_SUM_REL, FP32_REL, as_f64, check_bf16_bar, check_sum, gen, run_plan

pytestmark = pytest.mark.gpu


def labels_of(eq):
    ins, out = eq.split("->")[0].split(","), eq.split("->")[1]
    order = []
    for c in "".join(ins):
        if c not in order:
            order.append(c)
    return ins, out, order


CASES = [
    # eq, bounds (first-appearance order), d, options
    ("ij,jk->ik", [256, 192, 128], [2, 3, 3, 2], ""),               # K-major A, N-major B, split K keys
    ("ij,jk->ik", [384, 256, 512], [1, 1, 1, 1], ""),               # N tile 256
    ("ji,jk->ik", [128, 256, 192], [2, 1, 2, 3], ""),               # M-major A
    ("ij,kj->ik", [256, 128, 256], [2, 2, 2, 2], ""),               # K-major B
    ("ji,kj->ik", [128, 256, 128], [1, 2, 1, 1], ""),               # both MN / K majors swapped
    ("bij,bjk->bik", [3, 128, 128, 192], [3, 1, 2, 3, 2, 3], ""),   # batch label split into keys
    ("abef,cfed->abcd", [4, 32, 8, 64, 4, 64], [2, 1, 1, 1, 2, 1, 1, 1], ""),
    ("sa,ahd->shd", [256, 128, 2, 128], [2, 1, 1, 1, 1], ":out=bf16"),
    ("shd,thd->hst", [256, 2, 128, 256], [1, 2, 1, 1, 2, 1], ":alpha=0.08838834764831845"),
    ("hst,thd->shd", [2, 256, 256, 128], [2, 1, 1, 1, 2, 1], ":out=bf16"),
    ("shd,ahd->sa", [256, 2, 128, 128], [1, 1, 1, 1, 1, 1], ""),
]

# 256 x 256 tiles on a cluster of two CTAs: each CTA loads half of the X rows and half of
# the Y rows of a tile; the tensor-core instruction reads both CTAs' shared memory.
PAIR_CASES = [
    ("ij,jk->ik", [256, 192, 256], [2, 3, 3, 2], ""),               # one Y key block per CTA
    ("ij,jk->ik", [512, 256, 768], [1, 1, 1, 1], ""),               # 2 x 3 tiles
    ("ji,jk->ik", [128, 256, 256], [2, 1, 2, 2], ""),               # M-major A
    ("ij,kj->ik", [256, 128, 256], [2, 2, 2, 2], ""),               # K-major B
    ("ji,kj->ik", [64, 256, 512], [1, 2, 1, 1], ""),                # both majors swapped
    ("bij,bjk->bik", [3, 256, 128, 256], [3, 1, 2, 3, 2, 1], ""),   # batch label split into keys
    ("bij,bjk->bik", [24, 512, 64, 512], [1, 1, 1, 1, 1, 1], ""),   # 96 tiles: clusters take several
    ("abef,cfed->abcd", [4, 64, 8, 64, 4, 64], [2, 1, 1, 1, 2, 1, 1, 1], ""),
    ("sa,ahd->shd", [256, 128, 2, 128], [2, 1, 1, 1, 1], ":out=bf16"),
    ("shd,thd->hst", [256, 2, 128, 256], [1, 2, 1, 1, 2, 1], ":alpha=0.08838834764831845"),
    ("shd,ahd->sa", [256, 2, 128, 256], [1, 1, 1, 1, 1, 1], ""),
    # 256 x 128 tiles: each CTA loads 64 rows of Y per K step
    ("ij,jk->ik", [256, 128, 128], [2, 1, 1, 2], ""),               # N-major B, one 64-wide box
    ("ij,kj->ik", [512, 192, 384], [1, 3, 1, 3], ""),               # K-major B, 3 column tiles
    ("hst,thd->shd", [2, 256, 256, 128], [2, 1, 1, 1, 2, 1], ":out=bf16"),  # attention A.V
]


def _tc_case(lib, eq, bounds, d, opts, kernel):
    ins, out, order = labels_of(eq)
    B = dict(zip(order, bounds))
    X = gen(tuple(B[c] for c in ins[0]), 9, 0, bf16=True)
    Y = gen(tuple(B[c] for c in ins[1]), 9, 1, bf16=True)
    spec = f"{eq}:mul:sum:in=bf16{opts}"
    alpha = 1.0
    if "alpha=" in opts:
        alpha = float(opts.split("alpha=")[1].split(":")[0])
    p, g = run_plan(lib, spec, bounds, d, X, Y, out_bf16=":out=bf16" in opts)
    assert p.kernel == kernel
    r = oracle.einsum(eq, as_f64(X), as_f64(Y), alpha=alpha)
    S = oracle.einsum(eq, np.abs(as_f64(X)), np.abs(as_f64(Y))) * abs(alpha)
    check_bf16_bar(g, r)
    if ":out=bf16" in opts:
        # one bf16 rounding of the fp32 accumulator: within half a bf16 ulp plus the sum error
        assert np.all(np.abs(g - r) <= 2.0 ** -8 * np.abs(r) + FP32_REL * S)
    else:
        check_sum(g, r, S, FP32_REL)


def _store_or_skip(lib, spec, bounds, d):
    try:
        lib.Plan(spec, bounds, d)
    except lib.TraError as e:
        assert "TRA_ERR_UNSUPPORTED" in str(e)
        pytest.skip("no tiling with this epilogue / width")


@pytest.mark.parametrize("store", [":tc_store=tma", ":tc_store=lsu"])
@pytest.mark.parametrize("eq,bounds,d,opts", CASES)
def test_tc_parity(lib, cuda, eq, bounds, d, opts, store):
    # the epilogue stores through an output tensor map (TMA) or with warp stores
    _store_or_skip(lib, f"{eq}:mul:sum:in=bf16{opts}:tc=single{store}", bounds, d)
    _tc_case(lib, eq, bounds, d, opts + ":tc=single" + store, "tc_bf16")


@pytest.mark.parametrize("store", [":tc_store=tma", ":tc_store=lsu"])
@pytest.mark.parametrize("width", ["", ":tc_n=256", ":tc_n=128"])
@pytest.mark.parametrize("eq,bounds,d,opts", PAIR_CASES)
def test_tc_pair_parity(lib, cuda, eq, bounds, d, opts, width, store):
    # default width and both forced widths, each with both epilogues
    _store_or_skip(lib, f"{eq}:mul:sum:in=bf16{opts}:tc=pair{width}{store}", bounds, d)
    _tc_case(lib, eq, bounds, d, opts + ":tc=pair" + width + store, "tc_bf16_pair")


def test_tc_repeat_and_stream(lib, cuda):
    # back-to-back launches on a side stream reuse the persistent schedule correctly
    import torch

    X = gen((512, 256), 10, 0, bf16=True)
    Y = gen((256, 512), 10, 1, bf16=True)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        outs = [run_plan(lib, "ij,jk->ik:mul:sum:in=bf16", [512, 256, 512], [2, 2, 2, 2], X, Y)[1] for _ in range(3)]
    torch.cuda.synchronize()
    for o in outs[1:]:
        np.testing.assert_array_equal(o, outs[0])
    r = oracle.einsum("ij,jk->ik", as_f64(X), as_f64(Y))
    check_sum(outs[0], r, oracle.einsum("ij,jk->ik", np.abs(as_f64(X)), np.abs(as_f64(Y))), FP32_REL)


def test_bounded_wait_gives_up(lib, cuda):
    lib.ein_status()  # clean status word
    lib.ein_selftest_wait_timeout(2_000_000)  # 2 ms on a barrier nothing arrives on
    with pytest.raises(lib.TraError) as e:
        lib.ein_status()
    assert "TRA_ERR_TIMEOUT" in str(e.value)
    lib.ein_status()  # cleared; the context is still usable
    X = gen((128, 64), 11, 0, bf16=True)
    Y = gen((64, 128), 11, 1, bf16=True)
    _, g = run_plan(lib, "ij,jk->ik:mul:sum:in=bf16", [128, 64, 128], [1, 1, 1, 1], X, Y)
    check_sum(g, oracle.einsum("ij,jk->ik", as_f64(X), as_f64(Y)),
              oracle.einsum("ij,jk->ik", np.abs(as_f64(X)), np.abs(as_f64(Y))), FP32_REL)
