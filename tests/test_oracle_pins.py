"""Pins for the CPU oracle: each check compares it with something other than itself.

The oracle follows "EinDecomp: automatic tensor-parallel decomposition via
Einstein summation + tensor relational algebra" (sections 2.1, 2.2, 3.1, 3.2)
and the ColossalAI 2.5D page's block equations.  Pins used here: numpy /
scipy library routines on special cases, closed forms, invariants (result
independent of the partition vector, softmax rows summing to one), brute force
on tiny inputs and the hand-derived values under ``tests/golden``.
"""
import json
import math
import os

import numpy as np
import pytest

import datagen
import oracle
from oracle import tra, rounding, mha

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def rng_arrays(*shapes, seed=0):
    return [datagen.uniform_f32(s, seed, t) for t, s in enumerate(shapes)]


# ---------------------------------------------------------------- generator
def test_philox_known_answers():
    # Known-answer vectors published with the Random123 library (Salmon et al., SC'11).
    cases = [
        ([0, 0, 0, 0], [0, 0], [0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8]),
        ([0xFFFFFFFF] * 4, [0xFFFFFFFF] * 2, [0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD]),
        ([0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344], [0xA4093822, 0x299F31D0],
         [0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1]),
    ]
    for ctr, key, want in cases:
        assert list(datagen.philox4x32_10(ctr, key)) == want


def test_generator_distributions():
    u = datagen.uniform_f32((200000,), 0, 0)
    assert u.min() >= -1 and u.max() < 1 and abs(u.mean()) < 0.01
    n = datagen.normal_f32((200000,), 0, 1, 0.0, 0.02)
    assert abs(n.mean()) < 1e-3 and abs(n.std() - 0.02) < 1e-3
    b = datagen.normal_bf16((1000,), 3, 4)
    f = datagen.normal_f32((1000,), 3, 4)
    np.testing.assert_array_equal(datagen.bf16_bits_to_f32(b), rounding.to_bf16(f))


# ---------------------------------------------------------------- rounding
def test_bf16_round_to_nearest_even():
    vals = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -8 + 2.0 ** -20, -2.5, 3.0e38])
    got = rounding.to_bf16(vals)
    want = np.array([1.0, 1.0 + 2.0 ** -6, 1.0 + 2.0 ** -7, -2.5, np.float32(3.0e38)], dtype=np.float64)
    # 3.0e38 -> nearest bf16: 0x7F62 = 2.9980e38 (7 fraction bits)
    want[4] = float(np.uint32(0x7F620000).view(np.float32))
    np.testing.assert_array_equal(got.astype(np.float64), want)


# ---------------------------------------------------------------- extended EinSum (section 2.1)
@pytest.mark.parametrize("eq,shapes", [
    ("ij,jk->ik", [(7, 5), (5, 9)]),
    ("abef,cfed->abcd", [(3, 2, 4, 5), (2, 5, 4, 3)]),
    ("shd,thd->hst", [(6, 3, 4), (5, 3, 4)]),
    ("hst,thd->shd", [(3, 6, 5), (5, 3, 4)]),
    ("shd,ahd->sa", [(6, 3, 4), (7, 3, 4)]),
    ("sa,ahd->shd", [(6, 7), (7, 3, 4)]),
])
def test_sum_mul_matches_numpy_einsum(eq, shapes):
    X, Y = rng_arrays(*shapes, seed=11)
    got = oracle.einsum(eq, X, Y)
    want = np.einsum(eq, X.astype(np.float64), Y.astype(np.float64))
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_transposed_operand_is_caught():
    # a plausible mistake (operand used transposed) must not pass the pin above
    X, Y = rng_arrays((6, 6), (6, 6), seed=5)
    wrong = oracle.einsum("ij,jk->ik", X, Y.T.copy())
    want = np.einsum("ij,jk->ik", X.astype(np.float64), Y.astype(np.float64))
    assert np.abs(wrong - want).max() > 1e-3


def test_elementwise_broadcast_addition():
    # section 2.1 element-wise example Z[i,j] = X[i,j] + Y[i,j]; no label contracted
    X, Y = rng_arrays((5, 7), (5, 7), seed=2)
    got = oracle.einsum("ij,ij->ij", X, Y, op="add", agg="none")
    np.testing.assert_array_equal(got, X.astype(np.float64) + Y.astype(np.float64))
    with pytest.raises(ValueError):
        oracle.einsum("ij,jk->ik", X, Y.T.copy(), op="add", agg="none")


def test_squared_distance_closed_form():
    # D[i,k] = sum_j (X[i,j]-Y[j,k])^2 = |x_i|^2 + |y_k|^2 - 2 x_i . y_k
    X, Y = rng_arrays((9, 13), (13, 11), seed=3)
    got = oracle.einsum("ij,jk->ik", X, Y, op="sqdiff", agg="sum")
    x, y = X.astype(np.float64), Y.astype(np.float64)
    closed = (x * x).sum(1)[:, None] + (y * y).sum(0)[None, :] - 2 * x @ y
    np.testing.assert_allclose(got, closed, rtol=1e-12, atol=1e-12)
    brute = ((x[:, :, None] - y[None, :, :]) ** 2).sum(1)
    np.testing.assert_allclose(got, brute, rtol=1e-13)


@pytest.mark.parametrize("agg,red", [("max", np.max), ("min", np.min)])
def test_max_min_plus_exact(agg, red):
    X, Y = rng_arrays((8, 16), (16, 10), seed=4)
    got = oracle.einsum("ij,jk->ik", X, Y, op="add", agg=agg)
    # an fp32 + fp32 sum is exact in double; one rounding gives the fp32 result
    want = red(X[:, :, None].astype(np.float64) + Y[None, :, :].astype(np.float64), axis=1)
    np.testing.assert_array_equal(got, want)
    f32 = red(X[:, :, None] + Y[None, :, :], axis=1)
    np.testing.assert_array_equal(rounding.to_f32(got), f32)


def test_logsumexp_matches_scipy():
    from scipy.special import logsumexp

    X, Y = rng_arrays((6, 40), (40, 7), seed=6)
    X, Y = 30 * X, 30 * Y
    got = oracle.einsum("ij,jk->ik", X, Y, op="add", agg="lse")
    want = logsumexp(X[:, :, None].astype(np.float64) + Y[None, :, :].astype(np.float64), axis=1)
    np.testing.assert_allclose(got, want, rtol=1e-13)
    S = datagen.normal_f32((3, 4, 50), 0, 9) * 40
    np.testing.assert_allclose(oracle.einsum("hst->hs", S, agg="lse"), logsumexp(S.astype(np.float64), axis=2),
                               rtol=1e-13)


def test_expsub_broadcast_join():
    S = datagen.normal_f32((3, 4, 5), 0, 1)
    L = datagen.normal_f32((3, 4), 0, 2)
    got = oracle.einsum("hst,hs->hst", S, L, op="expsub", agg="none")
    np.testing.assert_allclose(got, np.exp(S.astype(np.float64) - L[:, :, None]), rtol=1e-15)


def test_alpha_applies_after_aggregation():
    X, Y = rng_arrays((4, 6), (6, 5), seed=8)
    mx = oracle.einsum("ij,jk->ik", X, Y, op="add", agg="max")
    np.testing.assert_array_equal(oracle.einsum("ij,jk->ik", X, Y, op="add", agg="max", alpha=-1.0), -mx)


@pytest.mark.parametrize("op,agg,lib_red", [
    ("mul", "sum", lambda v: np.sum(v, axis=1)),
    ("add", "max", lambda v: np.max(v, axis=1, initial=-np.inf)),
    ("add", "min", lambda v: np.min(v, axis=1, initial=np.inf)),
    ("add", "lse", None),
])
def test_empty_contraction_gives_the_identity(op, agg, lib_red):
    # aggregating an empty set gives the aggregation's identity: numpy's empty sum is 0 and its
    # max / min with an initial value return that value; logsumexp of nothing is log(0) = -inf
    from scipy.special import logsumexp

    X = np.zeros((3, 0), np.float32)
    Y = np.zeros((0, 4), np.float32)
    got = oracle.einsum("ij,jk->ik", X, Y, op=op, agg=agg)
    v = X[:, :, None].astype(np.float64) + Y[None, :, :].astype(np.float64)
    if lib_red is not None:
        want = lib_red(v)
    else:
        with np.errstate(divide="ignore"):
            want = logsumexp(v, axis=1)
    assert got.shape == (3, 4)
    np.testing.assert_array_equal(got, want)
    np.testing.assert_array_equal(oracle.einsum("ij,jk->ik", X, Y, op=op, agg=agg, alpha=-2.0), -2.0 * want)
    # an empty output label: no output element at all
    assert oracle.einsum("ij,jk->ik", np.zeros((0, 5), np.float32), np.ones((5, 4), np.float32), op=op,
                         agg=agg).shape == (0, 4)


def test_points_equal_full():
    X, Y = rng_arrays((9, 5, 4), (7, 5, 4), seed=9)
    full = oracle.einsum("shd,thd->hst", X, Y, alpha=0.25)
    pts = np.array([0, 3, 17, full.size - 1, 100])
    np.testing.assert_array_equal(oracle.einsum_points("shd,thd->hst", X, Y, pts, alpha=0.25), full.reshape(-1)[pts])


# ---------------------------------------------------------------- relations (section 2.2)
def test_key_range_and_block_layout_golden():
    g = json.load(open(os.path.join(GOLD, "block_layout_4x4.json")))
    T = np.arange(16, dtype=np.float32).reshape(4, 4)
    for c in g["cases"]:
        np.testing.assert_array_equal(tra.block(T, c["d"]), np.array(c["blocked"], dtype=np.float32))
        np.testing.assert_array_equal(tra.unblock(tra.block(T, c["d"]), (4, 4), c["d"]), T)
    for kr in g["key_range"]:
        r = tra.key_range(kr["k"], kr["B"], kr["D"])
        assert [r.start, r.stop] == kr["range"]
    with pytest.raises(ValueError):
        tra.key_range(0, 10, 4)


def test_repartition_roundtrip():
    T = datagen.uniform_f32((8, 4, 6), 1, 2)
    b = tra.block(T, [2, 1, 3])
    r = tra.repartition(b, T.shape, [2, 1, 3], [1, 4, 2])
    np.testing.assert_array_equal(r, tra.block(T, [1, 4, 2]))
    np.testing.assert_array_equal(tra.repartition(r, T.shape, [1, 4, 2], [2, 1, 3]), b)


# ---------------------------------------------------------------- plan, task count, cost (sections 3.1, 3.2)
def test_plan_golden_costs():
    g = json.load(open(os.path.join(GOLD, "cost_terms.json")))
    for c in g["cases"]:
        p = tra.plan_bruteforce(c["eq"], c["bounds"], c["d"])
        for k in ("n_tasks", "n_groups", "n_agg", "x_sub", "y_sub", "z_sub", "cost_join", "cost_agg"):
            assert p[k] == c[k], (c["eq"], c["d"], k)
        # closed forms of section 3.1 with P = number of join tuples
        P = p["n_tasks"]
        assert p["cost_join"] == P * (p["x_sub"] + p["y_sub"])
        assert p["cost_agg"] * p["n_agg"] == P * (p["n_agg"] - 1) * p["z_sub"]


def test_aggregation_cost_equals_reduce_traffic():
    # communication page, primitive table: a Reduce of an M-element message over N
    # participants moves (N-1)*M.  Row-split matmul (d=[1,P,P,1]) has n_agg = P and one
    # group of the whole output, so its aggregation term must equal (P-1)*|Z|.
    for P in (2, 4, 8):
        p = tra.plan_bruteforce("ij,jk->ik", {"i": 32, "j": 64, "k": 16}, [1, P, P, 1])
        assert p["n_agg"] == P and p["n_groups"] == 1
        assert p["cost_agg"] == (P - 1) * 32 * 16


def test_summa_2p5d_key_pairing():
    g = json.load(open(os.path.join(GOLD, "summa_2p5d_pairs.json")))
    p = tra.plan_bruteforce(g["eq"], {"i": 8, "j": 4, "k": 4}, g["d"])
    got = {}
    for kx, ky, kz in p["tasks"]:
        got.setdefault(",".join(map(str, kz)), []).append([list(kx), list(ky)])
    assert got == g["groups"]


def test_task_order_and_join_condition():
    p = tra.plan_bruteforce("abef,cfed->abcd", {c: 4 for c in "abcdef"}, [2, 1, 2, 1, 2, 1, 2, 1])
    assert p["n_tasks"] == 2 * 2 * 2 * 1 * 1 * 1 * 1  # a, e split (X); c, e(shared) (Y)
    for kx, ky, kz in p["tasks"]:
        assert kx[2] == ky[2]  # e shared: positions 2 in X (a,b,e,f) and 2 in Y (c,f,e,d)
        assert kx[3] == ky[1]  # f shared
        assert kz == (kx[0], kx[1], ky[0], ky[3])
    zs = [kz for _, _, kz in p["tasks"]]
    assert zs == sorted(zs)
    with pytest.raises(ValueError):
        tra.plan_bruteforce("ij,jk->ik", {"i": 4, "j": 4, "k": 4}, [1, 2, 4, 1])
    with pytest.raises(ValueError):
        tra.plan_bruteforce("ij,jk->ik", {"i": 4, "j": 6, "k": 4}, [1, 4, 4, 1])


# ---------------------------------------------------------------- literal TRA = definition, any d
@pytest.mark.parametrize("d", [[4, 1, 1, 4], [1, 4, 4, 1], [2, 2, 2, 2], [1, 1, 1, 1]])
@pytest.mark.parametrize("op,agg", [("mul", "sum"), ("add", "max"), ("add", "min"), ("add", "lse"), ("sqdiff", "sum")])
def test_partition_vector_invariance(d, op, agg):
    X, Y = rng_arrays((16, 16), (16, 16), seed=0)
    ref = oracle.einsum("ij,jk->ik", X, Y, op=op, agg=agg)
    got = tra.tra_literal("ij,jk->ik", X, Y, d, op=op, agg=agg)
    if agg in ("max", "min"):
        np.testing.assert_array_equal(got, ref)
    else:
        np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_literal_4d_contraction_and_unary():
    A, B = rng_arrays((4, 2, 4, 2), (4, 2, 4, 2), seed=1)
    ref = np.einsum("abef,cfed->abcd", A.astype(np.float64), B.astype(np.float64))
    got = tra.tra_literal("abef,cfed->abcd", A, B, [2, 1, 2, 1, 2, 1, 2, 1])
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)
    S = datagen.normal_f32((2, 4, 8), 0, 3)
    from scipy.special import logsumexp

    np.testing.assert_allclose(tra.tra_literal("hst->hs", S, None, [2, 2, 4], agg="lse"),
                               logsumexp(S.astype(np.float64), axis=2), rtol=1e-13)


# ---------------------------------------------------------------- repartition cost
def _divisor_vectors(shape):
    out = [[]]
    for B in shape:
        out = [v + [D] for v in out for D in range(1, B + 1) if B % D == 0]
    return out


def test_repartition_cost_scatter_gather_pin():
    # rkmt.cn/news/51250.html, traffic per communication primitive: Scatter (centralized ->
    # partitioned) and Gather (partitioned -> centralized) each move (N-1)/N of the variable.
    # d = all ones is the centralized tensor (one block, owned by block id 0); a d with
    # N = prod(D) blocks spreads it over N owners.  Every divisor vector of three tiny shapes,
    # both directions, element by element.
    for shape in [(4, 6), (2, 3, 4), (4, 4, 4, 4), (12,)]:
        ones = [1] * len(shape)
        n = int(np.prod(shape))
        for d in _divisor_vectors(shape):
            N = int(np.prod(d))
            want = (N - 1) * n // N
            assert (N - 1) * n % N == 0
            assert tra.repartition_cost_bruteforce(shape, ones, d) == want, (shape, d)
            assert tra.repartition_cost_bruteforce(shape, d, ones) == want, (shape, d)
    with open(os.path.join(GOLD, "repartition_scatter_gather.json")) as f:
        gold = json.load(f)
    for c in gold["cases"]:
        if c["M"] <= 1024:  # the brute force walks every element
            ones = [1] * len(c["shape"])
            assert tra.repartition_cost_bruteforce(c["shape"], ones, c["d"]) == c["cost"]
            assert tra.repartition_cost_bruteforce(c["shape"], c["d"], ones) == c["cost"]


def test_repartition_cost_pin_rejects_plausible_mistakes():
    # Negative controls for the pin above: rules a slip could produce, each evaluated by the
    # same element walk, must miss (N-1)/N * M on some divisor vector.
    def walk(shape, src, dst, rule):
        n = int(np.prod(shape))
        total = 0
        blocks = set()
        for flat in range(n):
            idx = np.unravel_index(flat, shape)
            own = []
            for d in (src, dst):
                key = [int(i) // (B // D) for i, B, D in zip(idx, shape, d)]
                lin = 0
                for k, D in zip(key, d):
                    lin = lin * D + k
                own.append((lin, int(np.prod(d))))
            if rule == "owner_from_first_index":  # the linear id dropped every dimension but the first
                k0 = [int(idx[0]) // (shape[0] // d[0]) for d in (src, dst)]
                changed = k0[0] != k0[1]
            else:
                changed = own[0][0] != own[1][0]
            if changed:
                total += 1
                blocks.add(own[1][0])
        return len(blocks) if rule == "count_blocks" else (2 * total if rule == "both_sides" else total)

    shape = (4, 6)
    for rule in ("owner_from_first_index", "count_blocks", "both_sides"):
        missed = False
        for d in _divisor_vectors(shape):
            N = int(np.prod(d))
            if walk(shape, [1, 1], d, rule) != (N - 1) * 24 // N:
                missed = True
        assert missed, rule


def test_repartition_cost_invariants():
    shape = (4, 4, 4, 4)
    ds = [[4, 1, 4, 1], [1, 4, 1, 4], [2, 2, 2, 2], [1, 1, 1, 1], [4, 4, 1, 1]]
    n = int(np.prod(shape))
    for a in ds:
        assert tra.repartition_cost_bruteforce(shape, a, a) == 0
        for b in ds:
            c = tra.repartition_cost_bruteforce(shape, a, b)
            assert 0 <= c <= n
            assert c == tra.repartition_cost_bruteforce(shape, b, a)
            if a != b:
                assert c > 0
    # [4,1,4,1] -> [1,4,1,4]: block L keeps the 1x1x1x1 corner it shares with block L
    assert tra.repartition_cost_bruteforce(shape, [4, 1, 4, 1], [1, 4, 1, 4]) == n - 16


# ---------------------------------------------------------------- attention chain (section 2.1)
def test_attention_chain_against_plain_softmax():
    s, a, h, d = 16, 24, 2, 8
    Q, K, V = [datagen.bf16_bits_to_f32(datagen.normal_bf16((s, a), 0, t)) for t in range(3)]
    WQ, WK, WV, WO = [datagen.bf16_bits_to_f32(datagen.normal_bf16((a, h, d), 0, 3 + t, 0, 0.2)) for t in range(4)]
    r = mha.chain(Q, K, V, WQ, WK, WV, WO)
    np.testing.assert_allclose(r["A"].astype(np.float64).sum(-1), 1.0, atol=2e-2)
    np.testing.assert_allclose(r["A"], mha.softmax_plain(r["S"]), rtol=8e-3, atol=1e-6)
    # the whole chain in plain double (no intermediate rounding), as a textbook MHA
    q = np.einsum("sa,ahd->shd", Q.astype(np.float64), WQ)
    k = np.einsum("sa,ahd->shd", K.astype(np.float64), WK)
    v = np.einsum("sa,ahd->shd", V.astype(np.float64), WV)
    sc = np.einsum("shd,thd->hst", q, k) / math.sqrt(d)
    o = np.einsum("hst,thd->shd", mha.softmax_plain(sc), v)
    out = np.einsum("shd,ahd->sa", o, WO)
    assert np.abs(r["out"] - out).max() <= 2e-2 * np.abs(out).max()
    rows = np.array([0, 5, 15])
    rr = mha.chain(Q, K, V, WQ, WK, WV, WO, rows=rows)
    np.testing.assert_array_equal(rr["out"], r["out"][rows])


def test_attention_engines_agree():
    # the library-matmul engine (used at full size) against the nested-loop engine
    s, a, h, d = 24, 32, 2, 16
    Q, K, V = [datagen.bf16_bits_to_f32(datagen.normal_bf16((s, a), 1, t)) for t in range(3)]
    WQ, WK, WV, WO = [datagen.bf16_bits_to_f32(datagen.normal_bf16((a, h, d), 1, 3 + t, 0, 0.2)) for t in range(4)]
    lo = mha.chain(Q, K, V, WQ, WK, WV, WO, engine="loops")
    bl = mha.chain(Q, K, V, WQ, WK, WV, WO, engine="blas")
    for k in ("Qp", "Kp", "Vp", "A", "O"):
        assert np.mean(lo[k] == bl[k]) > 0.99, k  # bf16 roundings agree except at rare ties
    np.testing.assert_allclose(bl["S"], lo["S"], rtol=1e-2, atol=1e-3)
    assert np.abs(bl["out"] - lo["out"]).max() <= 1e-2 * np.abs(lo["out"]).max()
