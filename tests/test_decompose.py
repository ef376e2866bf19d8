"""EinDecomp's partition-vector search over an EinGraph (sections 3.1-3.2), host only.

The library's dynamic programme is checked against the oracle's exhaustive search over every
combination of candidates: equal optimum on tree-shaped graphs, and on a graph where one node
feeds two consumers a result whose recounted cost matches the oracle's count of the same
assignment.  A hand-derived single-node case pins the oracle's search.
"""
import time

import pytest

from oracle import decomp as odec


def _tasks(eq, bounds, d):
    ins = eq.split("->")[0].split(",")
    order = []
    for s in ins:
        for c in s:
            if c not in order:
                order.append(c)
    D = {}
    for c, v in zip("".join(ins), d):
        assert D.setdefault(c, v) == v  # shared labels equal
    B = dict(zip(order, bounds))
    n = 1
    for c in order:
        assert B[c] % D[c] == 0
        n *= D[c]
    return n, D


CHAIN = [("ij,jk->ik:mul:sum", [4, 2, 4], (-1, -1)),
         ("ik,kl->il:mul:sum", [4, 4, 2], (0, -1)),
         ("il,lm->im:add:max", [4, 2, 4], (1, -1))]
TREE = [("ij,jk->ik:mul:sum", [4, 2, 4], (-1, -1)),
        ("ab,bc->ac:mul:sum", [4, 2, 4], (-1, -1)),
        ("ik,kl->il:mul:sum", [4, 4, 4], (0, 1))]


@pytest.mark.parametrize("graph", [CHAIN, TREE], ids=["chain", "binary-tree"])
@pytest.mark.parametrize("p_min,p_max,pow2", [(2, 2, False), (4, 4, False), (2, 8, True)])
def test_programme_matches_exhaustive_search_on_trees(lib, graph, p_min, p_max, pow2):
    r = lib.decompose(graph, p_min, p_max, pow2=pow2)
    best, _ = odec.search(graph, p_min, p_max, pow2)
    assert r["total_cost"] == best
    assert r["dp_cost"] == r["total_cost"]  # no node feeds two consumers
    eqs = [(s.split(":")[0], b, i) for s, b, i in graph]
    choice = [_tasks(eq, b, d)[1] for (eq, b, _), d in zip(eqs, r["d"])]
    assert odec.graph_cost(eqs, choice) == r["total_cost"]
    for (eq, b, _), d in zip(eqs, r["d"]):
        n, D = _tasks(eq, b, d)
        assert p_min <= n <= p_max
        if pow2:
            assert all(v & (v - 1) == 0 for v in D.values())


def test_dag_choice_is_counted_consistently(lib):
    # S feeds both the logsumexp and the broadcast join exp(S - L)
    dag = [("ij,jk->ik:mul:sum", [4, 2, 4], (-1, -1)),
           ("ik->i::lse", [4, 4], (0, -1)),
           ("ik,i->ik:expsub:none", [4, 4], (0, 1))]
    r = lib.decompose(dag, 2, 4)
    best, _ = odec.search(dag, 2, 4)
    eqs = [(s.split(":")[0], b, i) for s, b, i in dag]
    choice = [_tasks(eq, b, d)[1] for (eq, b, _), d in zip(eqs, r["d"])]
    assert odec.graph_cost(eqs, choice) == r["total_cost"]
    assert r["total_cost"] >= best
    assert sum(r["node_cost"]) == r["total_cost"]


def test_single_node_hand_derived():
    # ij,jk->ik with B = [4,4,4], P = 2: splitting i, j or k costs 2*(8+16)=48, 2*(8+8)+16=48,
    # 2*(16+8)=48 -- the minimum is 48
    best, d = odec.search([("ij,jk->ik:mul:sum", [4, 4, 4], (-1, -1))], 2, 2)
    assert best == 48
    assert d[0] in ([2, 1, 1, 1], [1, 2, 2, 1], [1, 1, 1, 2])


@pytest.mark.parametrize("nodes,p,code", [
    ([("ij,jk->ik:mul:sum", [4, 4, 4], (1, -1)), ("ij,jk->ik:mul:sum", [4, 4, 4], (-1, -1))], 2, "TRA_ERR_ARG"),
    ([("ij,jk->ik:mul:sum", [4, 4, 4], (-1, -1)), ("ij,jk->ik:mul:sum", [8, 4, 4], (0, -1))], 2, "TRA_ERR_ARG"),
    ([("ij,jk->ik:mul:sum", [4, 4, 4], (-1, -1))], 128, "TRA_ERR_UNSUPPORTED"),
    ([("ij,jk->ik:mul:pow", [4, 4, 4], (-1, -1))], 2, "TRA_ERR_PARSE"),
])
def test_errors(lib, nodes, p, code):
    with pytest.raises(lib.TraError) as e:
        lib.decompose(nodes, p)
    assert code in str(e.value)


def test_attention_eingraph_full_size(lib):
    # the pages' multi-head-attention EinGraph (s = a = 4096, h = 32, d = 128), P = 128 tasks
    s, a, h, d = 4096, 4096, 32, 128
    g = [("sa,ahd->shd:mul:sum", [s, a, h, d], (-1, -1)),       # 0 Q projection
         ("sa,ahd->shd:mul:sum", [s, a, h, d], (-1, -1)),       # 1 K projection
         ("sa,ahd->shd:mul:sum", [s, a, h, d], (-1, -1)),       # 2 V projection
         ("shd,thd->hst:mul:sum", [s, h, d, s], (0, 1)),        # 3 Scores
         ("hst->hs::lse", [h, s, s], (3, -1)),                  # 4 L
         ("hst,hs->hst:expsub:none", [h, s, s], (3, 4)),        # 5 Attn
         ("hst,thd->shd:mul:sum", [h, s, s, d], (5, 2)),        # 6 O
         ("shd,ahd->sa:mul:sum", [s, h, d, a], (6, -1))]        # 7 output projection
    t0 = time.perf_counter()
    r = lib.decompose(g, 128, pow2=True)
    assert time.perf_counter() - t0 < 60
    total = 0
    for (spec, bounds, inputs), dv, own in zip(g, r["d"], r["node_cost"]):
        n, _ = _tasks(spec.split(":")[0], bounds, dv)
        assert n == 128
        info = lib.Plan(spec, bounds, dv).info
        edge = own - info.cost_join - info.cost_agg
        assert edge >= 0
        total += own
    assert total == r["total_cost"]


# ---------------------------------------------------------------- cost-model variants (page section 4.3)

@pytest.mark.parametrize("shape,src,dst,want", [
    # [0,2),[2,4) -> [0,1),[1,2),[2,3),[3,4): overlapping pairs (0,0),(0,1),(1,2),(1,3); (0,0) keeps
    # its id -> 3 messages
    ([4], [2], [4], 3),
    # [0,3),[3,6) -> [0,2),[2,4),[4,6): pairs (0,0),(0,1),(1,1),(1,2); same-id (0,0),(1,1) -> 2
    ([6], [2], [3], 2),
    # row halves -> column halves of a 4 x 4: all four pairs overlap, ids 0->0 and 1->1 stay -> 2
    ([4, 4], [2, 1], [1, 2], 2),
    ([8, 6], [2, 3], [2, 3], 0),  # unchanged partition: nothing moves
])
def test_repartition_messages_hand_derived(lib, shape, src, dst, want):
    assert odec.repartition_messages_bruteforce(shape, src, dst) == want
    assert lib.repartition_messages(shape, src, dst) == want


def test_repartition_messages_match_bruteforce(lib):
    import numpy as np

    rng = np.random.default_rng(5)
    for _ in range(60):
        rank = int(rng.integers(1, 4))
        shape = [int(v) for v in rng.choice([2, 3, 4, 6, 8, 12], size=rank)]
        divs = lambda n: [v for v in range(1, n + 1) if n % v == 0]  # noqa: E731
        src = [int(rng.choice(divs(n))) for n in shape]
        dst = [int(rng.choice(divs(n))) for n in shape]
        assert lib.repartition_messages(shape, src, dst) == odec.repartition_messages_bruteforce(shape, src, dst), \
            (shape, src, dst)


@pytest.mark.parametrize("eq,bounds,d", [
    ("ij,jk->ik", [4, 6, 4], [2, 3, 3, 2]),
    ("ij,jk->ik", [4, 6, 4], [4, 1, 1, 2]),
    ("abef,cfed->abcd", [2, 2, 2, 4, 2, 2], [1, 2, 2, 2, 2, 2, 2, 1]),
    ("hst->hs", [2, 4, 6], [2, 2, 3]),
    ("i,j->ij", [4, 6], [2, 3]),
])
def test_plan_messages_and_memory_match_bruteforce(lib, eq, bounds, d):
    spec = eq + (":mul:sum" if "," in eq and "->ij" not in eq else "::sum" if "," not in eq else ":mul:none")
    p = lib.Plan(spec, bounds, d)
    _, D = _tasks(eq, bounds, d)
    assert p.msg_join + p.msg_agg == odec.node_messages(eq, bounds, D)
    assert p.mem_elems == odec.node_memory(eq, bounds, D)


MODELS = [
    {"latency": 3},
    {"min_block": 2},
    {"mem_weight": 2},
    {"mem_limit": 40},
    {"task_multiple": 4},
    {"latency": 5, "min_block": 2, "mem_weight": 1, "task_multiple": 2},
]


@pytest.mark.parametrize("model", MODELS, ids=lambda m: ",".join(f"{k}={v}" for k, v in m.items()))
@pytest.mark.parametrize("graph", [CHAIN, TREE], ids=["chain", "binary-tree"])
def test_variants_match_exhaustive_search(lib, graph, model):
    p_min, p_max = 2, 8
    r = lib.decompose(graph, p_min, p_max, model=model)
    best, _ = odec.search(graph, p_min, p_max, model=model)
    assert r["total_cost"] == best
    eqs = [(s.split(":")[0], b, i) for s, b, i in graph]
    choice = [_tasks(eq, b, d)[1] for (eq, b, _), d in zip(eqs, r["d"])]
    assert odec.graph_cost(eqs, choice, model) == r["total_cost"]
    for (eq, b, _), d in zip(eqs, r["d"]):
        n, D = _tasks(eq, b, d)
        assert D in odec.candidates(eq, b, p_min, p_max, model=model)


def test_variant_terms_take_effect(lib):
    # the latency and memory terms raise the optimum by at least their smallest possible value
    base = lib.decompose(CHAIN, 2, 8)["total_cost"]
    assert lib.decompose(CHAIN, 2, 8, model={"latency": 7})["total_cost"] >= base + 7 * 3 * 2 * 2
    # outputs of 4x4, 4x2 and 4x4 elements: at least 40 of memory (partials only add)
    assert lib.decompose(CHAIN, 2, 8, model={"mem_weight": 1})["total_cost"] >= base + 16 + 8 + 16
    # minimum granularity equal to the bounds leaves one task per node
    with pytest.raises(lib.TraError) as e:
        lib.decompose(CHAIN, 2, 8, model={"min_block": 4})
    assert "TRA_ERR_UNSUPPORTED" in str(e.value)
    r = lib.decompose(CHAIN, 1, 8, model={"min_block": 4})
    assert all(v == 1 for d in r["d"] for v in d)
    # a memory limit below every output prunes everything
    with pytest.raises(lib.TraError):
        lib.decompose(CHAIN, 2, 8, model={"mem_limit": 8})
    with pytest.raises(ValueError):
        lib.decompose(CHAIN, 2, 8, model={"latncy": 1})
