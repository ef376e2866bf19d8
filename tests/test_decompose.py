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
