"""EinDecomp's choice of partition vectors over an EinGraph, by exhaustive search.

TEST INFRASTRUCTURE -- NOT PART OF THE PRODUCT (see the package header).

"EinDecomp ... tensor relational algebra", section 3.1: the cost of an EinGraph under one
partition vector per node is the sum over nodes of the join cost and the aggregation cost,
plus, for every edge whose producer output and consumer input are partitioned differently,
the repartition cost.  Section 3.2 keeps, per node, the vectors whose task count meets the
parallelism constraint (here p_min <= tasks <= p_max) and whose entries divide the bounds
(optionally powers of two only).

This module enumerates every combination of every node's candidates and evaluates the
whole cost from its definition: the join and aggregation terms come from the enumerated
join (``tra.plan_bruteforce``), the repartition term from the element-wise count
(``tra.repartition_cost_bruteforce``; parity of that term with the pages is unpinned).
Exponential: tiny graphs only.  Graph inputs cost nothing (they arrive partitioned as their
consumer asks).
"""
import itertools

from .tra import _labels, plan_bruteforce, repartition_cost_bruteforce


def _divisors(n, pow2):
    return [v for v in range(1, n + 1) if n % v == 0 and (not pow2 or v & (v - 1) == 0)]


def candidates(eq, bounds, p_min, p_max, pow2=False):
    """Per-label partition counts {label: D} whose task count lies in [p_min, p_max]."""
    ins, out, order, contracted = _labels(eq)
    B = dict(zip(order, bounds))
    out_list = []
    for combo in itertools.product(*[_divisors(B[c], pow2) for c in order]):
        tasks = 1
        for v in combo:
            tasks *= v
        if p_min <= tasks <= p_max:
            out_list.append(dict(zip(order, combo)))
    return out_list


def d_vector(eq, D):
    ins, _, _, _ = _labels(eq)
    return [D[c] for s in ins for c in s]


def node_cost(eq, bounds, D):
    ins, out, order, contracted = _labels(eq)
    r = plan_bruteforce(eq, dict(zip(order, bounds)), d_vector(eq, D))
    return r["cost_join"] + r["cost_agg"]


def edge_cost(u_eq, u_D, v_eq, v_bounds, v_D, k):
    """Repartition of producer u's output into consumer v's input k."""
    _, u_out, _, _ = _labels(u_eq)
    v_ins, _, v_order, _ = _labels(v_eq)
    B = dict(zip(v_order, v_bounds))
    shape = [B[c] for c in v_ins[k]]
    src = [u_D[c] for c in u_out]
    dst = [v_D[c] for c in v_ins[k]]
    return repartition_cost_bruteforce(shape, src, dst)


def graph_cost(nodes, choice):
    """Every node's cost and every node-to-node edge's repartition cost, each once."""
    total = 0
    for v, (eq, bounds, inputs) in enumerate(nodes):
        total += node_cost(eq, bounds, choice[v])
        for k, u in enumerate(inputs):
            if u is not None and u >= 0:
                total += edge_cost(nodes[u][0], choice[u], eq, bounds, choice[v], k)
    return total


def search(nodes, p_min, p_max, pow2=False):
    """Minimum total cost over all assignments, and one assignment reaching it.
    nodes: (spec, bounds, (input_x, input_y)) with -1 for a graph input."""
    eqs = [(spec.split(":")[0], bounds, inputs) for spec, bounds, inputs in nodes]
    cands = [candidates(eq, bounds, p_min, p_max, pow2) for eq, bounds, _ in eqs]
    best, arg = None, None
    for choice in itertools.product(*cands):
        c = graph_cost(eqs, choice)
        if best is None or c < best:
            best, arg = c, choice
    return best, [d_vector(eq, D) for (eq, _, _), D in zip(eqs, arg)] if arg else None
