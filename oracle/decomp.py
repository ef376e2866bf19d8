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
(``tra.repartition_cost_bruteforce``; pinned to the pages' Scatter / Gather traffic only
between the centralized layout and a partitioned one).
Exponential: tiny graphs only.  Graph inputs cost nothing (they arrive partitioned as their
consumer asks).

Cost-model variants (the page's section 4.3, "troubleshooting"; ``model`` is a dict with the
keys latency, min_block, mem_limit, mem_weight, task_multiple, each off at 0), counted here from
their definitions:
  * messages of a node: one per operand sub-tensor sent to each enumerated join tuple, plus one
    per partial of a group that is combined into another (group size - 1);
  * messages of an edge: the distinct (source block, destination block) pairs, with different
    linear ids, that some element moves between (element by element);
  * memory of a node: the output's elements plus, when some group aggregates more than one
    partial, every join tuple's partial (z_sub elements each);
  * min_block: every label's block extent at least min(min_block, bound);
  * task_multiple: the task count is a multiple of it; mem_limit prunes by memory.
"""
import itertools

import numpy as np

from .tra import _labels, plan_bruteforce, repartition_cost_bruteforce


def _divisors(n, pow2):
    return [v for v in range(1, n + 1) if n % v == 0 and (not pow2 or v & (v - 1) == 0)]


def _m(model, key):
    return (model or {}).get(key, 0) or 0


def candidates(eq, bounds, p_min, p_max, pow2=False, model=None):
    """Per-label partition counts {label: D} whose task count lies in [p_min, p_max] (and that
    pass the model's min_block, task_multiple and mem_limit)."""
    ins, out, order, contracted = _labels(eq)
    B = dict(zip(order, bounds))
    out_list = []
    for combo in itertools.product(*[_divisors(B[c], pow2) for c in order]):
        tasks = 1
        for v in combo:
            tasks *= v
        if not p_min <= tasks <= p_max:
            continue
        D = dict(zip(order, combo))
        g = _m(model, "min_block")
        if g > 1 and any(B[c] // D[c] < min(g, B[c]) for c in order):
            continue
        k = _m(model, "task_multiple")
        if k > 1 and tasks % k:
            continue
        lim = _m(model, "mem_limit")
        if lim and node_memory(eq, bounds, D) > lim:
            continue
        out_list.append(D)
    return out_list


def d_vector(eq, D):
    ins, _, _, _ = _labels(eq)
    return [D[c] for s in ins for c in s]


def _plan(eq, bounds, D):
    ins, out, order, contracted = _labels(eq)
    return plan_bruteforce(eq, dict(zip(order, bounds)), d_vector(eq, D)), ins


def node_messages(eq, bounds, D):
    """Sub-tensors sent to the enumerated join tuples plus partials combined into others."""
    r, ins = _plan(eq, bounds, D)
    groups = {}
    for kx, ky, kz in r["tasks"]:
        groups[kz] = groups.get(kz, 0) + 1
    return len(r["tasks"]) * len(ins) + sum(n - 1 for n in groups.values())


def node_memory(eq, bounds, D):
    """Output elements plus every join tuple's partial when some group aggregates several."""
    r, ins = _plan(eq, bounds, D)
    ins_, out, order, _ = _labels(eq)
    B = dict(zip(order, bounds))
    z_total = 1
    for c in out:
        z_total *= B[c]
    groups = {}
    for kx, ky, kz in r["tasks"]:
        groups[kz] = groups.get(kz, 0) + 1
    partials = len(r["tasks"]) * r["z_sub"] if any(n > 1 for n in groups.values()) else 0
    return z_total + partials


def node_cost(eq, bounds, D, model=None):
    r, _ = _plan(eq, bounds, D)
    c = r["cost_join"] + r["cost_agg"]
    if _m(model, "latency"):
        c += _m(model, "latency") * node_messages(eq, bounds, D)
    if _m(model, "mem_weight"):
        c += _m(model, "mem_weight") * node_memory(eq, bounds, D)
    return c


def repartition_messages_bruteforce(shape, src_d, dst_d):
    """Distinct (source block, destination block) pairs with different row-major linear ids
    between which some element moves; element by element (tiny shapes only)."""
    pairs = set()
    for flat in range(int(np.prod(shape))):
        idx = np.unravel_index(flat, shape)
        own = []
        for d in (src_d, dst_d):
            lin = 0
            for i, B, D in zip(idx, shape, d):
                lin = lin * D + int(i) // (B // D)
            own.append(lin)
        if own[0] != own[1]:
            pairs.add(tuple(own))
    return len(pairs)


def edge_cost(u_eq, u_D, v_eq, v_bounds, v_D, k, model=None):
    """Repartition of producer u's output into consumer v's input k."""
    _, u_out, _, _ = _labels(u_eq)
    v_ins, _, v_order, _ = _labels(v_eq)
    B = dict(zip(v_order, v_bounds))
    shape = [B[c] for c in v_ins[k]]
    src = [u_D[c] for c in u_out]
    dst = [v_D[c] for c in v_ins[k]]
    c = repartition_cost_bruteforce(shape, src, dst)
    if _m(model, "latency"):
        c += _m(model, "latency") * repartition_messages_bruteforce(shape, src, dst)
    return c


def graph_cost(nodes, choice, model=None):
    """Every node's cost and every node-to-node edge's repartition cost, each once."""
    total = 0
    for v, (eq, bounds, inputs) in enumerate(nodes):
        total += node_cost(eq, bounds, choice[v], model)
        for k, u in enumerate(inputs):
            if u is not None and u >= 0:
                total += edge_cost(nodes[u][0], choice[u], eq, bounds, choice[v], k, model)
    return total


def search(nodes, p_min, p_max, pow2=False, model=None):
    """Minimum total cost over all assignments, and one assignment reaching it.
    nodes: (spec, bounds, (input_x, input_y)) with -1 for a graph input."""
    eqs = [(spec.split(":")[0], bounds, inputs) for spec, bounds, inputs in nodes]
    cands = [candidates(eq, bounds, p_min, p_max, pow2, model) for eq, bounds, _ in eqs]
    best, arg = None, None
    for choice in itertools.product(*cands):
        c = graph_cost(eqs, choice, model)
        if best is None or c < best:
            best, arg = c, choice
    return best, [d_vector(eq, D) for (eq, _, _), D in zip(eqs, arg)] if arg else None
