"""Tensor relations, the TRA plan by brute force, and a literal TRA execution.

TEST INFRASTRUCTURE (oracle) -- not product code; shares nothing with the
CUDA path.  Source: "EinDecomp: automatic tensor-parallel decomposition via
Einstein summation + tensor relational algebra".

Section 2.2, key definition: a tensor of shape [B1, B2, ...] under a partition
vector d = [D1, D2, ...] (each Di divides Bi) is a relation of D1*D2*...
sub-tensors of shape [B1/D1, B2/D2, ...]; the sub-tensor at key
k = [k1, k2, ...] holds the index range [k_i*B_i/D_i, (k_i+1)*B_i/D_i) in every
dimension i.

Section 2.2, join: every pair of sub-tensors whose keys agree on the shared
labels is joined through the kernel.  Aggregation: the join results are
grouped by the output (non-contracted) labels' key and reduced with the
aggregation operator.  Section 2.2, EinSum -> TRA: partition, join all
matching pairs, aggregate.  Section 3.2 (state pruning): the number of tasks
is the number of tuples the join produces.

Section 3.1 cost model (counted in elements moved):
  join          P * (|X_sub| + |Y_sub|)
  aggregation   (P / n_agg) * (n_agg - 1) * |Z_sub|
Readings of points the pages leave open:
  * d holds one entry per operand index position, X's then Y's (the matmul
    vector [d_i, d_jX, d_jY, d_k] of section 2.2), and shared labels must get
    equal entries;
  * P is the number of join tuples (the pages set P to the device count and
    ask for exactly P tasks, so the terms depend only on the EinSum, the bounds
    and d);
  * n_agg is the product of the contracted labels' partition counts;
  * the repartition term (section 3.1 gives no formula): elements whose owner
    changes when blocks are owned by their row-major linear key id.  Pinned to
    the Scatter / Gather traffic (N-1)/N * M of rkmt.cn/news/51250.html (table of
    traffic per communication primitive) between d all ones and N blocks; between
    two partitioned layouts parity is unpinned (invariants and brute force only).
Canonical task order (a tie-break the pages do not set): output key in
row-major order, then the contracted labels' key components (first-appearance
order, X then Y) in row-major order.  Keys are linearised row-major.
"""
from __future__ import annotations

import itertools

import numpy as np

from .einsum import einsum, parse


def key_range(k: int, B: int, D: int):
    """Index range [k*B/D, (k+1)*B/D) held by key component k (section 2.2)."""
    if D <= 0 or B % D:
        raise ValueError(f"partition count {D} does not divide extent {B}")
    return range(k * B // D, (k + 1) * B // D)


def keys(d):
    """All keys of a relation under d, row-major."""
    return list(itertools.product(*[range(D) for D in d]))


def relation(T: np.ndarray, d) -> dict:
    """Dense tensor -> {key: sub-tensor} (section 2.2 key definition)."""
    if len(d) != T.ndim:
        raise ValueError("d must have one entry per dimension")
    rel = {}
    for k in keys(d):
        sl = []
        for ki, B, D in zip(k, T.shape, d):
            r = key_range(ki, B, D)
            sl.append(slice(r.start, r.stop))
        rel[k] = np.array(T[tuple(sl)])
    return rel


def unrelation(rel: dict, shape, d, dtype=None) -> np.ndarray:
    """{key: sub-tensor} -> dense tensor."""
    dtype = dtype or next(iter(rel.values())).dtype
    T = np.empty(shape, dtype=dtype)
    for k in keys(d):
        sl = tuple(slice(key_range(ki, B, D).start, key_range(ki, B, D).stop) for ki, B, D in zip(k, shape, d))
        T[sl] = rel[k]
    return T


def block(T: np.ndarray, d) -> np.ndarray:
    """Blocked physical layout of a relation: sub-tensors in row-major key order,
    each sub-tensor row-major over its own indices, concatenated (flat array)."""
    rel = relation(T, d)
    return np.concatenate([rel[k].reshape(-1) for k in keys(d)])


def unblock(buf: np.ndarray, shape, d) -> np.ndarray:
    """Inverse of :func:`block`."""
    buf = np.asarray(buf).reshape(-1)
    sub = tuple(B // D for B, D in zip(shape, d))
    n = int(np.prod(sub)) if sub else 1
    rel = {k: buf[i * n:(i + 1) * n].reshape(sub) for i, k in enumerate(keys(d))}
    return unrelation(rel, shape, d, dtype=buf.dtype)


def repartition(buf: np.ndarray, shape, src_d, dst_d) -> np.ndarray:
    """Section 2.2 repartition: the same tensor, re-blocked from src_d to dst_d."""
    return block(unblock(buf, shape, src_d), dst_d)


def _labels(eq):
    ins, out = parse(eq)
    order = []
    for s in ins:
        for c in s:
            if c not in order:
                order.append(c)
    contracted = [c for c in order if c not in out]
    return ins, out, order, contracted


def plan_bruteforce(eq: str, bounds: dict, d) -> dict:
    """Enumerate the join of section 2.2 by brute force.

    bounds: {label: extent}.  d: partition counts per operand index position,
    X's then Y's.  Returns the per-label partition counts, the tasks in canonical
    order as (x_key, y_key, z_key) tuples, the counts and the cost terms."""
    ins, out, order, contracted = _labels(eq)
    if len(d) != sum(len(s) for s in ins):
        raise ValueError("d needs one entry per operand index position")
    dx = list(d[:len(ins[0])])
    dy = list(d[len(ins[0]):]) if len(ins) == 2 else []
    D = {}
    for s, ds in zip(ins, [dx, dy]):
        for c, v in zip(s, ds):
            if bounds[c] % v:
                raise ValueError(f"D={v} does not divide B={bounds[c]} for label {c}")
            if D.setdefault(c, v) != v:
                raise ValueError(f"shared label {c} partitioned differently")
    dz = [D[c] for c in out]
    sub = {s: int(np.prod([bounds[c] // D[c] for c in s])) if s else 1 for s in ins + [out]}
    tasks = []
    xs = keys(dx)
    ys = keys(dy) if len(ins) == 2 else [()]
    for kx in xs:
        for ky in ys:
            comp = {}
            ok = True
            for c, v in zip(ins[0], kx):
                comp[c] = v
            if len(ins) == 2:
                for c, v in zip(ins[1], ky):
                    if comp.setdefault(c, v) != v:
                        ok = False
                        break
            if not ok:
                continue
            kz = tuple(comp[c] for c in out)
            kc = tuple(comp[c] for c in contracted)
            tasks.append((kz, kc, kx, ky))
    tasks.sort(key=lambda t: (t[0], t[1]))
    groups = {}
    for kz, kc, kx, ky in tasks:
        groups.setdefault(kz, []).append(kc)
    n_tasks = len(tasks)
    x_sub, y_sub, z_sub = sub[ins[0]], (sub[ins[1]] if len(ins) == 2 else 0), sub[out]
    cost_join = sum(x_sub + y_sub for _ in tasks)
    cost_agg = sum((len(m) - 1) * z_sub for m in groups.values())
    n_aggs = {len(m) for m in groups.values()}
    return {
        "D": D,
        "dz": dz,
        "tasks": [(kx, ky, kz) for kz, kc, kx, ky in tasks],
        "n_tasks": n_tasks,
        "n_groups": len(groups),
        "n_agg": n_aggs.pop() if len(n_aggs) == 1 else None,
        "x_sub": x_sub,
        "y_sub": y_sub,
        "z_sub": z_sub,
        "cost_join": cost_join,
        "cost_agg": cost_agg,
    }


def _combine(agg, a, b):
    if agg == "sum":
        return a + b
    if agg == "max":
        return np.maximum(a, b)
    if agg == "min":
        return np.minimum(a, b)
    if agg == "lse":
        return np.logaddexp(a, b)
    raise ValueError("aggregation 'none' admits one join tuple per group")


def tra_literal(eq: str, X, Y, d, op="mul", agg="sum", alpha=1.0) -> np.ndarray:
    """Execute the EinSum exactly as the TRA of section 2.2 describes it.

    Inputs become relations under d; every key-matched pair is joined through the
    kernel (the same EinSum on the two sub-tensors, evaluated by the oracle's
    nested loops); join results are grouped by output key and combined with the
    aggregation in canonical order; alpha scales the aggregated result."""
    ins, out, order, contracted = _labels(eq)
    bounds = {}
    for s, T in zip(ins, [X, Y]):
        for c, n in zip(s, T.shape):
            bounds[c] = n
    plan = plan_bruteforce(eq, bounds, d)
    dx = list(d[:len(ins[0])])
    dy = list(d[len(ins[0]):])
    xr = relation(np.asarray(X, dtype=np.float64), dx)
    yr = relation(np.asarray(Y, dtype=np.float64), dy) if Y is not None else None
    zr = {}
    for kx, ky, kz in plan["tasks"]:
        part = einsum(eq, xr[kx], yr[ky] if yr is not None else None, op=op, agg=agg, alpha=1.0)
        zr[kz] = part if kz not in zr else _combine(agg, zr[kz], part)
    for kz in zr:
        zr[kz] = alpha * zr[kz]
    return unrelation(zr, tuple(bounds[c] for c in out), plan["dz"], dtype=np.float64)


def repartition_cost_bruteforce(shape, src_d, dst_d) -> int:
    """Elements whose owning block (row-major linear key id) differs between the
    two partitionings.  Evaluated element by element (tiny shapes only)."""
    n = int(np.prod(shape))
    moved = 0
    for flat in range(n):
        idx = np.unravel_index(flat, shape)
        own = []
        for d in (src_d, dst_d):
            lin = 0
            for i, B, D in zip(idx, shape, d):
                lin = lin * D + int(i) // (B // D)
            own.append(lin)
        moved += own[0] != own[1]
    return moved
