"""Python face of the oracle's extended EinSum (test infrastructure only).

The arithmetic lives in ``einsum_ref.c``: the definition of the extended EinSum
("EinDecomp ... tensor relational algebra", section 2.1) as plain nested loops
in double.  This module parses the index string, converts the inputs exactly to
double and calls it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "einsum_ref.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

# binary scalar functions (section 2.1: any binary scalar function, e.g. (x-y)^2)
OPS = {"mul": 0, "add": 1, "sqdiff": 2, "sub": 3, "expsub": 4, "id": 5}
# commutative, associative aggregations (section 2.1: sum, max, min, logsumexp)
AGGS = {"sum": 0, "max": 1, "min": 2, "lse": 3, "none": 4}


def build(force: bool = False) -> str:
    """Compile ``einsum_ref.c`` with the host gcc (OpenMP when available)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", _SRC, "-o", _LIB + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        vp, i32, i64, dbl = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
        lib.oracle_einsum.argtypes = [i32, vp, i32, vp, vp, i32, vp, vp, i32, vp, vp, i32, i32, dbl]
        lib.oracle_einsum.restype = i32
        lib.oracle_einsum_points.argtypes = [i32, vp, i32, vp, vp, i32, vp, vp, i32, vp, i64, vp, vp, i32, i32, dbl]
        lib.oracle_einsum_points.restype = i32
        lib.oracle_num_threads.restype = i32
        lib.oracle_set_num_threads.argtypes = [i32]
        lib.oracle_set_num_threads.restype = None
        _lib = lib
    return _lib


def num_threads() -> int:
    """Threads the oracle's OpenMP loops use on this host."""
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    """Threads for the oracle's OpenMP loops from now on (1: a single-core run)."""
    _load().oracle_set_num_threads(int(n))


def parse(eq: str):
    """Split "ij,jk->ik" (or "hst->hs") into label strings."""
    lhs, out = eq.replace(" ", "").split("->")
    ins = lhs.split(",")
    if len(ins) not in (1, 2):
        raise ValueError("one or two operands expected: " + eq)
    for s in ins + [out]:
        if len(set(s)) != len(s):
            raise ValueError("a label repeats within one operand: " + eq)
    if not set(out) <= set("".join(ins)):
        raise ValueError("output label missing from the inputs: " + eq)
    return ins, out


def _prepare(eq, X, Y):
    ins, out = parse(eq)
    if (Y is None) != (len(ins) == 1):
        raise ValueError("operand count does not match " + eq)
    order = []
    for s in ins:
        for c in s:
            if c not in order:
                order.append(c)
    bounds = {}
    for s, T in zip(ins, [X, Y]):
        if T.ndim != len(s):
            raise ValueError(f"rank of operand {s} is {T.ndim}")
        for c, n in zip(s, T.shape):
            if bounds.setdefault(c, n) != n:
                raise ValueError(f"label {c} has two extents")
    lid = {c: i for i, c in enumerate(order)}
    b = np.array([bounds[c] for c in order], dtype=np.int64)
    lx = np.array([lid[c] for c in ins[0]], dtype=np.int32)
    ly = np.array([lid[c] for c in ins[1]], dtype=np.int32) if Y is not None else np.zeros(1, np.int32)
    lz = np.array([lid[c] for c in out], dtype=np.int32) if out else np.zeros(1, np.int32)
    Xd = np.ascontiguousarray(X, dtype=np.float64)
    Yd = np.ascontiguousarray(Y, dtype=np.float64) if Y is not None else None
    shape = tuple(bounds[c] for c in out)
    return ins, out, b, lx, ly, lz, Xd, Yd, shape


def einsum(eq: str, X, Y=None, op: str = "mul", agg: str = "sum", alpha: float = 1.0) -> np.ndarray:
    """Dense extended EinSum in double.  X, Y: numpy arrays (any real dtype, converted exactly)."""
    ins, out, b, lx, ly, lz, Xd, Yd, shape = _prepare(eq, X, Y)
    Z = np.empty(shape, dtype=np.float64)
    opc = OPS["id"] if Y is None else OPS[op]
    rc = _load().oracle_einsum(len(b), b.ctypes.data, len(ins[0]), lx.ctypes.data, Xd.ctypes.data,
                               len(ins[1]) if Y is not None else -1, ly.ctypes.data,
                               Yd.ctypes.data if Yd is not None else None, len(out), lz.ctypes.data,
                               Z.ctypes.data, opc, AGGS[agg], float(alpha))
    if rc != 0:
        raise ValueError(f"oracle rejected {eq} {op} {agg}")
    return Z


def einsum_points(eq: str, X, Y, points, op: str = "mul", agg: str = "sum", alpha: float = 1.0) -> np.ndarray:
    """Selected outputs of the same EinSum.  ``points``: row-major positions in the dense output."""
    ins, out, b, lx, ly, lz, Xd, Yd, shape = _prepare(eq, X, Y)
    pts = np.ascontiguousarray(points, dtype=np.int64)
    vals = np.empty(pts.shape, dtype=np.float64)
    opc = OPS["id"] if Y is None else OPS[op]
    rc = _load().oracle_einsum_points(len(b), b.ctypes.data, len(ins[0]), lx.ctypes.data, Xd.ctypes.data,
                                      len(ins[1]) if Y is not None else -1, ly.ctypes.data,
                                      Yd.ctypes.data if Yd is not None else None, len(out), lz.ctypes.data,
                                      pts.size, pts.ctypes.data, vals.ctypes.data, opc, AGGS[agg], float(alpha))
    if rc != 0:
        raise ValueError(f"oracle rejected {eq} {op} {agg}")
    return vals
