"""ein_execute_sqdist_noalloc: the squared-distance EinSum with the library's built-in scratch.

Some callers cannot allocate device memory on their path (their memory belongs to
another allocator or a fixed budget, or they run where an allocation and the
synchronisation it brings are not allowed).  For them the library keeps the
squared-distance expansion's row / column norms and its guard words in a fixed device
array of its own.  These tests call that entry point through the C ABI, two calls in a
row and plans of different sizes one after another (the array keeps the last call's
contents), and compare each result with ein_execute's (caller workspace) and with the
CPU oracle.  The file is collected last.
"""
import ctypes

import numpy as np
import pytest

import oracle
from oracle import tra as otra

from gpu_helpers import FP32_REL, as_f64, from_dev, gen, relation_on_device

pytestmark = pytest.mark.gpu

MM = "ij,jk->ik"


def _entry(lib):
    so = lib.load()
    f = so.ein_execute_sqdist_noalloc
    f.argtypes = [ctypes.c_void_p] * 5
    f.restype = ctypes.c_int
    return f


def _rel_ok(g, r):
    err = np.abs(g - r)
    assert np.all(err <= FP32_REL * np.abs(r)), f"worst {np.max(err / np.maximum(np.abs(r), 1e-300)):.3e}"


def _noalloc(lib, f, eq, bounds, d, X, Y, calls=1):
    """Dense host inputs -> relations on the device -> the entry point `calls` times; returns the
    plan, the device inputs and each call's dense result (float64)."""
    import torch

    p = lib.Plan(f"{eq}:sqdiff:sum", bounds, d)
    rx = len(p.operands[0])
    xr = relation_on_device(lib, X, d[:rx])
    yr = relation_on_device(lib, Y, d[rx:])
    zshape = p.shape("z")
    stream = torch.cuda.current_stream().cuda_stream
    outs = []
    for _ in range(calls):
        z = torch.full((int(np.prod(zshape)),), float("nan"), dtype=torch.float32, device="cuda")
        rc = f(p.handle, xr.data_ptr(), yr.data_ptr(), z.data_ptr(), stream)
        assert rc == 0, lib.ein_last_error()
        outs.append(z)
    lib.ein_status()
    dense = [otra.unblock(from_dev(z), zshape, p.dvec("z")).astype(np.float64) for z in outs]
    return p, xr, yr, dense


def test_noalloc_matches_workspace_entry_and_oracle(lib, cuda):
    import torch

    f = _entry(lib)
    M, K, N = 640, 256, 384
    d = [2, 1, 1, 3]
    X = gen((M, K), 31, 0)
    Y = gen((K, N), 31, 1)
    p, xr, yr, outs = _noalloc(lib, f, MM, [M, K, N], d, X, Y, calls=2)
    assert p.workspace_bytes > 0
    ws = torch.empty(p.workspace_bytes, dtype=torch.uint8, device="cuda")
    ref = torch.empty(M * N, dtype=torch.float32, device="cuda")
    lib.ein_execute(p.handle, xr, yr, ref, ws, p.workspace_bytes)
    lib.ein_status()
    w = otra.unblock(from_dev(ref), (M, N), p.dvec("z")).astype(np.float64)
    r = oracle.einsum(MM, as_f64(X), as_f64(Y), op="sqdiff", agg="sum")
    for g in outs:
        _rel_ok(g, w)
        _rel_ok(g, r)


def test_noalloc_larger_then_smaller_then_batched(lib, cuda):
    # the shared array keeps the previous call's norms and guard words: a large plan, then a
    # smaller one of another shape, then one with a batch label (b is in X, Y and Z)
    f = _entry(lib)
    cases = [
        (MM, [2048, 128, 1536], [4, 1, 1, 3]),
        (MM, [200, 72, 136], [2, 3, 3, 2]),
        ("bij,bjk->bik", [3, 130, 40, 96], [3, 2, 1, 3, 1, 3]),
    ]
    for n, (eq, bounds, d) in enumerate(cases):
        xs, ys = eq.split("->")[0].split(",")
        B = dict(zip(dict.fromkeys(xs + ys), bounds))
        X = gen(tuple(B[c] for c in xs), 32 + n, 0)
        Y = gen(tuple(B[c] for c in ys), 32 + n, 1)
        _, _, _, outs = _noalloc(lib, f, eq, bounds, d, X, Y, calls=2)
        r = oracle.einsum(eq, as_f64(X), as_f64(Y), op="sqdiff", agg="sum")
        for g in outs:
            _rel_ok(g, r)


def test_noalloc_coincident_points(lib, cuda):
    # rows of X copied into Y's columns (D = 0) and moved by 1e-3 in three coordinates: the
    # expansion's guard words (in the built-in array) send those tiles to the direct form
    f = _entry(lib)
    M, K, N = 384, 256, 320
    X = gen((M, K), 34, 0)
    Y = gen((K, N), 34, 1).copy()
    Y[:, :128] = X[:128, :].T
    Y[5:8, 200] = X[300, 5:8] + np.float32(1e-3)
    Y[:5, 200], Y[8:, 200] = X[300, :5], X[300, 8:]
    _, _, _, outs = _noalloc(lib, f, MM, [M, K, N], [3, 1, 1, 5], X, Y, calls=2)
    r = oracle.einsum(MM, as_f64(X), as_f64(Y), op="sqdiff", agg="sum")
    assert (np.diag(r[:128, :128]) == 0).all() and 0 < r[300, 200] < 1e-5
    for g in outs:
        _rel_ok(g, r)


def test_noalloc_empty_ranges(lib, cuda):
    import torch

    f = _entry(lib)
    stream = torch.cuda.current_stream().cuda_stream
    fill = lib.Plan(MM + ":sqdiff:sum", [16, 0, 24], [1, 1, 1, 1])  # every output sums an empty set
    z = torch.full((16 * 24,), float("nan"), dtype=torch.float32, device="cuda")
    assert f(fill.handle, None, None, z.data_ptr(), stream) == 0, lib.ein_last_error()
    empty = lib.Plan(MM + ":sqdiff:sum", [0, 8, 24], [1, 1, 1, 1])  # no output element
    assert f(empty.handle, None, None, None, stream) == 0, lib.ein_last_error()
    lib.ein_status()
    assert (from_dev(z) == 0).all()


def test_noalloc_rejects_oversize_and_other_plans(lib, cuda):
    f = _entry(lib)
    big = lib.Plan(MM + ":sqdiff:sum", [262144, 4, 64], [1, 1, 1, 1])  # norms need 1 MiB + 256 B
    assert f(big.handle, 16, 16, 16, None) == -6  # TRA_ERR_WORKSPACE, checked before any launch
    assert "scratch" in lib.ein_last_error()
    other = lib.Plan(MM + ":add:max", [64, 64, 64], [1, 1, 1, 1])
    assert f(other.handle, 16, 16, 16, None) == -5  # TRA_ERR_UNSUPPORTED
    direct = lib.Plan(MM + ":sqdiff:sum:sqdiff=direct", [64, 64, 64], [1, 1, 1, 1])
    assert f(direct.handle, 16, 16, 16, None) == -5
