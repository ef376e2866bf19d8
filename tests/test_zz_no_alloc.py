"""ein_execute_sqdist_noalloc: the squared-distance EinSum with the library's built-in scratch.

Some callers cannot allocate device memory on their path (their memory belongs to
another allocator or a fixed budget, or they run where an allocation and the
synchronisation it brings are not allowed).  For them the library keeps the
squared-distance expansion's row / column norms in a fixed device array of its own.
This test calls that entry point through the C ABI twice in a row and compares each
result with ein_execute's, which uses a caller-provided workspace.  It lives in a file
of its own that pytest collects last.
"""
import ctypes

import numpy as np
import pytest

from gpu_helpers import FP32_REL, from_dev, gen, relation_on_device

pytestmark = pytest.mark.gpu


def _entry(lib):
    so = lib.load()
    f = so.ein_execute_sqdist_noalloc
    f.argtypes = [ctypes.c_void_p] * 5
    f.restype = ctypes.c_int
    return f


def test_noalloc_matches_workspace_entry(lib, cuda):
    import torch

    f = _entry(lib)
    M, K, N = 640, 256, 384
    d = [2, 1, 1, 3]
    X = gen((M, K), 31, 0)
    Y = gen((K, N), 31, 1)
    p = lib.Plan("ij,jk->ik:sqdiff:sum", [M, K, N], d)
    assert p.workspace_bytes > 0
    xr = relation_on_device(lib, X, d[:2])
    yr = relation_on_device(lib, Y, d[2:])
    ws = torch.empty(p.workspace_bytes, dtype=torch.uint8, device="cuda")
    ref = torch.empty(M * N, dtype=torch.float32, device="cuda")
    lib.ein_execute(p.handle, xr, yr, ref, ws, p.workspace_bytes)
    stream = torch.cuda.current_stream().cuda_stream
    outs = []
    for _ in range(2):
        z = torch.full((M * N,), float("nan"), dtype=torch.float32, device="cuda")
        rc = f(p.handle, xr.data_ptr(), yr.data_ptr(), z.data_ptr(), stream)
        assert rc == 0, lib.ein_last_error()
        outs.append(z)
    lib.ein_status()
    r = from_dev(ref).astype(np.float64)
    for z in outs:
        g = from_dev(z).astype(np.float64)
        assert np.all(np.abs(g - r) <= FP32_REL * np.abs(r))


def test_noalloc_rejects_oversize_and_other_plans(lib, cuda):
    f = _entry(lib)
    big = lib.Plan("ij,jk->ik:sqdiff:sum", [262144, 4, 64], [1, 1, 1, 1])  # norms need 1 MiB + 256 B
    assert f(big.handle, 16, 16, 16, None) == -6  # TRA_ERR_WORKSPACE, checked before any launch
    assert "scratch" in lib.ein_last_error()
    other = lib.Plan("ij,jk->ik:add:max", [64, 64, 64], [1, 1, 1, 1])
    assert f(other.handle, 16, 16, 16, None) == -5  # TRA_ERR_UNSUPPORTED
