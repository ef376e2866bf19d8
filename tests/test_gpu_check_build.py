"""The GPU suite once more under the check build (libtra_check.so, compiled with -DTRA_CHECK).

In that build every plain global load and store of the CUDA-core semiring, reduction,
element-wise, split and repartition kernels, and the warp stores of the tensor-core
epilogue, first tests its index against the extent of its buffer; an access outside is
skipped and recorded, and ein_status() (which every parity test calls) then fails with
TRA_ERR_BOUNDS.  Nothing traps.  The run below selects the library through TRA_CHECK=1 in a
child pytest over the other GPU test modules, so each parity case doubles as a bounds check
of the indices its kernels formed.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_gpu_suite_under_the_check_build(lib, cuda):
    from tensor_relational_algebra_gb300 import _build

    _build.build(check=True)
    env = dict(os.environ, TRA_CHECK="1")
    cmd = [sys.executable, "-m", "pytest", "-q", "-m", "gpu", "-p", "no:cacheprovider", "-x",
           "-k", "not check_build", os.path.join(ROOT, "tests")]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=1500)
    tail = (r.stdout + r.stderr)[-3000:]
    assert r.returncode == 0, tail
    assert " passed" in r.stdout, tail
