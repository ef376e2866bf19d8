"""Out-of-bounds writes: every output and workspace buffer framed by guard regions.

Each buffer a kernel writes (the output relation, the workspace, the repartition's
destination, the fused attention's O and L) is allocated with 64 KiB guard regions on both
sides, and the guards and the output itself are filled with a NaN bit pattern before the
call.  After the call and ein_status():
  * both guard regions still hold the pattern, bit for bit (no write left the buffer), and
  * no output element still holds it (every output was written).
The cases are the ones most exposed to stray writes: ragged CUDA-core tiles (cp.async and
register-staged kernels), the tensor-core epilogues (TMA stores, warp stores, the K split of
the last wave), the padded split=bf16x3 operands, both repartition kernels, the factored
logsumexp, literal mode and the fused attention with s != t.
"""
import numpy as np
import pytest

from gpu_helpers import gen, relation_on_device, to_dev

pytestmark = pytest.mark.gpu

GUARD_BYTES = 64 * 1024
PATTERN = {4: 0x7FA5A5A5, 2: 0x7FA5, 1: 0xA5, 8: 0x7FF5A5A5A5A5A5A5}


class Guarded:
    """n elements of a torch dtype between two guard regions, all filled with PATTERN."""

    def __init__(self, n, dtype):
        import torch

        self.dtype = dtype
        self.es = torch.empty(0, dtype=dtype).element_size()
        self.g = GUARD_BYTES // self.es
        self.n = n
        ibits = {1: torch.uint8, 2: torch.int16, 4: torch.int32, 8: torch.int64}[self.es]
        self.raw = torch.empty(self.g * 2 + max(n, 1), dtype=ibits, device="cuda")
        pat = PATTERN[self.es]
        if self.es == 2 and pat >= 1 << 15:
            pat -= 1 << 16
        if self.es == 4 and pat >= 1 << 31:
            pat -= 1 << 32
        self.raw.fill_(pat)
        self.pat = pat
        self.view = self.raw[self.g:self.g + n].view(dtype)

    def check(self, what, written=True):
        import torch

        torch.cuda.synchronize()
        raw = self.raw
        lo, hi = raw[:self.g], raw[self.g + self.n:]
        assert bool((lo == self.pat).all()), f"{what}: write below the buffer"
        assert bool((hi == self.pat).all()), f"{what}: write past the buffer"
        if written:
            mid = raw[self.g:self.g + self.n]
            left = int((mid == self.pat).sum())
            assert left == 0, f"{what}: {left} output elements never written"


def _run(lib, spec, bounds, d, X, Y, out_dtype="f32"):
    import torch

    p = lib.Plan(spec, bounds, d)
    rx = len(p.operands[0])
    xd = relation_on_device(lib, X, d[:rx])
    yd = relation_on_device(lib, Y, d[rx:]) if Y is not None else None
    nz = int(np.prod(p.shape("z")))
    z = Guarded(nz, torch.bfloat16 if out_dtype == "bf16" else torch.float32)
    ws = Guarded(p.workspace_bytes, torch.uint8) if p.workspace_bytes else None
    p.execute(xd, yd, z.view, ws.view if ws else None)
    lib.ein_status()
    z.check(spec)
    if ws:
        ws.check(spec + " workspace", written=False)
    return p


MM = "ij,jk->ik"


@pytest.mark.parametrize("spec,bounds,d", [
    (MM + ":add:max", [300, 96, 264], [3, 1, 1, 2]),            # cp.async kernel, ragged M and N tiles
    (MM + ":sqdiff:sum", [300, 96, 264], [3, 1, 1, 2]),         # expansion + guard words + fix-up pass
    (MM + ":mul:sum", [130, 36, 70], [2, 3, 3, 2]),             # contracted label split, tails everywhere
    ("ij,kj->ik:mul:sum", [300, 96, 264], [3, 1, 2, 1]),        # Y K-contiguous: register-staged kernel
    (MM + ":add:lse", [200, 64, 136], [2, 1, 1, 2]),            # factored logsumexp (workspace, fix-up)
    (MM + ":add:max:mode=literal", [96, 60, 70], [2, 3, 3, 2]),  # one partial per join tuple + combine
])
def test_guards_cuda_core(lib, cuda, spec, bounds, d):
    M, K, N = bounds
    ys = (N, K) if spec.startswith("ij,kj") else (K, N)
    X = gen((M, K), 81, 0)
    Y = gen(ys, 81, 1)
    if ":sqdiff" in spec:  # a tile of coincident points, so the fix-up pass writes too
        Y = Y.copy()
        Y[:, :64] = X[:64, :].T
    _run(lib, spec, bounds, d, X, Y)


def test_guards_cuda_core_bf16(lib, cuda):
    X = gen((300, 96), 82, 0, bf16=True)
    Y = gen((96, 264), 82, 1, bf16=True)
    _run(lib, MM + ":add:max:in=bf16", [300, 96, 264], [3, 1, 1, 2], X, Y)
    _run(lib, MM + ":mul:sum:in=bf16:out=bf16", [300, 96, 264], [3, 1, 1, 2], X, Y, out_dtype="bf16")


@pytest.mark.parametrize("spec,bounds,d,kernel", [
    (MM + ":mul:sum:in=bf16:tc_store=tma", [1024, 4096, 1024], [1, 1, 1, 1], "tc_bf16_pair"),  # K split tail
    (MM + ":mul:sum:in=bf16:tc_store=lsu", [1024, 4096, 1024], [1, 1, 1, 1], "tc_bf16_pair"),
    (MM + ":mul:sum:in=bf16:tc_store=lsu:out=bf16", [512, 512, 384], [2, 1, 1, 3], "tc_bf16_pair"),
    (MM + ":mul:sum:in=bf16:tc=single", [384, 512, 192], [1, 1, 1, 1], "tc_bf16"),
    (MM + ":mul:sum:in=bf16:tc=single:tc_store=lsu", [384, 1024, 320], [3, 2, 2, 1], "tc_bf16"),
    ("abef,cfed->abcd:mul:sum:in=bf16", [8, 64, 8, 64, 8, 64], [2, 1, 1, 1, 2, 1, 1, 1], "tc_bf16_pair"),
])
def test_guards_tensor_core(lib, cuda, spec, bounds, d, kernel):
    eq = spec.split(":")[0]
    xs, ys = eq.split("->")[0].split(",")
    B = dict(zip(dict.fromkeys(xs + ys), bounds))
    X = gen(tuple(B[c] for c in xs), 83, 0, bf16=True)
    Y = gen(tuple(B[c] for c in ys), 83, 1, bf16=True)
    p = _run(lib, spec, bounds, d, X, Y, out_dtype="bf16" if "out=bf16" in spec else "f32")
    assert p.kernel == kernel


@pytest.mark.parametrize("op,agg,bounds,d", [
    ("sqdiff", "sum", [300, 96, 256], [3, 1, 1, 2]),   # rows padded 300 -> 384, general form
    ("add", "lse", [300, 96, 256], [3, 1, 1, 2]),
    ("sqdiff", "sum", [256, 64, 384], [1, 1, 1, 1]),   # direct form: TMA-store epilogue
])
def test_guards_split3(lib, cuda, op, agg, bounds, d):
    M, K, N = bounds
    X = gen((M, K), 84, 0)
    Y = gen((K, N), 84, 1).copy()
    if op == "sqdiff":
        Y[:, :32] = X[:32, :].T
    p = _run(lib, f"{MM}:{op}:{agg}:split=bf16x3", bounds, d, X, Y)
    assert p.kernel == "tc_split3"


@pytest.mark.parametrize("shape,src_d,dst_d,dtype", [
    ((64, 128, 256), [2, 1, 4], [4, 2, 1], "f32"),          # TMA boxes
    ((1, 128, 64, 256), [1, 2, 1, 4], [1, 1, 4, 2], "bf16"),  # TMA boxes, a unit dimension
    ((6, 10, 12), [3, 2, 4], [1, 5, 6], "f32"),              # warp-cooperative kernel
    ((2, 6, 4, 10, 6), [2, 3, 2, 5, 3], [1, 2, 4, 2, 6], "f32"),  # five dimensions: warp-cooperative
    ((16, 16), [2, 4], [8, 2], "f64"),
])
def test_guards_repartition(lib, cuda, shape, src_d, dst_d, dtype):
    import torch

    n = int(np.prod(shape))
    tdt = {"f32": torch.float32, "bf16": torch.bfloat16, "f64": torch.float64}[dtype]
    src = torch.arange(n, dtype=torch.float64, device="cuda").to(tdt)
    dst = Guarded(n, tdt)
    lib.repartition(src, dst.view, list(shape), src_d, dst_d)
    lib.ein_status()
    dst.check(f"repartition {shape} {src_d}->{dst_d}")


def test_guards_fused_attention(lib, cuda):
    import torch

    import datagen

    s, t, h, d = 256, 384, 3, 128
    q, k, v = (to_dev(datagen.normal_bf16((h, n, d), 85, i)).reshape(-1) for i, n in enumerate((s, t, t)))
    o = Guarded(s * h * d, torch.bfloat16)
    lse = Guarded(h * s, torch.float32)
    lib.attention(q, k, v, o.view, s, t, h, d, lse=lse.view)
    lib.ein_status()
    o.check("attention O")
    lse.check("attention L")


@pytest.mark.parametrize("spec,bounds,d", [
    ("hst->hs::lse", [3, 40, 300], [3, 2, 3]),
    ("hst,hs->hst:expsub:none", [3, 40, 300], [3, 2, 3, 3, 2]),
])
def test_guards_unary_and_elementwise(lib, cuda, spec, bounds, d):
    X = gen(tuple(bounds), 86, 0)
    Y = gen(tuple(bounds[:2]), 86, 1) if "," in spec else None
    _run(lib, spec, bounds, d, X, Y)
