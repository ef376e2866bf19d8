"""The attention chain fused into one kernel (ein_attention) against the oracle and against
the unfused EinGraph nodes ("EinDecomp ... tensor relational algebra", section 2.1).

O is compared at the BF16 bar (2e-2 of max|ref|) with the oracle's chain evaluated in double
(S, L = logsumexp_t S, A = exp(S - L), O = A.V); L within 1e-4 of max(|L|, 1).  The cases
cover one key block, an odd number of key blocks with s != t, several heads, key blocks
whose maxima grow (the kernel's reference maximum moves) or fall, CTAs that take several query
tiles with an odd number of key blocks each, and the whole attention EinGraph with the fused
node against the unfused one.
"""
import numpy as np
import pytest

import datagen
import oracle
from oracle import mha

from gpu_helpers import as_f64, check_bf16_bar, from_dev

pytestmark = pytest.mark.gpu


def _scale_key_blocks(k, factors):
    """k (bf16 bits [h][t][d]) with key block j (128 keys) multiplied by factors[j], a power of
    two, so the product stays exact in bf16."""
    f = datagen.bf16_bits_to_f32(k).copy()
    for j, g in enumerate(factors):
        f[:, 128 * j:128 * (j + 1)] *= np.float32(g)
    return (f.view(np.uint32) >> 16).astype(np.uint16)


def _run(lib, s, t, h, seed, key_scale=None):
    import torch

    d = 128
    q = datagen.normal_bf16((h, s, d), seed, 0)
    k = datagen.normal_bf16((h, t, d), seed, 1)
    v = datagen.normal_bf16((h, t, d), seed, 2)
    if key_scale is not None:
        k = _scale_key_blocks(k, key_scale)
    dev = [torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda().reshape(-1) for a in (q, k, v)]
    o = torch.empty(s * h * d, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(h * s, dtype=torch.float32, device="cuda")
    lib.attention(dev[0], dev[1], dev[2], o, s, t, h, d, lse=lse)
    lib.ein_status()
    f = [datagen.bf16_bits_to_f32(a).astype(np.float64) for a in (q, k, v)]
    qs, ks, vs = (np.transpose(a, (1, 0, 2)) for a in f)  # [s|t][h][d]
    S = oracle.einsum("shd,thd->hst", qs, ks, alpha=1.0 / np.sqrt(d))
    L = oracle.einsum("hst->hs", S, agg="lse")
    A = oracle.einsum("hst,hs->hst", S, L, op="expsub", agg="none")
    O = oracle.einsum("hst,thd->shd", A, vs)
    return as_f64(from_dev(o)).reshape(s, h, d), as_f64(from_dev(lse)).reshape(h, s), O, L


@pytest.mark.parametrize("s,t,h", [(128, 128, 1), (256, 384, 3), (384, 1024, 2)])
def test_fused_attention_against_oracle(lib, cuda, s, t, h):
    o, lse, O, L = _run(lib, s, t, h, 40 + s + t + h)
    check_bf16_bar(o, O)
    assert np.all(np.abs(lse - L) <= 1e-4 * np.maximum(np.abs(L), 1.0))


@pytest.mark.parametrize("s,t,h", [(10240, 256, 2), (8192, 128, 3)])
def test_fused_attention_more_tiles_than_sms(lib, cuda, s, t, h):
    # more (128-row query tile, head) CTAs than SMs (160 and 192 of them, t = 128: a single key
    # block per tile), so CTAs of a later wave start while others run
    o, lse, O, L = _run(lib, s, t, h, 90 + t + h)
    check_bf16_bar(o, O)
    assert np.all(np.abs(lse - L) <= 1e-4 * np.maximum(np.abs(L), 1.0))


@pytest.mark.parametrize("factors", [[1, 2, 4, 8, 8, 16, 1, 16], [16, 8, 4, 2, 1, 1, 1, 1]])
def test_fused_attention_growing_and_falling_block_maxima(lib, cuda, factors):
    """Key blocks scaled so the row maxima jump by more than 2^8 between blocks (the reference
    maximum moves and O is rescaled, for some rows of a warp but not others) or only fall."""
    o, lse, O, L = _run(lib, 256, 1024, 2, 77, key_scale=factors)
    check_bf16_bar(o, O)
    assert np.all(np.abs(lse - L) <= 1e-4 * np.maximum(np.abs(L), 1.0))


@pytest.mark.parametrize("key_scale", [None, [1, 16, 1]])
def test_fused_attention_odd_blocks_several_units_per_cta(lib, cuda, key_scale):
    """Three key blocks per query tile and 160 tiles on at most 152 CTAs: the two sets of
    softmax warps take alternate key blocks, so a CTA's second tile starts on the other set,
    whose first block of that tile is its second.  With the middle block scaled by 16 the
    reference maximum moves on that block, for either set."""
    o, lse, O, L = _run(lib, 10240, 384, 2, 55, key_scale=key_scale)
    check_bf16_bar(o, O)
    assert np.all(np.abs(lse - L) <= 1e-4 * np.maximum(np.abs(L), 1.0))


def test_fused_node_in_the_attention_eingraph(lib, cuda):
    import torch

    from tensor_relational_algebra_gb300.eingraph import AttentionGraph

    s, a, h, d = 512, 256, 2, 128
    acts = [datagen.normal_bf16((s, a), 41, t) for t in range(3)]
    ws = [datagen.normal_bf16((a, h, d), 41, 3 + t, 0.0, 0.02) for t in range(4)]
    dev = [torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).cuda().reshape(-1) for b in acts + ws]
    unfused = AttentionGraph(s, a, h, d)
    fused = AttentionGraph(s, a, h, d, fused=True)
    dev[3:6] = [unfused.projection_weight(w) for w in dev[3:6]]  # relations under [1, h, 1]
    unfused(*dev)
    fused(*dev)
    torch.cuda.synchronize()
    lib.ein_status()
    ref = mha.chain(*[datagen.bf16_bits_to_f32(b) for b in acts + ws], engine="blas")
    check_bf16_bar(as_f64(from_dev(fused.O)).reshape(s, h, d), ref["O"])
    check_bf16_bar(as_f64(from_dev(fused.out)).reshape(s, a), ref["out"])
    # against the unfused nodes on the same device inputs
    check_bf16_bar(as_f64(from_dev(fused.O)), as_f64(from_dev(unfused.O)))
    Lf, Lu = as_f64(from_dev(fused.L)), as_f64(from_dev(unfused.L))
    assert np.all(np.abs(Lf - Lu) <= 1e-4 * np.maximum(np.abs(Lu), 1.0))


@pytest.mark.parametrize("args,code", [((128, 128, 1, 64), "TRA_ERR_UNSUPPORTED"),
                                       ((100, 128, 1, 128), "TRA_ERR_UNSUPPORTED"),
                                       ((128, 200, 1, 128), "TRA_ERR_UNSUPPORTED")])
def test_fused_attention_rejects_shapes(lib, cuda, args, code):
    import torch

    buf = torch.zeros(1 << 20, dtype=torch.bfloat16, device="cuda")
    s, t, h, d = args
    with pytest.raises(lib.TraError) as e:
        lib.ein_attention(s, t, h, d, 0.1, buf, buf, buf, buf)
    assert code in str(e.value)
