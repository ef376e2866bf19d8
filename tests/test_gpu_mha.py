"""The multi-head-attention EinGraph ("EinDecomp ... tensor relational algebra", section 2.1)
run node by node through the C ABI, against the oracle's node-by-node chain.

Every node's output is compared at the BF16 bar (2e-2 of max|ref|); the small
case checks every element of every node, the full-size case (s = a = 4096,
h = 32, d = 128) checks sampled query rows of the final output and of S / L.
"""
import numpy as np
import pytest

import datagen
from oracle import mha
from oracle import tra as otra

from gpu_helpers import as_f64, check_bf16_bar, from_dev

pytestmark = pytest.mark.gpu


def inputs(s, a, h, d, seed):
    acts = [datagen.normal_bf16((s, a), seed, t) for t in range(3)]
    ws = [datagen.normal_bf16((a, h, d), seed, 3 + t, 0.0, 0.02) for t in range(4)]
    return acts + ws


def run_gpu(lib, bits, s, a, h, d):
    import torch

    from tensor_relational_algebra_gb300.eingraph import AttentionGraph

    g = AttentionGraph(s, a, h, d)
    dev = [torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).cuda().reshape(-1) for b in bits]
    dev[3:6] = [g.projection_weight(w) for w in dev[3:6]]  # W_Q, W_K, W_V as relations under [1, h, 1]
    g(*dev)
    lib.ein_status()
    torch.cuda.synchronize()
    return g


def f32(bits):
    return datagen.bf16_bits_to_f32(bits)


def test_attention_small_every_node(lib, cuda):
    s, a, h, d = 512, 512, 4, 128
    bits = inputs(s, a, h, d, 21)
    g = run_gpu(lib, bits, s, a, h, d)
    ref = mha.chain(*[f32(b) for b in bits], engine="blas")
    # projections: head-major relations under [1, h, 1] (h split in the projection's d)
    check_bf16_bar(as_f64(otra.unblock(from_dev(g.qp), (s, h, d), [1, h, 1])), ref["Qp"])
    check_bf16_bar(as_f64(otra.unblock(from_dev(g.kp), (s, h, d), [1, h, 1])), ref["Kp"])
    check_bf16_bar(as_f64(from_dev(g.S)).reshape(h, s, s), ref["S"])
    check_bf16_bar(as_f64(from_dev(g.L)).reshape(h, s), ref["L"])
    A = as_f64(from_dev(g.A)).reshape(h, s, s)
    check_bf16_bar(A, ref["A"])
    np.testing.assert_allclose(A.sum(-1), 1.0, atol=3e-2)  # softmax rows sum to one
    check_bf16_bar(as_f64(from_dev(g.O)).reshape(s, h, d), ref["O"])
    check_bf16_bar(as_f64(from_dev(g.out)).reshape(s, a), ref["out"])


def test_attention_full_size_sampled_rows(lib, cuda):
    s, a, h, d = 4096, 4096, 32, 128
    bits = inputs(s, a, h, d, 0)
    g = run_gpu(lib, bits, s, a, h, d)
    rows = np.array([0, 1, 777, 2048, 4095])
    ref = mha.chain(*[f32(b) for b in bits], rows=rows, engine="blas")
    out = as_f64(from_dev(g.out)).reshape(s, a)[rows]
    check_bf16_bar(out, ref["out"])
    S = as_f64(from_dev(g.S)).reshape(h, s, s)[:, rows, :]
    check_bf16_bar(S, ref["S"])
    L = as_f64(from_dev(g.L)).reshape(h, s)[:, rows]
    check_bf16_bar(L, ref["L"])


@pytest.mark.parametrize("fused", [False, True])
def test_packed_projections_one_einsum(lib, cuda, fused):
    # Q, K, V (and the relations of W_Q, W_K, W_V) back to back in one buffer: the three
    # projections run as one EinSum with a batch label p = 3 split 3 ways; every node still
    # matches the oracle's chain, and the projections agree with the three separate launches
    import torch

    from tensor_relational_algebra_gb300.eingraph import AttentionGraph

    s, a, h, d = 512, 512, 4, 128
    bits = inputs(s, a, h, d, 22)
    dev = [torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).cuda().reshape(-1) for b in bits]
    g_sep = AttentionGraph(s, a, h, d, fused=fused)
    ws = [g_sep.projection_weight(w) for w in dev[3:6]]
    qkv = torch.cat(dev[:3])
    wqkv = torch.cat(ws)
    n, m = s * a, a * h * d
    packed = [qkv[:n], qkv[n:2 * n], qkv[2 * n:], wqkv[:m], wqkv[m:2 * m], wqkv[2 * m:], dev[6]]
    g = AttentionGraph(s, a, h, d, fused=fused)
    names = [nd[0] for nd in g.nodes(*packed)]
    assert names[0].startswith("proj Q, K, V") and not any(x in ("proj K", "proj V") for x in names)
    g(*packed)
    g_sep(*dev[:3], *ws, dev[6])
    lib.ein_status()
    torch.cuda.synchronize()
    ref = mha.chain(*[f32(b) for b in bits], engine="blas")
    for t, key in ((g.qp, "Qp"), (g.kp, "Kp"), (g.vp, "Vp")):
        check_bf16_bar(as_f64(otra.unblock(from_dev(t), (s, h, d), [1, h, 1])), ref[key])
    check_bf16_bar(as_f64(from_dev(g.O)).reshape(s, h, d), ref["O"])
    check_bf16_bar(as_f64(from_dev(g.out)).reshape(s, a), ref["out"])
    # against the three separate projections: the same EinSum, summed in another order only in
    # tiles whose K loop the last wave splits (bf16 outputs: within one bf16 rounding)
    for t_p, t_s in ((g.qp, g_sep.qp), (g.kp, g_sep.kp), (g.vp, g_sep.vp)):
        x, y = as_f64(from_dev(t_p)), as_f64(from_dev(t_s))
        assert np.all(np.abs(x - y) <= 2.0 ** -7 * np.maximum(np.abs(x), np.abs(y)) + 1e-4 * np.abs(y).max())
