"""An EinGraph step captured into one CUDA graph and replayed.

Every entry point enqueues on the caller's stream, never synchronises and never allocates
device memory, so a whole step of the multi-head-attention EinGraph ("EinDecomp ... tensor
relational algebra", section 2.1) can be captured once and replayed.  The kernels use no
atomics, so a replay must reproduce the eager run bit for bit, and follow new input values
written into the captured buffers.
"""
import numpy as np
import pytest

import datagen

pytestmark = pytest.mark.gpu


def _inputs(s, a, h, d, seed):
    acts = [datagen.normal_bf16((s, a), seed, t) for t in range(3)]
    ws = [datagen.normal_bf16((a, h, d), seed, 3 + t, 0.0, 0.02) for t in range(4)]
    return acts + ws


def _to_dev(torch, bits):
    return [torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).cuda().reshape(-1) for b in bits]


def test_attention_step_graph_replay(lib, cuda):
    import torch

    from tensor_relational_algebra_gb300.eingraph import AttentionGraph

    s, a, h, d = 512, 256, 2, 128
    g = AttentionGraph(s, a, h, d)
    dev = _to_dev(torch, _inputs(s, a, h, d, 31))
    dev[3:6] = [g.projection_weight(w) for w in dev[3:6]]  # relations under [1, h, 1]
    nodes = g.nodes(*dev)

    def step():
        for node in nodes:
            node[1]()

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()  # eager run on the stream the capture will use (also warms the plans)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    eager = [t.clone() for t in (g.S, g.L, g.A, g.out)]

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for t in (g.S, g.L, g.A, g.out):
        t.zero_()
    graph.replay()
    torch.cuda.synchronize()
    lib.ein_status()
    for got, want in zip((g.S, g.L, g.A, g.out), eager):
        assert torch.equal(got, want)

    # new inputs written into the captured buffers: the replay follows them
    fresh = _to_dev(torch, _inputs(s, a, h, d, 32))
    fresh[3:6] = [g.projection_weight(w) for w in fresh[3:6]]
    for dst, src in zip(dev, fresh):
        dst.copy_(src)
    graph.replay()
    torch.cuda.synchronize()
    replayed = g.out.clone()
    step()
    torch.cuda.synchronize()
    assert torch.equal(replayed, g.out)
    assert not torch.equal(replayed, eager[3])


def test_semiring_pair_graph_replay(lib, cuda):
    # the default workload's step (repartition of Y, squared distance, max-plus) captured once;
    # replays equal the eager run bit for bit and follow new inputs (the launch path queries
    # the output's memory type, which must be allowed while capturing)
    import torch

    M, K, N = 512, 256, 640
    d = [2, 1, 1, 2]
    p_sq = lib.Plan("ij,jk->ik:sqdiff:sum", [M, K, N], d)
    p_mx = lib.Plan("ij,jk->ik:add:max", [M, K, N], d)
    ws = torch.empty(max(p_sq.workspace_bytes, 256), dtype=torch.uint8, device="cuda")
    xs = [(datagen.normal_f32((M, K), s, 0), datagen.normal_f32((K, N), s, 1)) for s in (41, 42)]
    x = torch.empty(M * K, device="cuda")
    y = torch.empty(K * N, device="cuda")
    yr = torch.empty_like(y)
    zs = torch.empty(M * N, device="cuda")
    zm = torch.empty_like(zs)

    def step():
        lib.repartition(y, yr, [K, N], [1, 1], [1, 2])
        p_sq.execute(x, yr, zs, ws)
        p_mx.execute(x, yr, zm)

    eager = []
    for X, Y in xs:
        x.copy_(torch.from_numpy(X).reshape(-1))
        y.copy_(torch.from_numpy(Y).reshape(-1))
        step()
        eager.append((zs.cpu().clone(), zm.cpu().clone()))
    lib.ein_status()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        step()
    for i in (1, 0, 1):
        X, Y = xs[i]
        x.copy_(torch.from_numpy(X).reshape(-1))
        y.copy_(torch.from_numpy(Y).reshape(-1))
        zs.zero_()
        zm.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(zs.cpu(), eager[i][0]) and torch.equal(zm.cpu(), eager[i][1])
    lib.ein_status()
