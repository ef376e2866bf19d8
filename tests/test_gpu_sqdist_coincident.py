"""Squared distance at its own zero: coincident and near-coincident points.

"EinDecomp ... tensor relational algebra", section 2.1 (the squared-distance example):
D[i,k] = sum_j (X[i,j] - Y[j,k])^2 >= 0, and D = 0 exactly when row i of X equals column
k of Y.  The expanded form |x|^2 + |y|^2 - 2 x.y cancels there, so its rounding error
(about sqrt(K) u (|x|^2 + |y|^2)) is unbounded relative to D.  The library's guard marks
every 128 x 128 output tile in which the expansion fell below tau * (|x|^2 + |y|^2) and
recomputes those tiles in the direct form.  These cases check the fp32 bar
|g - r| <= 1e-5 |r| (so g == 0 wherever r == 0) on:
  * exact copies of X rows among Y's columns, one whole tile of them,
  * near copies (three coordinates moved by 1e-3, D about 3e-6 against |x|^2 + |y|^2 of 512),
  * a clustered set where every pair is close (every tile recomputed),
for the default (expanded) form, the direct form and split=bf16x3, at the semiring pair's
size (X 8192 x 256, Y 256 x 8192, d = [8,1,1,8]) and on ragged small shapes.
"""
import numpy as np
import pytest

import oracle

from gpu_helpers import FP32_REL, as_f64, gen, run_plan, sample_points

pytestmark = pytest.mark.gpu

MM = "ij,jk->ik"
U = 2.0 ** -16


def coincident_inputs(M, K, N, seed, n_pairs):
    """X N(0,1); Y N(0,1) with some columns replaced by rows of X: the first min(M, N, 128)
    columns are X's first rows (a tile of exact coincidences on its diagonal), then n_pairs
    columns elsewhere copy a random row, every second one moved by 1e-3 in three coordinates.
    Returns X, Y and the dense output positions of every planted pair."""
    X = gen((M, K), seed, 0)
    Y = gen((K, N), seed, 1).copy()
    rng = np.random.default_rng(seed)
    t = min(M, N, 128)
    Y[:, :t] = X[:t, :].T
    pts = [i * N + i for i in range(t)]
    cols = rng.choice(np.arange(t, N), size=min(n_pairs, N - t), replace=False)
    rows = rng.integers(0, M, size=cols.size)
    for n, (i, k) in enumerate(zip(rows, cols)):
        Y[:, k] = X[i, :]
        if n % 2:
            js = rng.choice(K, size=min(3, K), replace=False)
            Y[js, k] = (X[i, js].astype(np.float64) + 1e-3).astype(np.float32)
        pts.append(int(i) * N + int(k))
    return X, Y, np.array(pts, dtype=np.int64)


def _rel_ok(g, r, what):
    err = np.abs(g - r)
    bad = err > FP32_REL * np.abs(r)
    assert not bad.any(), f"{what}: {int(bad.sum())} outside 1e-5 |r|; worst {np.max(err / np.maximum(np.abs(r), 1e-300)):.3e}"


FORMS = [("expand", ":sqdiff=expand"), ("direct", ":sqdiff=direct"), ("split", ":split=bf16x3")]


@pytest.mark.parametrize("form,opt", FORMS)
@pytest.mark.parametrize("bounds,d", [([300, 96, 320], [3, 1, 1, 5]),      # ragged tiles in M and N
                                      ([130, 40, 160], [1, 2, 2, 1])])      # contracted label split
def test_coincident_points_small(lib, cuda, form, opt, bounds, d):
    M, K, N = bounds
    X, Y, pts = coincident_inputs(M, K, N, 71, 40)
    p, g = run_plan(lib, MM + ":sqdiff:sum" + opt, bounds, d, X, Y)
    r = oracle.einsum(MM, as_f64(X), as_f64(Y), op="sqdiff", agg="sum")
    assert (r.reshape(-1)[pts[:min(M, N, 128)]] == 0).all()
    gv, rv = g.reshape(-1), r.reshape(-1)
    _rel_ok(gv[pts], rv[pts], form + " planted pairs")
    if form == "split":
        S = oracle.einsum(MM, np.abs(as_f64(X)), np.abs(as_f64(Y)), op="mul", agg="sum")
        assert np.all(np.abs(g - r) <= FP32_REL * np.abs(r) + 6 * U * S)
    else:
        _rel_ok(g, r, form)


@pytest.mark.parametrize("form,opt", FORMS)
def test_clustered_points_every_tile_recomputed(lib, cuda, form, opt):
    # every row and column is the same point mu (|mu|^2 about 1.6e4) plus noise of 0.01: D / S is
    # about 1e-5 everywhere, so every tile is marked and the whole output takes the direct form
    M, K, N = 200, 64, 128
    mu = 16.0 * gen((1, K), 72, 2)
    X = (mu + 0.01 * gen((M, K), 72, 0)).astype(np.float32)
    Y = (mu.T + 0.01 * gen((K, N), 72, 1)).astype(np.float32)
    _, g = run_plan(lib, MM + ":sqdiff:sum" + opt, [M, K, N], [2, 1, 1, 2], X, Y)
    r = oracle.einsum(MM, as_f64(X), as_f64(Y), op="sqdiff", agg="sum")
    _rel_ok(g, r, form)


@pytest.mark.parametrize("form,opt", FORMS)
def test_coincident_points_pair_workload(lib, cuda, form, opt):
    # the semiring pair's squared distance with 128 + 512 planted pairs; sampled outputs, every
    # planted pair and the whole first tile against the oracle
    M, K, N = 8192, 256, 8192
    X, Y, pts = coincident_inputs(M, K, N, 73, 512)
    p, g = run_plan(lib, MM + ":sqdiff:sum" + opt, [M, K, N], [8, 1, 1, 8], X, Y)
    tile = np.array([i * N + j for i in range(128) for j in range(128)], dtype=np.int64)
    gv = g.reshape(-1)
    exact = np.unique(np.concatenate([pts, tile]))
    r = oracle.einsum_points(MM, as_f64(X), as_f64(Y), exact, op="sqdiff", agg="sum")
    _rel_ok(gv[exact], r, form + " planted pairs and first tile")
    others = sample_points((M, N), 4096, seed=3)
    others = np.setdiff1d(others, exact)
    r = oracle.einsum_points(MM, as_f64(X), as_f64(Y), others, op="sqdiff", agg="sum")
    _rel_ok(gv[others], r, form + " sampled outputs")
