"""Multi-head-attention EinGraph of section 2.1, node by node (test infrastructure).

Source: "EinDecomp ... tensor relational algebra", section 2.1 (the multi-head
attention example):
  Q_proj[s,h,d] = sum_a Q[s,a] * W_Q[a,h,d]         (same for K and V)
  Scores[h,s,t] = (1/sqrt(d_k)) * sum_d Q_proj[s,h,d] * K_proj[t,h,d]
  Attn          = softmax over t of Scores
  O[s,h,d]      = sum_t Attn[h,s,t] * V_proj[t,h,d]
  Output[s,a]   = sum_h sum_d O[s,h,d] * W_O[a,h,d]
Readings: the repeated "s" of the printed Scores/Attn is a second sequence
index t; no mask; d_k = the per-head width; the scale is applied after the sum
over d.  The softmax is written as two EinSums: L[h,s] = logsumexp_t Scores
(an aggregation whose evaluation takes the row maximum first) and
Attn = exp(Scores - L) (an element-wise join with a broadcast operand).

Each node is evaluated in double and then rounded to the storage type the GPU
chain uses: bf16 for tensors that feed a BF16 contraction (projections, Attn,
O), fp32 for Scores, L and Output.  Two engines compute the nodes:
  "loops" -- the oracle's nested-loop EinSum (einsum_ref.c) for every node;
  "blas"  -- the contractions as a library matmul (numpy float64 einsum) and the
             softmax nodes as numpy reductions, for sizes the loops cannot reach
             in seconds; pinned against "loops" on small shapes in the tests.
"""
from __future__ import annotations

import numpy as np

from .einsum import einsum
from .rounding import to_bf16, to_f32


def _contract(eq, X, Y, alpha, engine):
    if engine == "loops":
        return einsum(eq, X, Y, alpha=alpha)
    return alpha * np.einsum(eq, np.asarray(X, np.float64), np.asarray(Y, np.float64), optimize=True)


def _lse(S, engine):
    if engine == "loops":
        return einsum("hst->hs", S, agg="lse")
    S = np.asarray(S, np.float64)
    m = S.max(axis=-1)
    return m + np.log(np.exp(S - m[..., None]).sum(axis=-1))


def _expsub(S, L, engine):
    if engine == "loops":
        return einsum("hst,hs->hst", S, L, op="expsub", agg="none")
    return np.exp(np.asarray(S, np.float64) - np.asarray(L, np.float64)[..., None])


def projections(Q, K, V, WQ, WK, WV, engine="loops"):
    qp = to_bf16(_contract("sa,ahd->shd", Q, WQ, 1.0, engine))
    kp = to_bf16(_contract("sa,ahd->shd", K, WK, 1.0, engine))
    vp = to_bf16(_contract("sa,ahd->shd", V, WV, 1.0, engine))
    return qp, kp, vp


def attention_rows(qp_rows, kp, vp, WO, scale, engine="loops"):
    """The chain from Scores on, for a set of query rows (all of s, or a sample)."""
    S = to_f32(_contract("shd,thd->hst", qp_rows, kp, scale, engine))
    L = to_f32(_lse(S, engine))
    A = to_bf16(_expsub(S, L, engine))
    O = to_bf16(_contract("hst,thd->shd", A, vp, 1.0, engine))
    out = to_f32(_contract("shd,ahd->sa", O, WO, 1.0, engine))
    return {"S": S, "L": L, "A": A, "O": O, "out": out}


def chain(Q, K, V, WQ, WK, WV, WO, rows=None, engine="loops"):
    """Whole chain; ``rows`` restricts the query positions (sampled check)."""
    scale = 1.0 / np.sqrt(WQ.shape[2])
    qp, kp, vp = projections(Q if rows is None else Q[rows], K, V, WQ, WK, WV, engine)
    res = attention_rows(qp, kp, vp, WO, scale, engine)
    res.update({"Qp": qp, "Kp": kp, "Vp": vp})
    return res


def softmax_plain(S):
    """exp(s - max) / sum exp(s - max) over the last axis, in double (used as a pin)."""
    S = np.asarray(S, dtype=np.float64)
    e = np.exp(S - S.max(axis=-1, keepdims=True))
    return e / e.sum(axis=-1, keepdims=True)
