"""The multi-head-attention EinGraph of "EinDecomp ... tensor relational algebra" section 2.1,
run node by node through the C ABI (one ein_execute or ein_repartition per node).

  Q_proj[s,h,d] = sum_a Q[s,a] W_Q[a,h,d]        (K, V alike)        h split h ways
  S[h,s,t]      = (1/sqrt(d)) sum_d Q_proj[s,h,d] K_proj[t,h,d]        split h ways
  L[h,s]        = logsumexp_t S[h,s,t]                                 split h ways
  A[h,s,t]      = exp(S[h,s,t] - L[h,s])                               split h ways (bf16)
  O[s,h,d]      = sum_t A[h,s,t] V_proj[t,h,d]                         split h ways (bf16)
  repartition   O [1,h,1] -> [1,1,1]
  Out[s,a]      = sum_h sum_d O[s,h,d] W_O[a,h,d]                      d = all ones

The printed Scores[h,s,s] is read with a second sequence index t; the scale is applied
after the sum over d; there is no mask.  Buffers are allocated once (torch) and reused.

The projections take the partition vector that splits h (X = Q: [1, 1]; Y = W_Q: [1, h, 1]), as
EinDecomp's search would pick to avoid a repartition: their output relation under [1, h, 1] is
the head-major layout the next nodes read.  W_Q, W_K and W_V are therefore passed as relations
under [1, h, 1] (stored [h][a][d]; projection_weight converts a dense [a][h][d] weight); W_O is
dense [a][h][d].

With fused=True the four nodes Scores -> L -> A -> O and the repartition of O run as one
kernel (ein_attention), which writes O dense and L, never the scores or A.

When Q, K, V lie back to back in one buffer, and so do the relations of W_Q, W_K, W_V, the three
projections run as one EinSum with a batch label p of extent 3, split 3 ways:
  QKV_proj[p,s,h,d] = sum_a QKV[p,s,a] W[p,a,h,d]      d = [3,1,1, 3,1,h,1]
Its input and output relations are exactly the three separate ones laid end to end, so the
result per element is the same EinSum; the tensor-core kernel sees 3x the tiles in one launch
(fewer partly filled waves).
"""
from __future__ import annotations

import math

from . import Plan, attention, repartition


class AttentionGraph:
    def __init__(self, s: int, a: int, h: int, d: int, device="cuda", fused: bool = False):
        import torch

        self.s, self.a, self.h, self.d = s, a, h, d
        self.fused = fused
        t = s
        self.p_proj = Plan("sa,ahd->shd:mul:sum:in=bf16:out=bf16", [s, a, h, d], [1, 1, 1, h, 1])
        self.p_proj3 = Plan("psa,pahd->pshd:mul:sum:in=bf16:out=bf16", [3, s, a, h, d], [3, 1, 1, 3, 1, h, 1])
        self.p_scores = Plan(f"shd,thd->hst:mul:sum:in=bf16:alpha={1.0 / math.sqrt(d)!r}", [s, h, d, t],
                             [1, h, 1, 1, h, 1])
        self.p_lse = Plan("hst->hs::lse", [h, s, t], [h, 1, 1])
        self.p_exp = Plan("hst,hs->hst:expsub:none:out=bf16", [h, s, t], [h, 1, 1, h, 1])
        self.p_pv = Plan("hst,thd->shd:mul:sum:in=bf16:out=bf16", [h, s, t, d], [h, 1, 1, 1, h, 1])
        self.p_out = Plan("shd,ahd->sa:mul:sum:in=bf16", [s, h, d, a], [1, 1, 1, 1, 1, 1])
        bf, f32 = torch.bfloat16, torch.float32
        e = lambda n, dt: torch.empty(n, dtype=dt, device=device)  # noqa: E731
        self.qkvp = e(3 * s * h * d, bf)  # Q_proj, K_proj, V_proj back to back, each [h][s][d]
        n = s * h * d
        self.qp, self.kp, self.vp = self.qkvp[:n], self.qkvp[n:2 * n], self.qkvp[2 * n:]
        self.S = None if fused else e(h * s * t, f32)
        self.L = e(h * s, f32)
        self.A = None if fused else e(h * s * t, bf)
        self.Oh = e(s * h * d, bf)
        self.O = e(s * h * d, bf)
        self.out = e(s * a, f32)

    @staticmethod
    def back_to_back(*ts) -> bool:
        """True when the tensors are contiguous, of one dtype and size, and follow each other in memory."""
        t0 = ts[0]
        return all(t.is_contiguous() and t.dtype == t0.dtype and t.numel() == t0.numel() for t in ts) and all(
            ts[i + 1].data_ptr() == ts[i].data_ptr() + ts[i].numel() * ts[i].element_size() for i in range(len(ts) - 1))

    def nodes(self, Q, K, V, WQ, WK, WV, WO):
        """(name, callable, work, unit, bound, kernel launches[, bytes]) per node, in execution
        order.  Tensor-core nodes also give the bytes they must move at least (operands read
        once, output written once), from which a roofline can tell whether the node is bound by
        the tensor cores or by HBM."""
        s, a, h, d = self.s, self.a, self.h, self.d
        shd = [s, h, d]
        gemm = 2 * s * a * h * d
        att = 2 * h * s * s * d
        act = s * h * d * 2  # one bf16 activation of s x h x d (Q, K, V, O or a projection)
        proj_bytes = s * a * 2 + a * h * d * 2 + act
        if self.back_to_back(Q, K, V) and self.back_to_back(WQ, WK, WV):
            proj = [("proj Q, K, V (one EinSum, p = 3)", lambda: self.p_proj3.execute(Q, WQ, self.qkvp), 3 * gemm,
                     "flop", "tensor", 1, 3 * proj_bytes)]
        else:
            proj = [
                ("proj Q", lambda: self.p_proj.execute(Q, WQ, self.qp), gemm, "flop", "tensor", 1, proj_bytes),
                ("proj K", lambda: self.p_proj.execute(K, WK, self.kp), gemm, "flop", "tensor", 1, proj_bytes),
                ("proj V", lambda: self.p_proj.execute(V, WV, self.vp), gemm, "flop", "tensor", 1, proj_bytes),
            ]
        return proj + ([
            ("attention (Scores -> L -> exp -> A.V fused)",
             lambda: attention(self.qp, self.kp, self.vp, self.O, s, s, h, d, lse=self.L),
             2 * att, "flop", "tensor", 1, 4 * act + h * s * 4),
        ] if self.fused else [
            ("scores", lambda: self.p_scores.execute(self.qp, self.kp, self.S), att, "flop", "tensor", 1,
             2 * act + h * s * s * 4),
            ("logsumexp", lambda: self.p_lse.execute(self.S, None, self.L), h * s * s * 4 + h * s * 4, "bytes", "hbm", 1),
            ("exp(S-L)", lambda: self.p_exp.execute(self.S, self.L, self.A), h * s * s * (4 + 2) + h * s * 4, "bytes",
             "hbm", 1),
            ("A.V", lambda: self.p_pv.execute(self.A, self.vp, self.Oh), att, "flop", "tensor", 1,
             h * s * s * 2 + 2 * act),
            ("repartition O -> dense", lambda: repartition(self.Oh, self.O, shd, [1, h, 1], [1, 1, 1]),
             2 * s * h * d * 2, "bytes", "hbm", 1),
        ]) + [
            ("out proj", lambda: self.p_out.execute(self.O, WO, self.out), gemm, "flop", "tensor", 1,
             act + a * h * d * 2 + s * a * 4),
        ]

    def projection_weight(self, W):
        """The relation under [1, h, 1] of a dense [a][h][d] projection weight (device bf16)."""
        import torch

        out = torch.empty_like(W)
        repartition(W, out, [self.a, self.h, self.d], [1, 1, 1], [1, self.h, 1])
        return out

    def __call__(self, Q, K, V, WQ, WK, WV, WO):
        for n in self.nodes(Q, K, V, WQ, WK, WV, WO):
            n[1]()
        return self.out

    def flops(self) -> int:
        s, a, h, d = self.s, self.a, self.h, self.d
        return 4 * (2 * s * a * h * d) + 2 * (2 * h * s * s * d) + 2 * (2 * h * s * s)
