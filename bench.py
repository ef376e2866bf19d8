#!/usr/bin/env python3
"""Throughput of the TRA join + aggregate hot path on one GB300 (one JSON line).

Default workload (``c5``): the largest single-GPU configuration, the matrix multiply of
"EinDecomp ... tensor relational algebra" section 2.1 at 16384 x 16384 x 16384, BF16
inputs N(0,1), FP32 accumulate, partition vector d = [1,1,1,1] (``--d`` for the others):
one join + aggregate on the tcgen05 tensor cores per step.  In the same process, after
the headline line's own measurement, the default run also times (device-resident, same
timing rules) the extended-semiring pair (``pair``: squared distance and max-plus, X
8192x256, Y 256x8192 fp32, d = [8,1,1,8]) and the 4-D contraction with the repartition
of its output (``c3``); they are reported under ``extra_workloads`` (``--extra`` picks
them, ``--extra none`` skips them).

Other workloads (``--workload``): pair, c1 (64^3 fp32 matmul under three d), c3, c4
(multi-head-attention EinGraph; c4f the same with the attention chain fused into one
kernel), c5b (8192^3 logsumexp); c2s and c5bs run the squared distance of the pair and
the 8192^3 logsumexp with split=bf16x3 (tensor cores).

``--impl reference`` times the CPU oracle on a bounded sample of the same
workload (the reference arm).  Under torchrun (N > 1) every rank runs an
independent replica of the workload (weak scaling, no collective on the data
path); rank 0 prints the line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "EinSum TRA join+aggregate TFLOP/s & % of roofline (1×GB300), vs CPU oracle"
FP32_LANES_PER_SM = 128  # FP32 FMA lanes per SM (4 sub-partitions x 32)


def measured_peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except OSError:
        return {}


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples (every 50 ms, stamped by nvidia-smi itself) of SM clock and throttle
    reasons; only the samples stamped inside the timed region count."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = str(gpu_index)
        try:
            import torch

            u = str(torch.cuda.get_device_properties(gpu_index).uuid)
            self.gpu = u if u.startswith("GPU-") else "GPU-" + u
        except Exception:
            pass
        self.proc = None
        self.lines = []
        self.region = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
            return
        t0 = time.time()  # wait (at most 3 s) for the first sample so the region is covered
        while not self.lines and time.time() - t0 < 3.0:
            time.sleep(0.01)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def mark(self, t_begin: float, t_end: float):
        """Wall-clock (time.time()) bounds of the timed region."""
        self.region = (t_begin, t_end)

    @staticmethod
    def _stamp(text):
        import datetime

        try:
            return datetime.datetime.strptime(text.strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 10:
                continue
            try:
                rows.append((self._stamp(parts[0]), float(parts[2]), float(parts[3]), parts[6:10]))
            except ValueError:
                continue
        inside = rows
        if self.region:
            lo, hi = self.region
            inside = [r for r in rows if r[0] is not None and lo - 0.025 <= r[0] <= hi + 0.025]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in inside:
            for n, v in zip(names, r[3]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        sm = [r[1] for r in inside]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(r[2] for r in rows) if rows else None,
                "reasons": sorted(reasons), "samples": len(sm),
                "sm_mhz_min": min(sm) if sm else None, "sampled": "nvidia-smi every 50 ms inside the timed region"}


# ----------------------------------------------------------------------------- workloads
class Step:
    """One named launch group inside a step, with its algorithmic work per launch.

    A tensor-core node may also give the bytes it must move at least (operands read once,
    output written once).  Its roofline is then the resource that bounds it: HBM when those
    bytes at the measured copy peak take longer than its flops at the measured BF16 peak
    (arithmetic intensity below the ridge point), the tensor cores otherwise.  A node that
    turns out HBM-bound keeps its flops in tensor_work."""

    def __init__(self, name, fn, work, unit, bound, launches, min_bytes=None):
        self.name, self.fn, self.work, self.unit, self.bound, self.launches = name, fn, work, unit, bound, launches
        self.tensor_work = None
        if bound == "tensor" and min_bytes:
            pk = measured_peaks()
            t_flop = work / (float(pk.get("bf16_tflops", 1900.0)) * 1e12)
            t_byte = min_bytes / (float(pk.get("hbm_gbs", 6800.0)) * 1e9)
            if t_byte > t_flop:
                self.tensor_work, self.work, self.unit, self.bound = work, min_bytes, "bytes", "hbm"


def kernel_launches(plan) -> int:
    """Kernels one ein_execute of this plan launches."""
    n = {"semiring_f32": 1, "tc_bf16": 1, "tc_bf16_pair": 1, "row_reduce": 1, "elementwise": 1, "lse_factored": 4,
         "literal": 2, "tc_split3": 5}[plan.kernel]
    if plan.kernel == "tc_split3" and ":add:lse" in plan.spec:
        n += 1  # the underflow fix-up pass
    spec = plan.spec
    if plan.kernel == "semiring_f32" and ":sqdiff:sum" in spec and "sqdiff=direct" not in spec and "in=bf16" not in spec:
        n += 2  # row / column norms of the squared-distance expansion
    return n


def device_relation(tra, torch, dense_dev, shape, d):
    if all(v == 1 for v in d):
        return dense_dev
    out = torch.empty_like(dense_dev)
    tra.repartition(dense_dev, out, shape, [1] * len(shape), d)
    return out


class PairWorkload:
    """Squared distance and max-plus, X 8192x256, Y 256x8192 fp32, d = [8,1,1,8]."""

    name = "semiring pair: sqdist (x-y)^2/sum + max-plus (x+y)/max, X 8192x256, Y 256x8192 fp32, d=[8,1,1,8]"
    M, K, N = 8192, 256, 8192
    d = [8, 1, 1, 8]
    dtype = "f32"
    cpu_default = 3072  # output rows (about 10 s of the oracle on 16 host cores)
    ref_default = 32

    def __init__(self, seed_offset=0, d=None):
        self.seed_offset = seed_offset

    def host_inputs(self):
        import datagen

        X = datagen.normal_f32((self.M, self.K), 0 + self.seed_offset, 0)
        Y = datagen.normal_f32((self.K, self.N), 1 + self.seed_offset, 0)
        return [X, Y]

    def setup(self, tra, torch, inputs):
        X, Y = inputs
        dev = torch.device("cuda")
        self.tra, self.torch = tra, torch
        self.Xd = torch.from_numpy(X).to(dev).reshape(-1)  # [8,1] relation of X == dense X
        self.Yd = torch.from_numpy(Y).to(dev).reshape(-1)
        self.Yr = torch.empty_like(self.Yd)
        self.p_sq = tra.Plan("ij,jk->ik:sqdiff:sum", [self.M, self.K, self.N], self.d)
        self.p_mx = tra.Plan("ij,jk->ik:add:max", [self.M, self.K, self.N], self.d)
        self.Zs = torch.empty(self.M * self.N, dtype=torch.float32, device=dev)
        self.Zm = torch.empty_like(self.Zs)
        ops = 2 * self.M * self.K * self.N
        self.steps = [
            Step("repartition Y [1,1]->[1,8]", lambda: tra.repartition(self.Yd, self.Yr, [self.K, self.N], [1, 1], [1, 8]),
                 2 * self.K * self.N * 4, "bytes", "hbm", 1),
            Step("join+agg (x-y)^2/sum", lambda: self.p_sq.execute(self.Xd, self.Yr, self.Zs), ops, "flop", "alu",
                 kernel_launches(self.p_sq)),
            Step("join+agg (x+y)/max", lambda: self.p_mx.execute(self.Xd, self.Yr, self.Zm), ops, "flop", "alu",
                 kernel_launches(self.p_mx)),
        ]
        self.inputs_dev = [self.Xd, self.Yd]
        self.outputs_dev = [self.Zs, self.Zm]
        self.output_steps = [1, 2]  # the launch group that produces each output

    # end to end: the CUDA-core kernels store their results straight into pinned host memory
    # (device-addressable over the host link), so no staging copy follows them
    e2e_host_outputs = True

    def redirect_outputs(self, outs):
        self.Zs, self.Zm = outs

    def ops_per_step(self):
        return 2 * (2 * self.M * self.K * self.N)

    # reference arm: oracle on output rows [r0, r0+rows) of both EinSums
    def oracle_sample(self, inputs, r0, rows):
        import oracle

        X, Y = inputs
        Xd, Yd = X.astype(np.float64), Y.astype(np.float64)
        pts = (np.arange(rows, dtype=np.int64)[:, None] % self.M + r0) % self.M * self.N + np.arange(self.N)[None, :]
        pts = pts.reshape(-1)
        oracle.einsum_points("ij,jk->ik", Xd, Yd, pts, op="sqdiff", agg="sum")
        oracle.einsum_points("ij,jk->ik", Xd, Yd, pts, op="add", agg="max")
        return 2 * 2 * pts.size * self.K  # two EinSums, two ops per tuple

    def sample_text(self, rows):
        return f"{rows} of 8192 output rows (all 8192 columns) of both EinSums"

    def traffic_key(self, j):
        return ("k_semiring.cu", ["repartition", "semiring sqdiff/sum", "semiring add/max"][j])


class _PointsWorkload:
    """Shared pieces: inputs resident in relation layout, one or more plans per step, oracle on points."""

    cpu_default = 64  # output points per oracle sample
    ref_default = 8
    dtype = "bf16"

    def __init__(self, seed_offset=0, d=None):
        self.seed_offset = seed_offset
        if d is not None:
            self.d = list(d)

    def f64_inputs(self, inputs, bf16=True):
        """The oracle's double inputs, converted once (outside any timed oracle sample)."""
        if getattr(self, "_f64", None) is None:
            from datagen import bf16_bits_to_f32

            self._f64 = [(bf16_bits_to_f32(a) if bf16 else a).astype(np.float64) for a in inputs]
        return self._f64

    def oracle_points(self, eq, X, Y, op, agg, zshape, r0, n, alpha=1.0):
        import oracle

        total = int(np.prod(zshape))
        pts = (np.arange(n, dtype=np.int64) + r0 * n) % total
        oracle.einsum_points(eq, X, Y, pts, op=op, agg=agg, alpha=alpha)
        K = 1
        return pts.size, K


def _bf16_host(shape, seed, tensor, sigma=1.0):
    import datagen

    return datagen.normal_bf16(shape, seed, tensor, 0.0, sigma)


def _dev_bf16(torch, bits):
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda().reshape(-1)


class C1Workload(_PointsWorkload):
    dtype = "f32"
    name = "matmul 64x64x64 fp32 U[-1,1], d in {[4,1,1,4],[1,4,4,1],[2,2,2,2]} (three executions per step)"
    d = [[4, 1, 1, 4], [1, 4, 4, 1], [2, 2, 2, 2]]
    single_core_baseline = True  # the oracle is timed on all host cores and on one

    def host_inputs(self):
        import datagen

        return [datagen.uniform_f32((64, 64), 0 + self.seed_offset, 0), datagen.uniform_f32((64, 64), 0 + self.seed_offset, 1)]

    mode = "fused"

    def setup(self, tra, torch, inputs):
        X, Y = inputs
        self.Xd = torch.from_numpy(X).cuda().reshape(-1)
        self.Yd = torch.from_numpy(Y).cuda().reshape(-1)
        self.steps, self.outputs_dev = [], []
        for d in self.d:
            p = tra.Plan(f"ij,jk->ik:mul:sum:mode={self.mode}", [64, 64, 64], d)
            xr, yr = torch.empty_like(self.Xd), torch.empty_like(self.Yd)
            z = torch.empty(64 * 64, dtype=torch.float32, device="cuda")
            self.outputs_dev.append(z)

            def run(p=p, xr=xr, yr=yr, z=z, d=d):
                tra.repartition(self.Xd, xr, [64, 64], [1, 1], d[:2])
                tra.repartition(self.Yd, yr, [64, 64], [1, 1], d[2:])
                p.execute(xr, yr, z)

            self.steps.append(Step(f"partition + join+agg d={d}", run, 2 * 64 ** 3, "flop", "alu",
                                   kernel_launches(p) + 2))
        self.inputs_dev = [self.Xd, self.Yd]

    def ops_per_step(self):
        return 3 * 2 * 64 ** 3

    def oracle_sample(self, inputs, r0, n):
        X, Y = [a.astype(np.float64) for a in inputs]
        import oracle

        for _ in self.d:
            oracle.einsum("ij,jk->ik", X, Y)
        return 3 * 2 * 64 ** 3

    def sample_text(self, n):
        return "the whole workload (three 64^3 EinSums)"


class C1LiteralWorkload(C1Workload):
    """Config 1 executed as the literal TRA: one partial sub-tensor per join tuple, then the
    aggregation combines each output key's partials in canonical order (combine kernel)."""
    name = ("matmul 64x64x64 fp32 U[-1,1], d in {[4,1,1,4],[1,4,4,1],[2,2,2,2]}, literal TRA "
            "(one partial per join tuple, ordered combine; three executions per step)")
    mode = "literal"


class C3Workload(_PointsWorkload):
    name = "4-D contraction C[a,b,c,d]=sum_e,f A[a,b,e,f]B[c,f,e,d], 64^6 BF16 in / FP32 out, d=[4,1,1,1,4,1,1,1]; + repartition of C [4,1,4,1]->[1,4,1,4]"
    d = [4, 1, 1, 1, 4, 1, 1, 1]
    cpu_default = 4194304  # contraction outputs (about 8 s of the oracle on 16 host cores)

    def host_inputs(self):
        return [_bf16_host((64,) * 4, 0 + self.seed_offset, 0), _bf16_host((64,) * 4, 0 + self.seed_offset, 1)]

    def setup(self, tra, torch, inputs):
        A, B = inputs
        self.Ad, self.Bd = _dev_bf16(torch, A), _dev_bf16(torch, B)  # [4,1,1,1] relation == dense
        self.p = tra.Plan("abef,cfed->abcd:mul:sum:in=bf16", [64] * 6, self.d)
        self.C = torch.empty(64 ** 4, dtype=torch.float32, device="cuda")
        self.C2 = torch.empty_like(self.C)
        self.steps = [
            Step("join+agg 4-D contraction (tcgen05)", lambda: self.p.execute(self.Ad, self.Bd, self.C), 2 * 64 ** 6,
                 "flop", "tensor", kernel_launches(self.p)),
            Step("repartition C [4,1,4,1]->[1,4,1,4]",
                 lambda: tra.repartition(self.C, self.C2, [64] * 4, [4, 1, 4, 1], [1, 4, 1, 4]), 2 * 64 ** 4 * 4,
                 "bytes", "hbm", 1),
        ]
        self.inputs_dev = [self.Ad, self.Bd]
        self.outputs_dev = [self.C2]

    def ops_per_step(self):
        return 2 * 64 ** 6

    def oracle_sample(self, inputs, r0, n):
        A, B = self.f64_inputs(inputs)
        self.oracle_points("abef,cfed->abcd", A, B, "mul", "sum", (64,) * 4, r0, n)
        return 2 * n * 64 * 64

    def sample_text(self, n):
        return f"{n} of 64^4 outputs of the contraction"

    def traffic_key(self, j):
        return ("k_tc.cu", "tc_gemm 4-D contraction") if j == 0 else ("k_repart.cu", "repartition 64^4 fp32")


def _packed_dev(torch, inputs):
    """Q, K, V in one device buffer, back to back, and so the relations of W_Q, W_K, W_V (the graph then
    runs the three projections as one EinSum); W_O on its own."""
    qkv = _dev_bf16(torch, np.concatenate([x.reshape(-1) for x in inputs[:3]]))
    w = _dev_bf16(torch, np.concatenate([x.reshape(-1) for x in inputs[3:6]]))
    n, m = inputs[0].size, inputs[3].size
    return [qkv[:n], qkv[n:2 * n], qkv[2 * n:], w[:m], w[m:2 * m], w[2 * m:], _dev_bf16(torch, inputs[6])]


class C4Workload(_PointsWorkload):
    name = "multi-head attention EinGraph s=4096 a=4096 h=32 d=128, BF16 activations N(0,1), weights N(0,0.02)"
    d = "projections split h=32 (head-major outputs); scores/lse/exp/A.V split h=32; repartition of O to dense"
    cpu_default = 2457600  # Q-projection outputs (about 8 s of the oracle on 16 host cores)

    def host_inputs(self):
        s, a, h, d = 4096, 4096, 32, 128
        o = self.seed_offset
        ws = [_bf16_host((a, h, d), 0 + o, 3 + t, 0.02) for t in range(4)]
        # W_Q, W_K, W_V as the projections' relations under [1, h, 1]: stored [h][a][d]
        ws[:3] = [np.ascontiguousarray(w.reshape(a, h, d).transpose(1, 0, 2)).reshape(-1) for w in ws[:3]]
        return [_bf16_host((s, a), 0 + o, t) for t in range(3)] + ws

    def setup(self, tra, torch, inputs):
        from tensor_relational_algebra_gb300.eingraph import AttentionGraph

        self.g = AttentionGraph(4096, 4096, 32, 128)
        self.dev = _packed_dev(torch, inputs)
        self.steps = [Step(*n) for n in self.g.nodes(*self.dev)]
        self.inputs_dev = self.dev
        self.outputs_dev = [self.g.out]

    def ops_per_step(self):
        return self.g.flops()

    def oracle_sample(self, inputs, r0, n):
        from datagen import bf16_bits_to_f32

        Q = bf16_bits_to_f32(inputs[0]).astype(np.float64)
        WQ = bf16_bits_to_f32(inputs[3]).astype(np.float64).reshape(32, 4096, 128).transpose(1, 0, 2)  # dense [a][h][d]
        self.oracle_points("sa,ahd->shd", Q, WQ, "mul", "sum", (4096, 32, 128), r0, n)
        return 2 * n * 4096

    def sample_text(self, n):
        return f"{n} outputs of the Q projection node (4096 terms each)"


class C4fWorkload(C4Workload):
    name = ("multi-head attention EinGraph s=4096 a=4096 h=32 d=128, BF16 activations N(0,1), weights N(0,0.02), "
            "Scores -> L -> exp -> A.V -> repartition O fused in one kernel")
    d = "projections split h=32 (head-major outputs); fused attention over (s/128 row blocks) x h"

    def setup(self, tra, torch, inputs):
        from tensor_relational_algebra_gb300.eingraph import AttentionGraph

        self.g = AttentionGraph(4096, 4096, 32, 128, fused=True)
        self.dev = _packed_dev(torch, inputs)
        self.steps = [Step(*n) for n in self.g.nodes(*self.dev)]
        self.inputs_dev = self.dev
        self.outputs_dev = [self.g.out]

    def traffic_key(self, j):
        name = self.steps[j].name
        if name.startswith("proj Q, K, V"):
            return ("k_tc.cu", "tc_gemm projections QKV s=a=4096 h=32 d=128")
        return ("k_attn.cu", "attention s=4096 h=32 d=128" if name.startswith("attention") else "-")


class C5Workload(_PointsWorkload):
    name_fmt = "BF16 matmul Z[i,k]=sum_j X[i,j]Y[j,k] 16384^3, inputs N(0,1), FP32 accumulate, d={}"
    d = [1, 1, 1, 1]
    cpu_default = 262144  # output points (about 10 s of the oracle on 16 host cores)
    ref_default = 16384

    @property
    def name(self):
        return self.name_fmt.format(self.d)

    def host_inputs(self):
        n = 16384
        return [_bf16_host((n, n), 0 + self.seed_offset, 0), _bf16_host((n, n), 0 + self.seed_offset, 1)]

    def setup(self, tra, torch, inputs):
        n = 16384
        X, Y = inputs
        self.Xd, self.Yd = _dev_bf16(torch, X), _dev_bf16(torch, Y)
        self.Xr, self.Yr = device_relation(tra, torch, self.Xd, [n, n], self.d[:2]), device_relation(
            tra, torch, self.Yd, [n, n], self.d[2:])
        torch.cuda.synchronize()
        self.p = tra.Plan("ij,jk->ik:mul:sum:in=bf16", [n, n, n], self.d)
        self.Z = torch.empty(n * n, dtype=torch.float32, device="cuda")
        self.steps = [Step(f"join+agg matmul d={self.d} (tcgen05)", lambda: self.p.execute(self.Xr, self.Yr, self.Z),
                           2 * n ** 3, "flop", "tensor", kernel_launches(self.p))]
        self.inputs_dev = [self.Xr, self.Yr]
        self.outputs_dev = [self.Z]

    # end to end: the result goes straight into pinned host memory (the tensor-core kernel takes
    # its warp-store epilogue for a host output), so its 1 GiB crosses the host link while later
    # tiles compute, with no device staging buffer and no copy-engine pass
    e2e_host_outputs = True
    # inputs 2 x 512 MiB (larger than L2): step k + 1's copy in can run while step k computes
    e2e_pipeline = True

    def redirect_outputs(self, outs):
        self.Z = outs[0]

    def use_inputs(self, bufs):
        self.Xr, self.Yr = bufs

    def use_outputs(self, bufs):
        self.Z = bufs[0]

    def ops_per_step(self):
        return 2 * 16384 ** 3

    def oracle_sample(self, inputs, r0, n):
        X, Y = self.f64_inputs(inputs)
        self.oracle_points("ij,jk->ik", X, Y, "mul", "sum", (16384, 16384), r0, n)
        return 2 * n * 16384

    def sample_text(self, n):
        return f"{n} of 16384^2 outputs"

    def traffic_key(self, j):
        return ("k_tc.cu", f"tc_gemm 16384^3 d={self.d}")


class C5bWorkload(_PointsWorkload):
    dtype = "f32"
    name_fmt = "logsumexp-aggregated Z[i,k]=lse_j(X[i,j]+Y[j,k]) 8192^3 fp32, d={}"
    d = [1, 1, 1, 1]
    cpu_default = 64

    @property
    def name(self):
        return self.name_fmt.format(self.d)

    def host_inputs(self):
        import datagen

        n = 8192
        return [datagen.normal_f32((n, n), 0 + self.seed_offset, 0), datagen.normal_f32((n, n), 0 + self.seed_offset, 1)]

    def setup(self, tra, torch, inputs):
        n = 8192
        X, Y = inputs
        self.Xd, self.Yd = torch.from_numpy(X).cuda().reshape(-1), torch.from_numpy(Y).cuda().reshape(-1)
        self.Xr, self.Yr = device_relation(tra, torch, self.Xd, [n, n], self.d[:2]), device_relation(
            tra, torch, self.Yd, [n, n], self.d[2:])
        self.p = tra.Plan("ij,jk->ik:add:lse", [n, n, n], self.d)
        self.ws = torch.empty(self.p.workspace_bytes, dtype=torch.uint8, device="cuda")
        self.Z = torch.empty(n * n, dtype=torch.float32, device="cuda")
        self.steps = [Step(f"join+agg (x+y)/logsumexp d={self.d}", lambda: self.p.execute(self.Xr, self.Yr, self.Z, self.ws),
                           2 * n ** 3, "flop", "alu", kernel_launches(self.p))]
        self.inputs_dev = [self.Xr, self.Yr]
        self.outputs_dev = [self.Z]

    def ops_per_step(self):
        return 2 * 8192 ** 3

    def oracle_sample(self, inputs, r0, n):
        X, Y = self.f64_inputs(inputs, bf16=False)
        self.oracle_points("ij,jk->ik", X, Y, "add", "lse", (8192, 8192), r0, n)
        return 2 * n * 8192

    def sample_text(self, n):
        return f"{n} of 8192^2 outputs"


class C2sWorkload(PairWorkload):
    """Squared distance only, X 8192x256, Y 256x8192 fp32, d = [8,1,1,8], with split=bf16x3: the
    expansion's x.y on BF16 tensor cores as hi.hi + hi.lo + lo.hi (K' = 768)."""

    name = "squared distance (x-y)^2/sum, X 8192x256, Y 256x8192 fp32, d=[8,1,1,8], split=bf16x3 on tensor cores"
    e2e_host_outputs = False  # the tensor-core epilogue stores through a TMA tensor map: device memory only

    def traffic_key(self, j):
        return ("k_tc.cu", "-")  # no ncu record of the split GEMM's DRAM bytes: traffic stays null

    def setup(self, tra, torch, inputs):
        X, Y = inputs
        dev = torch.device("cuda")
        self.Xd = torch.from_numpy(X).to(dev).reshape(-1)
        self.Yd = torch.from_numpy(Y).to(dev).reshape(-1)
        self.Yr = torch.empty_like(self.Yd)
        self.p_sq = tra.Plan("ij,jk->ik:sqdiff:sum:split=bf16x3", [self.M, self.K, self.N], self.d)
        self.ws = torch.empty(self.p_sq.workspace_bytes, dtype=torch.uint8, device=dev)
        self.Zs = torch.empty(self.M * self.N, dtype=torch.float32, device=dev)
        # work of the split step: the GEMM's BF16 flops over K' = 3K (the EinSum's own 2MKN is the
        # headline value)
        self.steps = [
            Step("repartition Y [1,1]->[1,8]", lambda: tra.repartition(self.Yd, self.Yr, [self.K, self.N], [1, 1], [1, 8]),
                 2 * self.K * self.N * 4, "bytes", "hbm", 1),
            Step("join+agg (x-y)^2/sum, split bf16x3 (tcgen05)", lambda: self.p_sq.execute(self.Xd, self.Yr, self.Zs, self.ws),
                 3 * 2 * self.M * self.K * self.N, "flop", "tensor", kernel_launches(self.p_sq)),
        ]
        self.inputs_dev = [self.Xd, self.Yd]
        self.outputs_dev = [self.Zs]
        self.output_steps = [1]

    def ops_per_step(self):
        return 2 * self.M * self.K * self.N

    def oracle_sample(self, inputs, r0, rows):
        import oracle

        X, Y = inputs
        pts = (np.arange(rows, dtype=np.int64)[:, None] % self.M + r0) % self.M * self.N + np.arange(self.N)[None, :]
        oracle.einsum_points("ij,jk->ik", X.astype(np.float64), Y.astype(np.float64), pts.reshape(-1), op="sqdiff",
                             agg="sum")
        return 2 * pts.size * self.K

    def sample_text(self, rows):
        return f"{rows} of 8192 output rows (all 8192 columns)"


class C5bsWorkload(C5bWorkload):
    name_fmt = "logsumexp-aggregated Z[i,k]=lse_j(X[i,j]+Y[j,k]) 8192^3 fp32, d={}, split=bf16x3 on tensor cores"

    def setup(self, tra, torch, inputs):
        n = 8192
        X, Y = inputs
        self.Xd, self.Yd = torch.from_numpy(X).cuda().reshape(-1), torch.from_numpy(Y).cuda().reshape(-1)
        self.Xr, self.Yr = device_relation(tra, torch, self.Xd, [n, n], self.d[:2]), device_relation(
            tra, torch, self.Yd, [n, n], self.d[2:])
        self.p = tra.Plan("ij,jk->ik:add:lse:split=bf16x3", [n, n, n], self.d)
        self.ws = torch.empty(self.p.workspace_bytes, dtype=torch.uint8, device="cuda")
        self.Z = torch.empty(n * n, dtype=torch.float32, device="cuda")
        self.steps = [Step(f"join+agg (x+y)/logsumexp d={self.d}, split bf16x3 (tcgen05)",
                           lambda: self.p.execute(self.Xr, self.Yr, self.Z, self.ws), 3 * 2 * n ** 3, "flop", "tensor",
                           kernel_launches(self.p))]
        self.inputs_dev = [self.Xr, self.Yr]
        self.outputs_dev = [self.Z]


WORKLOADS = {"pair": PairWorkload, "c1": C1Workload, "c1l": C1LiteralWorkload, "c2s": C2sWorkload, "c3": C3Workload,
             "c4": C4Workload, "c4f": C4fWorkload, "c5": C5Workload, "c5b": C5bWorkload, "c5bs": C5bsWorkload}


# ----------------------------------------------------------------------------- measurement
def time_e2e_pipelined(torch, wl, pinned_in, pinned_out, steps, warmup, staged):
    """End to end as a stream of steps: step k + 1's inputs are copied in from pinned host memory
    on a copy stream while step k computes, into the other of two device input buffers (a buffer
    is reloaded only once the step that used it has finished).  The results reach pinned host
    memory either from the kernels themselves (staged=False: the workload's outputs already point
    there) or through two device output buffers copied out on a second copy stream while the next
    step computes (staged=True; a buffer is rewritten only once its copy has left).  Returns the
    ms from the start of the first copy in to the end of the last step's results."""
    comp = torch.cuda.current_stream()
    cin, cout = torch.cuda.Stream(), torch.cuda.Stream()
    bin_ = [list(wl.inputs_dev), [torch.empty_like(t) for t in wl.inputs_dev]]
    bout = [list(wl.outputs_dev), [torch.empty_like(t) for t in wl.outputs_dev]] if staged else None

    def event(stream):
        ev = torch.cuda.Event()
        ev.record(stream)
        return ev

    def run(n, record):
        done, left = [None, None], [None, None]

        def load(k):
            if done[k & 1] is not None:
                cin.wait_event(done[k & 1])
            with torch.cuda.stream(cin):
                for src, dst in zip(pinned_in, bin_[k & 1]):
                    dst.copy_(src, non_blocking=True)
            return event(cin)

        torch.cuda.synchronize()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if record:
            start.record(cin)
        ready = load(0)
        for k in range(n):
            comp.wait_event(ready)
            wl.use_inputs(bin_[k & 1])
            if staged:
                if left[k & 1] is not None:
                    comp.wait_event(left[k & 1])
                wl.use_outputs(bout[k & 1])
            for st in wl.steps:
                st.fn()
            done[k & 1] = event(comp)
            if staged:
                cout.wait_event(done[k & 1])
                with torch.cuda.stream(cout):
                    for src, dst in zip(bout[k & 1], pinned_out):
                        dst.copy_(src, non_blocking=True)
                left[k & 1] = event(cout)
            if k + 1 < n:
                ready = load(k + 1)
        if record:
            end.record(cout if staged else comp)
        torch.cuda.synchronize()
        return start.elapsed_time(end) if record else None

    run(warmup, False)
    ms = run(steps, True)
    wl.use_inputs(bin_[0])
    if staged:
        wl.use_outputs(bout[0])
    return ms


def time_steps(torch, wl, steps, warmup, flush, sampler=None, e2e_io=None):
    """Run warmup + timed steps; per-launch-group CUDA events on the launching stream."""
    stream = torch.cuda.current_stream()
    n = len(wl.steps)

    def one_step(record):
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1 + (2 if e2e_io else 0))] if record else None
        i = 0
        if record:
            evs[0].record(stream)
        if e2e_io:
            e2e_io["h2d"]()
            if record:
                evs[1].record(stream)
            i = 1
        for j, st in enumerate(wl.steps):
            st.fn()
            if record:
                evs[i + j + 1].record(stream)
            if e2e_io:
                e2e_io["after"](j)
        if e2e_io:
            e2e_io["d2h"]()
            if record:
                evs[-1].record(stream)
        return evs

    for _ in range(warmup):
        one_step(False)
        flush()
    torch.cuda.synchronize()
    recs = []
    if sampler:
        sampler.start()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    w0 = time.time()
    for _ in range(steps):
        recs.append(one_step(True))
        flush()
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    if sampler:
        sampler.mark(w0, time.time())
    clocks = sampler.stop() if sampler else None
    step_ms = [r[0].elapsed_time(r[-1]) for r in recs]
    off = 1 if e2e_io else 0
    per = [[r[off + j].elapsed_time(r[off + j + 1]) for r in recs] for j in range(n)]
    return step_ms, per, wall, clocks


def traffic_for(kernel_file: str, kernel_name: str, units_scale: float = 1.0):
    """DRAM bytes per launch from the committed ncu summary, if the kernel source is unchanged."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        rec = json.load(open(path))[kernel_name]
    except (OSError, KeyError, ValueError):
        return None
    src = os.path.join(ROOT, "tensor_relational_algebra_gb300", "csrc", kernel_file)
    try:
        h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    except OSError:
        return None
    if rec.get("source_sha256_16") != h:
        return None
    return rec["dram_bytes_per_launch"] * units_scale


def max_over_ranks(value_ms: float, world: int, device: str = "cuda") -> float:
    """Largest per-rank elapsed time (the job's time) -- an all-reduce MAX across ranks."""
    if world <= 1:
        return value_ms
    import torch
    import torch.distributed as dist

    t = torch.tensor([value_ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def plan_times(tra, wl, reps: int = 20) -> dict:
    """Host time (median of reps, ms) to build each plan the step executes: ein_plan runs once,
    before the timed region, and is reported here apart from it."""
    plans = []

    def collect(obj, depth):
        for v in vars(obj).values():
            if isinstance(v, tra.Plan):
                plans.append(v)
            elif depth == 0 and type(v).__module__.startswith("tensor_relational_algebra_gb300"):
                collect(v, 1)

    collect(wl, 0)
    out = {}
    for p in plans:
        ts = []
        for _ in range(reps):
            t0 = time.perf_counter()
            q = tra.Plan(p.spec, p.bounds, p.d)
            ts.append(time.perf_counter() - t0)
            del q
        out[f"{p.spec} d={p.d}"] = round(sorted(ts)[len(ts) // 2] * 1e3, 4)
    return out


def roofline_of(step, ms, peaks, props):
    """(achieved, peak, unit) of one launch group from its mean device time."""
    if step.bound == "alu":
        sm_max = float(peaks.get("sm_max_mhz", 2070.0))
        pk = props.multi_processor_count * FP32_LANES_PER_SM * 2 * sm_max * 1e6 / 1e12
        return step.work / (ms * 1e-3) / 1e12, pk, "TFLOP/s"
    if step.bound == "tensor":
        return step.work / (ms * 1e-3) / 1e12, float(peaks.get("bf16_tflops", 1900.0)), "TFLOP/s"
    return step.work / (ms * 1e-3) / 1e9, float(peaks.get("hbm_gbs", 6800.0)), "GB/s"


def fp32_mix_ceilings():
    """Fractions of the FP32 peak that the semiring inner step's instruction mix reaches by
    itself (profiles/fp32_ceilings.json, written by --probe fp32): {kind: frac}."""
    try:
        rec = json.load(open(os.path.join(ROOT, "profiles", "fp32_ceilings.json")))["record"]
        return {r["kind"]: r["of_fp32_peak_at_max_clock"] for r in rec["results"]}
    except (OSError, KeyError, ValueError):
        return {}


def mix_kind(step_name):
    """Probe kind whose loop is the node's inner step: 1 for max/min-plus, 0 for FFMA loops."""
    if "/max" in step_name or "/min" in step_name:
        return 1
    if "/sum" in step_name or "lse" in step_name or "logsumexp" in step_name:
        return 0
    return None


def roofline_nodes(wl, means, peaks, props):
    nodes = []
    mix = fp32_mix_ceilings()
    for step, ms in zip(wl.steps, means):
        a, pk, u = roofline_of(step, ms, peaks, props)
        node = {"name": step.name, "bound": step.bound, "ms": round(ms, 4), "achieved": round(a, 1),
                "unit": u, "frac": round(a / pk, 3)}
        if step.tensor_work:  # HBM-bound tensor-core node: its flops against the BF16 peak too
            tf = step.tensor_work / (ms * 1e-3) / 1e12
            node["tensor_achieved"] = round(tf, 1)
            node["tensor_frac"] = round(tf / float(peaks.get("bf16_tflops", 1900.0)), 3)
            node["flop_per_byte"] = round(step.tensor_work / step.work, 1)
        k = mix_kind(step.name) if step.bound == "alu" else None
        if k in mix:
            node["instruction_mix_ceiling_frac"] = round(mix[k], 3)
        nodes.append(node)
    return nodes


def peak_source(bound):
    pk = measured_peaks()
    if bound == "alu":
        return ("derived: SMs x 128 FP32 lanes x 2 x max SM clock (" +
                ("MEASURED_PEAKS sm_max_mhz" if "sm_max_mhz" in pk else "2070 MHz, of fallback") +
                "); the inner step's instruction-mix ceilings are measured in profiles/fp32_ceilings.json "
                "(bench.py --probe fp32)")
    key = "hbm_gbs" if bound == "hbm" else "bf16_tflops"
    return ("MEASURED_PEAKS.json (of measured)" if key in pk else
            "fallback 6.8 TB/s copy, 1.9 PFLOP/s BF16 (one earlier GB300 measurement; of fallback)")


def extra_workload(torch, tra, name, args, flush, local):
    """Device-resident timing of one more workload in this process (the same warm-up, step
    count, L2 flush and clock sampling as the headline), for the extra_workloads record."""
    wl = WORKLOADS[name]()
    wl.setup(tra, torch, wl.host_inputs())
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    step_ms, per, wall, clocks = time_steps(torch, wl, args.steps, args.warmup, flush, sampler)
    peaks, props = measured_peaks(), torch.cuda.get_device_properties(0)
    means = [statistics.mean(p) for p in per]
    dom = max(range(len(wl.steps)), key=lambda j: means[j])
    st = wl.steps[dom]
    achieved, peak, unit = roofline_of(st, means[dom], peaks, props)
    total = sum(step_ms)
    rec = {"workload": wl.name, "key": name, "d": wl.d, "dtype": wl.dtype, "steps": args.steps,
           "ms_per_step": total / args.steps, "value": job_throughput(wl.ops_per_step(), args.steps, 1, total),
           "unit": "TFLOP/s",
           "roofline": {"bound": st.bound, "kernel": st.name, "achieved": achieved, "peak": peak, "unit": unit,
                        "frac": achieved / peak,
                        "traffic": traffic_for(*wl.traffic_key(dom)) if hasattr(wl, "traffic_key") else None,
                        "peak_source": peak_source(st.bound)},
           "roofline_nodes": roofline_nodes(wl, means, peaks, props),
           "gpu_launches": args.steps * sum(s.launches for s in wl.steps),
           "clocks": clocks, "wall_s": round(wall, 3)}
    if st.bound == "alu" and clocks and clocks.get("sm_mhz"):
        pk = props.multi_processor_count * FP32_LANES_PER_SM * 2 * clocks["sm_mhz"] * 1e6 / 1e12
        rec["alu_peak_at_sampled_clock"] = {"sm_mhz": clocks["sm_mhz"], "peak": pk, "frac": achieved / pk}
    del wl
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return rec


def job_throughput(ops_per_step: int, steps: int, world: int, job_ms: float) -> float:
    """Whole-job TFLOP/s: every rank processed its own replica of the workload (weak scaling)."""
    return world * ops_per_step * steps / (job_ms * 1e-3) / 1e12


def run_ours(args):
    import torch

    import tensor_relational_algebra_gb300 as tra

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    tra.load()
    wl = WORKLOADS[args.workload](seed_offset=rank, d=args.d)
    host = wl.host_inputs()
    wl.setup(tra, torch, host)
    flush_buf = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device="cuda")

    def flush():
        flush_buf.zero_()

    def barrier():
        if world > 1:
            import torch.distributed as dist

            dist.barrier()
        torch.cuda.synchronize()

    # device-resident timing
    barrier()
    sampler = ClockSampler(local) if rank == 0 else None
    step_ms, per, wall, clocks = time_steps(torch, wl, args.steps, args.warmup, flush, sampler)
    barrier()
    total_ms = max_over_ranks(sum(step_ms), world)
    ops = wl.ops_per_step()
    value = job_throughput(ops, args.steps, world, total_ms)

    # end to end: pinned host inputs -> device, the step, results -> pinned host
    def pinned_host(h, like):
        """Pinned host copy of one input with the device tensor's dtype: bf16 inputs are kept as
        their bit patterns (uint16 viewed as bfloat16), so the copy is a plain byte transfer."""
        t = torch.from_numpy(np.ascontiguousarray(h).reshape(-1))
        if like.dtype == torch.bfloat16 and t.dtype == torch.uint16:
            t = t.view(torch.bfloat16)
        if t.dtype != like.dtype or t.numel() != like.numel():
            raise ValueError(f"host input {t.dtype}[{t.numel()}] does not match device {like.dtype}[{like.numel()}]")
        return t.pin_memory()

    pinned_in = [pinned_host(h, d) for h, d in zip(host, wl.inputs_dev)]
    pinned_out = [torch.empty(o.numel(), dtype=o.dtype).pin_memory() for o in wl.outputs_dev]

    def h2d():
        for src, dst in zip(pinned_in, wl.inputs_dev):
            dst.copy_(src, non_blocking=True)

    # each result leaves on a copy stream as soon as the launch group producing it is done,
    # overlapping the groups after it; the step ends when the copies have landed
    copy_stream = torch.cuda.Stream()
    out_steps = getattr(wl, "output_steps", [len(wl.steps) - 1] * len(wl.outputs_dev))

    def after(j):
        ready = [k for k, sj in enumerate(out_steps) if sj == j]
        if not ready:
            return
        copy_stream.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(copy_stream):
            for k in ready:
                pinned_out[k].copy_(wl.outputs_dev[k], non_blocking=True)

    def d2h():
        torch.cuda.current_stream().wait_stream(copy_stream)

    n_e2e = max(3, args.steps // 4)
    e2e_alt = None
    if getattr(wl, "e2e_pipeline", False):
        # results staged in device memory and copied out while the next step computes
        barrier()
        e2e_alt = max_over_ranks(time_e2e_pipelined(torch, wl, pinned_in, pinned_out, n_e2e, args.warmup, True),
                                 world)
    if getattr(wl, "e2e_host_outputs", False):
        # the step's kernels write pinned host memory themselves: the same bytes cross to the
        # host, with no device-side staging buffer and no copy engine pass
        wl.redirect_outputs(pinned_out)

        def after(j):
            return None

        def d2h():
            return None

    barrier()
    staged_method = ("pipelined: step k+1's inputs copied in on one copy stream and step k-1's results copied out "
                     "on another while step k computes (two device buffers each); no L2 flush (inputs larger than "
                     "L2); first copy in to last copy out")
    if getattr(wl, "e2e_pipeline", False):
        e2e_total, e2e_method = e2e_alt, staged_method
        e2e_alt = None
        if getattr(wl, "e2e_host_outputs", False):
            direct = max_over_ranks(time_e2e_pipelined(torch, wl, pinned_in, pinned_out, n_e2e, args.warmup, False),
                                    world)
            direct_method = ("pipelined: step k+1's inputs copied in on a copy stream while step k computes (two "
                             "device input buffers); results written into pinned host memory by the kernels; no "
                             "L2 flush (inputs larger than L2); first copy in to last kernel")
            e2e_alt = direct
            if direct < e2e_total:
                e2e_total, e2e_alt, e2e_method = direct, e2e_total, direct_method
    else:
        e2e_ms, _, _, _ = time_steps(torch, wl, n_e2e, args.warmup, flush, None,
                                     {"h2d": h2d, "after": after, "d2h": d2h})
        e2e_total = max_over_ranks(sum(e2e_ms), world)
        e2e_method = "per step: inputs copied in, the step, results out; L2 flushed between steps"
    barrier()
    e2e_value = job_throughput(ops, n_e2e, world, e2e_total)
    h2d_bytes = sum(t.numel() * t.element_size() for t in pinned_in)
    d2h_bytes = sum(t.numel() * t.element_size() for t in pinned_out)

    if rank != 0:
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()
        return

    # roofline of the dominant kernel
    peaks = measured_peaks()
    props = torch.cuda.get_device_properties(0)
    means = [statistics.mean(p) for p in per]
    dom = max(range(len(wl.steps)), key=lambda j: means[j])
    st = wl.steps[dom]
    achieved, peak, unit = roofline_of(st, means[dom], peaks, props)
    nodes = roofline_nodes(wl, means, peaks, props)
    traffic = traffic_for(*wl.traffic_key(dom)) if hasattr(wl, "traffic_key") else None
    gpu_launches = args.steps * sum(s.launches for s in wl.steps)
    plan_ms = plan_times(tra, wl)

    # the other workloads of the default run, each with its own timed region (device-resident)
    extras = []
    names = [] if args.extra == "none" else [n for n in args.extra.split(",") if n and n != args.workload]
    wl_name, wl_d, wl_dtype, wl_steps = wl.name, wl.d, wl.dtype, wl.steps
    if world == 1 and names:
        # release the headline workload's device and pinned buffers first (the oracle sample
        # below needs only its host inputs)
        for k, v in list(vars(wl).items()):
            if isinstance(v, torch.Tensor) or (isinstance(v, list) and v and isinstance(v[0], torch.Tensor)):
                delattr(wl, k)
        pinned_in = pinned_out = None
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        for n in names:
            extras.append(extra_workload(torch, tra, n, args, flush, local))

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        import oracle

        rows = args.cpu_rows or wl.cpu_default
        t0 = time.perf_counter()
        work = wl.oracle_sample(host, 0, rows)
        dt = time.perf_counter() - t0
        cpu = {"value": work / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
               "sample": wl.sample_text(rows), "seconds": round(dt, 2)}
        if getattr(wl, "single_core_baseline", False):
            # the same sample on one host core as well
            threads = oracle.num_threads()
            oracle.set_num_threads(1)
            t0 = time.perf_counter()
            wl.oracle_sample(host, 0, rows)
            dt1 = time.perf_counter() - t0
            oracle.set_num_threads(threads)
            cpu["single_core"] = {"value": work / dt1 / 1e12, "seconds": round(dt1, 3)}

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": wl_dtype, "data": "synthetic (Philox-4x32-10, seeded)",
        "config": {"workload": wl_name, "d": wl_d, "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "flushed between steps (512 MiB write outside the step's events)",
                   "per_launch_group_ms": {s.name: round(m, 4) for s, m in zip(wl_steps, means)}},
        "roofline": {"bound": st.bound, "kernel": st.name, "achieved": achieved, "peak": peak, "unit": unit,
                     "frac": achieved / peak, "traffic": traffic, "peak_source": peak_source(st.bound)},
        "roofline_nodes": nodes,
        "alu_peak_at_sampled_clock": (
            {"sm_mhz": clocks["sm_mhz"],
             "peak": props.multi_processor_count * FP32_LANES_PER_SM * 2 * clocks["sm_mhz"] * 1e6 / 1e12,
             "frac": achieved / (props.multi_processor_count * FP32_LANES_PER_SM * 2 * clocks["sm_mhz"] * 1e6 / 1e12)}
            if st.bound == "alu" and clocks and clocks.get("sm_mhz") else None),
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d_bytes,
                "d2h_bytes_per_step": d2h_bytes, "steps": n_e2e, "method": e2e_method,
                "other_method_value": (job_throughput(ops, n_e2e, world, e2e_alt) if e2e_alt else None)},
        "gpu_launches": gpu_launches,
        "plan_ms": plan_ms,
        "clocks": clocks,
        "wall_s": round(wall, 3),
        "extra_workloads": extras,
    }
    if wl_dtype == "bf16" and st.bound == "tensor":
        line["config"]["accumulate"] = "fp32"
    print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


def run_probe_fp32(args):
    """FP32 issue ceilings of the semiring kernels' inner step (ein_probe_fp32): one JSON record
    with tuples per clock per SM, the SM clock the loop ran at (clock64 over the global timer)
    and the absolute rate, for the sum of products (FFMA), max-plus (FADD + FADD + 3-input max)
    and max-plus with the packed add."""
    import torch

    import tensor_relational_algebra_gb300 as tra

    tra.load()
    props = torch.cuda.get_device_properties(0)
    sms = props.multi_processor_count
    ctas = 2 * sms  # the semiring kernels' occupancy
    sink = torch.empty(ctas * 256, dtype=torch.float32, device="cuda")
    cyc = torch.empty(ctas, dtype=torch.int64, device="cuda")
    nns = torch.empty(ctas, dtype=torch.int64, device="cuda")
    peaks = measured_peaks()
    sm_max = float(peaks.get("sm_max_mhz", 2070.0))
    kinds = [(0, "ffma: 2 FFMA per 2 tuples (sum of products)"),
             (1, "max-plus: FADD + FADD + 3-input max.f32 per 2 tuples"),
             (2, "max-plus: add.rn.f32x2 + 3-input max.f32 per 2 tuples")]
    sampler = ClockSampler(0)
    sampler.start()
    w0 = time.time()
    out = []
    for kind, name in kinds:
        for _ in range(2):  # warm-up launch
            tra.ein_probe_fp32(kind, 64, ctas, sink, cyc, nns)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        per_cta = tra.ein_probe_fp32(kind, args.probe_iters, ctas, sink, cyc, nns)
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
        c = cyc.cpu().numpy().astype(np.float64)
        n = nns.cpu().numpy().astype(np.float64)
        cmed = float(np.median(c))
        tpc = 2 * per_cta / cmed  # two CTAs per SM
        mhz = float(np.median(c / n * 1e3))
        rate = per_cta * ctas / (ms * 1e-3)
        out.append({"kind": kind, "loop": name, "tuples_per_clk_per_sm": round(tpc, 2),
                    "loop_cycles_min_median_max": [int(c.min()), int(cmed), int(c.max())],
                    "loop_ms_min_median_max": [round(float(n.min()) * 1e-6, 3), round(float(np.median(n)) * 1e-6, 3),
                                               round(float(n.max()) * 1e-6, 3)],
                    "flop_per_clk_per_sm": round(2 * tpc, 2), "of_issue_peak_256_flop_per_clk": round(2 * tpc / 256, 4),
                    "sm_mhz_in_loop": round(mhz, 1), "event_ms": round(ms, 3), "tuples_per_s": rate,
                    "tflops_2_per_tuple": 2 * rate / 1e12,
                    "of_fp32_peak_at_max_clock": 2 * rate / (sms * FP32_LANES_PER_SM * 2 * sm_max * 1e6)})
    sampler.mark(w0, time.time())
    rec = {"probe": "fp32", "sms": sms, "ctas": ctas, "threads_per_cta": 256, "iters": args.probe_iters,
           "fp32_peak_tflops_at_max_clock": sms * FP32_LANES_PER_SM * 2 * sm_max * 1e6 / 1e12,
           "peak_derivation": f"{sms} SMs x {FP32_LANES_PER_SM} FP32 lanes x 2 flop x {sm_max:.0f} MHz",
           "results": out, "clocks": sampler.stop(), "gpu": props.name}
    print(json.dumps(rec))


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle

    wl = WORKLOADS[args.workload](d=args.d)
    host = wl.host_inputs()
    rows = args.ref_rows or wl.ref_default
    for s in range(args.warmup):
        wl.oracle_sample(host, s * rows, rows)
    t0 = time.perf_counter()
    work = 0
    for s in range(args.steps):
        work += wl.oracle_sample(host, (args.warmup + s) * rows, rows)
    dt = time.perf_counter() - t0
    value = work / dt / 1e12
    cores = oracle.num_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (Philox-4x32-10 N(0,1), seeded)",
        "config": {"workload": wl.name, "d": wl.d},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": "per step: " + wl.sample_text(rows)},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="c5")
    ap.add_argument("--extra", default="pair,c3",
                    help="comma-separated workloads also timed (device-resident) in the same run, or 'none'")
    ap.add_argument("--d", type=lambda v: [int(x) for x in v.split(",")], default=None,
                    help="partition vector for c5 / c5b, e.g. 4,2,2,2")
    ap.add_argument("--cpu-rows", type=int, default=None, help="oracle sample size of the CPU baseline")
    ap.add_argument("--ref-rows", type=int, default=None, help="oracle sample size per reference-arm step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--probe", choices=["fp32"], default=None,
                    help="run a measurement probe instead of a workload (fp32: the semiring inner step's issue ceilings)")
    ap.add_argument("--probe-iters", type=int, default=4000)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.probe == "fp32":
        run_probe_fp32(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
