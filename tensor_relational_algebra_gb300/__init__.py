"""GB300-native tensor-relational-algebra (TRA) execution of one extended EinSum.

Python binding of ``libtra.so`` (C ABI in ``include/tra.h``): argument
marshalling only.  Every step of the path -- join, aggregation, repartition --
runs in the library's CUDA kernels; PyTorch supplies device memory and streams.
There is no CPU fallback: if the library cannot be loaded, every call raises.

Source of the operations: "EinDecomp: automatic tensor-parallel decomposition
via Einstein summation + tensor relational algebra" (sections 2.1, 2.2, 3.1, 3.2).
"""
from __future__ import annotations

import ctypes
import os

from ._build import LIB as _LIB_DEFAULT, LIB_CHECK as _LIB_CHECK, build as _build_lib

# TRA_CHECK=1 in the environment selects the check build (bounds tests in the kernels)
CHECK_BUILD = os.environ.get("TRA_CHECK", "") not in ("", "0")
_LIB_PATH = _LIB_CHECK if CHECK_BUILD else _LIB_DEFAULT

__all__ = [
    "TraError", "build_library", "load", "Plan", "ein_plan", "ein_plan_info", "ein_plan_keys", "ein_execute",
    "ein_repartition", "ein_repartition_cost", "ein_status", "ein_selftest_wait_timeout", "ein_plan_destroy",
    "ein_last_error", "ein_graph_decompose", "ein_attention", "attention", "ein_repartition_messages",
    "repartition", "repartition_cost", "repartition_messages", "decompose", "KERNELS", "ROLES",
]

TRA_MAX_RANK = 8
TRA_MAX_LABELS = 12
ERRORS = {
    -1: "TRA_ERR_PARSE", -2: "TRA_ERR_DIVISIBILITY", -3: "TRA_ERR_SHARED_LABEL_D", -4: "TRA_ERR_RANK",
    -5: "TRA_ERR_UNSUPPORTED", -6: "TRA_ERR_WORKSPACE", -7: "TRA_ERR_CUDA", -8: "TRA_ERR_TIMEOUT", -9: "TRA_ERR_ARG",
    -10: "TRA_ERR_BOUNDS",
}
KERNELS = {1: "semiring_f32", 2: "tc_bf16", 3: "row_reduce", 4: "elementwise", 5: "lse_factored", 6: "literal",
           7: "tc_bf16_pair", 8: "tc_split3", 9: "empty", 10: "fill"}
ROLES = {0: "batch", 1: "M", 2: "N", 3: "contracted"}


class TraError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{ERRORS.get(code, code)}: {msg}")
        self.code = code


class tra_plan_info(ctypes.Structure):
    _fields_ = [
        ("n_labels", ctypes.c_int32),
        ("labels", ctypes.c_char * TRA_MAX_LABELS),
        ("bound", ctypes.c_int64 * TRA_MAX_LABELS),
        ("part", ctypes.c_int32 * TRA_MAX_LABELS),
        ("sub_extent", ctypes.c_int64 * TRA_MAX_LABELS),
        ("role", ctypes.c_int32 * TRA_MAX_LABELS),
        ("rank_x", ctypes.c_int32), ("rank_y", ctypes.c_int32), ("rank_z", ctypes.c_int32),
        ("key_grid_x", ctypes.c_int32 * TRA_MAX_RANK),
        ("key_grid_y", ctypes.c_int32 * TRA_MAX_RANK),
        ("key_grid_z", ctypes.c_int32 * TRA_MAX_RANK),
        ("n_tasks", ctypes.c_uint64), ("n_groups", ctypes.c_uint64), ("n_agg", ctypes.c_uint64),
        ("x_sub", ctypes.c_uint64), ("y_sub", ctypes.c_uint64), ("z_sub", ctypes.c_uint64),
        ("cost_join", ctypes.c_uint64), ("cost_agg", ctypes.c_uint64),
        ("workspace_bytes", ctypes.c_uint64),
        ("in_dtype", ctypes.c_int32), ("out_dtype", ctypes.c_int32),
        ("kernel", ctypes.c_int32),
        ("msg_join", ctypes.c_uint64), ("msg_agg", ctypes.c_uint64), ("mem_elems", ctypes.c_uint64),
    ]


class tra_graph_node(ctypes.Structure):
    _fields_ = [("spec", ctypes.c_char_p), ("bounds", ctypes.POINTER(ctypes.c_int64)), ("n_bounds", ctypes.c_int32),
                ("input", ctypes.c_int32 * 2)]


class tra_graph_result(ctypes.Structure):
    _fields_ = [("total_cost", ctypes.c_uint64), ("dp_cost", ctypes.c_uint64), ("n_candidates", ctypes.c_uint64)]


class tra_cost_model(ctypes.Structure):
    _fields_ = [("latency", ctypes.c_uint64), ("min_block", ctypes.c_int64), ("mem_limit", ctypes.c_uint64),
                ("mem_weight", ctypes.c_uint64), ("task_multiple", ctypes.c_int64)]


TRA_DP_POW2 = 1

_lib = None


def build_library(force: bool = False, both: bool = False) -> str:
    """Compile libtra.so in-tree for sm_103a (no-op when up to date); under TRA_CHECK=1 the check
    build libtra_check.so instead; both=True builds the two."""
    return _build_lib(force=force, check=CHECK_BUILD, both=both)


def load():
    """Load libtra.so (building it first if needed) and declare the C signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        _build_lib(check=CHECK_BUILD)
    lib = ctypes.CDLL(_LIB_PATH)
    vp, i32, i64, u64p = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.POINTER(ctypes.c_uint64)
    lib.ein_plan.argtypes = [ctypes.c_char_p, vp, i32, vp, i32, ctypes.POINTER(vp)]
    lib.ein_plan_info.argtypes = [vp, ctypes.POINTER(tra_plan_info)]
    lib.ein_plan_keys.argtypes = [vp, vp, i64]
    lib.ein_execute.argtypes = [vp, vp, vp, vp, vp, ctypes.c_size_t, vp]
    lib.ein_repartition.argtypes = [i32, vp, vp, vp, i32, vp, vp, vp]
    lib.ein_repartition_cost.argtypes = [i32, vp, vp, vp, u64p]
    lib.ein_repartition_messages.argtypes = [i32, vp, vp, vp, u64p]
    lib.ein_status.argtypes = [vp]
    lib.ein_selftest_wait_timeout.argtypes = [ctypes.c_uint64, vp]
    lib.ein_selftest_wait_timeout.restype = ctypes.c_int
    lib.ein_plan_destroy.argtypes = [vp]
    lib.ein_plan_destroy.restype = None
    lib.ein_last_error.restype = ctypes.c_char_p
    lib.ein_graph_decompose.argtypes = [ctypes.POINTER(tra_graph_node), i32, i64, i64, i32,
                                        ctypes.POINTER(tra_cost_model), vp, i32, u64p,
                                        ctypes.POINTER(tra_graph_result)]
    lib.ein_attention.argtypes = [i32, i32, i32, i32, ctypes.c_float, vp, vp, vp, vp, vp, vp]
    lib.ein_build_flags.argtypes = []
    lib.ein_build_flags.restype = ctypes.c_int
    lib.ein_probe_fp32.argtypes = [i32, i32, i32, vp, vp, vp, u64p, vp]
    lib.ein_probe_fp32.restype = ctypes.c_int
    for f in ("ein_plan", "ein_plan_info", "ein_plan_keys", "ein_execute", "ein_repartition",
              "ein_repartition_cost", "ein_repartition_messages", "ein_status", "ein_graph_decompose",
              "ein_attention"):
        getattr(lib, f).restype = ctypes.c_int
    _lib = lib
    return lib


def _check(rc: int):
    if rc != 0:
        raise TraError(rc, load().ein_last_error().decode())


def _i64(vals):
    return (ctypes.c_int64 * max(1, len(vals)))(*vals)


def _i32(vals):
    return (ctypes.c_int32 * max(1, len(vals)))(*vals)


def _ptr(t):
    """Device (or host) address of a torch tensor / int / None."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ----------------------------------------------------------------- raw C names
def ein_plan(spec: str, bounds, d) -> int:
    h = ctypes.c_void_p()
    _check(load().ein_plan(spec.encode(), _i64(bounds), len(bounds), _i32(d), len(d), ctypes.byref(h)))
    return h.value


def ein_plan_info(plan: int) -> tra_plan_info:
    info = tra_plan_info()
    _check(load().ein_plan_info(plan, ctypes.byref(info)))
    return info


def ein_plan_keys(plan: int, n_tasks: int, width: int):
    buf = (ctypes.c_int32 * max(1, n_tasks * width))()
    _check(load().ein_plan_keys(plan, buf, n_tasks * width))
    return [tuple(buf[i * width:(i + 1) * width]) for i in range(n_tasks)]


def ein_execute(plan: int, in0, in1, out, workspace=None, workspace_bytes: int = 0, stream=None):
    _check(load().ein_execute(plan, _ptr(in0), _ptr(in1), _ptr(out), _ptr(workspace), workspace_bytes,
                              _stream(stream)))


def ein_repartition(shape, src_d, dst_d, elem_bytes: int, src, dst, stream=None):
    _check(load().ein_repartition(len(shape), _i64(shape), _i32(src_d), _i32(dst_d), elem_bytes, _ptr(src),
                                  _ptr(dst), _stream(stream)))


def ein_repartition_cost(shape, src_d, dst_d) -> int:
    c = ctypes.c_uint64()
    _check(load().ein_repartition_cost(len(shape), _i64(shape), _i32(src_d), _i32(dst_d), ctypes.byref(c)))
    return c.value


def ein_repartition_messages(shape, src_d, dst_d) -> int:
    c = ctypes.c_uint64()
    _check(load().ein_repartition_messages(len(shape), _i64(shape), _i32(src_d), _i32(dst_d), ctypes.byref(c)))
    return c.value


def _cost_model(model):
    if model is None:
        return None
    unknown = set(model) - {f for f, _ in tra_cost_model._fields_}
    if unknown:
        raise ValueError(f"unknown cost-model fields {sorted(unknown)}")
    return tra_cost_model(**model)


def ein_graph_decompose(nodes, p_min: int, p_max: int, flags: int = 0, model=None):
    """nodes: sequence of (spec, bounds, (input_x, input_y)) with -1 for a graph input.
    model: None or a dict of tra_cost_model fields (latency, min_block, mem_limit,
    mem_weight, task_multiple).  Returns (d per node, cost per node, total_cost, dp_cost,
    n_candidates)."""
    keep, arr = [], (tra_graph_node * len(nodes))()
    ranks = []
    for i, (spec, bounds, inputs) in enumerate(nodes):
        b = _i64(bounds)
        e = spec.encode()
        keep += [b, e]
        arr[i].spec, arr[i].bounds, arr[i].n_bounds = e, ctypes.cast(b, ctypes.POINTER(ctypes.c_int64)), len(bounds)
        arr[i].input[0], arr[i].input[1] = (list(inputs) + [-1, -1])[:2]
        lhs = spec.split("->")[0]
        ranks.append([len(x) for x in lhs.split(",")])
    n_d = sum(sum(r) for r in ranks)
    d = (ctypes.c_int32 * max(1, n_d))()
    costs = (ctypes.c_uint64 * len(nodes))()
    res = tra_graph_result()
    cm = _cost_model(model)
    _check(load().ein_graph_decompose(arr, len(nodes), p_min, p_max, flags, ctypes.byref(cm) if cm else None, d, n_d,
                                      costs, ctypes.byref(res)))
    out, pos = [], 0
    for r in ranks:
        out.append(list(d[pos:pos + sum(r)]))
        pos += sum(r)
    return out, list(costs), res.total_cost, res.dp_cost, res.n_candidates


def ein_attention(s: int, t: int, h: int, d: int, scale: float, q, k, v, o, lse=None, stream=None):
    _check(load().ein_attention(s, t, h, d, scale, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _stream(stream)))


def attention(q, k, v, o, s: int, t: int, h: int, d: int = 128, scale: float = None, lse=None, stream=None):
    """Fused Scores -> logsumexp -> exp -> A.V on device tensors (see ein_attention)."""
    ein_attention(s, t, h, d, (1.0 / d ** 0.5) if scale is None else scale, q, k, v, o, lse, stream)


def ein_probe_fp32(kind: int, iters: int, ctas: int, sink, cycles, nanos, stream=None) -> int:
    """Launch the FP32 issue-ceiling probe (see include/tra.h); returns tuples per CTA."""
    n = ctypes.c_uint64()
    _check(load().ein_probe_fp32(kind, iters, ctas, _ptr(sink), _ptr(cycles), _ptr(nanos), ctypes.byref(n),
                                 _stream(stream)))
    return n.value


def ein_status(stream=None):
    _check(load().ein_status(_stream(stream)))


def ein_selftest_wait_timeout(timeout_ns: int, stream=None):
    _check(load().ein_selftest_wait_timeout(timeout_ns, _stream(stream)))


def ein_plan_destroy(plan: int):
    load().ein_plan_destroy(plan)


def ein_last_error() -> str:
    return load().ein_last_error().decode()


# ----------------------------------------------------------------- convenience layer
class Plan:
    """A TRA plan of one EinSum under a partition vector (host object).

    ``bounds``: {label: extent} or a list in first-appearance order.
    ``d``: partition counts per operand index position, X's then Y's."""

    def __init__(self, spec: str, bounds, d):
        eq = spec.split(":")[0]
        lhs = eq.split("->")[0]
        order = []
        for c in lhs.replace(",", ""):
            if c not in order:
                order.append(c)
        if isinstance(bounds, dict):
            bounds = [bounds[c] for c in order]
        self.handle = None
        self.handle = ein_plan(spec, list(bounds), list(d))  # the library validates the spec
        self.info = ein_plan_info(self.handle)
        self.spec = spec
        self.labels = order
        self.operands = lhs.split(",")
        self.output = eq.split("->")[1]
        self.bounds = list(bounds)
        self.d = list(d)

    def __del__(self):
        h = getattr(self, "handle", None)
        if h and _lib is not None:
            _lib.ein_plan_destroy(h)
            self.handle = None

    # plan facts (bit-exact integers)
    @property
    def n_tasks(self):
        return self.info.n_tasks

    @property
    def n_groups(self):
        return self.info.n_groups

    @property
    def n_agg(self):
        return self.info.n_agg

    @property
    def cost_join(self):
        return self.info.cost_join

    @property
    def cost_agg(self):
        return self.info.cost_agg

    @property
    def msg_join(self):
        return self.info.msg_join

    @property
    def msg_agg(self):
        return self.info.msg_agg

    @property
    def mem_elems(self):
        return self.info.mem_elems

    @property
    def workspace_bytes(self):
        return self.info.workspace_bytes

    @property
    def kernel(self):
        return KERNELS.get(self.info.kernel, self.info.kernel)

    def part(self, label):
        return self.info.part[self.labels.index(label)]

    def shape(self, which: str):
        labs = {"x": self.operands[0], "y": self.operands[1] if len(self.operands) > 1 else "",
                "z": self.output}[which]
        return [self.bounds[self.labels.index(c)] for c in labs]

    def dvec(self, which: str):
        labs = {"x": self.operands[0], "y": self.operands[1] if len(self.operands) > 1 else "",
                "z": self.output}[which]
        return [self.info.part[self.labels.index(c)] for c in labs]

    def keys(self):
        w = self.info.rank_x + self.info.rank_y + self.info.rank_z
        rows = ein_plan_keys(self.handle, self.info.n_tasks, w)
        rx, ry = self.info.rank_x, self.info.rank_y
        return [(r[:rx], r[rx:rx + ry], r[rx + ry:]) for r in rows]

    def execute(self, x, y, z, workspace=None, stream=None):
        """Run the plan on device tensors in the relation layout of d.  When the plan needs
        scratch and none is given, a torch buffer is allocated once and kept with the plan, so
        calls of one plan that may overlap on the GPU (other streams) must each pass their own
        workspace."""
        if workspace is None and self.info.workspace_bytes:
            import torch

            # device scratch, on the inputs' device (z may be pinned host memory)
            dev = x.device if x is not None and x.is_cuda else (z.device if z.is_cuda else
                                                                 torch.device("cuda", torch.cuda.current_device()))
            ws = getattr(self, "_workspace", None)
            if ws is None or ws.device != dev:
                ws = torch.empty(self.info.workspace_bytes, dtype=torch.uint8, device=dev)
                self._workspace = ws
            workspace = ws
        ws_bytes = 0
        if workspace is not None:
            ws_bytes = workspace.numel() * workspace.element_size()
        ein_execute(self.handle, x, y, z, workspace, ws_bytes, stream)


def repartition(src, dst, shape, src_d, dst_d, stream=None):
    """Device permute-copy of a relation from src_d to dst_d (torch tensors)."""
    ein_repartition(shape, src_d, dst_d, src.element_size(), src, dst, stream)


def repartition_cost(shape, src_d, dst_d) -> int:
    return ein_repartition_cost(shape, src_d, dst_d)


def repartition_messages(shape, src_d, dst_d) -> int:
    return ein_repartition_messages(shape, src_d, dst_d)


def decompose(nodes, P: int, p_max: int = None, pow2: bool = False, model=None):
    """EinDecomp over an EinGraph (host only): a partition vector for every node with
    P..p_max join tuples (p_max defaults to P), minimising join + aggregation +
    repartition cost (plus the terms of the cost-model variants in model, a dict of
    tra_cost_model fields).  nodes: (spec, bounds, (input_x, input_y)) in topological
    order, -1 marking a graph input.  Returns a dict with "d", "node_cost",
    "total_cost", "dp_cost", "n_candidates"."""
    d, costs, total, dp, n = ein_graph_decompose(nodes, P, P if p_max is None else p_max,
                                                 TRA_DP_POW2 if pow2 else 0, model)
    return {"d": d, "node_cost": costs, "total_cost": total, "dp_cost": dp, "n_candidates": n}
