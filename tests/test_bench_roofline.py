"""bench.py's choice of roofline for tensor-core nodes (no GPU needed).

A node whose compulsory bytes take longer at the measured copy peak than its flops at the
measured BF16 peak (arithmetic intensity below the ridge point) is reported against HBM, with
its tensor fraction kept beside it; a node above the ridge stays tensor-bound."""
import types

import bench


def _props():
    return types.SimpleNamespace(multi_processor_count=152)


def test_gemm_above_the_ridge_stays_tensor_bound():
    n = 4096
    st = bench.Step("gemm", None, 2 * n ** 3, "flop", "tensor", 1, 3 * n * n * 2)
    assert st.bound == "tensor" and st.unit == "flop" and st.tensor_work is None
    assert st.work == 2 * n ** 3


def test_scores_node_below_the_ridge_is_hbm_bound():
    s, h, d = 4096, 32, 128
    flops = 2 * h * s * s * d
    nbytes = 2 * s * h * d * 2 + h * s * s * 4  # Q and K read, fp32 scores written
    st = bench.Step("scores", None, flops, "flop", "tensor", 1, nbytes)
    assert st.bound == "hbm" and st.unit == "bytes" and st.work == nbytes and st.tensor_work == flops
    peaks = bench.measured_peaks()
    ms = 0.369
    node = bench.roofline_nodes(types.SimpleNamespace(steps=[st]), [ms], peaks, _props())[0]
    assert node["bound"] == "hbm" and node["unit"] == "GB/s"
    assert abs(node["achieved"] - nbytes / (ms * 1e-3) / 1e9) < 0.1
    assert abs(node["tensor_frac"] - flops / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"]) < 1e-3
    assert abs(node["flop_per_byte"] - flops / nbytes) < 0.1


def test_ridge_point_decides():
    peaks = bench.measured_peaks()
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)  # flop per byte
    work = 10 ** 12
    below = bench.Step("b", None, work, "flop", "tensor", 1, int(work / (0.9 * ridge)))
    above = bench.Step("a", None, work, "flop", "tensor", 1, int(work / (1.1 * ridge)))
    assert below.bound == "hbm" and above.bound == "tensor"
    # the other kinds of node are left as declared
    assert bench.Step("r", None, 100, "bytes", "hbm", 1).bound == "hbm"
    assert bench.Step("s", None, 100, "flop", "alu", 1, 10 ** 9).bound == "alu"
