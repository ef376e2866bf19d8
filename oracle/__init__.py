"""CPU oracle for the tensor-relational-algebra (TRA) hot path.

TEST INFRASTRUCTURE -- NOT PART OF THE PRODUCT.  Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference arm may
import it.  It shares no code with the CUDA path (the package
``tensor_relational_algebra_gb300``) and never imports it.

Source: "EinDecomp: automatic tensor-parallel decomposition via Einstein
summation + tensor relational algebra".

* ``einsum`` / ``einsum_points`` -- the extended EinSum of section 2.1, the
  definition written out as nested loops in double (``einsum_ref.c``).
* ``tra`` -- the tensor relation of section 2.2 (key -> sub-tensor, key -> index
  range), the join / aggregation / repartition operators, the brute-force
  plan enumeration and the communication-cost terms of section 3.1, and a
  literal TRA execution (relation dictionaries, join, GROUP BY aggregate).
* ``mha`` -- the multi-head-attention EinGraph of section 2.1, node by node.
* ``decomp`` -- the partition-vector choice of sections 3.1-3.2 by exhaustive search
  over every combination of every node's candidates (tiny graphs), with the cost-model
  variants of section 4.3 counted from their definitions (messages element by element).
* ``rounding`` -- fp32 / bf16 round-to-nearest-even.

Parity pins: every function above is checked in ``tests/test_oracle_pins.py``
against closed forms, library routines on special cases, brute force and the
pages' own formulas.  The repartition-cost term (section 3.1 gives no formula) is
pinned where the pages fix it -- between the centralized layout (d all ones) and N
blocks, the Scatter / Gather traffic (N-1)/N * M of the communication-primitive
table on rkmt.cn/news/51250.html -- and by invariants elsewhere: between two
partitioned layouts it is "parity unpinned".
"""
from .einsum import OPS, AGGS, einsum, einsum_points, num_threads, set_num_threads, build  # noqa: F401
from . import tra, rounding, mha  # noqa: F401
