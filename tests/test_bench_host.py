"""Host-side pieces of bench.py, on the CPU.

- The algorithmic bytes of the measured workloads are the figures the metric is defined on.
- The committed ncu summary of the bench's dominant kernel was taken on the current device code and
  the launch shape AUTO picks for the bench's workload, so the bench reports its DRAM traffic instead
  of null.  A change to that kernel's device code or launch shape fails here until its counters are
  taken again.
"""
import bench
import tensor_allreduce_residual_gb300 as ar
import workloads
from tensor_allreduce_residual_gb300 import _build


def test_algorithmic_bytes_of_the_workloads():
    # TP prefill: 8 partials + residual + 2 outputs of 8192 x 8192 bf16, bias and weight of 8192
    assert bench.algorithmic_bytes(8, 8192, 8192, 2) == 1_476_427_776
    assert workloads.fused_algorithmic_bytes(8, 8192, 8192, "bf16", True) == 1_476_427_776
    # R=8 decode without bias, one token; TP decode R=2 fp16 with bias, one token
    assert workloads.fused_algorithmic_bytes(8, 1, 8192, "bf16", False) == 196_608
    assert workloads.fused_algorithmic_bytes(2, 1, 4096, "fp16", True) == 57_344
    # reduce-only R=4 fp16 at 2^27 elements
    assert workloads.sum_algorithmic_bytes(4, 1 << 27, "fp16") == 1_342_177_280


def test_committed_counters_match_the_bench_kernel():
    _build.build()
    plan = ar.ar_query_launch(bench.R, bench.HIDDEN, bench.TOKENS, ar.AR_BF16, "AUTO")
    traffic = bench.profiled_traffic(plan["kernel_name"], bench.plan_key(plan))
    assert traffic is not None, ("no committed ncu summary matches the current device code "
                                 f"({bench.kernel_sources_hash()}) and launch plan ({bench.plan_key(plan)})")
    # DRAM traffic within a few percent of the algorithmic bytes (no re-reads)
    assert 0.95 < traffic / bench.algorithmic_bytes(bench.R, bench.TOKENS, bench.HIDDEN, 2) < 1.05
