"""Host-side arithmetic of bench.py, checked without a GPU.

The canonical Newton-Schulz flop count behind the reported NS TFLOP/s and the CPU
baseline's extrapolation is counted in bench.py independently of the oracle; here it
must equal the oracle's counts (which the oracle tests pin).  The oracle sample behind
cpu_baseline must stay inside its flop budget.
"""

import bench
import oracle
import synth

SHAPES = [(128, 256), (4096, 11008), (11008, 4096), (768, 768), (1408, 2048), (1024, 4096)]


def test_canonical_flops_match_oracle():
    for method, count in (("gram", oracle.flops_gram), ("standard", oracle.flops_standard)):
        want = sum(count(min(r, c), max(r, c), 5) for r, c in SHAPES)
        assert bench._canonical_ns_flops(SHAPES, method) == want, method


def test_oracle_sample_keeps_to_its_flop_budget():
    wl = synth.workload("tiny")  # four 128 x 256 matrices: one shape, one sampled matrix
    ms, desc = bench.cpu_oracle_sample(wl, "gram", budget_s=5.0, max_flops=1e9)
    assert ms > 0
    assert "on 1 matrices (128x256)" in desc
    # a budget below the smallest matrix still samples that one matrix
    ms, desc = bench.cpu_oracle_sample(wl, "gram", budget_s=5.0, max_flops=1.0)
    assert ms > 0 and "on 1 matrices" in desc
