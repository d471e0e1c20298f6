"""Host-side arithmetic of bench.py, checked without a GPU.

The Newton-Schulz flop counts behind the reported TFLOP/s are counted in bench.py
independently of the oracle; here they must equal the oracle's counts (which the oracle
tests pin): the canonical count is the gram form without re-anchoring, the dense count
the chain as the library runs it.  The oracle sample behind cpu_baseline covers the
distinct shapes of the table and scales each by its count.
"""

import bench
import oracle
import synth

SHAPES = [(128, 256), (4096, 11008), (11008, 4096), (768, 768), (1408, 2048), (1024, 4096)]


def test_canonical_flops_match_oracle():
    for m, n in [(min(r, c), max(r, c)) for r, c in SHAPES]:
        assert oracle.flops_gram(m, n, 5, restart_every=0) == 4 * m * m * n + 34 * m ** 3
    want = sum(oracle.flops_gram(min(r, c), max(r, c), 5, restart_every=0) for r, c in SHAPES)
    assert bench._canonical_ns_flops(SHAPES, "gram") == want
    want = sum(oracle.flops_standard(min(r, c), max(r, c), 5) for r, c in SHAPES)
    assert bench._canonical_ns_flops(SHAPES, "standard") == want
    assert bench._dense_ns_flops(SHAPES, "standard") == want


def test_dense_flops_match_oracle():
    want = sum(oracle.flops_gram(min(r, c), max(r, c), 5) for r, c in SHAPES)
    assert bench._dense_ns_flops(SHAPES, "gram") == want


def test_oracle_sample_covers_shapes_and_scales_by_count():
    wl = synth.custom([(16, 32), (16, 32), (16, 32), (24, 8)], seed=1)
    shapes = bench._shape_counts(wl)
    assert [(sh, cnt) for sh, _, cnt in shapes] == [((24, 8), 1), ((16, 32), 3)]
    ms, desc = bench.cpu_oracle_sample(wl, "gram", budget_s=30.0)
    assert ms > 0
    assert "2 of the 2 distinct shapes" in desc
    # a budget below the smallest matrix still times that one shape, and scales it to
    # the whole table by the matrix count
    ms1, desc1 = bench.cpu_oracle_sample(wl, "gram", budget_s=0.0)
    assert ms1 > 0 and "1 of the 2 distinct shapes" in desc1


def test_owner_split_covers_the_table_once():
    # bench.py --split owners: every matrix of the table on exactly one rank (the library's
    # LPT owner plan), the AdamW group on rank 0 only, the hyperparameters kept
    import newton_schulz_orthogonalized_gb300 as nsm
    nsm.lib()
    full = synth.workload("gpt2small")
    for world in (1, 2, 3, 8):
        parts = [bench.owner_workload(nsm, "gpt2small", r, world, "gram") for r in range(world)]
        names = sorted(n for p in parts for n in p.muon_names)
        assert names == sorted(full.muon_names)
        for p in parts:
            assert [full.muon_shapes[full.muon_names.index(n)] for n in p.muon_names] == p.muon_shapes
            assert (p.lr, p.wd, p.mu) == (full.lr, full.wd, full.mu)
        assert parts[0].adam_elements == full.adam_elements
        assert all(p.adam_elements == 0 for p in parts[1:])
        owner, load = nsm.assign_owners(full.muon_shapes, world, "gram")
        assert [len(p.muon_shapes) for p in parts] == [int((owner == r).sum()) for r in range(world)]
