"""Dedicated ownership on the host: the owner planner against the oracle's plain LPT
(bit-exact), its balance bound, per-owner tables, and the DMuon page's arithmetic."""

import json
import os

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def nsm():
    import newton_schulz_orthogonalized_gb300 as m
    if not os.path.exists(m.LIB_PATH):
        from newton_schulz_orthogonalized_gb300 import _build
        _build.build()
    m.lib()
    return m


def _costs(shapes, method):
    out = []
    for r, c in shapes:
        m, n = min(r, c), max(r, c)
        out.append(oracle.flops_gram(m, n) if method == "gram" else oracle.flops_standard(m, n))
    return out


@pytest.mark.parametrize("name", ["layer1024", "gpt2small", "llama7b", "split_moe"])
@pytest.mark.parametrize("method", ["standard", "gram"])
@pytest.mark.parametrize("world", [1, 2, 3, 8])
def test_owners_match_plain_lpt(nsm, name, method, world):
    shapes = synth.workload(name).muon_shapes
    owner, load = nsm.assign_owners(shapes, world, method)
    ref_owner, ref_load = oracle.lpt_assign(_costs(shapes, method), world)
    assert list(owner) == ref_owner
    assert list(load) == ref_load


@pytest.mark.parametrize("world", [2, 4, 8, 16])
def test_owner_balance_bound(nsm, world):
    shapes = synth.workload("split_moe").muon_shapes
    owner, load = nsm.assign_owners(shapes, world, "gram")
    costs = _costs(shapes, "gram")
    assert sum(load) == sum(costs)
    # LPT: no owner exceeds the average by more than the largest single matrix
    assert max(load) <= sum(costs) / world + max(costs)
    assert set(int(o) for o in owner) == set(range(world))


def test_owner_tables_partition_the_table(nsm):
    shapes = synth.workload("llama7b").muon_shapes
    owner, _ = nsm.assign_owners(shapes, 4, "standard")
    seen = []
    for rank in range(4):
        idx, sub, offs, total = nsm.owner_table(shapes, owner, rank)
        assert [shapes[i] for i in idx] == sub
        ro, rt = oracle.pack_offsets(sub, 64)
        assert list(offs) == ro and total == rt
        seen += idx
    assert sorted(seen) == list(range(len(shapes)))


def test_owner_errors(nsm):
    with pytest.raises(nsm.NsmError):
        nsm.assign_owners([(4, 4)], 0)
    with pytest.raises(nsm.NsmError):
        nsm.assign_owners([(4, 0)], 2)


def test_dmuon_page_arithmetic(nsm):
    g = json.load(open(os.path.join(GOLDEN, "pages_constants.json"), encoding="utf-8"))
    d = g["dmuon_z2_example"]
    per_rank = nsm.dmuon_packed_memory_elements("dmuon_z2", d["shards"], d["params_muon"])
    assert per_rank * d["bytes_per_elem"] / 1e6 == d["per_rank_mb"]
    n, pm = 8, 1000.0
    # DMuon drops the gradient all-gather of the naive scheme in both modes, and Z2 also
    # drops the backward re-broadcast (communication-optimal 2(N-1)/N P_M)
    assert nsm.dmuon_comm_elements("naive_z2", n, pm) - nsm.dmuon_comm_elements("dmuon_z2", n, pm) == pytest.approx((n - 1) / n * pm)
    assert nsm.dmuon_comm_elements("naive_z3", n, pm) - nsm.dmuon_comm_elements("dmuon_z3", n, pm) == pytest.approx((n - 1) / n * pm)
    assert nsm.dmuon_comm_elements("dmuon_z3", n, pm) - nsm.dmuon_comm_elements("dmuon_z2", n, pm) == pytest.approx((n - 1) / n * pm)
    assert nsm.dmuon_comm_elements("dmuon_z2", n, pm) == pytest.approx(2 * 7 / 8 * pm)
    assert nsm.dmuon_packed_memory_elements("dmuon_z3", n, pm, max_layer_p_m=37.0) == 37.0
