"""The small-matrix kernel: whole Newton-Schulz chains of matrices with m <= 128 in one launch.

Matrices whose short side is at most 128 (Muon-Split head blocks, small projections) run
their entire chain in one CTA, with every m x m iterate in shared memory.  These tests hold
that kernel to the oracle in the method's storage precision, at more matrices than the
GPU has SMs (each CTA runs several chains), at every step count the interface allows,
and to the grouped path, which computes the same products in other launches.
"""

import numpy as np
import pytest
import torch

import oracle
import synth

from test_gpu_parity import TOL_NS, Step, compare, orthogonalize_gpu, rel

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nsm():
    import newton_schulz_orthogonalized_gb300 as m
    m.lib()
    return m


SMALL_MIX = [(64, 192), (192, 64), (128, 128), (100, 300), (128, 4096), (17, 40), (128, 129)]


@pytest.mark.parametrize("method", ["gram", "standard", "standard_bf16"])
def test_more_matrices_than_sms(nsm, method):
    # 350 chains on at most one CTA per SM: every CTA runs several matrices in a row
    # (bf16 storage on near-low-rank inputs is chaotic at the percent level, so that form
    # runs on well-conditioned inputs, where any correct implementation lands within 1e-2)
    shapes = [SMALL_MIX[i % len(SMALL_MIX)] for i in range(350)]
    wl = synth.custom(shapes, seed=41, lowrank=method != "standard_bf16")
    s = Step(nsm, wl, method)
    s.check(indices=list(range(0, 350, 7)) + list(range(343, 350)))


@pytest.mark.parametrize("method", ["gram", "standard"])
@pytest.mark.parametrize("steps", [1, 2, 3, 4, 6, 16])
def test_step_counts(nsm, method, steps):
    wl = synth.custom([(128, 256), (96, 500), (33, 65), (500, 96)], seed=43, lowrank=False)
    s = Step(nsm, wl, method, steps=steps)
    s.check()


@pytest.mark.parametrize("method", ["gram", "standard"])
def test_mixed_small_and_grouped(nsm, method):
    # one table with matrices for both the small kernel and the grouped launches; both
    # apply the step in their last product
    wl = synth.custom([(128, 512), (512, 128), (64, 300), (256, 384), (100, 100), (129, 700),
                       (4096, 128)], seed=47)
    s = Step(nsm, wl, method)
    s.check()


def test_small_table_is_one_chain_launch(nsm):
    # momentum, norm, normalise, the whole chain in one launch, then the apply pass
    wl = synth.workload("tiny")
    nsm.timing_reset()
    nsm.timing_enable(True)
    try:
        Step(nsm, wl, "gram")
        torch.cuda.synchronize()
        launches = nsm.last_launch_count()
        _, n_small, flops = nsm.timing_read(nsm.KIND_SMALL)
        _, n_gemm, _ = nsm.timing_read(nsm.KIND_GEMM)
    finally:
        nsm.timing_enable(False)
    assert launches == 5
    assert n_small == 1 and n_gemm == 0
    # bytes: the re-anchored gram chain (re-anchored after step 3) reads X in R0 = X X^T,
    # in the re-anchoring pass and in the final pass, and writes it in those two passes
    # (2 bytes each)
    assert flops == pytest.approx(4 * 128 * 256 * 2 * (3 + 2))


@pytest.mark.parametrize("method", ["gram", "standard"])
def test_orthogonalize_small_vs_exact(nsm, method):
    # well-conditioned inputs: the fp16 iteration stays close to the exact one
    wl = synth.custom([(128, 1024), (64, 64), (1000, 96)], seed=53, lowrank=False)
    offsets, inp, out = orthogonalize_gpu(nsm, wl, method)
    for i, (r, c) in enumerate(wl.muon_shapes):
        o = int(offsets[i])
        x = inp[o:o + r * c].reshape(r, c)
        got = out[o:o + r * c].reshape(r, c)
        want = oracle.orthogonalize(x, method)
        compare(got, want, TOL_NS, f"small/vs_exact/{method}/{(r, c)}")


def _orthogonalize_both_forms(nsm):
    wl = synth.custom([(128, 1024), (96, 333), (128, 128), (700, 64)], seed=59, lowrank=False)
    offsets, total = nsm.pack(wl.muon_shapes)
    res = {}
    for method in ("gram", "standard"):
        inp = torch.zeros(total, dtype=torch.bfloat16, device="cuda")
        synth.fill_packed_grads(wl, offsets, inp)
        out = torch.zeros_like(inp)
        ws = torch.empty(nsm.workspace_bytes(wl.muon_shapes, method), dtype=torch.uint8, device="cuda")
        nsm.muon_orthogonalize(inp, out, offsets, wl.muon_shapes, method, 5, ws)
        assert nsm.device_status() == nsm.NSM_OK
        res[method] = out.cpu()
    return res


def test_small_kernel_agrees_with_grouped_path(nsm):
    # The option that turns the small-matrix kernel off sends the same matrices through
    # the grouped launches: the same products and storage points, summed in another order
    assert nsm.get_option(nsm.OPT_SMALL_KERNEL) == 1
    a = _orthogonalize_both_forms(nsm)
    nsm.set_option(nsm.OPT_SMALL_KERNEL, 0)
    try:
        b = _orthogonalize_both_forms(nsm)
    finally:
        nsm.set_option(nsm.OPT_SMALL_KERNEL, 1)
    for method in a:
        x, y = a[method].double().numpy(), b[method].double().numpy()
        assert rel(x, y) <= 5e-3, (method, rel(x, y))
