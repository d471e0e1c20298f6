"""Parity at the full workload sizes, in the launch configuration the benchmark times.

One muon_step runs over the whole packed group (224 matrices / 5.67B elements for the
Llama-7B-shaped set, 3584 matrices / 9.13B elements for the Split/MoE set).  A sample of
matrices (one of each working shape) is then checked against the oracle in the method's
storage precision.  On every matrix the properties that hold at any size are checked:
the update is finite, and ||O||_F <= 1.2 sqrt(m), because every singular value of the
five-step output lies in [0, 1.2].
"""

import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module")
def nsm():
    import newton_schulz_orthogonalized_gb300 as m
    m.lib()
    return m


def rel(a, b):
    return np.linalg.norm(a - b) / np.linalg.norm(b)


def _run_fullsize(nsm, name, method, sample_shapes, last_too=()):
    wl = synth.workload(name)
    shapes = wl.muon_shapes
    offsets, total = nsm.pack(shapes)
    dev = "cuda"
    grads = torch.empty(total, dtype=torch.bfloat16, device=dev)
    params = torch.zeros(total, dtype=torch.float32, device=dev)
    mom = torch.zeros(total, dtype=torch.float32, device=dev)
    synth.fill_packed_grads(wl, offsets, grads)
    synth.fill_packed_params(wl, offsets, params)
    p0 = params.clone()
    ws = torch.empty(nsm.workspace_bytes(shapes, method), dtype=torch.uint8, device=dev)
    copy = torch.empty(total, dtype=torch.bfloat16, device=dev)
    nsm.muon_step(grads, params, mom, offsets, shapes, wl.lr, wl.wd, wl.mu, method, 5, True, ws,
                  params_bf16=copy)
    assert nsm.device_status() == nsm.NSM_OK
    del ws
    # properties on every matrix: O = (p0 (1 - lr wd) - p1) / (lr scale)
    decay = np.float32(1.0) - np.float32(wl.lr) * np.float32(wl.wd)
    for i, (r, c) in enumerate(shapes):
        o = int(offsets[i])
        d = p0[o:o + r * c] * float(decay) - params[o:o + r * c]
        assert torch.isfinite(d).all()
        onorm = float(d.double().norm()) / (wl.lr * oracle.update_scale(r, c))
        assert onorm <= 1.2 * np.sqrt(min(r, c)) * 1.01, (i, onorm)
    # sampled matrices against the oracle: each shape's first occurrence and, where asked,
    # its last (at the far end of the packed buffers and of the class slots, where 64-bit
    # offsets matter)
    picked = []
    for want in sample_shapes:
        where = [i for i, sh in enumerate(shapes) if sh == want]
        picked.append(where[0])
        if len(where) > 1 and want in last_too:
            picked.append(where[-1])
    # the bf16 copy (the owner's broadcast payload) is the rounding of the updated params,
    # here on the sampled matrices and on the table's last one (the largest offsets)
    for i in picked + [len(shapes) - 1]:
        r, c = shapes[i]
        o = int(offsets[i])
        assert torch.equal(copy[o:o + r * c], params[o:o + r * c].to(torch.bfloat16)), i
    del copy
    for i in picked:
        r, c = shapes[i]
        o = int(offsets[i])
        g = grads[o:o + r * c].double().cpu().numpy().reshape(r, c)
        p = p0[o:o + r * c].double().cpu().numpy().reshape(r, c)
        (pn,), (mn,), _ = oracle.muon_step([g], [p], [np.zeros_like(g)], wl.lr, wl.wd, wl.mu, method,
                                           storage="method")
        got_p = params[o:o + r * c].double().cpu().numpy().reshape(r, c)
        got_m = mom[o:o + r * c].double().cpu().numpy().reshape(r, c)
        assert rel(got_m, mn) <= 1e-5
        assert rel(got_p - p, pn - p) <= 1e-2, ((r, c), rel(got_p - p, pn - p))


@pytest.mark.parametrize("method", ["gram", "standard"])
def test_llama7b_fullsize(nsm, method):
    _run_fullsize(nsm, "llama7b", method, [(1024, 4096), (4096, 4096)], last_too=[(1024, 4096)])


@pytest.mark.parametrize("method", ["gram"])
def test_split_moe_fullsize(nsm, method):
    _run_fullsize(nsm, "split_moe", method, [(128, 4096), (1408, 2048), (2048, 1408)],
                  last_too=[(1408, 2048)])
