"""Parity at the full workload sizes, in the launch configuration the benchmark times.

One muon_step runs over the whole packed group (224 matrices / 5.67B elements for the
Llama-7B-shaped set, 3584 matrices / 9.13B elements for the Split/MoE set); then one
muon_orthogonalize runs over the same table, with the same grouped launches.

* On every matrix: the update is finite, ||O||_F <= 1.2 sqrt(m) (every singular value of
  the five-step output lies in [0, 1.2]), and every m x m iterate the chain left in the
  workspace is kept as its upper 256 x 256 tiles (every launch of these tables runs on
  the 2-SM kernel): the tiles on and above the diagonal are finite, the diagonal tiles
  exactly symmetric, and the tiles below it never written (the workspace starts as NaN).
* On a sample that covers every working shape, the first and the last matrix of the large
  classes (the far ends of the packed buffers and of the class slots, where 64-bit offsets
  matter): the momentum at 1e-5 and the parameter delta at 1e-2 against the oracle in the
  method's storage precision, and the orthogonalised output at 2e-2 against it, each with
  the element-wise bounds of the parity tests.  The same outputs are compared with the
  exact float64 iteration too: the measured distance is recorded, and held to 2e-2.
"""

import numpy as np
import pytest
import torch

import oracle
import parity_log
import synth
from test_gpu_parity import TOL_DELTA, TOL_FP32, TOL_NS, compare, elementwise, rel

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

TOL_EXACT = {"gram": TOL_NS, "standard": TOL_NS}


@pytest.fixture(scope="module")
def nsm():
    import newton_schulz_orthogonalized_gb300 as m
    m.lib()
    return m


def _pick(shapes, picks):
    """Indices: for each (shape, which) in picks, its first ('first') or last ('last')
    occurrence in the table."""
    out = []
    for want, which in picks:
        where = [i for i, sh in enumerate(shapes) if sh == want]
        i = where[0] if which == "first" else where[-1]
        if i not in out:
            out.append(i)
    return out


def _iterates_symmetric(nsm, shapes, method, ws, upper_tiles=False):
    """Every m x m block of the workspace is untouched (NaN bits) or finite and exactly
    symmetric; at least one block of every grouped-launch matrix was written.  With
    upper_tiles (iterates kept as their upper 256 x 256 tiles): in a written block the
    tiles on and above the diagonal are finite, the diagonal tiles exactly symmetric and
    the tiles below it untouched."""
    bits = ws.view(torch.int16)
    vals = ws.view(torch.float16 if method != "standard_bf16" else torch.bfloat16)
    for i in range(len(shapes)):
        written = 0
        for b in range(nsm.mm_buffers(method)):
            off, m, ld = nsm.workspace_iterate(shapes, i, b, method)
            if m == 0:
                break
            e0 = off // 2
            blk = bits[e0:e0 + m * ld].view(m, ld)[:, :m]
            if bool((blk == -1).all()):
                continue
            v = vals[e0:e0 + m * ld].view(m, ld)[:, :m]
            if not upper_tiles:
                assert bool(torch.isfinite(v).all()), (i, b)
                assert torch.equal(blk, blk.t()), (i, shapes[i], b)
            else:
                tile = torch.arange(m, device=blk.device) // 256
                lower = tile[:, None] > tile[None, :]
                diag = tile[:, None] == tile[None, :]
                assert bool((blk[lower] == -1).all()), (i, shapes[i], b)
                assert bool(torch.isfinite(v[~lower]).all()), (i, shapes[i], b)
                assert bool((blk == blk.t())[diag].all()), (i, shapes[i], b)
            written += 1
        off, m, _ = nsm.workspace_iterate(shapes, i, 0, method)
        assert m == 0 or written > 0, i


def _fullsize(nsm, name, method, step_picks, ortho_picks):
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
    ws = torch.full((nsm.workspace_bytes(shapes, method),), 255, dtype=torch.uint8, device=dev)
    copy = torch.empty(total, dtype=torch.bfloat16, device=dev)
    nsm.muon_step(grads, params, mom, offsets, shapes, wl.lr, wl.wd, wl.mu, method, 5, True, ws,
                  params_bf16=copy)
    assert nsm.device_status() == nsm.NSM_OK
    _iterates_symmetric(nsm, shapes, method, ws, upper_tiles=True)
    # properties on every matrix: O = (p0 (1 - lr wd) - p1) / (lr scale)
    decay = np.float32(1.0) - np.float32(wl.lr) * np.float32(wl.wd)
    for i, (r, c) in enumerate(shapes):
        o = int(offsets[i])
        d = p0[o:o + r * c] * float(decay) - params[o:o + r * c]
        assert torch.isfinite(d).all()
        onorm = float(d.double().norm()) / (wl.lr * oracle.update_scale(r, c))
        assert onorm <= 1.2 * np.sqrt(min(r, c)) * 1.01, (i, onorm)
    step_idx = _pick(shapes, step_picks)
    # the bf16 copy (the owner's broadcast payload) is the rounding of the updated params,
    # on the sampled matrices and on the table's last one (the largest offsets)
    for i in step_idx + [len(shapes) - 1]:
        r, c = shapes[i]
        o = int(offsets[i])
        assert torch.equal(copy[o:o + r * c], params[o:o + r * c].to(torch.bfloat16)), i
    del copy
    for i in step_idx:
        r, c = shapes[i]
        o = int(offsets[i])
        g = grads[o:o + r * c].double().cpu().numpy().reshape(r, c)
        p = p0[o:o + r * c].double().cpu().numpy().reshape(r, c)
        (pn,), (mn,), _ = oracle.muon_step([g], [p], [np.zeros_like(g)], wl.lr, wl.wd, wl.mu, method,
                                           storage="method")
        got_p = params[o:o + r * c].double().cpu().numpy().reshape(r, c)
        got_m = mom[o:o + r * c].double().cpu().numpy().reshape(r, c)
        assert rel(got_m, mn) <= TOL_FP32
        compare(got_p - p, pn - p, TOL_DELTA, f"fullsize/{name}/{method}/step/{(r, c)}/{i}")
    del params, mom, p0

    # the orthogonalisation alone over the same table: O as the chain computes it
    out = torch.empty_like(grads)
    ws.fill_(255)
    nsm.muon_orthogonalize(grads, out, offsets, shapes, method, 5, ws)
    assert nsm.device_status() == nsm.NSM_OK
    _iterates_symmetric(nsm, shapes, method, ws, upper_tiles=True)
    del ws
    for i in _pick(shapes, ortho_picks):
        r, c = shapes[i]
        o = int(offsets[i])
        g = grads[o:o + r * c].double().cpu().numpy().reshape(r, c)
        got = out[o:o + r * c].double().cpu().numpy().reshape(r, c)
        ref = oracle.orthogonalize(g, method, storage="method")
        compare(got, ref, TOL_NS, f"fullsize/{name}/{method}/ortho/{(r, c)}/{i}")
        exact = oracle.orthogonalize(g, method)
        e = rel(got, exact)
        emax, ep = elementwise(got, exact)
        parity_log.record(f"fullsize/{name}/{method}/ortho_vs_exact/{(r, c)}/{i}", rel=e, max_over_rms=emax,
                          p999_over_rms=ep, tol=TOL_EXACT[method])
        assert e <= TOL_EXACT[method], ((r, c), i, e)


LLAMA_STEP = [((1024, 4096), "first"), ((1024, 4096), "last"), ((4096, 4096), "first"),
              ((11008, 4096), "first"), ((11008, 4096), "last"), ((4096, 11008), "last")]
LLAMA_ORTHO = [((11008, 4096), "first"), ((4096, 11008), "first"), ((4096, 4096), "last"),
               ((1024, 4096), "last")]


@pytest.mark.parametrize("method", ["gram", "standard"])
def test_llama7b_fullsize(nsm, method):
    _fullsize(nsm, "llama7b", method, LLAMA_STEP, LLAMA_ORTHO)


@pytest.mark.parametrize("method", ["gram"])
def test_split_moe_fullsize(nsm, method):
    picks = [((128, 4096), "first"), ((128, 4096), "last"), ((1408, 2048), "first"),
             ((1408, 2048), "last"), ((2048, 1408), "last")]
    _fullsize(nsm, "split_moe", method, picks, [((2048, 1408), "first"), ((1408, 2048), "last"),
                                                ((128, 4096), "last")])
