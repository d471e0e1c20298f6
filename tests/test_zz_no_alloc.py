"""The allocation-free orthogonalisation against the regular one.

muon_orthogonalize_noalloc is for callers that cannot call cudaMalloc: a framework whose
own caching pool owns all device memory (an allocation outside it can fail or fragment
the pool), or a latency-critical loop that cannot take the device synchronisation an
allocation may imply.  It keeps its workspace and launch plan in a fixed array of device
memory that belongs to the library.

It runs the same kernels on the same plan as muon_orthogonalize with a caller workspace,
so the outputs must be identical bit for bit.  The calls in a row use different tables,
then the first table again: the shared array keeps the last call's contents, and neither
a stale workspace nor a stale plan may leak into the next result.  This file is
collected last so that a failure here leaves every other result standing; it passes on
its own in a fresh process too.
"""

import ctypes

import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nsm():
    import newton_schulz_orthogonalized_gb300 as m
    m.lib()
    return m


def _inputs(nsm, wl):
    offsets, total = nsm.pack(wl.muon_shapes)
    inp = torch.zeros(total, dtype=torch.bfloat16, device="cuda")
    synth.fill_packed_grads(wl, offsets, inp)
    return offsets, inp


def _regular(nsm, wl, offsets, inp, method):
    out = torch.full_like(inp, float("nan"))
    ws = torch.empty(nsm.workspace_bytes(wl.muon_shapes, method), dtype=torch.uint8, device="cuda")
    nsm.muon_orthogonalize(inp, out, offsets, wl.muon_shapes, method, 5, ws)
    torch.cuda.synchronize()
    return out


def _noalloc(nsm, wl, offsets, inp, method):
    # straight through the C ABI
    out = torch.full_like(inp, float("nan"))
    L = nsm.lib()
    s = np.ascontiguousarray(np.asarray(wl.muon_shapes, dtype=np.int32).reshape(-1, 2))
    o = np.ascontiguousarray(np.asarray(offsets, dtype=np.int64))
    rc = L.muon_orthogonalize_noalloc(inp.data_ptr(), out.data_ptr(),
                                      o.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                                      s.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), s.shape[0],
                                      nsm.method_code(method), 5,
                                      int(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, nsm.last_error()
    torch.cuda.synchronize()
    return out


def _same_bits(nsm, wl, offsets, got, ref):
    for i, (r, c) in enumerate(wl.muon_shapes):
        o = int(offsets[i])
        x, y = got[o:o + r * c], ref[o:o + r * c]
        assert torch.isfinite(x.float()).all(), (i, (r, c))
        assert torch.equal(x, y), (i, (r, c))


@pytest.mark.parametrize("method", ["gram", "standard"])
def test_noalloc_matches_regular_two_calls(nsm, method):
    first = synth.custom([(256, 512), (512, 256), (130, 260), (64, 64)], seed=31)
    second = synth.custom([(1024, 1024), (384, 96), (3, 5)], seed=32)
    for wl in (first, second, first):
        offsets, inp = _inputs(nsm, wl)
        ref = _regular(nsm, wl, offsets, inp, method)
        got = _noalloc(nsm, wl, offsets, inp, method)
        _same_bits(nsm, wl, offsets, got, ref)
        # the same table again: the plan already in the array is reused as it stands
        again = _noalloc(nsm, wl, offsets, inp, method)
        _same_bits(nsm, wl, offsets, again, ref)
    assert nsm.device_status() == nsm.NSM_OK


def test_noalloc_rejects_tables_beyond_its_array(nsm):
    wl = synth.custom([(4096, 4096)] * 3, seed=0)  # ~100 MB of workspace > 64 MiB
    offsets, total = nsm.pack(wl.muon_shapes)
    inp = torch.zeros(total, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros_like(inp)
    with pytest.raises(nsm.NsmError) as e:
        nsm.muon_orthogonalize_noalloc(inp, out, offsets, wl.muon_shapes, "gram")
    assert e.value.code == nsm.NSM_ERR_WORKSPACE
    assert "bytes" in nsm.last_error()
