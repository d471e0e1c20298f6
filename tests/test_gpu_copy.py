"""The library's host-to-device copy by SM loads (nsm_copy_to_device): the bytes of a
page-locked host buffer arrive unchanged, whatever the byte count, on the given stream;
memory the SMs cannot read through a device mapping is refused before any launch."""

import ctypes

import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nsm():
    import newton_schulz_orthogonalized_gb300 as m
    m.lib()
    return m


@pytest.mark.parametrize("nbytes", [16, 4096, 1 << 20, (1 << 26) + 48, (1 << 26) + 7])
def test_copy_is_exact(nsm, nbytes):
    g = torch.Generator().manual_seed(nbytes)
    src = torch.randint(0, 256, (nbytes,), dtype=torch.uint8, generator=g).pin_memory()
    dst = torch.zeros(nbytes + 32, dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    nsm.copy_to_device(dst[:nbytes], src, s)
    s.synchronize()
    assert torch.equal(dst[:nbytes].cpu(), src)
    assert int(dst[nbytes:].count_nonzero()) == 0  # nothing written past the end


def test_copy_of_bf16_grads_matches_engine_copy(nsm):
    src = (torch.randn(3 * 1024 * 1024 + 5) * 0.01).to(torch.bfloat16).pin_memory()
    a = torch.empty(src.numel(), dtype=torch.bfloat16, device="cuda")
    nsm.copy_to_device(a, src, torch.cuda.current_stream(), ctas=38)
    b = src.to("cuda")
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_copy_refuses_memory_without_device_mapping(nsm):
    L = nsm.lib()
    dst = torch.empty(4096, dtype=torch.uint8, device="cuda")
    pageable = torch.empty(4096, dtype=torch.uint8)
    assert L.nsm_copy_to_device(dst.data_ptr(), pageable.data_ptr(), 4096, 0, None) == nsm.NSM_ERR_ARG
    device_src = torch.empty(4096, dtype=torch.uint8, device="cuda")
    assert L.nsm_copy_to_device(dst.data_ptr(), device_src.data_ptr(), 4096, 0, None) == nsm.NSM_ERR_ARG
    assert nsm.device_status() == nsm.NSM_OK


def test_step_reads_grads_in_place_from_page_locked_memory(nsm):
    # muon_step takes its grads from page-locked host memory as well as from device
    # memory: the step's first pass reads them through their device mapping, and the
    # result is the same to the bit
    import synth
    wl = synth.custom([(256, 512), (640, 192), (96, 200), (130, 260)], seed=31)
    offsets, total = nsm.pack(wl.muon_shapes)
    g_dev = torch.zeros(total, dtype=torch.bfloat16, device="cuda")
    synth.fill_packed_grads(wl, offsets, g_dev)
    g_host = g_dev.cpu().pin_memory()
    results = []
    for grads in (g_dev, g_host):
        p = torch.zeros(total, dtype=torch.float32, device="cuda")
        synth.fill_packed_params(wl, offsets, p)
        m = torch.zeros(total, dtype=torch.float32, device="cuda")
        copy = torch.zeros(total, dtype=torch.bfloat16, device="cuda")
        ws = torch.zeros(nsm.workspace_bytes(wl.muon_shapes, "gram"), dtype=torch.uint8, device="cuda")
        for _ in range(2):  # the second step reads the exponents the first one left
            nsm.muon_step(grads, p, m, offsets, wl.muon_shapes, wl.lr, wl.wd, wl.mu, "gram", 5, True, ws,
                          params_bf16=copy)
        torch.cuda.synchronize()
        assert nsm.device_status() == nsm.NSM_OK
        results.append((p.cpu(), m.cpu(), copy.cpu()))
    for a, b in zip(results[0], results[1]):
        assert torch.equal(a.view(torch.int32) if a.dtype == torch.float32 else a.view(torch.int16),
                           b.view(torch.int32) if b.dtype == torch.float32 else b.view(torch.int16))


def test_step_refuses_pageable_grads(nsm):
    wl_shapes = [(64, 128)]
    offsets, total = nsm.pack(wl_shapes)
    pageable = torch.zeros(total, dtype=torch.bfloat16)
    p = torch.zeros(total, dtype=torch.float32, device="cuda")
    m = torch.zeros(total, dtype=torch.float32, device="cuda")
    ws = torch.zeros(nsm.workspace_bytes(wl_shapes, "gram"), dtype=torch.uint8, device="cuda")
    with pytest.raises(RuntimeError, match="page-locked"):
        nsm.muon_step(pageable, p, m, offsets, wl_shapes, 0.02, 0.0, 0.95, "gram", 5, True, ws)
    assert nsm.device_status() == nsm.NSM_OK
