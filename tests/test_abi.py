"""CPU-side checks of the C ABI: the library loads, exports every declared symbol, and
its host-only functions (routing, packing, workspace sizing, argument validation)
behave as documented.  Nothing here touches a GPU: every validation failure is
returned before the library makes a CUDA call."""

import ctypes
import json
import os
import re

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nsmuon.h")


@pytest.fixture(scope="module")
def nsm():
    import newton_schulz_orthogonalized_gb300 as m
    if not os.path.exists(m.LIB_PATH):
        from newton_schulz_orthogonalized_gb300 import _build
        _build.build()
    m.lib()
    return m


def _declared_functions():
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z_][a-z0-9_]*)\s*\(",
                       text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = _declared_functions()
    for required in ("muon_step", "adamw_step", "muon_orthogonalize", "muon_workspace_bytes",
                     "nsm_route", "nsm_pack", "nsm_version", "nsm_last_error"):
        assert required in names


def test_library_exports_every_declared_symbol(nsm):
    L = nsm.lib()
    for name in _declared_functions():
        assert hasattr(L, name), name


def test_version(nsm):
    assert nsm.version() >= 100


def test_route_matches_oracle_and_prose(nsm):
    with open(os.path.join(ROOT, "tests", "golden", "routing_cases.json"), encoding="utf-8") as f:
        cases = json.load(f)["cases"]
    for name, ndim, expected, _ in cases:
        assert nsm.route(name, ndim) is expected
        assert nsm.route(name, ndim) == oracle.route(name, ndim)
    assert nsm.lib().nsm_route(None, 2) == nsm.NSM_ERR_NULL


@pytest.mark.parametrize("align", [1, 8, 64, 128])
def test_pack_matches_oracle(nsm, align):
    rng = np.random.default_rng(align)
    shapes = [tuple(int(x) for x in rng.integers(1, 300, 2)) for _ in range(37)]
    offs, total = nsm.pack(shapes, align)
    ro, rt = oracle.pack_offsets(shapes, align)
    assert list(offs) == ro and total == rt


def test_pack_rejects_bad_shapes(nsm):
    with pytest.raises(nsm.NsmError) as e:
        nsm.pack([(4, 0)])
    assert e.value.code == nsm.NSM_ERR_SHAPE


def test_workspace_bytes(nsm):
    a = nsm.workspace_bytes([(128, 256)] * 4, "standard")
    b = nsm.workspace_bytes([(128, 256)] * 4, "gram")
    assert a > 0 and b > a  # gram keeps four m x m buffers
    # depends on shapes, not their order of equal classes
    assert nsm.workspace_bytes([(256, 128), (128, 256)], "standard") == \
        nsm.workspace_bytes([(128, 256), (256, 128)], "standard")
    with pytest.raises(nsm.NsmError):
        nsm.workspace_bytes([(128, 256)], 7)
    with pytest.raises(nsm.NsmError):
        nsm.workspace_bytes([(128, 256)], "standard", 99)


def _call_step(nsm, shapes, offsets=None, grads=0x10000, params=0x20000000, mom=0x40000000,
               ws=0x80000000, ws_bytes=None, method=0, steps=5, n=None):
    L = nsm.lib()
    s = np.ascontiguousarray(np.asarray(shapes, dtype=np.int32).reshape(-1, 2))
    if offsets is None:
        offsets, _ = nsm.pack(shapes)
    o = np.ascontiguousarray(np.asarray(offsets, dtype=np.int64))
    if ws_bytes is None:
        ws_bytes = 16
    return L.muon_step(grads, params, mom, o.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                       s.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                       s.shape[0] if n is None else n, 0.02, 0.1, 0.95, method, steps, 1,
                       ws, ws_bytes, None)


def test_step_validation_errors_without_gpu(nsm):
    shapes = [(128, 256), (64, 64)]
    assert _call_step(nsm, shapes, grads=0) == nsm.NSM_ERR_NULL
    assert _call_step(nsm, [(128, 0)], offsets=[0]) == nsm.NSM_ERR_SHAPE
    assert _call_step(nsm, shapes, n=0) == nsm.NSM_ERR_SHAPE
    assert _call_step(nsm, shapes, method=3) == nsm.NSM_ERR_METHOD
    assert _call_step(nsm, shapes, method=2) == nsm.NSM_ERR_WORKSPACE  # standard_bf16 is valid
    assert _call_step(nsm, shapes, steps=-1) == nsm.NSM_ERR_METHOD
    # overlapping matrices
    assert _call_step(nsm, shapes, offsets=[0, 64]) == nsm.NSM_ERR_OFFSET
    assert _call_step(nsm, shapes, offsets=[-64, 40000]) == nsm.NSM_ERR_OFFSET
    # offsets must be multiples of 8 elements
    assert _call_step(nsm, shapes, offsets=[0, 32772]) == nsm.NSM_ERR_ALIGN
    # misaligned device pointer
    assert _call_step(nsm, shapes, grads=0x10002) == nsm.NSM_ERR_ALIGN
    # aliasing grads and params
    assert _call_step(nsm, shapes, grads=0x20000000) == nsm.NSM_ERR_ARG
    # workspace too small / NULL / misaligned
    assert _call_step(nsm, shapes) == nsm.NSM_ERR_WORKSPACE
    assert _call_step(nsm, shapes, ws=0, ws_bytes=1 << 40) == nsm.NSM_ERR_WORKSPACE
    assert _call_step(nsm, shapes, ws=0x80000010, ws_bytes=1 << 40) == nsm.NSM_ERR_ALIGN
    assert "workspace" in nsm.last_error()


def test_adamw_validation_without_gpu(nsm):
    L = nsm.lib()
    assert L.adamw_step(0, 0, 0, 0, 0, 1e-3, 0.9, 0.95, 1e-8, 0.0, 1, None) == 0  # empty group
    assert L.adamw_step(0, 0x1000, 0x2000, 0x3000, 8, 1e-3, 0.9, 0.95, 1e-8, 0.0, 1, None) == nsm.NSM_ERR_NULL
    assert L.adamw_step(0x100, 0x1000, 0x2000, 0x3000, -1, 1e-3, 0.9, 0.95, 1e-8, 0.0, 1, None) == nsm.NSM_ERR_SHAPE
    assert L.adamw_step(0x100, 0x1000, 0x2000, 0x3000, 8, 1e-3, 0.9, 0.95, 1e-8, 0.0, 0, None) == nsm.NSM_ERR_ARG
    assert L.adamw_step(0x100, 0x1000, 0x2000, 0x3000, 8, 1e-3, 1.5, 0.95, 1e-8, 0.0, 1, None) == nsm.NSM_ERR_ARG
    assert L.adamw_step(0x104, 0x1000, 0x2000, 0x3000, 8, 1e-3, 0.9, 0.95, 1e-8, 0.0, 1, None) == nsm.NSM_ERR_ALIGN
    assert L.adamw_step(0x100, 0x1000, 0x1000, 0x3000, 8, 1e-3, 0.9, 0.95, 1e-8, 0.0, 1, None) == nsm.NSM_ERR_ARG


def test_orthogonalize_validation_without_gpu(nsm):
    L = nsm.lib()
    s = np.array([[16, 32]], dtype=np.int32)
    o = np.array([0], dtype=np.int64)
    P32 = ctypes.POINTER(ctypes.c_int32)
    P64 = ctypes.POINTER(ctypes.c_int64)
    args = (o.ctypes.data_as(P64), s.ctypes.data_as(P32), 1, 0, 5)
    assert L.muon_orthogonalize(0, 0x2000, *args, 0x100000, 1 << 30, None) == nsm.NSM_ERR_NULL
    assert L.muon_orthogonalize(0x1000, 0x1000, *args, 0x100000, 1 << 30, None) == nsm.NSM_ERR_ARG
    assert L.muon_orthogonalize(0x1000, 0x9000, *args, 0x100000, 8, None) == nsm.NSM_ERR_WORKSPACE


def test_optimizer_wrapper_routing(nsm):
    # routing and grouping only; constructing device buffers needs a GPU
    named = [("model.embed_tokens.weight", (100, 16)), ("layers.0.q_proj.weight", (16, 16)),
             ("layers.0.norm.weight", (16,)), ("lm_head.weight", (100, 16)),
             ("conv.weight", (8, 3, 3, 3))]
    muon = [n for n, s in named if nsm.route(n, len(s))]
    assert muon == ["layers.0.q_proj.weight", "conv.weight"]
    assert oracle.matrix_view_shape((8, 3, 3, 3)) == (8, 27)


def test_status_selftest_validation_without_gpu(nsm):
    L = nsm.lib()
    assert L.nsm_status_selftest(0, None) == nsm.NSM_ERR_ARG
    assert L.nsm_status_selftest(2000001, None) == nsm.NSM_ERR_ARG


def test_options_set_get_and_reject(nsm):
    # host-only: the defaults, a round trip, and validation (no GPU call is made)
    assert nsm.get_option(nsm.OPT_PAIR_KERNELS) == 1
    assert nsm.get_option(nsm.OPT_SMALL_KERNEL) == 1
    assert nsm.get_option(nsm.OPT_PDL) == 2  # auto
    assert nsm.get_option(nsm.OPT_SYM_STORAGE) == 1
    nsm.set_option(nsm.OPT_SYM_STORAGE, 0)
    try:
        assert nsm.get_option(nsm.OPT_SYM_STORAGE) == 0
    finally:
        nsm.set_option(nsm.OPT_SYM_STORAGE, 1)
    nsm.set_option(nsm.OPT_PDL, 1)
    try:
        assert nsm.get_option(nsm.OPT_PDL) == 1
    finally:
        nsm.set_option(nsm.OPT_PDL, 2)
    with pytest.raises(nsm.NsmError) as e:
        nsm.set_option(nsm.OPT_PDL, 3)
    assert e.value.code == nsm.NSM_ERR_ARG
    with pytest.raises(nsm.NsmError):
        nsm.set_option(nsm.OPT_SMALL_KERNEL, 2)
    with pytest.raises(nsm.NsmError):
        nsm.set_option(99, 1)
    with pytest.raises(nsm.NsmError):
        nsm.get_option(99)


@pytest.mark.parametrize("method", ["gram", "standard", "standard_bf16"])
def test_workspace_iterate_layout(nsm, method):
    # every m x m block lies inside the workspace, blocks of one buffer do not overlap,
    # matrices of the same working shape share the block size, and the small-matrix
    # kernel's matrices report m = 0 (their iterates stay in shared memory)
    shapes = [(256, 512), (512, 256), (130, 260), (64, 1000), (1024, 1024), (300, 520), (520, 300)]
    total = nsm.workspace_bytes(shapes, method)
    nbuf = nsm.mm_buffers(method)
    for b in range(nbuf):
        spans = []
        for i, (r, c) in enumerate(shapes):
            off, m, ld = nsm.workspace_iterate(shapes, i, b, method)
            if min(r, c) <= 128:
                assert m == 0
                continue
            assert m == min(r, c) and ld >= m and ld % 64 == 0
            assert off % 2 == 0 and off + m * ld * 2 <= total
            spans.append((off, off + m * ld * 2))
        spans.sort()
        for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
            assert a1 <= b0
    with pytest.raises(nsm.NsmError):
        nsm.workspace_iterate(shapes, 0, nbuf, method)
    with pytest.raises(nsm.NsmError):
        nsm.workspace_iterate(shapes, len(shapes), 0, method)


def test_checked_build_exports_the_same_symbols_and_reports_itself(nsm):
    # the bounds-checked twin library: same ABI; NSM_OPT_BOUNDS_CHECKS reads 1 there and
    # 0 in the regular build, and is read only in both (host-only calls, no GPU)
    if not os.path.exists(nsm.LIB_CHECKED):
        from newton_schulz_orthogonalized_gb300 import _build
        _build.build(checked=True)
    C = ctypes.CDLL(nsm.LIB_CHECKED)
    for name in _declared_functions():
        assert hasattr(C, name), name
    assert C.nsm_get_option(nsm.OPT_BOUNDS_CHECKS) == 1
    assert C.nsm_set_option(nsm.OPT_BOUNDS_CHECKS, 0) == nsm.NSM_ERR_ARG
    assert nsm.get_option(nsm.OPT_BOUNDS_CHECKS) == 0
    assert not nsm.checked_build()
    with pytest.raises(nsm.NsmError):
        nsm.set_option(nsm.OPT_BOUNDS_CHECKS, 1)


def test_copy_to_device_validation_without_gpu(nsm):
    L = nsm.lib()
    buf = ctypes.create_string_buffer(64)
    base = (ctypes.addressof(buf) + 15) // 16 * 16
    assert L.nsm_copy_to_device(None, base, 16, 0, None) == nsm.NSM_ERR_NULL
    assert L.nsm_copy_to_device(base, None, 16, 0, None) == nsm.NSM_ERR_NULL
    assert L.nsm_copy_to_device(base + 8, base, 16, 0, None) == nsm.NSM_ERR_ALIGN
    assert L.nsm_copy_to_device(base, base + 4, 16, 0, None) == nsm.NSM_ERR_ALIGN
    assert L.nsm_copy_to_device(base, base, 16, -1, None) == nsm.NSM_ERR_ARG
    assert L.nsm_copy_to_device(base, base, 16, 1025, None) == nsm.NSM_ERR_ARG
    assert L.nsm_copy_to_device(base, base, 0, 0, None) == nsm.NSM_OK  # nothing to copy
