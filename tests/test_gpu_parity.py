"""Parity of the CUDA path with the oracle, through the C ABI.

The oracle runs the method in the storage precision of its form (fp16 for the standard
and gram forms, bf16 for standard_bf16: it rounds where the method stores an iterate and
accumulates in float64).  Tolerances (relative Frobenius norms): orthogonalised output
<= 2e-2, final parameter delta <= 1e-2, momentum and AdamW <= 1e-5.  Routing and
offsets are bit-exact (tests/test_abi.py).  Where the exact float64 iteration is within
reach of half-precision storage (well-conditioned inputs, and the re-anchored gram form)
the GPU is also held to it.  Inputs come from the seeded generators in ``synth``: the GPU
draws them, the oracle reads the same bf16 values decoded exactly.
"""


import numpy as np
import pytest
import torch

import oracle
import parity_log
import synth

pytestmark = pytest.mark.gpu

TOL_NS = 2e-2
TOL_DELTA = 1e-2
TOL_FP32 = 1e-5


@pytest.fixture(scope="module")
def nsm():
    import newton_schulz_orthogonalized_gb300 as m
    m.lib()
    return m


def rel(a, b):
    nb = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (nb if nb > 0 else 1.0)


# Element-wise bounds, checked beside every relative Frobenius norm: max |GPU - oracle|
# and its 99.9th percentile, in units of the oracle's rms value.  The entries of O spread
# to about 7 times their rms, and a wrong, zeroed, stale or misplaced 32 x 32 block moves
# its entries by about their own size (>= 1 rms on average), which these bounds catch even
# where the Frobenius norm of a 4096 x 4096 output would not (one block is 0.8% of it).
# Measured against the storage-precision oracle on the 4096-row classes (O exported in
# bf16): worst entry 0.40 rms, 99.9th percentile 0.09 rms.  The bf16 form is chaotic at
# the 1-2% level and gets its own bounds.
ELEM_MAX, ELEM_P999 = 0.75, 0.25
ELEM_MAX_BF16, ELEM_P999_BF16 = 2.0, 0.6


def elementwise(got, ref):
    """(max |got - ref|, 99.9th percentile of |got - ref|) over rms(ref)."""
    d = np.abs(np.asarray(got, np.float64) - np.asarray(ref, np.float64)).ravel()
    rms = float(np.sqrt(np.mean(np.square(ref)))) if np.size(ref) else 0.0
    if rms == 0.0:
        return (0.0, 0.0) if d.size == 0 or d.max() == 0 else (np.inf, np.inf)
    return float(d.max()) / rms, float(np.quantile(d, 0.999)) / rms


def compare(got, ref, tol, what, bf16=False):
    """Relative Frobenius error <= tol and the element-wise bounds; records the numbers."""
    e = rel(got, ref)
    emax, ep = elementwise(got, ref)
    parity_log.record(what, rel=e, max_over_rms=emax, p999_over_rms=ep, tol=tol)
    lim_max, lim_p = (ELEM_MAX_BF16, ELEM_P999_BF16) if bf16 else (ELEM_MAX, ELEM_P999)
    assert e <= tol, (what, e)
    assert emax <= lim_max and ep <= lim_p, (what, emax, ep)
    return e


class Step:
    """Runs muon_step on a workload and keeps host copies for the oracle."""

    def __init__(self, nsm, wl, method, steps=5, nesterov=True, momentum_init=None,
                 zero_grads=()):
        self.wl = wl
        self.method = method
        self.steps = steps
        self.nesterov = nesterov
        self.offsets, total = nsm.pack(wl.muon_shapes)
        dev = "cuda"
        self.grads = torch.zeros(total, dtype=torch.bfloat16, device=dev)
        synth.fill_packed_grads(wl, self.offsets, self.grads)
        for i in zero_grads:
            r, c = wl.muon_shapes[i]
            o = int(self.offsets[i])
            self.grads[o:o + r * c].zero_()
        self.params = torch.zeros(total, dtype=torch.float32, device=dev)
        synth.fill_packed_params(wl, self.offsets, self.params)
        if momentum_init is None:
            self.mom = torch.zeros(total, dtype=torch.float32, device=dev)
        else:
            self.mom = momentum_init.to(dev).clone()
        self.p0 = self.params.double().cpu().numpy()
        self.m0 = self.mom.double().cpu().numpy()
        self.g = self.grads.double().cpu().numpy()
        ws = torch.empty(nsm.workspace_bytes(wl.muon_shapes, method, steps), dtype=torch.uint8,
                         device=dev)
        nsm.muon_step(self.grads, self.params, self.mom, self.offsets, wl.muon_shapes, wl.lr,
                      wl.wd, wl.mu, method, steps, nesterov, ws)
        assert nsm.device_status() == nsm.NSM_OK
        self.p1 = self.params.double().cpu().numpy()
        self.m1 = self.mom.double().cpu().numpy()

    def matrix(self, arr, i):
        r, c = self.wl.muon_shapes[i]
        o = int(self.offsets[i])
        return arr[o:o + r * c].reshape(r, c)

    def check(self, indices=None, tol_delta=TOL_DELTA):
        wl = self.wl
        idx = range(len(wl.muon_shapes)) if indices is None else indices
        worst = {"delta": 0.0, "mom": 0.0}
        for i in idx:
            g = self.matrix(self.g, i)
            p = self.matrix(self.p0, i)
            m = self.matrix(self.m0, i)
            (pn,), (mn,), _ = oracle.muon_step([g], [p], [m], wl.lr, wl.wd, wl.mu, self.method,
                                               self.steps, self.nesterov, storage="method")
            e_m = rel(self.matrix(self.m1, i), mn)
            assert e_m <= TOL_FP32, (i, e_m)
            e_d = compare(self.matrix(self.p1, i) - p, pn - p, tol_delta,
                          f"step/{wl.name}/{self.method}/{wl.muon_shapes[i]}/{i}",
                          bf16=self.method == "standard_bf16")
            worst["mom"] = max(worst["mom"], e_m)
            worst["delta"] = max(worst["delta"], e_d)
        return worst


def orthogonalize_gpu(nsm, wl, method, steps=5):
    offsets, total = nsm.pack(wl.muon_shapes)
    inp = torch.zeros(total, dtype=torch.bfloat16, device="cuda")
    synth.fill_packed_grads(wl, offsets, inp)
    out = torch.zeros_like(inp)
    ws = torch.empty(nsm.workspace_bytes(wl.muon_shapes, method, steps), dtype=torch.uint8,
                     device="cuda")
    nsm.muon_orthogonalize(inp, out, offsets, wl.muon_shapes, method, steps, ws)
    assert nsm.device_status() == nsm.NSM_OK
    return offsets, inp.double().cpu().numpy(), out.double().cpu().numpy()


RAGGED = [(130, 260), (3, 5), (257, 129), (64, 1000), (1, 8), (200, 200), (8, 8), (384, 96),
          (136, 72)]


# ------------------------------------------------------------------ orthogonalisation

@pytest.mark.parametrize("method", ["standard", "gram"])
@pytest.mark.parametrize("steps", [0, 1, 5])
def test_orthogonalize_ragged(nsm, method, steps):
    wl = synth.custom(RAGGED, seed=3, lowrank=False)
    offsets, g, o = orthogonalize_gpu(nsm, wl, method, steps)
    for i, (r, c) in enumerate(wl.muon_shapes):
        off = int(offsets[i])
        gi = g[off:off + r * c].reshape(r, c)
        ref = oracle.orthogonalize(gi, method, steps, storage="method")
        got = o[off:off + r * c].reshape(r, c)
        compare(got, ref, TOL_NS, f"ortho/ragged/{method}/{steps}/{(r, c)}")


@pytest.mark.parametrize("method", ["standard", "gram"])
def test_orthogonalize_layer1024(nsm, method):
    wl = synth.workload("layer1024")
    offsets, g, o = orthogonalize_gpu(nsm, wl, method)
    for i, (r, c) in enumerate(wl.muon_shapes):
        off = int(offsets[i])
        ref = oracle.orthogonalize(g[off:off + r * c].reshape(r, c), method, storage="method")
        got = o[off:off + r * c].reshape(r, c)
        compare(got, ref, TOL_NS, f"ortho/layer1024/{method}/{(r, c)}")


@pytest.mark.parametrize("method", ["standard", "gram"])
def test_orthogonalize_well_conditioned_vs_exact(nsm, method):
    # singular values in a band where the iteration is not steep: half-precision storage
    # stays within 2e-2 of the exact float64 iteration
    rng = np.random.default_rng(17)
    shapes = [(96, 160), (256, 256), (300, 130)]
    mats = []
    for r, c in shapes:
        m, n = min(r, c), max(r, c)
        uu, _ = np.linalg.qr(rng.standard_normal((m, m)))
        vv, _ = np.linalg.qr(rng.standard_normal((n, m)))
        x = (uu * np.linspace(1.0, 0.35, m)) @ vv.T
        mats.append(x.T if r > c else x)
    offsets, total = nsm.pack(shapes)
    host = np.zeros(total, dtype=np.float32)
    for (r, c), o, x in zip(shapes, offsets, mats):
        host[int(o):int(o) + r * c] = x.reshape(-1)
    inp = torch.from_numpy(host).to("cuda", torch.bfloat16)
    out = torch.zeros_like(inp)
    ws = torch.empty(nsm.workspace_bytes(shapes, method), dtype=torch.uint8, device="cuda")
    nsm.muon_orthogonalize(inp, out, offsets, shapes, method, 5, ws)
    torch.cuda.synchronize()
    g = inp.double().cpu().numpy()
    o = out.double().cpu().numpy()
    for (r, c), off in zip(shapes, offsets):
        sl = slice(int(off), int(off) + r * c)
        ref = oracle.orthogonalize(g[sl].reshape(r, c), method)
        compare(o[sl].reshape(r, c), ref, TOL_NS, f"ortho/well_conditioned_vs_exact/{method}/{(r, c)}")


@pytest.mark.parametrize("method", ["standard", "gram"])
def test_fp16_forms_close_to_exact_on_workload(nsm, method):
    # both fp16 forms stay within 2e-2 of the exact float64 iteration even on the
    # near-low-rank inputs, the input being stored as U 2^k (11 significant bits at any
    # magnitude, no subnormals); the bf16 form is ~18% away
    wl = synth.workload("layer1024")
    offsets, g, o = orthogonalize_gpu(nsm, wl, method)
    for i, (r, c) in enumerate(wl.muon_shapes):
        off = int(offsets[i])
        ref = oracle.orthogonalize(g[off:off + r * c].reshape(r, c), method)
        compare(o[off:off + r * c].reshape(r, c), ref, TOL_NS, f"ortho/layer1024_vs_exact/{method}/{(r, c)}")


@pytest.mark.parametrize("wl_name", ["tiny", "gpt2small"])
@pytest.mark.parametrize("method", ["standard", "gram"])
def test_orthogonalize_vs_exact_small_workloads(nsm, wl_name, method):
    # The exact float64 iteration on the tiny and GPT-2-small tables (one matrix of each
    # shape), recorded beside the storage-precision comparison; the one-layer table is
    # covered above and the Llama-7B and Split/MoE tables at full size.  Both fp16 forms
    # stay within 2e-2 of it.
    wl = synth.workload(wl_name)
    offsets, g, o = orthogonalize_gpu(nsm, wl, method)
    seen = set()
    for i, (r, c) in enumerate(wl.muon_shapes):
        if (r, c) in seen:
            continue
        seen.add((r, c))
        off = int(offsets[i])
        x = g[off:off + r * c].reshape(r, c)
        got = o[off:off + r * c].reshape(r, c)
        compare(got, oracle.orthogonalize(x, method, storage="method"), TOL_NS,
                f"ortho/{wl_name}/{method}/{(r, c)}")
        compare(got, oracle.orthogonalize(x, method), TOL_NS, f"ortho/{wl_name}_vs_exact/{method}/{(r, c)}")


# ------------------------------------------------------------------ full step

# The bf16 form of the standard iteration: two correct bf16 implementations that round at
# the same points but accumulate differently differ by up to ~1.5% on near-low-rank
# inputs (the iteration amplifies small singular directions ~487x), so its step delta is
# held at the same 2e-2 as its output; the fp16 forms meet 1e-2.
TOL_DELTA_BF16 = 2e-2


@pytest.mark.parametrize("wl_name", ["tiny", "layer1024"])
def test_step_standard_bf16(nsm, wl_name):
    Step(nsm, synth.workload(wl_name), "standard_bf16").check(tol_delta=TOL_DELTA_BF16)


def test_orthogonalize_standard_bf16(nsm):
    wl = synth.custom(RAGGED + [(1024, 1024), (768, 3072)], seed=4)
    offsets, g, o = orthogonalize_gpu(nsm, wl, "standard_bf16")
    for i, (r, c) in enumerate(wl.muon_shapes):
        off = int(offsets[i])
        ref = oracle.orthogonalize(g[off:off + r * c].reshape(r, c), "standard_bf16", storage="method")
        compare(o[off:off + r * c].reshape(r, c), ref, TOL_NS, f"ortho/bf16/{(r, c)}", bf16=True)


@pytest.mark.parametrize("method", ["standard", "gram"])
def test_step_tiny(nsm, method):
    Step(nsm, synth.workload("tiny"), method).check()


@pytest.mark.parametrize("method", ["standard", "gram"])
def test_step_ragged(nsm, method):
    Step(nsm, synth.custom(RAGGED, seed=5), method).check()


@pytest.mark.parametrize("method", ["standard", "gram"])
def test_orthogonalize_extreme_aspect_ratios(nsm, method):
    # Rows or columns past 2^16 (257 column tiles of 256, more than 1024 natural 64-wide
    # tiles in a row), the tall transpose included: every tile index and coordinate of the
    # layout and GEMM paths must stay exact.  With K = n of 65600 to 70000 in X X^T, the
    # GPU's fp32 sums and the oracle's float64 sums round to different fp16 values often
    # enough that the two fp16 iterations drift apart (about 1.4% for the standard form,
    # 0.7-0.9% for gram).  Measured against the exact iteration: standard 1.25-1.27% (the
    # oracle 1.23-1.25%), gram 0.60-0.74% (the oracle 0.38-0.44%).  Held here: within
    # 2e-2 of the exact iteration and within twice the oracle's own distance plus 1e-3.
    shapes = [(130, 65600), (65600, 130), (260, 70000)]
    wl = synth.custom(shapes, seed=19)
    offsets, g, o = orthogonalize_gpu(nsm, wl, method)
    for i, (r, c) in enumerate(shapes):
        off = int(offsets[i])
        gi = g[off:off + r * c].reshape(r, c)
        got = o[off:off + r * c].reshape(r, c)
        ref = oracle.orthogonalize(gi, method, 5, storage="method")
        exact = oracle.orthogonalize(gi, method, 5)
        name = f"ortho/extreme/{method}/{(r, c)}"
        parity_log.record(name + "/vs_exact", rel=rel(got, exact), tol=rel(ref, exact))
        assert rel(got, exact) <= min(TOL_NS, 2 * rel(ref, exact) + 1e-3), (name, rel(got, exact), rel(ref, exact))
        compare(got, ref, TOL_NS, name)


# Direct matrices whose width is a multiple of 64 (slot stride = width) take flat
# 4096-element runs in the layout and apply passes; other direct matrices keep 64 x 64
# tiles, and tall ones the transposing tiles.  200x192 ends in a partial run; 256x1000 is
# 8-aligned (vector accesses) but on tiles.
FLAT = [(200, 192), (136, 4096), (4096, 136), (256, 1000), (192, 320), (1000, 256)]


@pytest.mark.parametrize("method", ["standard", "gram"])
def test_step_flat_runs(nsm, method):
    Step(nsm, synth.custom(FLAT, seed=71), method).check()


def test_orthogonalize_flat_runs(nsm):
    # the export of O to the natural layout takes the same runs and tiles
    wl = synth.custom(FLAT, seed=73)
    offsets, g, o = orthogonalize_gpu(nsm, wl, "gram")
    for i, (r, c) in enumerate(wl.muon_shapes):
        off = int(offsets[i])
        ref = oracle.orthogonalize(g[off:off + r * c].reshape(r, c), "gram", storage="method")
        compare(o[off:off + r * c].reshape(r, c), ref, TOL_NS, f"ortho/flat/{(r, c)}")


@pytest.mark.parametrize("method", ["standard", "gram"])
def test_step_layer1024(nsm, method):
    Step(nsm, synth.workload("layer1024"), method).check()


@pytest.mark.parametrize("method", ["standard", "gram"])
def test_step_gpt2small_one_per_shape(nsm, method):
    wl = synth.workload("gpt2small")
    s = Step(nsm, wl, method)
    s.check(indices=[0, 1, 2, 3, 45, 46, 47])


@pytest.mark.parametrize("nesterov", [True, False])
@pytest.mark.parametrize("steps", [1, 2, 3])
def test_step_variants(nsm, nesterov, steps):
    wl = synth.custom([(256, 384), (384, 256), (128, 128)], seed=11)
    for method in ("standard", "gram"):
        Step(nsm, wl, method, steps=steps, nesterov=nesterov).check()


def test_step_zero_grads_with_momentum(nsm):
    # matrices whose gradient is zero still decay, and move along their momentum
    wl = synth.custom([(128, 256), (256, 128), (192, 64)], seed=2)
    _, total = nsm.pack(wl.muon_shapes)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(99)
    m_init = 0.01 * torch.randn(total, generator=gen, device="cuda")
    for method in ("standard", "gram"):
        s = Step(nsm, wl, method, momentum_init=m_init, zero_grads=(0, 2))
        s.check()


def test_step_all_zero(nsm):
    # G = 0 and M = 0: U = 0, the orthogonalised update is 0, only the decay acts
    wl = synth.custom([(128, 256), (64, 64)], seed=0)
    for method in ("standard", "gram"):
        s = Step(nsm, wl, method, zero_grads=(0, 1))
        lr, wd = wl.lr, wl.wd
        np.testing.assert_allclose(s.p1, s.p0 * np.float32(1 - np.float32(lr) * np.float32(wd)),
                                   rtol=1e-6, atol=0)
        assert np.all(s.m1 == 0)


def test_packed_equals_per_matrix_bitwise(nsm):
    shapes = [(128, 256), (256, 128), (96, 320), (128, 256)]
    wl = synth.custom(shapes, seed=21)
    for method in ("standard", "gram"):
        packed = Step(nsm, wl, method)
        for i, sh in enumerate(shapes):
            offs, total = nsm.pack([sh])
            grads = torch.from_numpy(packed.matrix(packed.g, i).reshape(-1)).to("cuda", torch.bfloat16)
            params = torch.from_numpy(packed.matrix(packed.p0, i).reshape(-1)).to("cuda", torch.float32)
            mom = torch.zeros_like(params)
            ws = torch.empty(nsm.workspace_bytes([sh], method), dtype=torch.uint8, device="cuda")
            nsm.muon_step(grads, params, mom, offs, [sh], wl.lr, wl.wd, wl.mu, method, 5, True, ws)
            torch.cuda.synchronize()
            assert np.array_equal(params.double().cpu().numpy(), packed.matrix(packed.p1, i).reshape(-1)), i


def test_deterministic_bitwise(nsm):
    wl = synth.workload("layer1024")
    for method in ("standard", "gram"):
        a = Step(nsm, wl, method)
        b = Step(nsm, wl, method)
        assert np.array_equal(a.p1, b.p1) and np.array_equal(a.m1, b.m1)


def test_two_steps_accumulate_momentum(nsm):
    # second step with a new gradient: the momentum path through two calls
    wl = synth.custom([(256, 512), (512, 256)], seed=7)
    offsets, total = nsm.pack(wl.muon_shapes)
    dev = "cuda"
    grads = torch.zeros(total, dtype=torch.bfloat16, device=dev)
    params = torch.zeros(total, dtype=torch.float32, device=dev)
    mom = torch.zeros(total, dtype=torch.float32, device=dev)
    synth.fill_packed_params(wl, offsets, params)
    ws = torch.empty(nsm.workspace_bytes(wl.muon_shapes, "gram"), dtype=torch.uint8, device=dev)
    p = [params.double().cpu().numpy()]
    m = [mom.double().cpu().numpy()]
    g = []
    for k in range(2):
        synth.fill_packed_grads(wl, offsets, grads, seed_offset=k)
        g.append(grads.double().cpu().numpy())
        nsm.muon_step(grads, params, mom, offsets, wl.muon_shapes, wl.lr, wl.wd, wl.mu, "gram", 5,
                      True, ws)
        torch.cuda.synchronize()
        p.append(params.double().cpu().numpy())
        m.append(mom.double().cpu().numpy())
    for i, (r, c) in enumerate(wl.muon_shapes):
        o = int(offsets[i])
        sl = slice(o, o + r * c)
        pr, mr = p[0][sl].reshape(r, c), m[0][sl].reshape(r, c)
        for k in range(2):
            (pr,), (mr,), _ = oracle.muon_step([g[k][sl].reshape(r, c)], [pr], [mr], wl.lr, wl.wd,
                                               wl.mu, "gram", storage="method")
        assert rel(m[2][sl].reshape(r, c), mr) <= TOL_FP32
        compare(p[2][sl].reshape(r, c) - p[0][sl].reshape(r, c), pr - p[0][sl].reshape(r, c), TOL_DELTA,
                f"step/two_steps/{(r, c)}")


# ------------------------------------------------------------------ AdamW

@pytest.mark.parametrize("numel", [1, 7, 8, 1000, 1000003])
def test_adamw(nsm, numel):
    gen = torch.Generator(device="cuda")
    gen.manual_seed(numel)
    g = (0.01 * torch.randn(numel, generator=gen, device="cuda")).to(torch.bfloat16)
    p = 0.02 * torch.randn(numel, generator=gen, device="cuda")
    m = 1e-3 * torch.randn(numel, generator=gen, device="cuda")
    v = 1e-5 * torch.rand(numel, generator=gen, device="cuda")
    host = [t.double().cpu().numpy() for t in (g, p, m, v)]
    for step in (1, 2, 10):
        nsm.adamw_step(g, p, m, v, 3e-4, 0.9, 0.95, 1e-8, 0.1, step)
        torch.cuda.synchronize()
        pr, mr, vr = oracle.adamw_step(host[0], host[1], host[2], host[3], 3e-4, 0.9, 0.95, 1e-8,
                                       0.1, step)
        host = [host[0], pr, mr, vr]
        assert rel(p.double().cpu().numpy(), pr) <= TOL_FP32
        assert rel(m.double().cpu().numpy(), mr) <= TOL_FP32
        assert rel(v.double().cpu().numpy(), vr) <= TOL_FP32


def test_adamw_group_of_workload(nsm):
    wl = synth.workload("gpt2small")
    g, p = synth.make_adam_group(wl, "cuda")
    n = p.numel()
    m = torch.zeros(n, device="cuda")
    v = torch.zeros(n, device="cuda")
    p0 = p.double().cpu().numpy()
    nsm.adamw_step(g, p, m, v, 3e-4, 0.9, 0.95, 1e-10, wl.wd, 1)
    torch.cuda.synchronize()
    pr, mr, vr = oracle.adamw_step(g.double().cpu().numpy(), p0, np.zeros(n), np.zeros(n), 3e-4,
                                   0.9, 0.95, 1e-10, wl.wd, 1)
    assert rel(p.double().cpu().numpy() - p0, pr - p0) <= TOL_FP32 * 10
    assert rel(m.double().cpu().numpy(), mr) <= TOL_FP32


# ------------------------------------------------------------------ boundary on a GPU

def test_errors_launch_nothing(nsm):
    wl = synth.workload("tiny")
    offsets, total = nsm.pack(wl.muon_shapes)
    g = torch.zeros(total, dtype=torch.bfloat16, device="cuda")
    p = torch.zeros(total, device="cuda")
    m = torch.zeros(total, device="cuda")
    small = torch.empty(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(nsm.NsmError) as e:
        nsm.muon_step(g, p, m, offsets, wl.muon_shapes, workspace=small)
    assert e.value.code == nsm.NSM_ERR_WORKSPACE
    with pytest.raises(nsm.NsmError) as e:
        nsm.muon_step(g, p, p, offsets, wl.muon_shapes, workspace=small)
    assert e.value.code == nsm.NSM_ERR_ARG
    torch.cuda.synchronize()
    assert nsm.device_status() == nsm.NSM_OK


def test_step_bf16_copy(nsm):
    # the bf16 copy is the round-to-nearest-even bf16 of the updated fp32 parameters, and
    # writing it changes nothing else (grouped launches and the small-matrix kernel)
    wl = synth.custom([(256, 384), (384, 256), (130, 260), (64, 192), (300, 100), (128, 128), (7, 1),
                       (200, 192)], seed=13)
    offsets, total = nsm.pack(wl.muon_shapes)
    dev = "cuda"
    grads = torch.zeros(total, dtype=torch.bfloat16, device=dev)
    synth.fill_packed_grads(wl, offsets, grads)
    p_a = torch.zeros(total, dtype=torch.float32, device=dev)
    synth.fill_packed_params(wl, offsets, p_a)
    p_b = p_a.clone()
    m_a = torch.zeros(total, device=dev)
    m_b = torch.zeros(total, device=dev)
    copy = torch.full((total,), float("nan"), dtype=torch.bfloat16, device=dev)
    for method in ("gram", "standard"):
        ws = torch.empty(nsm.workspace_bytes(wl.muon_shapes, method), dtype=torch.uint8, device=dev)
        nsm.muon_step(grads, p_a, m_a, offsets, wl.muon_shapes, wl.lr, wl.wd, wl.mu, method, 5, True, ws)
        nsm.muon_step(grads, p_b, m_b, offsets, wl.muon_shapes, wl.lr, wl.wd, wl.mu, method, 5, True, ws,
                      params_bf16=copy)
        torch.cuda.synchronize()
        assert torch.equal(p_a, p_b) and torch.equal(m_a, m_b)
        inside = torch.zeros(total, dtype=torch.bool, device=dev)
        for i, (r, c) in enumerate(wl.muon_shapes):
            o = int(offsets[i])
            assert torch.equal(copy[o:o + r * c], p_b[o:o + r * c].to(torch.bfloat16))
            inside[o:o + r * c] = True
        # nothing written between the matrices (the packing's padding)
        assert torch.isnan(copy[~inside].float()).all()
        assert (p_b[~inside] == 0).all() and (m_b[~inside] == 0).all()


@pytest.mark.parametrize("table", ["tiny", "pair"])
@pytest.mark.parametrize("method", ["gram", "standard"])
def test_step_replays_in_cuda_graph(nsm, method, table):
    # After a first call has built the plan, muon_step launches only kernels on the given
    # stream: a CUDA graph of it replays bit-identically to direct calls (the remedy for
    # launch-bound small tables).  "tiny" runs the small-matrix kernel, "pair" the grouped
    # launches on the 2-SM kernel with upper-tile iterates.
    wl = synth.workload("tiny") if table == "tiny" else synth.custom(PAIR_TABLE, seed=41, name="pair")
    offsets, total = nsm.pack(wl.muon_shapes)
    dev = "cuda"
    grads = torch.zeros(total, dtype=torch.bfloat16, device=dev)
    synth.fill_packed_grads(wl, offsets, grads)
    p0 = torch.zeros(total, device=dev)
    synth.fill_packed_params(wl, offsets, p0)
    ws = torch.empty(nsm.workspace_bytes(wl.muon_shapes, method), dtype=torch.uint8, device=dev)

    def run(p, m, stream=None):
        nsm.muon_step(grads, p, m, offsets, wl.muon_shapes, wl.lr, wl.wd, wl.mu, method, 5, True, ws,
                      stream)

    p_direct, m_direct = p0.clone(), torch.zeros(total, device=dev)
    for _ in range(3):
        run(p_direct, m_direct)
    p_graph, m_graph = p0.clone(), torch.zeros(total, device=dev)
    warm_p, warm_m = p0.clone(), torch.zeros(total, device=dev)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        run(warm_p, warm_m, s)  # builds and caches the plan outside capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run(p_graph, m_graph, torch.cuda.current_stream())
    p_graph.copy_(p0)
    m_graph.zero_()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert nsm.device_status() == nsm.NSM_OK
    assert torch.equal(p_graph, p_direct) and torch.equal(m_graph, m_direct)


def test_expired_wait_is_reported_and_context_survives(nsm):
    # a bounded in-kernel wait on a barrier nothing completes runs out after 20 ms,
    # records the timeout in the status word and returns: the status read reports it
    # once, and the same context still computes a correct step
    import time
    assert nsm.device_status() == nsm.NSM_OK
    t0 = time.perf_counter()
    nsm.status_selftest(20000)
    assert nsm.device_status() == nsm.NSM_ERR_TIMEOUT
    assert time.perf_counter() - t0 >= 0.02
    assert nsm.device_status() == nsm.NSM_OK
    # the detailed read names the kernel and the barrier that gave up
    nsm.status_selftest(1000)
    assert nsm.device_status_detail() == (nsm.NSM_ERR_TIMEOUT, nsm.NSM_KERNEL_SELFTEST, 0, nsm.NSM_SITE_SELFTEST)
    assert nsm.device_status_detail() == (nsm.NSM_OK, 0, 0, 0)
    Step(nsm, synth.workload("tiny"), "gram").check()


def test_checkpoint_resume_bitwise(nsm):
    # the step's whole state is the fp32 params and momentum (plus the caller's step
    # count): saving them mid-run and resuming gives bit-identical later steps
    wl = synth.custom([(256, 384), (384, 256), (128, 128)], seed=23)
    offsets, total = nsm.pack(wl.muon_shapes)
    dev = "cuda"
    grads = torch.zeros(total, dtype=torch.bfloat16, device=dev)
    p = torch.zeros(total, device=dev)
    synth.fill_packed_params(wl, offsets, p)
    m = torch.zeros(total, device=dev)
    ws = torch.empty(nsm.workspace_bytes(wl.muon_shapes, "gram"), dtype=torch.uint8, device=dev)

    def step(k, p, m):
        synth.fill_packed_grads(wl, offsets, grads, seed_offset=k)
        nsm.muon_step(grads, p, m, offsets, wl.muon_shapes, wl.lr, wl.wd, wl.mu, "gram", 5, True, ws)

    for k in range(2):
        step(k, p, m)
    saved = {"p": p.cpu().clone(), "m": m.cpu().clone()}
    for k in range(2, 4):
        step(k, p, m)
    p2, m2 = saved["p"].to(dev), saved["m"].to(dev)
    for k in range(2, 4):
        step(k, p2, m2)
    torch.cuda.synchronize()
    assert torch.equal(p, p2) and torch.equal(m, m2)


@pytest.mark.parametrize("method", ["gram", "standard"])
def test_degenerate_and_extreme_shapes(nsm, method):
    shapes = [(1, 1), (7, 1), (1, 8), (256, 262144)]
    wl = synth.custom(shapes, seed=29, lowrank=False)
    s = Step(nsm, wl, method)
    s.check()


def _two_steps_each_form(nsm, wl=None):
    if wl is None:
        wl = synth.custom([(256, 384), (384, 256), (130, 260), (96, 96)], seed=31)
    offsets, total = nsm.pack(wl.muon_shapes)
    out = {}
    for method in ("gram", "standard", "standard_bf16"):
        grads = torch.zeros(total, dtype=torch.bfloat16, device="cuda")
        synth.fill_packed_grads(wl, offsets, grads)
        p = torch.zeros(total, device="cuda")
        synth.fill_packed_params(wl, offsets, p)
        m = torch.zeros(total, device="cuda")
        copy = torch.zeros(total, dtype=torch.bfloat16, device="cuda")
        ws = torch.empty(nsm.workspace_bytes(wl.muon_shapes, method), dtype=torch.uint8, device="cuda")
        for _ in range(2):
            nsm.muon_step(grads, p, m, offsets, wl.muon_shapes, wl.lr, wl.wd, wl.mu, method, 5, True, ws,
                          params_bf16=copy)
        assert nsm.device_status() == nsm.NSM_OK
        out[method] = (p.cpu(), m.cpu(), copy.cpu())
    return out


def test_overlapped_launches_match_plain_order_bitwise(nsm):
    # With the PDL option every kernel is launched with programmatic stream serialisation
    # (each waits for the previous grid before touching its outputs): the same bits
    default = nsm.get_option(nsm.OPT_PDL)
    nsm.set_option(nsm.OPT_PDL, 0)
    try:
        plain = _two_steps_each_form(nsm)
        nsm.set_option(nsm.OPT_PDL, 1)
        overlapped = _two_steps_each_form(nsm)
    finally:
        nsm.set_option(nsm.OPT_PDL, default)
    for method in plain:
        for a, b in zip(overlapped[method], plain[method]):
            assert torch.equal(a, b), method


def test_one_cta_kernel_matches_pair_kernel_bitwise(nsm):
    # The option that keeps every grouped launch on the 1-CTA kernel gives the same bits:
    # both kernels sum each output element over K in the same order of 16-wide MMAs
    assert nsm.get_option(nsm.OPT_PAIR_KERNELS) == 1
    pair = _two_steps_each_form(nsm)
    nsm.set_option(nsm.OPT_PAIR_KERNELS, 0)
    try:
        single = _two_steps_each_form(nsm)
    finally:
        nsm.set_option(nsm.OPT_PAIR_KERNELS, 1)
    for method in pair:
        for a, b in zip(single[method], pair[method]):
            assert torch.equal(a, b), method


# tables on which every grouped launch takes the 2-SM kernel (every order >= 256,
# ragged orders, and the narrow last tiles of order 1408)
PAIR_TABLE = [(256, 384), (384, 256), (300, 520), (520, 300), (1408, 2048), (700, 700)]


def _stored_iterates(nsm, shapes, method, store_whole):
    from test_gpu_fullsize import _iterates_symmetric
    wl = synth.custom(shapes, seed=83)
    offsets, total = nsm.pack(shapes)
    grads = torch.zeros(total, dtype=torch.bfloat16, device="cuda")
    synth.fill_packed_grads(wl, offsets, grads)
    params = torch.zeros(total, device="cuda")
    mom = torch.zeros(total, device="cuda")
    ws = torch.full((nsm.workspace_bytes(shapes, method),), 255, dtype=torch.uint8, device="cuda")
    if store_whole:
        nsm.set_option(nsm.OPT_SYM_STORAGE, 0)
    try:
        nsm.muon_step(grads, params, mom, offsets, shapes, wl.lr, wl.wd, wl.mu, method, 5, True, ws)
    finally:
        nsm.set_option(nsm.OPT_SYM_STORAGE, 1)
    assert nsm.device_status() == nsm.NSM_OK
    _iterates_symmetric(nsm, shapes, method, ws, upper_tiles=not store_whole)


@pytest.mark.parametrize("method", ["gram", "standard", "standard_bf16"])
def test_stored_iterates_exactly_symmetric(nsm, method):
    # Every m x m iterate of the chain (A, B; R, H, Q, T) is a polynomial in X X^T, and
    # the engine computes only its upper-triangle tiles and mirrors them: what it stores
    # must be symmetric bit for bit, for ragged orders too.  The workspace starts as NaN,
    # so a block the chain never wrote shows as untouched rather than as symmetric.  This
    # table mixes orders below 256, so its launches run on the 1-CTA kernel and store whole
    # iterates; PAIR_TABLE with whole storage forced covers the 2-SM kernel's mirror.
    _stored_iterates(nsm, [(130, 260), (257, 129), (200, 200), (300, 520), (520, 300), (96, 500)], method,
                     store_whole=False)
    _stored_iterates(nsm, PAIR_TABLE, method, store_whole=True)


@pytest.mark.parametrize("method", ["gram", "standard", "standard_bf16"])
def test_upper_tile_storage_layout(nsm, method):
    # With every launch on the 2-SM kernel the iterates are kept as their upper 256 x 256
    # tiles: those are finite, the diagonal tiles exactly symmetric, and no tile below the
    # diagonal is ever written (it keeps the NaN the workspace started with).
    _stored_iterates(nsm, PAIR_TABLE, method, store_whole=False)


def test_upper_tile_storage_matches_whole_storage_bitwise(nsm):
    # A product reads a block below the diagonal of an operand from its mirror image above
    # it (an MN-major operand): the same values in the same order of 16-wide MMAs, so the
    # same bits as with whole iterates, for every form.
    wl = synth.custom(PAIR_TABLE, seed=37)
    assert nsm.get_option(nsm.OPT_SYM_STORAGE) == 1
    upper = _two_steps_each_form(nsm, wl)
    nsm.set_option(nsm.OPT_SYM_STORAGE, 0)
    try:
        whole = _two_steps_each_form(nsm, wl)
    finally:
        nsm.set_option(nsm.OPT_SYM_STORAGE, 1)
    for method in upper:
        for a, b in zip(upper[method], whole[method]):
            assert torch.equal(a, b), method


@pytest.mark.parametrize("steps", [1, 2, 3, 4, 5, 7])
def test_grouped_gram_chain_runs_one_launch_per_product_of_the_oracle(nsm, steps):
    # The library's gram chain and the oracle's take the same re-anchoring schedule:
    # one grouped GEMM launch per product the oracle's chain forms (flops_gram counts
    # 2 m^2 n per product with X and 2 m^3 per square product, so at m = n = 1 it is
    # twice the number of products), and the same executed work in flops.
    wl = synth.custom([(256, 512), (512, 256)], seed=71, name="pair")
    nsm.timing_reset()
    nsm.timing_enable(True)
    try:
        Step(nsm, wl, "gram", steps=steps)
        torch.cuda.synchronize()
        _, n_gemm, _ = nsm.timing_read(nsm.KIND_GEMM)
    finally:
        nsm.timing_enable(False)
    assert n_gemm == oracle.flops_gram(1, 1, steps) // 2
