"""The stored input of the chain, U 2^k, and the exponent the step keeps in its workspace.

muon_step stores the normalised input X = s U as U 2^k rounded once to the storage
format, with s 2^-k entering the products that read it.  It knows U's norm and largest
entry only after its pass over G and M, so it stores U with the exponent the previous call
on the same table and workspace chose (the first 4n bytes of the workspace) and stores U
again, in a second pass, only for the matrices where that exponent put max|U| 2^k outside
[2^4, 2^15).  These tests hold the step to what that design promises: the result does
not depend on the exponent bytes (a power of two commutes with the rounding), the bytes
end up holding 12 - e for max|U| = f 2^e (f in [0.5, 1)), and a jump in the gradients'
magnitude is caught and stored again, at parity with the oracle.
"""

import math

import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

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


class Table:
    """One workload's device buffers and a workspace kept from call to call."""

    def __init__(self, nsm, wl, method, steps=5, grad_scale=1.0):
        self.nsm, self.wl, self.method, self.steps = nsm, wl, method, steps
        self.offsets, total = nsm.pack(wl.muon_shapes)
        self.grads = torch.zeros(total, dtype=torch.bfloat16, device="cuda")
        synth.fill_packed_grads(wl, self.offsets, self.grads)
        if grad_scale != 1.0:
            self.grads = (self.grads.float() * grad_scale).to(torch.bfloat16)
        self.params = torch.zeros(total, dtype=torch.float32, device="cuda")
        synth.fill_packed_params(wl, self.offsets, self.params)
        self.mom = torch.zeros(total, dtype=torch.float32, device="cuda")
        self.ws = torch.zeros(nsm.workspace_bytes(wl.muon_shapes, method, steps), dtype=torch.uint8,
                              device="cuda")

    def hints(self):
        n = len(self.wl.muon_shapes)
        return self.ws[:4 * n].view(torch.int32).cpu().numpy().copy()

    def set_hints(self, values):
        n = len(self.wl.muon_shapes)
        self.ws[:4 * n].view(torch.int32).copy_(torch.as_tensor(np.asarray(values, np.int32)))

    def step(self, grads=None):
        nsm, wl = self.nsm, self.wl
        nsm.muon_step(self.grads if grads is None else grads, self.params, self.mom, self.offsets,
                      wl.muon_shapes, wl.lr, wl.wd, wl.mu, self.method, self.steps, True, self.ws)
        assert nsm.device_status() == nsm.NSM_OK

    def matrix(self, arr, i):
        r, c = self.wl.muon_shapes[i]
        o = int(self.offsets[i])
        return arr[o:o + r * c].reshape(r, c)


def frexp_exponent(x):
    return int(np.frexp(np.float64(x))[1])


def expected_hints(t, g, m_new):
    """12 - e for each matrix's max|U| = f 2^e (Nesterov U = G + mu M_new), skipping the
    matrices whose largest |U| lies within float32 rounding of a power of two."""
    out = {}
    for i in range(len(t.wl.muon_shapes)):
        u = t.matrix(g, i) + t.wl.mu * t.matrix(m_new, i)
        mx = float(np.max(np.abs(u)))
        if mx == 0.0:
            continue
        f, e = np.frexp(mx)
        if abs(f - 0.5) < 1e-6 or abs(f - 1.0) < 1e-6:
            continue
        out[i] = 12 - int(e)
    return out


@pytest.mark.parametrize("method", ["gram", "standard", "standard_bf16"])
def test_result_does_not_depend_on_the_exponent_bytes(nsm, method):
    wl = synth.custom([(256, 512), (640, 192), (96, 200), (130, 260), (8, 24)], seed=21)
    n = len(wl.muon_shapes)
    results = []
    rng = np.random.default_rng(3)
    # zeros, garbage, the exponents a step on this table leaves, and those shifted by one
    # (still in range: no second pass for them)
    for fill in ("zeros", "garbage", "steady", "steady+1", "steady-1"):
        t = Table(nsm, wl, method)
        if fill == "garbage":
            t.set_hints(rng.integers(-2 ** 31, 2 ** 31 - 1, size=n, dtype=np.int64).astype(np.int32))
        elif fill.startswith("steady"):
            t.step()                      # leaves this table's exponents in the workspace
            h = t.hints()
            p0 = torch.zeros_like(t.params)
            synth.fill_packed_params(wl, t.offsets, p0)
            t.params.copy_(p0)
            t.mom.zero_()
            t.set_hints(h + (1 if fill == "steady+1" else -1 if fill == "steady-1" else 0))
        t.step()
        results.append((fill, t.params.cpu().numpy(), t.mom.cpu().numpy()))
    _, p_ref, m_ref = results[0]
    for fill, p, m in results[1:]:
        assert np.array_equal(p, p_ref), fill
        assert np.array_equal(m, m_ref), fill


def test_exponent_bytes_after_a_step(nsm):
    wl = synth.custom([(256, 512), (640, 192), (96, 200), (130, 260)], seed=22)
    t = Table(nsm, wl, "gram")
    t.set_hints([77, -77, 3, 0])         # whatever they were, the step leaves 12 - e
    g = t.grads.double().cpu().numpy()
    t.step()
    want = expected_hints(t, g, t.mom.double().cpu().numpy())
    got = t.hints()
    assert want, "no matrix to check"
    for i, k in want.items():
        assert got[i] == k, (i, got[i], k)


@pytest.mark.parametrize("jump", [2.0 ** 20, 2.0 ** -20])
def test_jump_in_gradient_magnitude_is_stored_again(nsm, jump):
    # the first step leaves exponents for gradients of one magnitude; before the second,
    # gradients and momentum are 2^20 times larger (or smaller), so U 2^k with the old
    # exponent would overflow fp16 (or sink into its subnormals): the step must store U
    # again, and match the oracle from the state it started from
    wl = synth.custom([(256, 512), (640, 192), (96, 200)], seed=23)
    shift = int(round(math.log2(jump)))
    for method in ("gram", "standard"):
        t = Table(nsm, wl, method)
        t.step()
        h1 = t.hints()
        g2 = (t.grads.float() * jump).to(torch.bfloat16)   # a power of two: exact
        t.mom.mul_(jump)
        p1 = t.params.double().cpu().numpy()
        m1 = t.mom.double().cpu().numpy()
        g = g2.double().cpu().numpy()
        t.step(g2)
        p2 = t.params.double().cpu().numpy()
        m2 = t.mom.double().cpu().numpy()
        h2 = t.hints()
        want = expected_hints(t, g, m2)
        for i, k in want.items():
            assert h2[i] == k, (method, i, h2[i], k)
            # the old exponent was out of range for the new magnitude
            assert not (5 <= (12 - k) + h1[i] <= 15), (method, i, h1[i], k)
        assert np.all(np.abs(h2 - h1 + shift) <= 2), (h1, h2)
        for i in range(len(wl.muon_shapes)):
            (pn,), (mn,), _ = oracle.muon_step([t.matrix(g, i)], [t.matrix(p1, i)], [t.matrix(m1, i)],
                                               wl.lr, wl.wd, wl.mu, method, 5, True, storage="method")
            assert rel(t.matrix(m2, i), mn) <= TOL_FP32, (method, i)
            e = rel(t.matrix(p2, i) - t.matrix(p1, i), pn - t.matrix(p1, i))
            assert e <= TOL_DELTA, (method, i, e)


@pytest.mark.parametrize("method", ["gram", "standard"])
def test_zero_steps_apply_the_normalised_input(nsm, method):
    # with no Newton-Schulz step the update is the stored input itself, times its factor
    wl = synth.custom([(256, 512), (640, 192), (96, 200), (130, 260)], seed=24)
    t = Table(nsm, wl, method, steps=0)
    p0 = t.params.double().cpu().numpy()
    g = t.grads.double().cpu().numpy()
    t.step()
    p1 = t.params.double().cpu().numpy()
    for i in range(len(wl.muon_shapes)):
        (pn,), _, _ = oracle.muon_step([t.matrix(g, i)], [t.matrix(p0, i)],
                                       [np.zeros_like(t.matrix(p0, i))], wl.lr, wl.wd, wl.mu, method, 0,
                                       True, storage="method")
        # p is stored in fp32: its half-ulp (about 1e-9 at these parameters' size) against an
        # update of about 5e-5 rms bounds what the delta can show, near 2e-5
        e = rel(t.matrix(p1, i) - t.matrix(p0, i), pn - t.matrix(p0, i))
        assert e <= 1e-4, (i, e)


def test_orthogonalize_keeps_entries_far_below_the_largest(nsm):
    # bf16 entries spread over 2^-24 .. 2^0 of the largest: stored as G 2^k, every one is
    # an fp16 number (none below 2^-26 of the largest), so X = s G exactly and, with no
    # step, the export is bf16(s G) up to the one rounding of s G to fp32
    rng = np.random.default_rng(9)
    rows, cols = 64, 256
    mag = np.ldexp(1.0, -rng.integers(0, 25, size=(rows, cols)))
    g = (mag * rng.choice([-1.0, 1.0], size=(rows, cols)) * (1 + rng.integers(0, 128, size=(rows, cols)) / 128))
    g_bf = torch.from_numpy(g.astype(np.float32)).to(torch.bfloat16)
    shapes = [(rows, cols)]
    offsets, total = nsm.pack(shapes)
    inp = torch.zeros(total, dtype=torch.bfloat16, device="cuda")
    inp[:rows * cols] = g_bf.reshape(-1).cuda()
    out = torch.zeros_like(inp)
    ws = torch.empty(nsm.workspace_bytes(shapes, "gram", 0), dtype=torch.uint8, device="cuda")
    nsm.muon_orthogonalize(inp, out, offsets, shapes, "gram", 0, ws)
    assert nsm.device_status() == nsm.NSM_OK
    got = out[:rows * cols].double().cpu().numpy().reshape(rows, cols)
    x = g_bf.double().numpy()
    want = oracle.orthogonalize(x, "gram", 0, storage="fp16")
    # one bf16 rounding of values that went through fp32: equal, or one bf16 ulp apart
    ulp = np.ldexp(1.0, np.frexp(np.abs(want))[1] - 8)
    assert np.all(np.abs(got - want) <= ulp), np.max(np.abs(got - want) / ulp)
    assert np.count_nonzero(got) == np.count_nonzero(x)
