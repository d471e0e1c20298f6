"""Pins of the float64 oracle against facts fixed outside the oracle itself.

Each test checks the oracle against one of: values the pages print (tests/golden/),
hand-derived arithmetic on exactly representable inputs, the closed form of
Newton-Schulz on a matrix with a known SVD, brute-force pure-Python loops on tiny
shapes, algebraic identities (gram form == standard form), or special cases.
No expected value here comes from the CUDA path.
"""

import json
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        return json.load(f)


# ---------------------------------------------------------------- constants (pages)

def test_coefficients_match_pages():
    g = _golden("pages_constants.json")
    c = g["ns_coefficients"]
    assert (oracle.NS_A, oracle.NS_B, oracle.NS_C) == (c["a"], c["b"], c["c"])
    assert oracle.NS_STEPS == c["steps"]
    assert set(oracle.NS_METHODS) == set(g["ns_methods"]["methods"])
    assert oracle.muon_ref.NS_METHOD_DEFAULT == g["ns_methods"]["default"]
    d = g["muon_defaults"]
    assert oracle.muon_ref.MUON_LR_DEFAULT == d["lr"]
    assert oracle.muon_ref.MUON_MOMENTUM_DEFAULT == d["momentum"]
    a = g["adam_defaults"]
    assert oracle.muon_ref.ADAM_LR_DEFAULT == a["lr"]
    assert list(oracle.muon_ref.ADAM_BETAS_DEFAULT) == a["betas"]
    assert oracle.muon_ref.ADAM_EPS_DEFAULT == a["eps"]


# ---------------------------------------------------------------- routing

def test_routing_cases_from_prose():
    cases = _golden("routing_cases.json")["cases"]
    for name, ndim, expected, why in cases:
        assert oracle.route(name, ndim) is expected, (name, ndim, why)


def test_matrix_view_shape():
    assert oracle.matrix_view_shape((6, 4)) == (6, 4)
    assert oracle.matrix_view_shape((8, 3, 3, 2)) == (8, 18)
    with pytest.raises(ValueError):
        oracle.matrix_view_shape((5,))


# ---------------------------------------------------------------- packing (hand values)

def test_pack_offsets_by_hand():
    # 2x3 = 6 elements at 0, next start rounds 6 up to 64; 4x4 = 16 at 64 ends at 80 ->
    # 128; 1x65 at 128 ends at 193 -> total rounds to 256.
    offs, total = oracle.pack_offsets([(2, 3), (4, 4), (1, 65)], align=64)
    assert offs == [0, 64, 128] and total == 256
    offs, total = oracle.pack_offsets([(2, 3), (4, 4), (1, 65)], align=1)
    assert offs == [0, 6, 22] and total == 87
    offs, total = oracle.pack_offsets([(8, 8)], align=64)
    assert offs == [0] and total == 64
    with pytest.raises(ValueError):
        oracle.pack_offsets([(0, 3)])


# ---------------------------------------------------------------- momentum (hand values)

def test_momentum_by_hand():
    g = np.array([1.0, -2.0, 0.5, 0.0])
    m = np.array([0.5, 0.25, -1.0, 2.0])
    mu = 0.5
    # M_new = mu*M + G = [1.25, -1.875, 0.0, 1.0]
    # Nesterov U = G + mu*M_new = [1.625, -2.9375, 0.5, 0.5]; plain U = M_new
    m_new, u = oracle.momentum_update(g, m, mu, nesterov=True)
    assert np.array_equal(m_new, [1.25, -1.875, 0.0, 1.0])
    assert np.array_equal(u, [1.625, -2.9375, 0.5, 0.5])
    m_new2, u2 = oracle.momentum_update(g, m, mu, nesterov=False)
    assert np.array_equal(m_new2, m_new) and np.array_equal(u2, m_new)


def test_normalize_by_hand():
    u = np.array([[3.0, 0.0], [0.0, 4.0]])
    x = oracle.frobenius_normalize(u, eps=0.0)
    assert np.array_equal(x, u / 5.0)
    x = oracle.frobenius_normalize(np.zeros((2, 2)), eps=1e-7)
    assert np.array_equal(x, np.zeros((2, 2)))


# ---------------------------------------------------------------- scalar polynomial

def test_scalar_polynomial_by_hand():
    # p(1) = a + b + c = 3.4445 - 4.7750 + 2.0315 = 0.701
    assert oracle.ns_poly(1.0) == pytest.approx(0.701, abs=1e-15)
    # p(0.5) = 1.72225 - 0.596875 + 0.063484375 = 1.188859375
    assert oracle.ns_poly(0.5) == pytest.approx(1.188859375, abs=1e-15)
    assert oracle.ns_poly(0.0) == 0.0
    xs = np.linspace(-1, 1, 11)
    assert np.allclose(oracle.ns_poly(-xs), -oracle.ns_poly(xs))
    # composition: p5(1) = p(p(p(p(0.701))))
    y = 1.0
    for _ in range(5):
        y = 3.4445 * y - 4.7750 * y ** 3 + 2.0315 * y ** 5
    assert oracle.ns_poly_iterated(1.0) == pytest.approx(y, abs=1e-15)


def test_iterated_polynomial_band():
    # Singular values in [0.01, 1] land in a band around 1 after five steps: the
    # iteration's purpose (orthogonalisation up to a bounded spread).
    xs = np.linspace(0.01, 1.0, 2000)
    ys = oracle.ns_poly_iterated(xs)
    assert ys.min() > 0.68 and ys.max() < 1.14


# ---------------------------------------------------------------- NS closed form via SVD

def _known_svd(m, n, sigmas, seed):
    rng = np.random.default_rng(seed)
    uu, _ = np.linalg.qr(rng.standard_normal((m, m)))
    vv, _ = np.linalg.qr(rng.standard_normal((n, m)))
    return uu, np.asarray(sigmas, dtype=np.float64), vv


@pytest.mark.parametrize("method", ["standard", "gram"])
@pytest.mark.parametrize("m,n", [(4, 4), (5, 9), (16, 40), (32, 32)])
def test_ns_closed_form(method, m, n):
    # For X = U diag(s) V^T every step maps singular values through p and keeps the
    # singular vectors; so NS(X) = U diag(p^5(s)) V^T.
    rng = np.random.default_rng(m * 100 + n)
    sig = np.sort(rng.uniform(0.02, 1.0, m))[::-1] * np.logspace(0, -2, m)
    uu, s, vv = _known_svd(m, n, sig, seed=m + n)
    x = (uu * s) @ vv.T
    x = x / np.linalg.norm(x)  # singular values now s/||s||
    s_n = s / np.linalg.norm(s)
    expected = (uu * oracle.ns_poly_iterated(s_n)) @ vv.T
    got = oracle.newton_schulz(x, method)
    assert np.max(np.abs(got - expected)) < 1e-10


@pytest.mark.parametrize("method", ["standard", "gram"])
def test_orthogonalize_closed_form_with_norm(method):
    # orthogonalize divides by ||U||_F + eps before iterating.
    m, n = 6, 10
    uu, s, vv = _known_svd(m, n, [5.0, 3.0, 2.0, 1.0, 0.5, 0.01], seed=7)
    g = (uu * s) @ vv.T
    expected = (uu * oracle.ns_poly_iterated(s / (np.linalg.norm(s) + 1e-7))) @ vv.T
    assert np.max(np.abs(oracle.orthogonalize(g, method) - expected)) < 1e-10
    # tall input takes the transposed path and comes back in the input's shape
    got_t = oracle.orthogonalize(g.T, method)
    assert got_t.shape == (n, m)
    assert np.max(np.abs(got_t - expected.T)) < 1e-10


def test_transpose_rule_is_strict():
    # square: no transpose; mathematically NS(X) == NS(X^T)^T for square X too, so
    # check the rule through shapes of a wide and a tall case instead.
    rng = np.random.default_rng(3)
    wide = rng.standard_normal((3, 7))
    tall = wide.T.copy()
    ow = oracle.orthogonalize(wide, "standard")
    ot = oracle.orthogonalize(tall, "standard")
    assert np.max(np.abs(ot - ow.T)) < 1e-12


# ---------------------------------------------------------------- special cases

@pytest.mark.parametrize("method", ["standard", "gram"])
def test_zero_gradient(method):
    o = oracle.orthogonalize(np.zeros((4, 8)), method)
    assert np.array_equal(o, np.zeros((4, 8)))


@pytest.mark.parametrize("method", ["standard", "gram"])
def test_rank_one(method):
    rng = np.random.default_rng(11)
    u = rng.standard_normal(5)
    v = rng.standard_normal(9)
    u /= np.linalg.norm(u)
    v /= np.linalg.norm(v)
    sigma = 3.7
    g = sigma * np.outer(u, v)
    expected = oracle.ns_poly_iterated(sigma / (sigma + 1e-7)) * np.outer(u, v)
    assert np.max(np.abs(oracle.orthogonalize(g, method) - expected)) < 1e-12


@pytest.mark.parametrize("method", ["standard", "gram"])
def test_orthonormal_rows(method):
    rng = np.random.default_rng(5)
    q, _ = np.linalg.qr(rng.standard_normal((12, 4)))
    rows = q.T  # 4 x 12 with orthonormal rows
    scale = 2.5
    g = scale * rows
    # ||g||_F = scale*sqrt(4): every singular value of X is scale/(2*scale + eps)
    s = scale / (scale * 2.0 + 1e-7)
    expected = oracle.ns_poly_iterated(s) * rows
    assert np.max(np.abs(oracle.orthogonalize(g, method) - expected)) < 1e-12


# ---------------------------------------------------------------- gram == standard

@pytest.mark.parametrize("m,n", [(8, 8), (8, 64), (24, 40), (1, 5)])
def test_gram_equals_standard(m, n):
    rng = np.random.default_rng(m * 7 + n)
    x = rng.standard_normal((m, n))
    x /= np.linalg.norm(x)
    a = oracle.ns_standard(x)
    b = oracle.ns_gram(x)
    assert np.max(np.abs(a - b)) < 1e-10


@pytest.mark.parametrize("steps", [1, 2, 3, 7])
def test_gram_equals_standard_other_step_counts(steps):
    rng = np.random.default_rng(steps)
    x = rng.standard_normal((6, 13))
    x /= np.linalg.norm(x)
    assert np.max(np.abs(oracle.ns_standard(x, steps) - oracle.ns_gram(x, steps))) < 1e-10


# ---------------------------------------------------------------- brute force loops

def _mm(a, b):
    n, k, m = len(a), len(b), len(b[0])
    return [[sum(a[i][t] * b[t][j] for t in range(k)) for j in range(m)] for i in range(n)]


def _tr(a):
    return [list(r) for r in zip(*a)]


def _brute_ns(x, steps, a, b, c):
    for _ in range(steps):
        aa = _mm(x, _tr(x))
        aa2 = _mm(aa, aa)
        bb = [[b * aa[i][j] + c * aa2[i][j] for j in range(len(aa))] for i in range(len(aa))]
        bx = _mm(bb, x)
        x = [[a * x[i][j] + bx[i][j] for j in range(len(x[0]))] for i in range(len(x))]
    return x


@pytest.mark.parametrize("shape", [(2, 3), (3, 5), (4, 4), (5, 2), (1, 4)])
def test_brute_force_tiny(shape):
    rng = np.random.default_rng(sum(shape))
    g = rng.standard_normal(shape)
    rows, cols = shape
    x = g.T if rows > cols else g
    nrm = math.sqrt(sum(v * v for row in x.tolist() for v in row))
    xl = [[v / (nrm + 1e-7) for v in row] for row in x.tolist()]
    o = np.array(_brute_ns(xl, 5, 3.4445, -4.7750, 2.0315))
    if rows > cols:
        o = o.T
    for method in ("standard", "gram"):
        assert np.max(np.abs(oracle.orthogonalize(g, method) - o)) < 1e-12


# ---------------------------------------------------------------- apply (hand values)

def test_apply_by_hand():
    p = np.array([[1.0, -2.0, 0.5, 4.0]])           # 1 x 4: scale sqrt(max(1, 1/4)) = 1
    o = np.array([[0.5, 0.25, -1.0, 0.0]])
    lr, wd = 0.5, 0.5                                # p*(1 - 0.25) - 0.5*o
    expected = np.array([[0.5, -1.625, 0.875, 3.0]])
    assert np.array_equal(oracle.apply_update(p, o, lr, wd), expected)
    # 4 x 1: scale sqrt(4) = 2 -> p*0.75 - 1.0*o
    expected_t = np.array([[0.25], [-1.75], [1.375], [3.0]])
    assert np.array_equal(oracle.apply_update(p.T, o.T, lr, wd), expected_t)
    assert oracle.update_scale(9, 4) == 1.5
    assert oracle.update_scale(4, 9) == 1.0


def test_muon_step_closed_form_row_vector():
    # one 1x4 gradient [3,0,4,0], M=0, mu=0.5, Nesterov: M_new = g, U = 1.5 g,
    # ||U|| = 7.5, X has the single singular value 7.5/(7.5+eps) with right vector g/5.
    g = np.array([[3.0, 0.0, 4.0, 0.0]])
    p = np.array([[1.0, 1.0, 1.0, 1.0]])
    m = np.zeros((1, 4))
    lr, wd = 0.1, 0.2
    s = oracle.ns_poly_iterated(7.5 / (7.5 + 1e-7))
    o = s * g / 5.0
    for method in ("standard", "gram"):
        (pn,), (mn,), (on,) = oracle.muon_step([g], [p], [m], lr, wd, mu=0.5, method=method)
        assert np.array_equal(mn, g)
        assert np.max(np.abs(on - o)) < 1e-14
        assert np.max(np.abs(pn - (p * (1 - lr * wd) - lr * o))) < 1e-14
        # tall version: scale 2 and the result is the transpose
        (pt,), _, (ot,) = oracle.muon_step([g.T], [p.T], [m.T], lr, wd, mu=0.5, method=method)
        assert np.max(np.abs(ot - o.T)) < 1e-14
        assert np.max(np.abs(pt - (p.T * (1 - lr * wd) - lr * 2.0 * o.T))) < 1e-14


# ---------------------------------------------------------------- AdamW (hand values)

def test_adamw_two_steps_by_hand():
    lr, b1, b2, eps, wd = 0.5, 0.5, 0.5, 0.0, 0.5
    p, m, v = np.array([1.0]), np.array([0.0]), np.array([0.0])
    # step 1, g = 2: m = 1, v = 2; m_hat = 2, v_hat = 4; step = 2/2 = 1
    # p = 1*(1 - 0.25) - 0.5*1 = 0.25
    p, m, v = oracle.adamw_step(np.array([2.0]), p, m, v, lr, b1, b2, eps, wd, 1)
    assert (p[0], m[0], v[0]) == (0.25, 1.0, 2.0)
    # step 2, g = -2: m = 0.5 - 1 = -0.5, v = 1 + 2 = 3; m_hat = -0.5/0.75 = -2/3,
    # v_hat = 3/0.75 = 4; step = (-2/3)/2 = -1/3; p = 0.25*0.75 + 0.5/3
    p, m, v = oracle.adamw_step(np.array([-2.0]), p, m, v, lr, b1, b2, eps, wd, 2)
    assert m[0] == -0.5 and v[0] == 3.0
    assert p[0] == pytest.approx(0.1875 + 0.5 / 3.0, abs=1e-15)


def test_adamw_eps_outside_sqrt():
    # with v = 0 the step is m_hat / eps exactly (eps outside the square root)
    p, m, v = oracle.adamw_step(np.array([0.0]), np.array([0.0]), np.array([1.0]),
                                np.array([0.0]), 1.0, 0.5, 0.5, 0.25, 0.0, 1)
    # m = 0.5, m_hat = 1, v_hat = 0 -> step = 1/0.25 = 4
    assert p[0] == -4.0


# ---------------------------------------------------------------- bf16 decode, flops

def test_bf16_decode():
    bits = np.array([0x3F80, 0xBF80, 0x4049, 0x0000, 0x7F80], dtype=np.uint16)
    vals = oracle.bf16_bits_to_f64(bits)
    assert vals[0] == 1.0 and vals[1] == -1.0 and vals[3] == 0.0 and np.isinf(vals[4])
    assert vals[2] == 3.140625


def _count_macs_standard(m, n, steps):
    macs = 0
    for _ in range(steps):
        macs += m * m * n        # X X^T
        macs += m * m * m        # A A
        macs += m * m * n        # B X
    return 2 * macs


def test_flop_counts():
    for m, n in [(2, 3), (128, 4096), (4096, 11008)]:
        assert oracle.flops_standard(m, n) == _count_macs_standard(m, n, 5)
    # gram, 5 steps, never re-anchored: R0 and Q X0 (m^2 n MACs each); R R x5; H Q x4;
    # H R H = 2 per step x4
    m, n = 7, 11
    assert oracle.flops_gram(m, n, restart_every=0) == 2 * (2 * m * m * n + (5 + 4 + 8) * m ** 3)
    # re-anchored after step 3 (the default): products with X are R0, Q X and X X^T,
    # and the final Q X = 4; squares: step1 R R, T, R; step2 R R, H Q, T, R; step3 R R,
    # H Q; step4 R R, T, R; step5 R R, H Q = 14
    assert oracle.GRAM_RESTART_EVERY == 3
    assert oracle.flops_gram(m, n) == 2 * (4 * m * m * n + 14 * m ** 3)
    # re-anchored after steps 2 and 4: products with X are R0, (Q X, X X^T) twice and the
    # final Q X = 6; squares: step1 R R, T, R; step2 R R, H Q; step3 R R, T, R;
    # step4 R R, H Q; step5 R R = 11
    assert oracle.flops_gram(m, n, restart_every=2) == 2 * (6 * m * m * n + 11 * m ** 3)
    assert oracle.flops_gram(m, n, steps=1) == 2 * (2 * m * m * n + 1 * m ** 3)


def _mac_count_gram(m, n, steps, restart_every):
    """Counts MACs by running the gram iteration on shape placeholders."""
    macs = m * m * n  # R0
    q_identity = True
    for step in range(1, steps + 1):
        macs += m ** 3
        if not q_identity:
            macs += m ** 3
        q_identity = False
        if step < steps:
            if restart_every and step % restart_every == 0:
                macs += 2 * m * m * n
                q_identity = True
            else:
                macs += 2 * m ** 3
    if not q_identity:
        macs += m * m * n
    return 2 * macs


def test_flop_counts_gram_schedules():
    for steps in range(0, 8):
        for every in (0, 1, 2, 3):
            if steps == 0:
                assert oracle.flops_gram(9, 13, steps, every) == 0
            else:
                assert oracle.flops_gram(9, 13, steps, every) == _mac_count_gram(9, 13, steps, every)


# ---------------------------------------------------------------- storage rounding

def test_round_to_ties_by_hand():
    # bf16 keeps 8 significant bits: neighbours of 1 are 1 and 1 + 2^-7
    assert oracle.round_to(1 + 2 ** -8, "bf16") == 1.0             # tie -> even
    assert oracle.round_to(1 + 3 * 2 ** -8, "bf16") == 1 + 2 ** -6  # tie -> even
    assert oracle.round_to(1 + 2 ** -8 + 2 ** -20, "bf16") == 1 + 2 ** -7
    # fp16 keeps 11 significant bits, largest finite 65504, subnormal spacing 2^-24
    assert oracle.round_to(1 + 2 ** -11, "fp16") == 1.0
    assert oracle.round_to(65504.0, "fp16") == 65504.0
    assert np.isinf(oracle.round_to(65520.0, "fp16"))              # ties away to inf
    assert oracle.round_to(3 * 2 ** -25, "fp16") == 2 ** -23       # subnormal tie -> even
    assert oracle.round_to(2 ** -26, "fp16") == 0.0
    assert oracle.round_to(-0.0, "bf16") == 0.0


def test_round_to_matches_library_conversions():
    import torch
    rng = np.random.default_rng(0)
    # float32 inputs (exact in float64), spanning normal, subnormal and overflow ranges
    for scale in (1.0, 1e-3, 1e-30, 1e-39, 1e30, 1e38):
        x32 = (rng.standard_normal(20000) * scale).astype(np.float32)
        x = x32.astype(np.float64)
        bf = torch.from_numpy(x32).to(torch.bfloat16).double().numpy()
        assert np.array_equal(oracle.round_to(x, "bf16"), bf), scale
        f16 = x32.astype(np.float16).astype(np.float64)
        assert np.array_equal(oracle.round_to(x, "fp16"), f16), scale


def test_round_significand_by_hand():
    # the format's significant bits, at any exponent: no subnormal spacing, no overflow
    for e in (-60, -30, 0, 20, 70):
        two = 2.0 ** e
        assert oracle.round_significand(two * (1 + 2 ** -11), "fp16") == two            # tie -> even
        assert oracle.round_significand(two * (1 + 3 * 2 ** -11), "fp16") == two * (1 + 2 ** -9)
        assert oracle.round_significand(two * (1 + 2 ** -8), "bf16") == two             # tie -> even
        assert oracle.round_significand(-two * (1 + 2 ** -8 + 2 ** -20), "bf16") == -two * (1 + 2 ** -7)
    assert oracle.round_significand(65520.0, "fp16") == 65536.0   # halfway to 2^16, no overflow
    assert oracle.round_significand(3 * 2 ** -40, "fp16") == 3 * 2 ** -40
    assert oracle.round_significand(0.0, "fp16") == 0.0


def test_round_significand_is_power_of_two_scaled_library_rounding():
    import torch
    rng = np.random.default_rng(3)
    for scale in (1e-30, 1e-3, 1.0, 1e4, 1e30):
        x32 = (rng.standard_normal(20000) * scale).astype(np.float32)
        x = x32.astype(np.float64)
        # a power of two that puts the largest magnitude in [2^11, 2^12): the library's
        # fp16 rounding of 2^k x, scaled back, wherever 2^k x is a normal fp16 number
        _, e = np.frexp(np.max(np.abs(x)))
        k = 12 - int(e)
        y = np.ldexp(x, k)
        normal = np.abs(y) >= 2.0 ** -14
        f16 = np.ldexp(y.astype(np.float16).astype(np.float64), -k)
        got = oracle.round_significand(x, "fp16")
        assert np.array_equal(got[normal], f16[normal]), scale
        assert normal.mean() > 0.999
        bf = np.ldexp(torch.from_numpy(y.astype(np.float32)).to(torch.bfloat16).double().numpy(), -k)
        assert np.array_equal(oracle.round_significand(x, "bf16"), bf), scale


def test_orthogonalize_stores_the_input_as_rounded_u_times_its_scale():
    # with no Newton-Schulz step the result is the stored input itself: U rounded to
    # fp16's 11 significant bits, times s = 1/(||U||_F + eps) of the unrounded U.  Entries
    # far below fp16's normal range after normalisation keep their 11 bits.
    u = np.array([[1.0 + 2 ** -12, 2.0 ** -30, -3.0],
                  [0.5, -(2.0 ** -36) * (1 + 2 ** -9), 0.0]])
    s = 1.0 / (math.sqrt(float(np.sum(u * u))) + 1e-7)
    want = s * np.array([[1.0, 2.0 ** -30, -3.0],
                         [0.5, -(2.0 ** -36) * (1 + 2 ** -9), 0.0]])
    got = oracle.orthogonalize(u, "standard", 0, storage="fp16")
    assert np.array_equal(got, want)
    # the entry of magnitude 2^-30 s (about 1e-9) is below fp16's smallest subnormal:
    # rounding after the scale would have flushed it
    assert got[0, 1] != 0 and oracle.round_to(s * u[0, 1], "fp16") == 0.0
    # tall matrices are stored transposed, then transposed back
    assert np.array_equal(oracle.orthogonalize(u.T, "gram", 0, storage="fp16"), want.T)


@pytest.mark.parametrize("method", ["standard", "gram", "standard_bf16"])
def test_storage_mode_invariant_under_power_of_two_scale(method):
    # eps = 0: s scales inversely with U, and rounding U to its significand commutes with
    # a power of two, so the stored iteration gives the same bits at any magnitude
    rng = np.random.default_rng(5)
    u = rng.standard_normal((6, 11))
    want = oracle.orthogonalize(u, method, eps=0.0, storage="method")
    for j in (-70, -20, 15, 60):
        assert np.array_equal(oracle.orthogonalize(np.ldexp(u, j), method, eps=0.0, storage="method"), want), j


def test_method_storage_formats():
    assert oracle.method_storage("standard") == "fp16"
    assert oracle.method_storage("gram") == "fp16"
    assert oracle.method_storage("standard_bf16") == "bf16"
    # the bf16 variant is the same mathematical iteration
    rng = np.random.default_rng(2)
    g = rng.standard_normal((5, 8))
    assert np.array_equal(oracle.orthogonalize(g, "standard_bf16"), oracle.orthogonalize(g, "standard"))


@pytest.mark.parametrize("every", [0, 1, 2, 3])
@pytest.mark.parametrize("steps", [1, 2, 5, 6])
def test_gram_reanchoring_is_exact_noop(every, steps):
    rng = np.random.default_rng(steps * 10 + every)
    x = rng.standard_normal((12, 31))
    x /= np.linalg.norm(x)
    assert np.max(np.abs(oracle.ns_gram(x, steps, restart_every=every) -
                         oracle.ns_standard(x, steps))) < 1e-10


@pytest.mark.parametrize("method", ["standard", "gram", "standard_bf16"])
def test_storage_mode_close_on_well_conditioned_input(method):
    # singular values of X in [0.2, 0.6]: the iteration is not in its steep region, so
    # half-precision storage stays within a few units of its rounding of the exact map
    m, n = 24, 40
    uu, s, vv = _known_svd(m, n, np.linspace(1.0, 0.35, m), seed=4)
    g = (uu * s) @ vv.T
    exact = oracle.orthogonalize(g, method)
    stored = oracle.orthogonalize(g, method, storage="method")
    err = np.linalg.norm(stored - exact) / np.linalg.norm(exact)
    assert 0 < err < 2e-2
    # the result is a value of the storage format
    fmt = oracle.method_storage(method)
    assert np.array_equal(oracle.round_to(stored, fmt), stored)


def test_storage_mode_none_is_exact():
    rng = np.random.default_rng(8)
    g = rng.standard_normal((6, 9))
    for method in ("standard", "gram"):
        assert np.array_equal(oracle.orthogonalize(g, method, storage=None),
                              oracle.orthogonalize(g, method))


# ---------------------------------------------------------------- page arithmetic

def test_page_memory_arithmetic():
    g = _golden("pages_constants.json")
    mem = g["memory_per_param_bytes"]
    w = mem["world"]
    assert 2 + 2 + 4 + 4 + 4 == mem["no_shard"]
    assert 2 + 2 + (4 + 4 + 4) / w == mem["zero1"]
    assert 2 + (2 + 4 + 4 + 4) / w == mem["zero2"]
    assert (2 + 2 + 4 + 4 + 4) / w == mem["zero3"]
    d = g["dmuon_z2_example"]
    assert d["params_muon"] * d["bytes_per_elem"] / d["shards"] / 1e6 == d["per_rank_mb"]


# ---------------------------------------------------------------- storage-point placement
#
# tests/golden/storage_points.json holds a 3x5 case worked in exact rational arithmetic
# with its own fp16 rounding (tests/golden/make_storage_points.py: no numpy, no oracle):
# the expected fp16 results of 1-2 standard steps and 1-4 gram steps (re-anchored every 3
# steps: the fourth covers a re-anchoring), and the results with any one rounding point dropped or one plausible
# extra rounding point added, each of which differs from the expected one.  The oracle
# must give the expected bits, round exactly as many times, and change its result when
# any one of its own rounding points is skipped.

def _hexmat(rows):
    return np.array([[float.fromhex(v) for v in r] for r in rows])


_SP = _golden("storage_points.json")


def test_storage_points_use_the_oracles_reanchoring_interval():
    assert _SP["gram_restart_every"] == oracle.GRAM_RESTART_EVERY


def _ns_fp16(method, x, steps):
    if method == "standard":
        return oracle.ns_standard(x, steps, storage="fp16")
    return oracle.ns_gram(x, steps, storage="fp16")


@pytest.mark.parametrize("case", _SP["cases"], ids=lambda c: f"{c['method']}{c['steps']}")
def test_storage_points_give_the_worked_bits(case):
    x = _hexmat(_SP["x"])
    want = _hexmat(case["expected"])
    assert np.array_equal(_ns_fp16(case["method"], x, case["steps"]), want)
    for alt in case["dropped"] + list(case["added"].values()):
        assert not np.array_equal(_hexmat(alt), want)


@pytest.mark.parametrize("case", _SP["cases"], ids=lambda c: f"{c['method']}{c['steps']}")
def test_storage_points_count_and_each_matters(case, monkeypatch):
    x = _hexmat(_SP["x"])
    want = _hexmat(case["expected"])
    from oracle import muon_ref
    real_store = muon_ref._store
    calls = {"n": 0, "skip": None}

    def counting_store(v, storage):
        k = calls["n"]
        calls["n"] += 1
        if storage is not None and k == calls["skip"]:
            return np.asarray(v, dtype=np.float64)
        return real_store(v, storage)

    monkeypatch.setattr(muon_ref, "_store", counting_store)
    _ns_fp16(case["method"], x, case["steps"])
    assert calls["n"] == case["rounding_points"]
    for k in range(1, case["rounding_points"]):
        calls["n"], calls["skip"] = 0, k
        assert not np.array_equal(_ns_fp16(case["method"], x, case["steps"]), want), k
