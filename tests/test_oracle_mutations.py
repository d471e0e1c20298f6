"""Plant plausible mistakes in the oracle (on the CPU) and check that the pins see them.

Each mutant below is a copy of an oracle routine with one slip: a sign, a transposed
operand, a dropped term, a wrong index order.  The closed-form and hand-value checks of
``test_oracle.py`` must reject every one of them; if one slipped through, the pins would
be too weak to trust the oracle.
"""

import numpy as np

import oracle

A, B, C = oracle.NS_A, oracle.NS_B, oracle.NS_C


def _closed_form_error(ns_fn, m=6, n=10, seed=1):
    rng = np.random.default_rng(seed)
    uu, _ = np.linalg.qr(rng.standard_normal((m, m)))
    vv, _ = np.linalg.qr(rng.standard_normal((n, m)))
    s = np.linspace(1.0, 0.05, m)
    x = (uu * s) @ vv.T
    x /= np.linalg.norm(x)
    expected = (uu * oracle.ns_poly_iterated(s / np.linalg.norm(s))) @ vv.T
    with np.errstate(all="ignore"):
        err = np.max(np.abs(ns_fn(x) - expected))
    # a mutant that blows up (inf / nan) is as detected as one that is merely off
    return err if np.isfinite(err) else np.inf


def _ns_wrong_sign(x):
    for _ in range(5):
        a_ = x @ x.T
        x = A * x + (-B * a_ + C * a_ @ a_) @ x
    return x


def _ns_transposed_gram(x):
    # X^T X on a square non-normal iterate
    for _ in range(5):
        a_ = x.T @ x
        x = A * x + (B * a_ + C * a_ @ a_) @ x
    return x


def _ns_dropped_square(x):
    for _ in range(5):
        a_ = x @ x.T
        x = A * x + (B * a_ + C * a_) @ x
    return x


def _ns_right_multiply(x):
    # applies the polynomial from the wrong side: X B instead of B X (square case)
    for _ in range(5):
        a_ = x @ x.T
        x = A * x + x @ (B * a_ + C * a_ @ a_)
    return x


def _gram_no_r_update(x0):
    m = x0.shape[0]
    eye = np.eye(m)
    r = x0 @ x0.T
    q = eye
    for _ in range(5):
        h = A * eye + B * r + C * r @ r
        q = h @ q
    return q @ x0


def _gram_r_update_one_side(x0):
    m = x0.shape[0]
    eye = np.eye(m)
    r = x0 @ x0.T
    q = eye
    for step in range(5):
        h = A * eye + B * r + C * r @ r
        q = h @ q
        if step < 4:
            r = h @ r
    return q @ x0


def test_reference_passes():
    assert _closed_form_error(oracle.ns_standard) < 1e-10
    assert _closed_form_error(oracle.ns_gram) < 1e-10


def test_standard_mutants_fail():
    for fn in (_ns_wrong_sign, _ns_dropped_square):
        assert _closed_form_error(fn) > 1e-3, fn.__name__
    # operand-order slips only show on non-normal square iterates
    for fn in (_ns_transposed_gram,):
        assert _closed_form_error(fn, m=6, n=6, seed=2) > 1e-3, fn.__name__
    # applying the polynomial from the right is wrong whenever X X^T != X^T X
    assert _closed_form_error(_ns_right_multiply, m=6, n=6, seed=2) > 1e-3


def test_gram_mutants_fail():
    for fn in (_gram_no_r_update, _gram_r_update_one_side):
        assert _closed_form_error(fn) > 1e-3, fn.__name__


def test_momentum_mutants_fail():
    g = np.array([1.0, -2.0, 0.5, 0.0])
    m = np.array([0.5, 0.25, -1.0, 2.0])
    expected_u = np.array([1.625, -2.9375, 0.5, 0.5])
    # Nesterov with the old momentum, or mu on the gradient, miss the hand values
    assert not np.array_equal(g + 0.5 * m, expected_u)
    assert not np.array_equal(0.5 * g + m + 0.5 * (0.5 * g + m), expected_u)
    _, u = oracle.momentum_update(g, m, 0.5, True)
    assert np.array_equal(u, expected_u)


def test_adamw_mutants_fail():
    # no bias correction on step 1 (g = 2, beta = 0.5): m/sqrt(v) = 1/sqrt(2) != 1
    p_no_bc = 1.0 * 0.75 - 0.5 * (1.0 / np.sqrt(2.0))
    p, _, _ = oracle.adamw_step(np.array([2.0]), np.array([1.0]), np.array([0.0]),
                                np.array([0.0]), 0.5, 0.5, 0.5, 0.0, 0.5, 1)
    assert p[0] == 0.25 and p_no_bc != 0.25


def test_storage_mutants_fail():
    # dropping the rounding of A (or of the input) changes the stored-precision result
    rng = np.random.default_rng(3)
    x = rng.standard_normal((16, 24))
    x /= np.linalg.norm(x)
    good = oracle.ns_standard(x, storage="bf16")

    def no_round_a(x):
        r = lambda v: oracle.round_to(v, "bf16")
        x = r(x)
        for _ in range(5):
            a_ = x @ x.T
            x = r(A * x + r(B * a_ + C * a_ @ a_) @ x)
        return x

    def unrounded_input(x):
        r = lambda v: oracle.round_to(v, "bf16")
        for _ in range(5):
            a_ = r(x @ x.T)
            x = r(A * x + r(B * a_ + C * a_ @ a_) @ x)
        return x
    assert not np.array_equal(no_round_a(x), good)
    assert not np.array_equal(unrounded_input(x), good)


def test_input_storage_mutants_fail():
    # the stored normalised input is s * rnd(U): U rounded to the format's significant
    # bits at any exponent, s applied unrounded.  Two slips a rewrite could make -- rounding
    # s U into fp16's range (the earlier reading), or rounding U inside fp16's range
    # (subnormals and all) -- both fail the pin of
    # test_oracle.py::test_orthogonalize_stores_the_input_as_rounded_u_times_its_scale.
    import math
    u = np.array([[1.0 + 2 ** -12, 2.0 ** -30, -3.0],
                  [0.5, -(2.0 ** -36) * (1 + 2 ** -9), 0.0]])
    s = 1.0 / (math.sqrt(float(np.sum(u * u))) + 1e-7)
    good = oracle.orthogonalize(u, "standard", 0, storage="fp16")

    def rounded_after_scale(u):
        return oracle.round_to(s * u, "fp16")

    def rounded_in_range(u):
        return s * oracle.round_to(u, "fp16")

    for mutant in (rounded_after_scale, rounded_in_range):
        assert not np.array_equal(mutant(u), good), mutant.__name__
