"""The exponent rule of the step's stored input, on the host (nsm_input_exponent).

The kernels store a matrix's normalised input as U 2^k rounded once to the storage
format and apply the same function (in_exponent) to choose and accept k.  These tests
hold it to its definition, checked in float64 with numpy's frexp/ldexp, on the CPU:
- without a hint, max|U| 2^k lies in [2^11, 2^12);
- with a hint, the stored values stand exactly when max|U| 2^hint lies in [2^4, 2^15),
  otherwise k is the exponent above and the matrix is stored again;
- the next hint is always that exponent;
- zero, infinite and NaN maxima yield no exponent (the hint stands), and exponents are
  clamped to [-120, 120] so that 2^k and 2^-k stay normal floats.
"""

import math

import numpy as np
import pytest

import newton_schulz_orthogonalized_gb300 as nsm

CLAMP = 120


@pytest.fixture(scope="module")
def lib():
    return nsm.lib()


def target_k(m):
    """The exponent that puts m 2^k in [2^11, 2^12), clamped."""
    _, e = math.frexp(m)
    return max(-CLAMP, min(CLAMP, 12 - e))


def test_without_hint_puts_the_largest_entry_in_range(lib):
    rng = np.random.default_rng(1)
    for m in np.float32(10.0) ** rng.uniform(-30, 30, size=2000).astype(np.float32):
        m = float(np.float32(m))
        k, nxt, store = nsm.input_exponent(m)
        assert store and nxt == k == target_k(m), (m, k)
        assert 2.0 ** 11 <= math.ldexp(m, k) < 2.0 ** 12, (m, k)


def test_with_hint_the_stored_values_stand_exactly_inside_the_accepted_range(lib):
    rng = np.random.default_rng(2)
    ms = np.float32(10.0) ** rng.uniform(-20, 20, size=400).astype(np.float32)
    for m in ms:
        m = float(np.float32(m))
        for hint in rng.integers(-80, 80, size=8):
            hint = int(hint)
            k, nxt, store = nsm.input_exponent(m, hint)
            scaled = math.ldexp(m, hint)
            accepted = 2.0 ** 4 <= scaled < 2.0 ** 15
            assert store == (not accepted), (m, hint, scaled)
            assert k == (hint if accepted else target_k(m)), (m, hint, k)
            assert nxt == target_k(m)


def test_range_edges(lib):
    # for max|U| = f 2^e the accepted hints are those with 5 <= e + hint <= 15
    for m, e in ((1.0, 1), (0.75, 0), (65504.0, 16), (2.0 ** -40, -39)):
        assert math.frexp(m)[1] == e
        assert nsm.input_exponent(m, 5 - e) == (5 - e, target_k(m), False)     # m 2^hint = 2^4 f'
        assert nsm.input_exponent(m, 4 - e)[2]                                 # below 2^4
        assert nsm.input_exponent(m, 15 - e) == (15 - e, target_k(m), False)   # under 2^15
        assert nsm.input_exponent(m, 16 - e)[2]                                # 2^15 and above
    # exactly 2^4 stands, exactly 2^15 does not
    assert not nsm.input_exponent(2.0 ** 4, 0)[2]
    assert nsm.input_exponent(2.0 ** 15, 0)[2]


def test_no_exponent_from_zero_or_non_finite_maxima(lib):
    for m in (0.0, -0.0, math.inf, math.nan):
        assert nsm.input_exponent(m, 7) == (7, 7, False)
        assert nsm.input_exponent(m, 500) == (CLAMP, CLAMP, False)
        assert nsm.input_exponent(m) == (0, 0, True)


def test_exponents_are_clamped(lib):
    assert nsm.input_exponent(1.0, 2 ** 31 - 1) == (target_k(1.0), target_k(1.0), True)
    assert nsm.input_exponent(1.0, -(2 ** 31)) == (target_k(1.0), target_k(1.0), True)
    # a largest entry near the float range's ends: the exponent stops at the clamp
    assert nsm.input_exponent(float(np.float32(1e-40)))[0] == CLAMP       # subnormal
    assert nsm.input_exponent(float(np.finfo(np.float32).max))[0] == 12 - 128
    assert nsm.input_exponent(float(np.finfo(np.float32).tiny))[0] == CLAMP


def test_null_outputs_refused(lib):
    import ctypes
    k = ctypes.c_int(0)
    assert lib.nsm_input_exponent(1.0, 0, 0, None, ctypes.byref(k), ctypes.byref(k)) == nsm.NSM_ERR_NULL


def test_stored_input_is_the_oracles_rounding_for_every_accepted_exponent(lib):
    # The step stores U as fp16(U 2^k) and multiplies by 2^-k (inside s 2^-k).  For every
    # k the rule accepts, that is the oracle's rnd(U) -- U rounded to fp16's 11
    # significant bits at any exponent -- on every entry within 2^18 of the matrix's
    # largest (numpy's float16 conversion is the rounding here, not the oracle's code);
    # smaller entries may land in fp16's subnormals.  bf16 storage has no such range.
    import torch

    import oracle
    rng = np.random.default_rng(7)
    for scale in (1e-30, 1e-6, 1.0, 3e4, 1e30):
        u = (rng.standard_normal(4096) * scale * np.exp(rng.uniform(-8, 0, size=4096))).astype(np.float32)
        u = u.astype(np.float64)
        m = float(np.max(np.abs(u)))
        want16 = oracle.round_significand(u, "fp16")
        want_bf = oracle.round_significand(u, "bf16")
        k0 = nsm.input_exponent(m)[0]
        accepted = [k for k in range(k0 - 12, k0 + 12) if not nsm.input_exponent(m, k)[2]]
        assert accepted and k0 in accepted, (scale, k0, accepted)
        big = np.abs(u) >= m * 2.0 ** -18
        for k in accepted:
            stored = np.ldexp(np.ldexp(u, k).astype(np.float16).astype(np.float64), -k)
            assert np.all(np.isfinite(stored)), (scale, k)
            assert np.array_equal(stored[big], want16[big]), (scale, k)
            y = torch.from_numpy(np.ldexp(u, k).astype(np.float32)).to(torch.bfloat16).double().numpy()
            assert np.array_equal(np.ldexp(y, -k), want_bf), (scale, k)
