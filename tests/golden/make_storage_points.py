"""Writes storage_points.json: a 3x5 Newton-Schulz case worked in exact arithmetic.

The oracle's storage mode rounds every matrix the method stores to fp16: the standard
form stores X, A = X X^T and B = b A + c A A; the gram form stores R, H, Q, T, the
re-anchored X and the result ("DeepSpeed 集成 Muon 优化器实战" §核心算子 gives the two
forms and their half precision; the rounding points are the reading written in the
oracle's docstrings).  This script computes the same steps independently of the oracle
and of numpy: Python fractions hold every value exactly, and each stored value is rounded
to the nearest fp16 number (ties to even) by its own exact routine.  It writes the input,
the expected results for 1-2 standard steps and 1-4 gram steps (re-anchored every 3
steps, so the fourth covers a re-anchoring), and, for every case, the
results with one rounding point dropped or one extra rounding point added; the input is
chosen (first seed that works) so that every one of those variants differs from the
expected result, so a test that demands the expected bits pins the placement.

Run from the repository root:  python tests/golden/make_storage_points.py
"""

import json
import os
import random
from fractions import Fraction

# quintic coefficients, as the float64 values of the printed decimals
A_ = Fraction(3.4445)
B_ = Fraction(-4.7750)
C_ = Fraction(2.0315)


def round_fp16(q):
    """Nearest fp16 value to the rational q (ties to even); beyond 65504 -> overflow."""
    if q == 0:
        return Fraction(0)
    sign = -1 if q < 0 else 1
    a = abs(q)
    e = 0
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, -14)                      # subnormals share the spacing of the smallest binade
    ulp = Fraction(2) ** (e - 10)        # 11 significant bits
    t = a / ulp
    n = t.numerator // t.denominator     # floor
    rem = t - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    r = n * ulp
    if r > 65504:
        raise OverflowError("fp16 overflow")
    return sign * r


def matmul(x, y):
    return [[sum(x[i][k] * y[k][j] for k in range(len(y))) for j in range(len(y[0]))] for i in range(len(x))]


def transpose(x):
    return [list(r) for r in zip(*x)]


def lin(*terms):
    """sum of coef * matrix."""
    rows, cols = len(terms[0][1]), len(terms[0][1][0])
    return [[sum(c * m[i][j] for c, m in terms) for j in range(cols)] for i in range(rows)]


def eye(m):
    return [[Fraction(int(i == j)) for j in range(m)] for i in range(m)]


class Store:
    """Rounds stored matrices; `drop` = index of the stored matrix left unrounded,
    `extra` = an additional rounding point by name."""

    def __init__(self, drop=None, extra=None):
        self.drop, self.extra, self.count = drop, extra, 0

    def __call__(self, x):
        k = self.count
        self.count += 1
        if k == self.drop:
            return x
        return [[round_fp16(v) for v in row] for row in x]

    def maybe(self, name, x):
        return [[round_fp16(v) for v in row] for row in x] if name == self.extra else x


def standard(x, steps, st):
    x = st(x)
    for _ in range(steps):
        a = st(matmul(x, transpose(x)))
        aa = st.maybe("AA", matmul(a, a))
        b = st(lin((B_, a), (C_, aa)))
        bx = st.maybe("BX", matmul(b, x))
        x = st(lin((A_, x), (Fraction(1), bx)))
    return x


# gram form: R is re-anchored from the explicit iterate every EVERY steps
EVERY = 3


def gram(x, steps, st, every=EVERY):
    x = st(x)
    m = len(x)
    r = st(matmul(x, transpose(x)))
    q = None
    for step in range(1, steps + 1):
        rr = st.maybe("RR", matmul(r, r))
        h = st(lin((A_, eye(m)), (B_, r), (C_, rr)))
        q = h if q is None else st(matmul(h, q))
        if step < steps:
            if every and step % every == 0:
                x = st(matmul(q, x))
                q = None
                r = st(matmul(x, transpose(x)))
            else:
                t = st(matmul(h, r))
                r = st(matmul(t, h))
    if q is None:
        return x
    return st(matmul(q, x))


CASES = [("standard", 1), ("standard", 2), ("gram", 1), ("gram", 2), ("gram", 3), ("gram", 4)]
# extra rounding points a slip could add: A A or B X rounded before they are combined
# (standard), R R rounded before H is formed (gram)
EXTRAS = {"standard": ["AA", "BX"], "gram": ["RR"]}
ROWS, COLS = 3, 5  # the smallest shape found whose every rounding point shows in the result


def run(method, steps, x, drop=None, extra=None):
    st = Store(drop, extra)
    out = (standard if method == "standard" else gram)(x, steps, st)
    return out, st.count


def hexs(x):
    return [[float(v).hex() for v in row] for row in x]


def try_seed(seed):
    rnd = random.Random(seed)
    scale = 2.0 / (ROWS * COLS) ** 0.5  # Frobenius norm about 0.7, as after normalisation
    x = [[round_fp16(Fraction(rnd.uniform(-0.6, 0.6) * scale)) for _ in range(COLS)] for _ in range(ROWS)]
    cases = []
    for method, steps in CASES:
        want, npoints = run(method, steps, x)
        dropped = []
        for k in range(1, npoints):  # point 0 is the input, already an fp16 value
            got, _ = run(method, steps, x, drop=k)
            if got == want:
                return None
            dropped.append(hexs(got))
        added = {}
        for name in EXTRAS[method]:
            got, _ = run(method, steps, x, extra=name)
            if got == want:
                return None
            added[name] = hexs(got)
        cases.append({"method": method, "steps": steps, "rounding_points": npoints,
                      "expected": hexs(want), "dropped": dropped, "added": added})
    return x, cases


def main():
    for seed in range(1000):
        found = try_seed(seed)
        if found:
            break
    else:
        raise SystemExit("no seed makes every rounding point visible")
    x, cases = found
    doc = {
        "_source": ("Written by tests/golden/make_storage_points.py (exact rational arithmetic, "
                    "its own fp16 rounding; no numpy, no oracle).  The Newton-Schulz steps and "
                    "coefficients are those of \"DeepSpeed 集成 Muon 优化器实战\" §核心算子; the "
                    "rounding points are the storage-precision reading of the oracle."),
        "seed": seed,
        "gram_restart_every": EVERY,
        "x": hexs(x),
        "cases": cases,
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "storage_points.json")
    with open(path, "w") as f:
        json.dump(doc, f, indent=1)
    print(path, "seed", seed)


if __name__ == "__main__":
    main()
