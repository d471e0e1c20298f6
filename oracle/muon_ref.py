"""Float64 CPU oracle of the owner-side Muon step and of the auxiliary AdamW step.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  This module is the independent checker of the
CUDA path.  Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline /
reference legs of ``bench.py`` may import it.  It imports nothing from the product
package and the product package never imports it.

Every routine is plain numpy in float64, written from what the pages state, in the
order the pages give the steps; a library matmul is the only primitive used.  Inputs
that arrive as bf16 are decoded exactly to float64 by the caller before they get here.

Sources (web pages; cited by title and section):

[DSM]  "DeepSpeed 集成 Muon 优化器实战：从正交化原理到 ZeRO 微调配置"
       (dpshk.com news article on DeepSpeed's Muon integration)
[DMZ]  "Z2 与 Z3 模式" (DMuon guide, x-square-robot.github.io/dmuon)
[FSDP] "FSDP-Zero123分片简介" (solus-sano.com)

Readings taken where the pages are silent (each is listed again in the design notes):

* momentum convention: ``M <- mu*M + G``; Nesterov update ``U = G + mu*M_new``;
  plain update ``U = M_new``; no dampening.
* normalisation: ``X = U / (||U||_F + eps)`` with ``eps = 1e-7``, per table entry.
* transpose rule: work on ``U^T`` when ``rows > cols`` (strictly), so that the
  iterate always has ``m = min(rows, cols)`` rows.
* the same (a, b, c) on every Newton-Schulz step.
* gram form: iterate on ``R = X X^T`` and accumulate the left polynomial ``Q``
  (derivation in :func:`ns_gram`), re-anchoring ``R`` from the explicit iterate every
  three steps (exact-arithmetic no-op; keeps the fp16 iteration accurate).
* storage precision: fp16 for both forms (the page calls the standard form stable in
  bf16 and gives fp16 to the gram form for accuracy); "standard_bf16" keeps bf16;
  ``storage="method"`` rounds at exactly the points where the method stores.
* the normalised input in storage precision: ``X = s * rnd(U)``, with ``s = 1/(||U||_F +
  eps)`` and ``rnd`` rounding U to the format's significant bits at any exponent; the
  scalar s multiplies the products that read X, unrounded (:func:`round_significand`).
* update scale ``sqrt(max(1, rows/cols))`` of the original (untransposed) matrix.
* AdamW: the textbook decoupled form with bias correction, eps outside the square
  root, step counter starting at 1.

Parity status: every public function here is pinned by ``tests/test_oracle.py``
against closed forms, hand-derived values, brute force or values the pages print.
"""

from __future__ import annotations

import math
from typing import Iterable, List, Sequence, Tuple

import numpy as np

# --- constants the pages fix -------------------------------------------------------

# [DSM] §核心算子：牛顿-舒尔茨正交化内核 — quintic coefficients of the five-step
# Newton-Schulz iteration, chosen to maximise the slope at zero.
NS_A = 3.4445
NS_B = -4.7750
NS_C = 2.0315
NS_STEPS = 5
# gram form: steps between re-anchorings of R from the explicit iterate (see ns_gram)
GRAM_RESTART_EVERY = 3

# [DSM] §如何用配置启用 — defaults filled in by the hybrid optimizer when the config
# omits them: Muon group lr 0.02, momentum 0.95, ns_method "gram"; Adam group
# lr 3e-4, betas (0.9, 0.95), eps 1e-10.
MUON_LR_DEFAULT = 0.02
MUON_MOMENTUM_DEFAULT = 0.95
NS_METHOD_DEFAULT = "gram"
ADAM_LR_DEFAULT = 3e-4
ADAM_BETAS_DEFAULT = (0.9, 0.95)
ADAM_EPS_DEFAULT = 1e-10

# [DSM] §核心算子 — the two methods the dispatcher accepts.
NS_METHODS = ("standard", "gram")
# The standard form stored in bf16, the precision the page calls stable.
NS_METHOD_VARIANTS = ("standard_bf16",)

# Reading (pages silent): the epsilon added to the Frobenius norm.
NORM_EPS = 1e-7


# --- storage formats -------------------------------------------------------------------
#
# [DSM] §核心算子 describes the precision the method stores its iterates in: the
# five-step iteration is stable in bf16, and the gram variant uses fp16 for better
# half-precision accuracy.  Reading taken: both forms store in fp16 (the normalised
# iterate, X X^T and the quintic's matrices stay within fp16's range, and fp16 carries
# three more significant bits at the same tensor-core rate); the bf16 form of the
# standard iteration is kept as the method "standard_bf16".  With ``storage`` set, the
# routines below round every intermediate the method stores to that format (round to
# nearest, ties to even) and accumulate everything else in float64.  With
# ``storage=None`` they are the exact float64 iteration.

_FORMATS = {
    # significant bits, smallest normal exponent, largest finite value
    "bf16": (8, -126, float.fromhex("0x1.fep127")),
    "fp16": (11, -14, 65504.0),
}


def round_to(x, fmt):
    """Round float64 values to the nearest ``fmt`` value (ties to even), exactly.

    The spacing of ``fmt`` values around ``x`` is ``2**(e - p + 1)`` for
    ``2**e <= |x| < 2**(e+1)`` (``p`` significant bits), never finer than the subnormal
    spacing ``2**(emin - p + 1)``; scaling by a power of two and ``np.rint`` (ties to
    even) are exact in float64.  Values beyond the largest finite one become inf.
    """
    if fmt is None:
        return np.asarray(x, dtype=np.float64)
    p, emin, vmax = _FORMATS[fmt]
    x = np.asarray(x, dtype=np.float64)
    out = np.array(x, dtype=np.float64, copy=True)
    finite = np.isfinite(x) & (x != 0)
    xf = x[finite]
    _, e2 = np.frexp(np.abs(xf))          # |x| = f * 2**e2 with f in [0.5, 1)
    e = np.maximum(e2 - 1, emin)           # exponent of the leading bit, clamped
    ulp = np.ldexp(1.0, (e - (p - 1)).astype(np.int64))
    r = np.rint(xf / ulp) * ulp
    r[np.abs(r) > vmax] = np.inf * np.sign(r[np.abs(r) > vmax])
    out[finite] = r
    return out


def round_significand(x, fmt):
    """Round float64 values to ``fmt``'s significant bits (ties to even) at any exponent.

    This is :func:`round_to` without the format's exponent range: no subnormal spacing,
    no overflow.  It is what storing ``2**k x`` in ``fmt`` and scaling back by ``2**-k``
    gives whenever ``2**k x`` lies in the format's normal range, since a power of two
    commutes with the rounding there.
    """
    if fmt is None:
        return np.asarray(x, dtype=np.float64)
    p = _FORMATS[fmt][0]
    x = np.asarray(x, dtype=np.float64)
    out = np.array(x, dtype=np.float64, copy=True)
    finite = np.isfinite(x) & (x != 0)
    xf = x[finite]
    _, e2 = np.frexp(np.abs(xf))           # |x| = f * 2**e2 with f in [0.5, 1)
    ulp = np.ldexp(1.0, (e2 - p).astype(np.int64))
    out[finite] = np.rint(xf / ulp) * ulp
    return out


def method_storage(method):
    """Storage format of each ns_method: fp16 (standard, gram), bf16 (standard_bf16)."""
    return {"standard": "fp16", "gram": "fp16", "standard_bf16": "bf16"}[method]


def _store(x, storage):
    return x if storage is None else round_to(x, storage)


# --- a0: routing ---------------------------------------------------------------------

def route(name: str, ndim: int) -> bool:
    """True when a parameter goes to the Muon group, False when it goes to AdamW.

    [DSM] §use_muon参数打标：谁是 2D 隐藏权重？ — a parameter is tagged for Muon when it
    has at least two dimensions and its lower-cased name contains neither "embed" nor
    "lm_head"; every other parameter (embeddings, layer norms, biases, lm_head) falls
    back to AdamW.
    """
    lowered = name.lower()
    if ndim < 2:
        return False
    for keyword in ("embed", "lm_head"):
        if keyword in lowered:
            return False
    return True


def matrix_view_shape(shape: Sequence[int]) -> Tuple[int, int]:
    """Rows and columns of the 2D matrix a Muon parameter is treated as.

    [DSM] §use_muon参数打标 states the orthogonalisation needs a 2D weight; for a
    parameter with more than two dimensions the plainest reading keeps the first
    dimension as rows and flattens the rest into columns.
    """
    if len(shape) < 2:
        raise ValueError("a Muon parameter needs at least two dimensions")
    rows = int(shape[0])
    cols = 1
    for d in shape[1:]:
        cols *= int(d)
    return rows, cols


# --- a1: packing ---------------------------------------------------------------------

def pack_offsets(shapes: Sequence[Tuple[int, int]], align: int = 64) -> Tuple[List[int], int]:
    """Element offsets of each matrix inside one contiguous packed buffer.

    [DMZ] §两种packed buffer生命周期 — all Muon-target parameters of one owner are packed
    into one contiguous buffer.  The page fixes no layout; the reading taken: matrices in
    table order, each starting on a multiple of ``align`` elements.  Returns the offsets and
    the total number of elements (the end of the last matrix, rounded up likewise).
    """
    if align <= 0:
        raise ValueError("align must be positive")
    offsets: List[int] = []
    cursor = 0
    for rows, cols in shapes:
        if rows <= 0 or cols <= 0:
            raise ValueError("matrix dimensions must be positive")
        offsets.append(cursor)
        end = cursor + rows * cols
        cursor = ((end + align - 1) // align) * align
    return offsets, cursor


# --- a2: momentum ----------------------------------------------------------------------

def momentum_update(grad: np.ndarray, momentum: np.ndarray, mu: float,
                    nesterov: bool = True) -> Tuple[np.ndarray, np.ndarray]:
    """One momentum step: returns ``(M_new, U)``.

    [DSM] §什么是 Muon 优化器？ — Muon first forms the momentum of the gradient, then
    orthogonalises it; the coefficient 0.95 is the default of §如何用配置启用.  The
    accumulation ``M <- mu*M + G`` and the Nesterov look-ahead ``U = G + mu*M_new`` are
    the readings taken here (the pages do not spell them out).
    """
    grad = np.asarray(grad, dtype=np.float64)
    momentum = np.asarray(momentum, dtype=np.float64)
    m_new = mu * momentum + grad
    if nesterov:
        update = grad + mu * m_new
    else:
        update = m_new
    return m_new, update


# --- a3: normalisation -------------------------------------------------------------

def frobenius_normalize(u: np.ndarray, eps: float = NORM_EPS) -> np.ndarray:
    """``X = U / (||U||_F + eps)`` — puts every singular value of X in [0, 1)."""
    u = np.asarray(u, dtype=np.float64)
    return u / (math.sqrt(float(np.sum(u * u))) + eps)


# --- a4: Newton-Schulz, scalar polynomial ------------------------------------------

def ns_poly(x, a: float = NS_A, b: float = NS_B, c: float = NS_C):
    """The quintic ``p(x) = a x + b x^3 + c x^5`` that one step applies to each
    singular value ([DSM] §核心算子)."""
    x = np.asarray(x, dtype=np.float64)
    return a * x + b * x ** 3 + c * x ** 5


def ns_poly_iterated(x, steps: int = NS_STEPS, a: float = NS_A, b: float = NS_B,
                     c: float = NS_C):
    """``p`` composed ``steps`` times: the map NS applies to singular values."""
    y = np.asarray(x, dtype=np.float64)
    for _ in range(steps):
        y = ns_poly(y, a, b, c)
    return y


# --- a4: Newton-Schulz, standard form -----------------------------------------------

def ns_standard(x: np.ndarray, steps: int = NS_STEPS, a: float = NS_A, b: float = NS_B,
                c: float = NS_C, storage=None, input_stored: bool = False) -> np.ndarray:
    """Standard quintic Newton-Schulz on an already normalised ``m x n`` iterate.

    [DSM] §核心算子 (``zeropower_via_newtonschulz5``): each step forms
    ``A = X X^T``, ``B = b A + c A A`` and replaces ``X`` by ``a X + B X``.  With
    ``storage`` the input (unless ``input_stored``: the caller has stored it already),
    ``A``, ``B`` and every new ``X`` are rounded to that format.
    """
    x = np.array(x, dtype=np.float64)
    if not input_stored:
        x = _store(x, storage)
    for _ in range(steps):
        gram_a = _store(x @ x.T, storage)
        poly_b = _store(b * gram_a + c * (gram_a @ gram_a), storage)
        x = _store(a * x + poly_b @ x, storage)
    return x


# --- a4': Newton-Schulz, gram form ----------------------------------------------------

def ns_gram(x: np.ndarray, steps: int = NS_STEPS, a: float = NS_A, b: float = NS_B,
            c: float = NS_C, storage=None, restart_every: int = GRAM_RESTART_EVERY,
            input_stored: bool = False) -> np.ndarray:
    """Gram-form Newton-Schulz: iterate on the small square ``R = X X^T``.

    [DSM] §核心算子 (``zeropower_via_gram_newtonschulz``) says the variant iterates on
    the Gram matrix ``R = X @ X.T`` to save FLOPs on wide matrices, in fp16.  Reading of
    the steps: every iterate of the standard form is ``X_k = Q_k X_0`` with ``Q_k`` a
    polynomial in ``R_0 = X_0 X_0^T``, hence ``X_k X_k^T = Q_k R_0 Q_k``.  One step with
    ``H = a I + b R + c R R`` sends ``Q -> H Q`` and ``R -> H R H`` (formed as
    ``T = H R``, ``R = T H``); the result is ``Q X``.  The last step needs no ``R``.

    Re-anchoring: every ``restart_every`` steps (when more steps follow) the iterate is
    formed explicitly, ``X <- Q X``, ``Q <- I`` and ``R <- X X^T``.  In exact arithmetic
    this changes nothing (``X X^T = Q R Q``); in fp16 it keeps the small eigenvalues of
    ``R`` from drowning in the rounding of the large ones.  ``restart_every=0`` never
    re-anchors.  With ``storage`` every stored matrix (``X``, ``R``, ``H``, ``Q``,
    ``T``, the result) is rounded to that format.

    The interval is a reading (the page gives none): on the near-low-rank inputs of the
    workloads, fp16 storage with re-anchoring every 3 steps lands as close to the exact
    iteration as every 2 steps (about 1.8-2.0% on shapes from 128 x 4096 to
    4096 x 11008), every 4 steps about 2.5%, and never re-anchoring 10-47%.  Counting
    each symmetric product (``X X^T`` and every square one) at half its cost, since one
    triangle determines it, a five-step chain costs ``3 m^2 (n - m)`` flops less with
    every 3 than with every 2.
    """
    x = np.array(x, dtype=np.float64)
    if not input_stored:
        x = _store(x, storage)
    m = x.shape[0]
    eye = np.eye(m)
    r = _store(x @ x.T, storage)
    q = None  # None stands for the identity
    for step in range(1, steps + 1):
        h = _store(a * eye + b * r + c * (r @ r), storage)
        q = h if q is None else _store(h @ q, storage)
        if step < steps:
            if restart_every and step % restart_every == 0:
                x = _store(q @ x, storage)
                q = None
                r = _store(x @ x.T, storage)
            else:
                t = _store(h @ r, storage)
                r = _store(t @ h, storage)
    return x if q is None else _store(q @ x, storage)


def newton_schulz(x: np.ndarray, method: str = NS_METHOD_DEFAULT, steps: int = NS_STEPS,
                  a: float = NS_A, b: float = NS_B, c: float = NS_C, storage=None,
                  input_stored: bool = False) -> np.ndarray:
    """Dispatch on ``ns_method`` ([DSM] §核心算子: ``NS_METHODS = {standard, gram}``)."""
    if method in ("standard", "standard_bf16"):
        return ns_standard(x, steps, a, b, c, storage, input_stored=input_stored)
    if method == "gram":
        return ns_gram(x, steps, a, b, c, storage, input_stored=input_stored)
    raise ValueError(f"unknown ns_method {method!r}")


def _resolve_storage(storage, method):
    if storage == "method":
        return method_storage(method)
    return storage


def orthogonalize(u: np.ndarray, method: str = NS_METHOD_DEFAULT, steps: int = NS_STEPS,
                  eps: float = NORM_EPS, storage=None) -> np.ndarray:
    """Normalise, transpose when tall, run Newton-Schulz, transpose back.

    Returns ``O`` with the shape of ``u``.  ``storage="method"`` stores the iterates in
    the method's format (:func:`method_storage`); ``None`` is exact.

    In storage precision the normalised input ``X = U / (||U||_F + eps)`` ([DSM]
    §核心算子: the normalisation before the iteration) is held as ``s * rnd(U)``: U
    rounded once to the format's significant bits (:func:`round_significand`) and the
    scalar ``s = 1/(||U||_F + eps)``, of the unrounded U, multiplying it in float64.
    """
    u = np.asarray(u, dtype=np.float64)
    if u.ndim != 2:
        raise ValueError("orthogonalize takes a 2D matrix")
    storage = _resolve_storage(storage, method)
    rows, cols = u.shape
    transposed = rows > cols
    x = u.T if transposed else u
    if storage is None:
        o = newton_schulz(frobenius_normalize(x, eps), method, steps)
    else:
        scale = 1.0 / (math.sqrt(float(np.sum(x * x))) + eps)
        o = newton_schulz(scale * round_significand(x, storage), method, steps, storage=storage,
                          input_stored=True)
    return o.T if transposed else o


# --- a5: decoupled weight decay and apply -------------------------------------------

def update_scale(rows: int, cols: int) -> float:
    """``sqrt(max(1, rows/cols))`` — the shape factor of the applied update."""
    return math.sqrt(max(1.0, rows / cols))


def apply_update(param: np.ndarray, ortho: np.ndarray, lr: float, wd: float) -> np.ndarray:
    """[DSM] §核心算子 (the wrapper's step): ``p.mul_(1 - lr*wd)`` then
    ``p.add_(update, alpha=-lr)``, with the update being the orthogonalised momentum
    times the shape factor.  Both terms use the old ``p``."""
    param = np.asarray(param, dtype=np.float64)
    rows, cols = param.shape
    return param * (1.0 - lr * wd) - lr * update_scale(rows, cols) * np.asarray(ortho, np.float64)


def muon_step(grads: Sequence[np.ndarray], params: Sequence[np.ndarray],
              momenta: Sequence[np.ndarray], lr: float, wd: float,
              mu: float = MUON_MOMENTUM_DEFAULT, method: str = NS_METHOD_DEFAULT,
              steps: int = NS_STEPS, nesterov: bool = True, eps: float = NORM_EPS,
              storage=None):
    """The owner-side Muon step over a list of matrices.

    [DSM] §什么是 Muon 优化器？ — momentum, then Newton-Schulz orthogonalisation of the
    momentum matrix, then the weight update; [DMZ] §两种packed buffer生命周期 — the
    owner runs it once per matrix of its packed buffer.  Returns
    ``(new_params, new_momenta, orthos)`` as float64 arrays.
    """
    new_params, new_momenta, orthos = [], [], []
    for g, p, m in zip(grads, params, momenta):
        m_new, u = momentum_update(g, m, mu, nesterov)
        o = orthogonalize(u, method, steps, eps, storage)
        new_params.append(apply_update(p, o, lr, wd))
        new_momenta.append(m_new)
        orthos.append(o)
    return new_params, new_momenta, orthos


# --- a6: AdamW for the routed-out parameters -----------------------------------------

def adamw_step(grad: np.ndarray, param: np.ndarray, exp_avg: np.ndarray,
               exp_avg_sq: np.ndarray, lr: float, beta1: float, beta2: float,
               eps: float, wd: float, step: int):
    """One decoupled-weight-decay Adam step on a flat group; ``step`` counts from 1.

    [DSM] §混合优化器的参数组构造 — parameters without ``use_muon`` go to the auxiliary
    Adam optimizer, in AdamW mode by default (``ADAM_W_MODE_DEFAULT = True``).  The
    update written here is the textbook AdamW: exponential moving averages of ``g`` and
    ``g^2``, bias correction by ``1 - beta^t``, eps added outside the square root, and
    the decay applied to the old parameter.  Returns ``(param, exp_avg, exp_avg_sq)``.
    """
    if step < 1:
        raise ValueError("step counts from 1")
    g = np.asarray(grad, dtype=np.float64)
    p = np.asarray(param, dtype=np.float64)
    m = beta1 * np.asarray(exp_avg, dtype=np.float64) + (1.0 - beta1) * g
    v = beta2 * np.asarray(exp_avg_sq, dtype=np.float64) + (1.0 - beta2) * g * g
    m_hat = m / (1.0 - beta1 ** step)
    v_hat = v / (1.0 - beta2 ** step)
    p_new = p * (1.0 - lr * wd) - lr * m_hat / (np.sqrt(v_hat) + eps)
    return p_new, m, v


# --- helpers for decoding bf16 / fp16 storage ---------------------------------------

def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact decode of bf16 bit patterns (uint16) to float64."""
    bits = np.asarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def flops_standard(m: int, n: int, steps: int = NS_STEPS) -> int:
    """Canonical flop count of the standard form on an ``m x n`` iterate (m <= n):
    per step ``2 m^2 n`` for ``X X^T``, ``2 m^3`` for ``A A`` and ``2 m^2 n`` for ``B X``."""
    return steps * (4 * m * m * n + 2 * m ** 3)


def flops_gram(m: int, n: int, steps: int = NS_STEPS, restart_every: int = GRAM_RESTART_EVERY) -> int:
    """Flop count of :func:`ns_gram` as written: ``2 m^2 n`` for each product with
    ``X`` (``R_0``, every re-anchoring ``Q X`` and ``X X^T``, the final ``Q X``) and
    ``2 m^3`` for each square product (``R R``; ``H Q`` unless ``Q`` is the identity;
    the two products of ``H R H``)."""
    if steps <= 0:
        return 0
    wide = 1          # R_0
    cubes = 0
    q_identity = True
    for step in range(1, steps + 1):
        cubes += 1                      # R R inside H
        if not q_identity:
            cubes += 1                  # H Q
        q_identity = False
        if step < steps:
            if restart_every and step % restart_every == 0:
                wide += 2               # X <- Q X, R <- X X^T
                q_identity = True
            else:
                cubes += 2              # T = H R, R = T H
    wide += 0 if q_identity else 1      # final Q X (skipped when Q is the identity)
    return 2 * wide * m * m * n + 2 * cubes * m ** 3


# --- dedicated ownership (planner check) ------------------------------------------------

def lpt_assign(costs: Sequence[int], world: int) -> Tuple[List[int], List[int]]:
    """Longest processing time first, written out plainly.

    [DMZ] §每步通信字节数 — under dedicated ownership each Muon-target matrix has one owner
    that runs its Newton-Schulz chain once.  The build balances owners with LPT: take the
    matrices from the heaviest down (equal costs in index order), give each to the owner
    with the smallest load so far (equal loads: the lowest rank).  Returns the owner of
    every matrix and the load of every owner.
    """
    order = sorted(range(len(costs)), key=lambda i: (-costs[i], i))
    load = [0] * world
    owner = [0] * len(costs)
    for i in order:
        best = min(range(world), key=lambda w: (load[w], w))
        owner[i] = best
        load[best] += costs[i]
    return owner, load
