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
  (derivation in :func:`ns_gram`); no restarts.
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

# Reading (pages silent): the epsilon added to the Frobenius norm.
NORM_EPS = 1e-7


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
    into one contiguous buffer.  The layout is this build's choice: matrices in table
    order, each starting on a multiple of ``align`` elements.  Returns the offsets and
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
                c: float = NS_C) -> np.ndarray:
    """Standard quintic Newton-Schulz on an already normalised ``m x n`` iterate.

    [DSM] §核心算子 (``zeropower_via_newtonschulz5``): each step forms
    ``A = X X^T``, ``B = b A + c A A`` and replaces ``X`` by ``a X + B X``.
    """
    x = np.array(x, dtype=np.float64)
    for _ in range(steps):
        gram_a = x @ x.T
        poly_b = b * gram_a + c * (gram_a @ gram_a)
        x = a * x + poly_b @ x
    return x


# --- a4': Newton-Schulz, gram form ----------------------------------------------------

def ns_gram(x: np.ndarray, steps: int = NS_STEPS, a: float = NS_A, b: float = NS_B,
            c: float = NS_C) -> np.ndarray:
    """Gram-form Newton-Schulz: iterate only on the small square ``R = X X^T``.

    [DSM] §核心算子 (``zeropower_via_gram_newtonschulz``) says the variant iterates on
    the Gram matrix ``R = X @ X.T`` to save FLOPs on wide matrices.  Reading of the
    steps: every iterate of the standard form is ``X_k = Q_k X_0`` with ``Q_k`` a
    polynomial in ``R_0 = X_0 X_0^T``, hence ``X_k X_k^T = Q_k R_0 Q_k``.  One step with
    ``H = a I + b R + c R R`` sends ``Q -> H Q`` and ``R -> H R H``; the final result is
    ``Q X_0``.  The last step does not need the ``R`` update.
    """
    x0 = np.array(x, dtype=np.float64)
    m = x0.shape[0]
    eye = np.eye(m)
    r = x0 @ x0.T
    q = eye.copy()
    for step in range(steps):
        h = a * eye + b * r + c * (r @ r)
        q = h @ q
        if step + 1 < steps:
            r = h @ r @ h
    return q @ x0


def newton_schulz(x: np.ndarray, method: str = NS_METHOD_DEFAULT, steps: int = NS_STEPS,
                  a: float = NS_A, b: float = NS_B, c: float = NS_C) -> np.ndarray:
    """Dispatch on ``ns_method`` ([DSM] §核心算子: ``NS_METHODS = {standard, gram}``)."""
    if method == "standard":
        return ns_standard(x, steps, a, b, c)
    if method == "gram":
        return ns_gram(x, steps, a, b, c)
    raise ValueError(f"unknown ns_method {method!r}")


def orthogonalize(u: np.ndarray, method: str = NS_METHOD_DEFAULT, steps: int = NS_STEPS,
                  eps: float = NORM_EPS) -> np.ndarray:
    """Normalise, transpose when tall, run Newton-Schulz, transpose back.

    Returns ``O`` with the shape of ``u``.
    """
    u = np.asarray(u, dtype=np.float64)
    if u.ndim != 2:
        raise ValueError("orthogonalize takes a 2D matrix")
    rows, cols = u.shape
    transposed = rows > cols
    x = u.T if transposed else u
    x = frobenius_normalize(x, eps)
    o = newton_schulz(x, method, steps)
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
              steps: int = NS_STEPS, nesterov: bool = True, eps: float = NORM_EPS):
    """The owner-side Muon step over a list of matrices.

    [DSM] §什么是 Muon 优化器？ — momentum, then Newton-Schulz orthogonalisation of the
    momentum matrix, then the weight update; [DMZ] §两种packed buffer生命周期 — the
    owner runs it once per matrix of its packed buffer.  Returns
    ``(new_params, new_momenta, orthos)`` as float64 arrays.
    """
    new_params, new_momenta, orthos = [], [], []
    for g, p, m in zip(grads, params, momenta):
        m_new, u = momentum_update(g, m, mu, nesterov)
        o = orthogonalize(u, method, steps, eps)
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


def flops_gram(m: int, n: int, steps: int = NS_STEPS) -> int:
    """Canonical flop count of the gram form: ``R_0`` and the final ``Q X_0``
    (``2 m^2 n`` each) plus ``2 m^3`` for each of ``R R``, ``H Q`` (not on the first
    step, where ``Q = H``) and the two products of ``H R H`` (not on the last step)."""
    if steps <= 0:
        return 0
    n_cubes = steps + (steps - 1) + 2 * (steps - 1)
    return 4 * m * m * n + 2 * n_cubes * m ** 3
