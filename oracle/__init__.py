"""Float64 CPU oracle of the owner-side Muon step (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline and
reference legs may import this package.  The product package never imports it, and it
imports nothing from the product.
"""

from .muon_ref import *  # noqa: F401,F403
from .muon_ref import (  # noqa: F401
    NS_A, NS_B, NS_C, NS_STEPS, NORM_EPS, NS_METHODS, GRAM_RESTART_EVERY,
    route, matrix_view_shape, pack_offsets, momentum_update, frobenius_normalize,
    ns_poly, ns_poly_iterated, ns_standard, ns_gram, newton_schulz, orthogonalize,
    update_scale, apply_update, muon_step, adamw_step, bf16_bits_to_f64,
    flops_standard, flops_gram, round_to, method_storage, lpt_assign,
)
