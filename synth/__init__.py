"""Seeded synthetic workloads for the Muon step: shapes, names and random tensors.

This module only makes inputs.  It holds none of the optimizer's arithmetic, so both
the CUDA path's tests/benchmark and the float64 oracle can draw the same inputs from it
without sharing any of the method.

Workloads (transformer-shaped gradient sets; no datasets or trained weights):

* ``tiny``      — 4 matrices of 128x256, N(0,1) gradients, plus a 256-element AdamW
                  vector.
* ``layer1024`` — one transformer layer of hidden size 1024: q/k/v/o 1024x1024,
                  gate/up 4096x1024, down 1024x4096; AdamW on two norm vectors and a
                  32000x1024 token embedding.
* ``gpt2small`` — 12 layers of hidden 768: 2304x768 qkv, 768x768 proj, 3072x768 fc,
                  768x3072 out; AdamW on the embeddings, lm_head, norms and biases.
* ``llama7b``   — 32 layers of hidden 4096: q/o 4096x4096, k/v 1024x4096 (GQA),
                  gate/up 11008x4096, down 4096x11008.  ``llama7b_layer`` is its first
                  layer alone (for profiler captures).
* ``split_moe`` — 16 layers, each with 32 per-head 128x4096 query blocks (Muon Split:
                  every head block is its own table entry) and 64 experts with gate/up
                  1408x2048 and down 2048x1408.  ``split_moe_heads`` is its 512 head
                  blocks alone, ``split_moe_layer`` its first layer.

Gradients other than ``tiny`` are near low-rank with a high condition number:
``G = sum_{i<32} 0.7^i u_i v_i^T + 0.01 N(0,1)`` with raw N(0,1) vectors ``u_i, v_i``,
rounded to bf16 (round to nearest even).  Every matrix draws from its own generator,
seeded ``seed * 1000003 + matrix_index``.  Parameters are N(0, 0.02) in fp32 and the
momentum starts at zero.
"""

from __future__ import annotations

from dataclasses import dataclass, field
from typing import Dict, List, Optional, Sequence, Tuple

import torch


@dataclass
class Workload:
    name: str
    seed: int
    muon_names: List[str]
    muon_shapes: List[Tuple[int, int]]
    adam_names: List[str] = field(default_factory=list)
    adam_shapes: List[Tuple[int, ...]] = field(default_factory=list)
    lr: float = 0.02
    wd: float = 0.1
    mu: float = 0.95
    lowrank: bool = True

    @property
    def muon_elements(self) -> int:
        return sum(r * c for r, c in self.muon_shapes)

    @property
    def adam_elements(self) -> int:
        total = 0
        for s in self.adam_shapes:
            n = 1
            for d in s:
                n *= d
            total += n
        return total


def _tiny() -> Workload:
    names = [f"model.layers.{i}.mlp.proj.weight" for i in range(4)]
    return Workload("tiny", 0, names, [(128, 256)] * 4,
                    ["model.norm.weight"], [(256,)], lowrank=False)


def _layer1024() -> Workload:
    h, f = 1024, 4096
    p = "model.layers.0."
    names = [p + "self_attn.q_proj.weight", p + "self_attn.k_proj.weight",
             p + "self_attn.v_proj.weight", p + "self_attn.o_proj.weight",
             p + "mlp.gate_proj.weight", p + "mlp.up_proj.weight", p + "mlp.down_proj.weight"]
    shapes = [(h, h), (h, h), (h, h), (h, h), (f, h), (f, h), (h, f)]
    adam_names = [p + "input_layernorm.weight", p + "post_attention_layernorm.weight",
                  "model.embed_tokens.weight"]
    adam_shapes = [(h,), (h,), (32000, h)]
    return Workload("layer1024", 1, names, shapes, adam_names, adam_shapes)


def _gpt2small() -> Workload:
    h = 768
    names, shapes, an, ash = [], [], [], []
    for l in range(12):
        p = f"transformer.h.{l}."
        names += [p + "attn.c_attn.weight", p + "attn.c_proj.weight",
                  p + "mlp.c_fc.weight", p + "mlp.c_proj.weight"]
        shapes += [(3 * h, h), (h, h), (4 * h, h), (h, 4 * h)]
        an += [p + "ln_1.weight", p + "ln_1.bias", p + "ln_2.weight", p + "ln_2.bias",
               p + "attn.c_attn.bias", p + "attn.c_proj.bias", p + "mlp.c_fc.bias",
               p + "mlp.c_proj.bias"]
        ash += [(h,), (h,), (h,), (h,), (3 * h,), (h,), (4 * h,), (h,)]
    # GPT-2 calls its embeddings wte/wpe; the names here carry "embed" so that the
    # routing rule sends them to AdamW, as the pages intend for embeddings.
    an += ["transformer.embed_tokens.weight", "transformer.embed_positions.weight",
           "transformer.ln_f.weight", "transformer.ln_f.bias", "lm_head.weight"]
    ash += [(50257, h), (1024, h), (h,), (h,), (50257, h)]
    return Workload("gpt2small", 2, names, shapes, an, ash)


def _llama7b() -> Workload:
    h, kv, f = 4096, 1024, 11008
    names, shapes = [], []
    for l in range(32):
        p = f"model.layers.{l}."
        names += [p + "self_attn.q_proj.weight", p + "self_attn.k_proj.weight",
                  p + "self_attn.v_proj.weight", p + "self_attn.o_proj.weight",
                  p + "mlp.gate_proj.weight", p + "mlp.up_proj.weight",
                  p + "mlp.down_proj.weight"]
        shapes += [(h, h), (kv, h), (kv, h), (h, h), (f, h), (f, h), (h, f)]
    return Workload("llama7b", 3, names, shapes, lr=1e-4)


def _llama7b_layer() -> Workload:
    """One layer of the Llama-7B-shaped set (7 matrices, 177M elements): small enough
    for profiler captures, with operands larger than L2."""
    full = _llama7b()
    return Workload("llama7b_layer", 3, full.muon_names[:7], full.muon_shapes[:7], lr=1e-4)


def _split_moe() -> Workload:
    names, shapes = [], []
    for l in range(16):
        p = f"model.layers.{l}."
        for hd in range(32):
            names.append(p + f"self_attn.q_proj.weight.head{hd}")
            shapes.append((128, 4096))
        for e in range(64):
            q = p + f"mlp.experts.{e}."
            names += [q + "gate_proj.weight", q + "up_proj.weight", q + "down_proj.weight"]
            shapes += [(1408, 2048), (1408, 2048), (2048, 1408)]
    return Workload("split_moe", 4, names, shapes)


def _split_moe_heads() -> Workload:
    """The Split/MoE set's query head blocks alone (512 blocks of 128x4096, 268M
    elements): the small-matrix kernel's share of that set, small enough for profiler
    captures."""
    full = _split_moe()
    keep = [i for i, s in enumerate(full.muon_shapes) if s == (128, 4096)]
    return Workload("split_moe_heads", 4, [full.muon_names[i] for i in keep],
                    [full.muon_shapes[i] for i in keep])


def _split_moe_layer() -> Workload:
    """The Split/MoE set's first layer (32 head blocks and 192 expert matrices, 570M
    elements): a small case of the same launches, for profiler captures."""
    full = _split_moe()
    n = 32 + 64 * 3
    return Workload("split_moe_layer", 4, full.muon_names[:n], full.muon_shapes[:n])


WORKLOADS = {
    "tiny": _tiny,
    "layer1024": _layer1024,
    "gpt2small": _gpt2small,
    "llama7b": _llama7b,
    "llama7b_layer": _llama7b_layer,
    "split_moe": _split_moe,
    "split_moe_heads": _split_moe_heads,
    "split_moe_layer": _split_moe_layer,
}


def workload(name: str) -> Workload:
    return WORKLOADS[name]()


def custom(shapes: Sequence[Tuple[int, int]], seed: int = 0, lowrank: bool = True,
           name: str = "custom") -> Workload:
    names = [f"layers.{i}.proj.weight" for i in range(len(shapes))]
    return Workload(name, seed, names, [tuple(s) for s in shapes], lowrank=lowrank)


def matrix_generator(seed: int, index: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1000003 + index)
    return g


def make_grad(rows: int, cols: int, seed: int, index: int, device="cpu",
              lowrank: bool = True, rank: int = 32, decay: float = 0.7,
              noise: float = 0.01) -> torch.Tensor:
    """One bf16 gradient matrix (see the module docstring for the recipe)."""
    gen = matrix_generator(seed, index, device)
    if not lowrank:
        return torch.randn(rows, cols, generator=gen, device=device,
                           dtype=torch.float32).to(torch.bfloat16)
    u = torch.randn(rows, rank, generator=gen, device=device, dtype=torch.float32)
    v = torch.randn(cols, rank, generator=gen, device=device, dtype=torch.float32)
    w = decay ** torch.arange(rank, device=device, dtype=torch.float32)
    g = (u * w) @ v.T
    g += noise * torch.randn(rows, cols, generator=gen, device=device, dtype=torch.float32)
    return g.to(torch.bfloat16)


def fill_packed_grads(wl: Workload, offsets: Sequence[int], out: torch.Tensor,
                      seed_offset: int = 0) -> None:
    """Write every gradient of ``wl`` into the packed bf16 buffer ``out``."""
    for i, (r, c) in enumerate(wl.muon_shapes):
        o = int(offsets[i])
        g = make_grad(r, c, wl.seed + seed_offset, i, out.device, wl.lowrank)
        out[o:o + r * c].copy_(g.reshape(-1))


def fill_packed_params(wl: Workload, offsets: Sequence[int], out: torch.Tensor,
                       std: float = 0.02) -> None:
    """fp32 N(0, std) parameters, one generator per matrix (index offset 500000)."""
    for i, (r, c) in enumerate(wl.muon_shapes):
        o = int(offsets[i])
        gen = matrix_generator(wl.seed, 500000 + i, out.device)
        out[o:o + r * c].copy_(
            std * torch.randn(r * c, generator=gen, device=out.device, dtype=torch.float32))


def make_adam_group(wl: Workload, device="cpu", seed_offset: int = 0):
    """Flat AdamW group: bf16 grads N(0,1)*0.01-ish and fp32 params N(0,0.02)."""
    n = wl.adam_elements
    gen = matrix_generator(wl.seed + seed_offset, 900000, device)
    grads = (0.01 * torch.randn(n, generator=gen, device=device)).to(torch.bfloat16)
    gen2 = matrix_generator(wl.seed, 900001, device)
    params = 0.02 * torch.randn(n, generator=gen2, device=device)
    return grads, params


def random_matrix(rows: int, cols: int, seed: int, device="cpu",
                  dtype=torch.bfloat16) -> torch.Tensor:
    gen = matrix_generator(seed, 0, device)
    return torch.randn(rows, cols, generator=gen, device=device).to(dtype)
