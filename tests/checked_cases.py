"""Cases run through both builds of the library, for tests/test_gpu_checked.py.

`run(nsm)` runs every case on cuda:0 through the binding `nsm` and returns the outputs
(name -> numpy array) and the device status read after each case (name -> (status,
kernel, role, site)).  The cases cover every kernel and every access path the library
has:
- muon_step on tables that take the small-matrix kernel, the 1-CTA GEMM kernel and the
  2-SM GEMM kernel (with narrow tiles: order 1408), in the three forms; rows that are not
  a whole number of 16-byte units (the direct epilogue and the scalar layout paths); tall
  matrices (the transposed layout); the grouped path for small matrices; plain momentum;
  the bf16 parameter copy; two steps in a row;
- muon_orthogonalize (the export of O);
- nsm_gemm with aux, MN-major B, a symmetric output of odd order and the 2-SM kernel;
- adamw_step on a group whose length is not a multiple of 8.

`fullsize_digest(nsm, name)` runs one muon_step (gram, with the bf16 parameter copy) over
a whole benchmark table (llama7b: 5.67B elements; split_moe: 9.13B) and returns exact
integer digests of the updated parameters, momentum and copy, and the device status.

Run as a script (`python tests/checked_cases.py OUT.npz`), it writes the outputs and the
statuses to OUT.npz / OUT.json (`python tests/checked_cases.py --fullsize NAME OUT.json`:
the digests); with NSM_CHECKED=1 in the environment the binding loads the bounds-checked
build.
"""

from __future__ import annotations

import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

STEP_TABLES = {
    # m <= 128 (small kernel), m = 129 / 130 (1-CTA kernel), rows of 130 (direct epilogue
    # of the m x m products), 257 x 129 and 300 x 130 tall (transposed layout), 3 x 5 and
    # 1 x 8 (scalar layout paths)
    "odd": [(3, 5), (130, 260), (257, 129), (1, 8), (96, 160), (300, 130)],
    # every m >= 256: the 2-SM kernel; order 1408 = 5.5 x 256 takes narrow tiles
    "pair": [(256, 512), (512, 256), (1408, 2048)],
    # m = 192 and a tall 4096 x 136: the 1-CTA kernel
    "single": [(192, 384), (4096, 136)],
}


def _status(nsm):
    return tuple(int(v) for v in nsm.device_status_detail())


def _step(nsm, torch, wl, method, steps=1, nesterov=True, copy=False):
    import synth
    shapes = wl.muon_shapes
    offsets, total = nsm.pack(shapes)
    grads = torch.zeros(total, dtype=torch.bfloat16, device="cuda")
    params = torch.zeros(total, dtype=torch.float32, device="cuda")
    mom = torch.zeros(total, dtype=torch.float32, device="cuda")
    synth.fill_packed_params(wl, offsets, params)
    out_bf16 = torch.zeros(total, dtype=torch.bfloat16, device="cuda") if copy else None
    ws = torch.empty(nsm.workspace_bytes(shapes, method), dtype=torch.uint8, device="cuda")
    for k in range(steps):
        synth.fill_packed_grads(wl, offsets, grads, seed_offset=k)
        nsm.muon_step(grads, params, mom, offsets, shapes, wl.lr, wl.wd, wl.mu, method, 5, nesterov, ws,
                      params_bf16=out_bf16)
    res = {"params": params, "momentum": mom}
    if copy:
        res["params_bf16"] = out_bf16.view(torch.int16)
    return res


def run(nsm):
    import torch

    import synth

    nsm.lib()
    out, status = {}, {}

    def record(name, tensors):
        torch.cuda.synchronize()
        for k, t in tensors.items():
            out[f"{name}/{k}"] = np.ascontiguousarray(t.detach().cpu().numpy())
        status[name] = _status(nsm)

    for tname, shapes in STEP_TABLES.items():
        wl = synth.custom(shapes, seed=31, name=tname)
        for method in ("gram", "standard", "standard_bf16"):
            record(f"step/{tname}/{method}", _step(nsm, torch, wl, method))
    wl = synth.custom(STEP_TABLES["odd"], seed=32, name="odd")
    record("step/odd/gram/two_steps_plain_copy", _step(nsm, torch, wl, "gram", steps=2, nesterov=False, copy=True))
    nsm.set_option(nsm.OPT_SMALL_KERNEL, 0)
    try:
        record("step/odd/gram/grouped", _step(nsm, torch, wl, "gram"))
    finally:
        nsm.set_option(nsm.OPT_SMALL_KERNEL, 1)

    for tname in ("odd", "pair"):
        wl = synth.custom(STEP_TABLES[tname], seed=33, name=tname)
        offsets, total = nsm.pack(wl.muon_shapes)
        inp = torch.zeros(total, dtype=torch.bfloat16, device="cuda")
        synth.fill_packed_grads(wl, offsets, inp)
        o = torch.zeros_like(inp)
        ws = torch.empty(nsm.workspace_bytes(wl.muon_shapes, "gram"), dtype=torch.uint8, device="cuda")
        nsm.muon_orthogonalize(inp, o, offsets, wl.muon_shapes, "gram", 5, ws)
        record(f"ortho/{tname}", {"out": o.view(torch.int16)})

    def padded(rows, cols, dt, seed):
        # rows padded to a whole number of 16-byte units, the library's stride rule
        ld = (cols + 7) // 8 * 8
        full = synth.random_matrix(rows, ld, seed, "cuda", dt)
        return full[:, :cols]

    # (M, N, K, dtype, b_mn_major, aux, symmetric, pair); order 130 is not a whole number
    # of 16-byte units (the direct epilogue), 1408 takes narrow tiles on the 2-SM kernel
    gemm_cases = [
        (300, 200, 136, torch.bfloat16, False, True, False, False),
        (130, 130, 72, torch.float16, False, True, True, False),
        (512, 384, 256, torch.float16, True, False, False, True),
        (1408, 1408, 704, torch.float16, False, True, True, True),
        (264, 330, 200, torch.bfloat16, True, True, False, False),
    ]
    for i, (M, N, K, dt, mn, has_aux, sym, pair) in enumerate(gemm_cases):
        a = padded(M, K, dt, 40 + i)
        b = a if sym else (padded(K, N, dt, 50 + i) if mn else padded(N, K, dt, 50 + i))
        aux = None
        if has_aux:
            aux = padded(M, N, dt, 60 + i)
            if sym:
                aux.copy_(((aux.float() + aux.float().T) * 0.5).to(dt))
        c = torch.zeros(M, (N + 7) // 8 * 8, dtype=dt, device="cuda")[:, :N]
        nsm.gemm(a, b, c, aux=aux, b_mn_major=mn, alpha=0.5, beta=-1.25 if has_aux else 0.0,
                 diag=2.0 if sym else 0.0, symmetric=sym, pair=pair)
        record(f"gemm/{i}", {"out": c.view(torch.int16)})

    n = 1_000_003
    gen = synth.matrix_generator(34, 7, "cuda")
    g = (0.01 * torch.randn(n, generator=gen, device="cuda")).to(torch.bfloat16)
    p = 0.02 * torch.randn(n, generator=gen, device="cuda")
    m = torch.zeros(n, device="cuda")
    v = torch.zeros(n, device="cuda")
    for step in (1, 2):
        nsm.adamw_step(g, p, m, v, 3e-4, 0.9, 0.95, 1e-10, 0.1, step)
    record("adamw", {"p": p, "m": m, "v": v})
    return out, status


def _digest(t):
    """Exact digest of a tensor's bits: per chunk of 2^26 elements, the sum of its 16- or
    32-bit words and their sum weighted by position (int64 arithmetic on the device)."""
    import torch
    words = t.view(torch.int32) if t.element_size() == 4 else t.view(torch.int16)
    out = []
    chunk = 1 << 26
    for i in range(0, words.numel(), chunk):
        w = words[i:i + chunk].to(torch.int64)
        pos = torch.arange(1, w.numel() + 1, device=w.device, dtype=torch.int64) % 65521 + 1
        out.append([int(w.sum()), int((w * pos).sum())])
        del w, pos
    return out


def fullsize_digest(nsm, name):
    import torch

    import synth

    nsm.lib()
    wl = synth.workload(name)
    shapes = wl.muon_shapes
    offsets, total = nsm.pack(shapes)
    grads = torch.zeros(total, dtype=torch.bfloat16, device="cuda")
    params = torch.zeros(total, dtype=torch.float32, device="cuda")
    mom = torch.zeros(total, dtype=torch.float32, device="cuda")
    copy = torch.zeros(total, dtype=torch.bfloat16, device="cuda")
    synth.fill_packed_grads(wl, offsets, grads)
    synth.fill_packed_params(wl, offsets, params)
    ws = torch.empty(nsm.workspace_bytes(shapes, "gram"), dtype=torch.uint8, device="cuda")
    nsm.muon_step(grads, params, mom, offsets, shapes, wl.lr, wl.wd, wl.mu, "gram", 5, True, ws,
                  params_bf16=copy)
    torch.cuda.synchronize()
    status = _status(nsm)
    del ws, grads
    res = {"status": status, "params": _digest(params), "momentum": _digest(mom), "copy": _digest(copy)}
    del params, mom, copy
    torch.cuda.empty_cache()
    return res


if __name__ == "__main__":
    import newton_schulz_orthogonalized_gb300 as nsm_mod

    if sys.argv[1] == "--fullsize":
        res = fullsize_digest(nsm_mod, sys.argv[2])
        res.update(checked=nsm_mod.checked_build(), lib=nsm_mod.LIB_PATH)
        with open(sys.argv[3], "w") as f:
            json.dump(res, f)
        sys.exit(0)
    path = sys.argv[1]
    outs, stats = run(nsm_mod)
    np.savez(path, **outs)
    with open(os.path.splitext(path)[0] + ".json", "w") as f:
        json.dump({"status": stats, "checked": nsm_mod.checked_build(), "lib": nsm_mod.LIB_PATH}, f)
