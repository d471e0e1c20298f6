"""MuonAdamW, the hybrid optimizer over named parameters, against the oracle.

The wrapper routes parameters by the rule of "DeepSpeed 集成 Muon 优化器实战"
§use_muon参数打标 (ndim >= 2 and no "embed"/"lm_head" in the name: Muon; everything else:
AdamW, §混合优化器的参数组构造), packs each group, and steps both.  Two steps on the
GPT-2-small parameter set are compared with the oracle (Muon: one matrix of every shape,
parameter delta <= 1e-2 and momentum <= 1e-5; AdamW: the whole group <= 1e-5), and a
checkpoint taken through the wrapper resumes bit for bit in a fresh optimizer.
"""

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


def _named_params():
    wl = synth.workload("gpt2small")
    named = list(zip(wl.muon_names, wl.muon_shapes)) + list(zip(wl.adam_names, wl.adam_shapes))
    # model order is not group order: interleave the two groups deterministically
    order = np.random.default_rng(0).permutation(len(named))
    return wl, [named[i] for i in order]


def _fill(opt, named, seed, what):
    for idx, (name, shape) in enumerate(named):
        gen = synth.matrix_generator(seed, idx, "cuda")
        if what == "param":
            opt.param(name).copy_(0.02 * torch.randn(shape, generator=gen, device="cuda"))
        elif len(shape) == 2 and name in opt.muon_names:
            r, c = shape
            opt.grad(name).copy_(synth.make_grad(r, c, seed, idx, "cuda").view(shape))
        else:
            opt.grad(name).copy_((0.01 * torch.randn(shape, generator=gen, device="cuda")).to(torch.bfloat16))


def _make(nsm, named, wl):
    return nsm.MuonAdamW(named, muon_lr=wl.lr, adam_lr=3e-4, momentum=wl.mu, weight_decay=wl.wd,
                         ns_method="gram")


def test_routing_follows_the_pages_rule(nsm):
    wl, named = _named_params()
    opt = _make(nsm, named, wl)
    want_muon = [n for n, s in named if oracle.route(n, len(s))]
    assert opt.muon_names == want_muon
    assert opt.adam_names == [n for n, s in named if not oracle.route(n, len(s))]
    assert sorted(opt.muon_names) == sorted(wl.muon_names)
    for n in opt.adam_names:
        shape = dict(named)[n]
        assert len(shape) < 2 or "embed" in n.lower() or "lm_head" in n.lower()


def test_two_steps_against_oracle_and_resume_bitwise(nsm):
    wl, named = _named_params()
    opt = _make(nsm, named, wl)
    _fill(opt, named, 7, "param")
    # one matrix of every working shape, checked against the oracle
    picked, seen = [], set()
    for n, (r, c) in zip(opt.muon_names, opt.muon_shapes):
        if (r, c) not in seen:
            seen.add((r, c))
            picked.append(n)
    for k in range(2):
        _fill(opt, named, 100 + k, "grad")
        before = {n: (opt.param(n).double().cpu().numpy(),
                      opt._view(n, opt.muon_momentum, opt.adam_exp_avg).double().cpu().numpy(),
                      opt.grad(n).double().cpu().numpy()) for n in picked}
        a_p = opt.adam_params.double().cpu().numpy()
        a_m = opt.adam_exp_avg.double().cpu().numpy()
        a_v = opt.adam_exp_avg_sq.double().cpu().numpy()
        a_g = opt.adam_grads.double().cpu().numpy()
        opt.step()
        assert nsm.device_status() == nsm.NSM_OK
        for n in picked:
            p, m, g = before[n]
            (pn,), (mn,), _ = oracle.muon_step([g], [p], [m], wl.lr, wl.wd, wl.mu, "gram", storage="method")
            got_p = opt.param(n).double().cpu().numpy()
            got_m = opt._view(n, opt.muon_momentum, opt.adam_exp_avg).double().cpu().numpy()
            assert rel(got_m, mn) <= TOL_FP32, (n, rel(got_m, mn))
            assert rel(got_p - p, pn - p) <= TOL_DELTA, (n, rel(got_p - p, pn - p))
        pr, mr, vr = oracle.adamw_step(a_g, a_p, a_m, a_v, 3e-4, 0.9, 0.95, 1e-10, wl.wd, k + 1)
        assert rel(opt.adam_exp_avg.double().cpu().numpy(), mr) <= TOL_FP32
        assert rel(opt.adam_exp_avg_sq.double().cpu().numpy(), vr) <= TOL_FP32
        got = opt.adam_params.double().cpu().numpy()
        assert rel(got, pr) <= TOL_FP32
        # the fp32 parameter itself is rounded once per step: about 1e-9 absolute at
        # |p| ~ 0.02 against a step of ~3e-4, a few 1e-6 of the step in relative terms
        assert rel(got - a_p, pr - a_p) <= 10 * TOL_FP32

    # checkpoint through the wrapper, two more steps, then the same two steps from the
    # checkpoint in a fresh optimizer: the same bits
    saved = {k: (v.cpu().clone() if torch.is_tensor(v) else v) for k, v in opt.state_dict().items()}
    for k in range(2, 4):
        _fill(opt, named, 100 + k, "grad")
        opt.step()
    fresh = _make(nsm, named, wl)
    fresh.load_state_dict(saved)
    assert fresh.step_count == 2
    for k in range(2, 4):
        _fill(fresh, named, 100 + k, "grad")
        fresh.step()
    torch.cuda.synchronize()
    for key in ("muon_params", "muon_momentum", "adam_params", "adam_exp_avg", "adam_exp_avg_sq"):
        assert torch.equal(getattr(fresh, key), getattr(opt, key)), key


def test_state_dict_carries_master_weights(nsm):
    wl, named = _named_params()
    opt = _make(nsm, named, wl)
    sd = opt.state_dict()
    for key in ("muon_params", "muon_momentum", "adam_params", "adam_exp_avg", "adam_exp_avg_sq", "step"):
        assert key in sd
    other = nsm.MuonAdamW(named[:-1], ns_method="gram")
    with pytest.raises(ValueError):
        other.load_state_dict(sd)
