"""The GRPO loss oracle against independent pins (no GPU).

Routes: a hand-worked example with exact values (tests/golden); the same
equations written with torch primitives (torch.std, torch.clamp,
torch.minimum) and differentiated by autograd; closed forms (ratio 1 on
equal-length rollouts gives a zero policy term, a reference equal to the
policy gives a zero KL term); central finite differences; and planted
mistakes that at least one pin must catch.
"""
import json
import math
import os
import types

import numpy as np
import pytest
import torch

import oracle.grpo_ref as ref

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(os.path.dirname(HERE), "oracle", "grpo_ref.py")


def rand_case(seed, groups=3, G=4, lo=1, hi=40, beta=0.05):
    rng = np.random.default_rng(seed)
    lens = rng.integers(lo, hi + 1, groups * G)
    cu = np.concatenate([[0], np.cumsum(lens)])
    T = int(cu[-1])
    logp_old = -rng.gamma(2.0, 1.0, T)
    logp = logp_old + rng.normal(0, 0.4, T)
    logp_ref = logp_old + rng.normal(0, 0.3, T)
    mask = (rng.random(T) < 0.8).astype(np.uint8)
    rewards = rng.integers(0, 3, groups * G).astype(np.float64)
    return dict(logp=logp, logp_old=logp_old, logp_ref=logp_ref, mask=mask, rewards=rewards, cu_tokens=cu,
                group_size=G, clip_eps=0.2, adv_eps=1e-6, kl_beta=beta)


def torch_loss(c):
    """Equations (3)-(7) with torch primitives; gradient by autograd."""
    lp = torch.tensor(c["logp"], dtype=torch.float64, requires_grad=True)
    old = torch.tensor(c["logp_old"], dtype=torch.float64)
    lref = torch.tensor(c["logp_ref"], dtype=torch.float64)
    m = torch.tensor(c["mask"] != 0)
    R = torch.tensor(c["rewards"], dtype=torch.float64).view(-1, c["group_size"])
    adv = ((R - R.mean(1, keepdim=True)) / (R.std(1, unbiased=False, keepdim=True) + c["adv_eps"])).reshape(-1)
    lens = torch.tensor(np.diff(c["cu_tokens"]))
    A = torch.repeat_interleave(adv, lens)
    rho = torch.exp(lp - old)
    J = torch.minimum(rho * A, torch.clamp(rho, 1 - c["clip_eps"], 1 + c["clip_eps"]) * A)
    r = lref - lp
    k3 = torch.exp(r) - r - 1
    N = m.sum()
    loss = -(J * m).sum() / N + c["kl_beta"] * (k3 * m).sum() / N
    loss.backward()
    return float(loss), lp.grad.numpy()


def check_hand(mod):
    with open(os.path.join(HERE, "golden", "grpo_hand_example.json")) as f:
        g = json.load(f)
    logp = np.array([math.log(1.5), math.log(0.5)])
    out = mod.grpo_loss(logp, np.array(g["logp_old"]), None, np.ones(2, np.uint8), np.array(g["rewards"]),
                        np.array(g["cu_tokens"]), g["group_size"], g["clip_eps"], g["adv_eps"], 0.0)
    ok = (abs(out["loss"] - g["loss"]) < 1e-12 and np.allclose(out["dlogp"], g["dlogp"], atol=1e-12)
          and abs(out["clip_frac"] - g["clip_frac"]) < 1e-12 and np.allclose(out["adv"], g["adv"], atol=1e-12))
    return None if ok else f"hand example: {out['loss']} {out['dlogp']} {out['clip_frac']}"


def check_autograd(mod):
    for seed in range(4):
        c = rand_case(seed)
        out = mod.grpo_loss(**c)
        loss, grad = torch_loss(c)
        if abs(out["loss"] - loss) > 1e-12 or np.max(np.abs(out["dlogp"] - grad)) > 1e-12:
            return f"autograd seed {seed}: loss {out['loss']} vs {loss}, grad err {np.max(np.abs(out['dlogp'] - grad))}"
    return None


def check_closed_forms(mod):
    c = rand_case(7, lo=9, hi=9)
    c["logp"] = c["logp_old"].copy()        # ratio 1 everywhere
    c["logp_ref"] = c["logp"].copy()        # reference = policy
    c["mask"] = np.ones_like(c["mask"])
    out = mod.grpo_loss(**c)
    if abs(out["policy"]) > 1e-12 or abs(out["kl"]) > 1e-15:
        return f"closed forms: policy {out['policy']}, kl {out['kl']}"
    adv = mod.advantages(c["rewards"], c["group_size"], 0.0).reshape(-1, c["group_size"])
    nz = adv.std(1) > 0
    if np.max(np.abs(adv.mean(1))) > 1e-12 or np.max(np.abs(adv.std(1)[nz] - 1.0)) > 1e-12:
        return "advantages are not zero-mean / unit population std"
    return None


def check_finite_differences(mod):
    c = rand_case(11, groups=2, G=3, hi=12)
    out = mod.grpo_loss(**c)
    h = 1e-6
    for t in range(0, len(c["logp"]), 3):
        lp = c["logp"].copy()
        lp[t] += h
        up = mod.grpo_loss(**{**c, "logp": lp})["loss"]
        lp[t] -= 2 * h
        dn = mod.grpo_loss(**{**c, "logp": lp})["loss"]
        fd = (up - dn) / (2 * h)
        if abs(fd - out["dlogp"][t]) > 1e-6:
            return f"finite difference at token {t}: {fd} vs {out['dlogp'][t]}"
    return None


def check_empty_mask(mod):
    c = rand_case(3)
    c["mask"] = np.zeros_like(c["mask"])
    out = mod.grpo_loss(**c)
    return None if out["loss"] == 0.0 and not np.any(out["dlogp"]) else "empty mask must give zero loss and gradient"


CHECKS = [check_hand, check_autograd, check_closed_forms, check_finite_differences, check_empty_mask]


@pytest.mark.parametrize("check", CHECKS, ids=lambda f: f.__name__)
def test_grpo_oracle_pin(check):
    msg = check(ref)
    assert msg is None, msg


MUTATIONS = {
    "sample_std": ("sigma = np.sqrt(((grp - mu) ** 2).sum() / G)", "sigma = np.sqrt(((grp - mu) ** 2).sum() / (G - 1))"),
    "clip_side": ("clipped = ((A > 0) & (rho > hi)) | ((A < 0) & (rho < lo))",
                  "clipped = ((A > 0) & (rho < lo)) | ((A < 0) & (rho > hi))"),
    "no_clip_grad_zero": ("dJ = np.where(clipped, 0.0, rho * A)", "dJ = rho * A"),
    "grad_without_rho": ("dJ = np.where(clipped, 0.0, rho * A)", "dJ = np.where(clipped, 0.0, A)"),
    "mean_over_rollouts": ("N = int(np.count_nonzero(m))", "N = max(1, R)"),
    "mask_ignored": ("policy = -float(np.sum(J[m])) / N", "policy = -float(np.sum(J)) / N"),
    "kl_sign": ("r = np.asarray(logp_ref, dtype=np.float64) - logp", "r = logp - np.asarray(logp_ref, dtype=np.float64)"),
    "max_not_min": ("J = np.minimum(rho * A, np.clip(rho, lo, hi) * A)", "J = np.maximum(rho * A, np.clip(rho, lo, hi) * A)"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_grpo_mutation_is_caught(name):
    old, new = MUTATIONS[name]
    with open(SRC) as f:
        text = f.read()
    assert text.count(old) == 1, old
    mod = types.ModuleType("grpo_mutant")
    exec(compile(text.replace(old, new), "grpo_mutant", "exec"), mod.__dict__)
    failed = []
    for check in CHECKS:
        try:
            if check(mod) is not None:
                failed.append(check.__name__)
        except Exception:
            failed.append(check.__name__)
    assert failed, f"planted mistake {name!r} passed every pin"
