"""CPU float64 oracle for the GRPO token loss and its gradient.

TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's CPU
baseline may import or run this module.  The product path never calls it.

Source: "Efficient Reinforcement Learning for Long-Horizon Tool-Use Agentic
Tasks" (SinkFlex-RL), zh page, "Policy update", equations (3)-(7):

* (3) group-normalised advantage of rollout i among the G rollouts of one
  prompt: A_i = (R_i - mu(R_1..G)) / (sigma(R_1..G) + eps_A), given to every
  optimised token of the rollout;
* (4) importance ratio rho_{i,t} = pi_theta / pi_old of the sampled token,
  i.e. exp(logp - logp_old);
* (5) clipped ratio clip(rho, 1 - eps_c, 1 + eps_c);
* (6) J_{i,t} = min(rho A_i, clip(rho) A_i);
* (7) L = -(1 / sum_i T_i) sum_i sum_t J_{i,t} + beta D_KL(pi_theta || pi_ref),
  T_i = number of optimised tokens of rollout i.

Readings where the pages are silent:
* sigma is the population standard deviation of the group's G rewards;
* the KL term is estimated per optimised token with
  k3 = exp(r) - r - 1, r = logp_ref - logp, and averaged with the same
  1 / sum_i T_i as the policy term;
* the gradient of J with respect to logp is rho A where J follows the
  unclipped branch (including rho exactly on a clip boundary) and 0 where
  the clipped branch is strictly smaller; d k3 / d logp = 1 - exp(r);
* with no optimised token at all the loss and every gradient are 0.

Arrays (float64 NumPy): logp, logp_old, logp_ref [T]; mask [T] (nonzero =
optimised token); rewards [num_rollouts]; cu_tokens [num_rollouts + 1]
(token offsets of the rollouts, consecutive groups of ``group_size``).
"""
from __future__ import annotations

import numpy as np


def advantages(rewards, group_size, adv_eps):
    """Equation (3) for every rollout (population standard deviation)."""
    r = np.asarray(rewards, dtype=np.float64)
    G = int(group_size)
    assert r.size % G == 0
    out = np.empty_like(r)
    for g0 in range(0, r.size, G):
        grp = r[g0:g0 + G]
        mu = grp.sum() / G
        sigma = np.sqrt(((grp - mu) ** 2).sum() / G)
        out[g0:g0 + G] = (grp - mu) / (sigma + adv_eps)
    return out


def grpo_loss(logp, logp_old, logp_ref, mask, rewards, cu_tokens, group_size, clip_eps=0.2, adv_eps=1e-6,
              kl_beta=0.0):
    """Returns dict(loss, policy, kl, clip_frac, n_tokens, adv [R], dlogp [T]).

    policy = -(1/N) sum J, kl = (1/N) sum k3 (unscaled), loss = policy + beta kl,
    clip_frac = fraction of optimised tokens whose gradient the clip removes.
    """
    logp = np.asarray(logp, dtype=np.float64)
    logp_old = np.asarray(logp_old, dtype=np.float64)
    m = np.asarray(mask) != 0
    cu = np.asarray(cu_tokens, dtype=np.int64)
    R = len(cu) - 1
    assert cu[0] == 0 and cu[-1] == logp.size and np.all(np.diff(cu) >= 0)
    adv = advantages(rewards, group_size, adv_eps)
    A = np.repeat(adv, np.diff(cu))                     # advantage of each token's rollout
    N = int(np.count_nonzero(m))
    rho = np.exp(logp - logp_old)
    lo, hi = 1.0 - clip_eps, 1.0 + clip_eps
    J = np.minimum(rho * A, np.clip(rho, lo, hi) * A)
    clipped = ((A > 0) & (rho > hi)) | ((A < 0) & (rho < lo))
    dJ = np.where(clipped, 0.0, rho * A)
    if kl_beta != 0.0:
        r = np.asarray(logp_ref, dtype=np.float64) - logp
        k3 = np.exp(r) - r - 1.0
        dk3 = 1.0 - np.exp(r)
    else:
        k3 = np.zeros_like(logp)
        dk3 = np.zeros_like(logp)
    if N == 0:
        return dict(loss=0.0, policy=0.0, kl=0.0, clip_frac=0.0, n_tokens=0, adv=adv, dlogp=np.zeros_like(logp))
    policy = -float(np.sum(J[m])) / N
    kl = float(np.sum(k3[m])) / N
    dlogp = np.where(m, (-dJ + kl_beta * dk3) / N, 0.0)
    return dict(loss=policy + kl_beta * kl, policy=policy, kl=kl, clip_frac=float(np.count_nonzero(clipped & m)) / N,
                n_tokens=N, adv=adv, dlogp=dlogp)
