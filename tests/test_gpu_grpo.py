"""GRPO token loss: CUDA path vs the CPU float64 oracle (needs a GB300).

The clip decision is taken in fp32 on the GPU and in fp64 by the oracle;
tokens whose ratio lies within 1e-5 (relative) of a clip boundary may fall
on either side, so the elementwise gradient comparison skips them and the
clipped fraction may differ by their share.
"""
import numpy as np
import pytest
import torch

import oracle.grpo_ref as ref
import workloads as W

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def built():
    from sink_aware_masked_gb300 import build

    build.build()


def run(inp, clip_eps=0.2, adv_eps=1e-6, kl_beta=0.04, mask=None, rewards=None):
    import sink_aware_masked_gb300 as sa

    mask = inp.mask if mask is None else mask
    rewards = inp.rewards if rewards is None else rewards
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)  # noqa: E731
    stats, dlogp, adv = sa.grpo_loss(t(inp.logp), t(inp.logp_old), t(mask), t(rewards), t(inp.cu_tokens),
                                     [int(x) for x in inp.cu_tokens], group_size=inp.wl.group_size,
                                     clip_eps=clip_eps, adv_eps=adv_eps, kl_beta=kl_beta,
                                     logp_ref=t(inp.logp_ref) if kl_beta else None)
    want = ref.grpo_loss(inp.logp.astype(np.float64), inp.logp_old.astype(np.float64),
                         inp.logp_ref.astype(np.float64), mask, rewards.astype(np.float64), inp.cu_tokens,
                         inp.wl.group_size, clip_eps, adv_eps, kl_beta)
    return stats.cpu().numpy().astype(np.float64), dlogp.cpu().numpy().astype(np.float64), adv.cpu().numpy(), want


def check(inp, **kw):
    stats, dlogp, adv, want = run(inp, **kw)
    clip_eps = kw.get("clip_eps", 0.2)
    rho = np.exp(inp.logp.astype(np.float64) - inp.logp_old.astype(np.float64))
    near = (np.abs(rho - (1 + clip_eps)) < 1e-5 * (1 + clip_eps)) | (np.abs(rho - (1 - clip_eps)) < 1e-5)
    N = max(1, want["n_tokens"])
    for got, key in zip(stats[:3], ("loss", "policy", "kl")):
        assert abs(got - want[key]) <= 1e-5 * max(1.0, abs(want[key])) + 2.0 * np.count_nonzero(near) / N, key
    assert abs(stats[3] - want["clip_frac"]) <= (np.count_nonzero(near) + 0.5) / N
    scale = max(1e-30, np.max(np.abs(want["dlogp"])))
    err = np.max(np.abs(dlogp - want["dlogp"])[~near], initial=0.0)
    assert err <= 1e-5 * scale, err
    np.testing.assert_allclose(adv, want["adv"], rtol=1e-6, atol=1e-6)


CASES = [
    W.GrpoWorkload("small", 3, 4, 1, 300, 1),
    W.GrpoWorkload("single_rollout_groups", 5, 1, 10, 2000, 2),   # G = 1: every advantage is 0
    W.GrpoWorkload("wide_groups", 2, 16, 0, 700, 3),              # zero-length rollouts allowed
    W.GrpoWorkload("many_short", 100, 6, 1, 40, 4),               # 600 rollouts, many crossing a 4-token vector
    W.GrpoWorkload("warp_groups", 3, 48, 0, 200, 6),              # G > 32: one warp per group
    W.GrpoWorkload("unstaged_rollouts", 1000, 8, 1, 64, 5),       # 8000 rollouts: offsets and advantages not staged
    W.GrpoWorkload("long_rollouts", 64, 8, 8192, 16384, 7),       # > 4 stages per CTA: the ring refills
]


@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
@pytest.mark.parametrize("beta", [0.0, 0.04])
def test_grpo_matches_oracle(wl, beta):
    check(W.make_grpo_inputs(wl), kl_beta=beta)


def test_grpo_empty_mask_and_equal_rewards():
    inp = W.make_grpo_inputs(CASES[0])
    stats, dlogp, adv, want = run(inp, mask=np.zeros_like(inp.mask))
    assert not np.any(stats) and not np.any(dlogp)
    stats, dlogp, adv, want = run(inp, rewards=np.ones_like(inp.rewards))
    assert not np.any(adv) and abs(stats[1]) == 0.0


@pytest.mark.parametrize("name", sorted(W.GRPO_WORKLOADS))
def test_grpo_workload(name):
    wl = W.GRPO_WORKLOADS[name]
    check(W.make_grpo_inputs(wl), clip_eps=wl.clip_eps, adv_eps=wl.adv_eps, kl_beta=wl.kl_beta)


def test_grpo_barrier_timeout_reports_and_recovers():
    """The grid barrier's wait is bounded: with an arrival word that can never
    complete (its count already past the grid size), every CTA gives up after
    about a second, the status word reports TIMEOUT, and a later call on a
    zero-filled workspace is correct again."""
    import sink_aware_masked_gb300 as sa

    inp = W.make_grpo_inputs(CASES[3])
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)  # noqa: E731
    cu_host = [int(x) for x in inp.cu_tokens]
    cu = t(inp.cu_tokens)
    ws = torch.zeros(sa.grpo_workspace_bytes(cu, cu_host, group_size=inp.wl.group_size), dtype=torch.uint8, device=DEV)
    assert sa.sinkattn_get_device_status() == 0
    ws[:8] = torch.tensor([1 << 19], dtype=torch.int64).view(torch.uint8).to(DEV)  # arrivals: 2^19, never grid - 1
    args = (t(inp.logp), t(inp.logp_old), t(inp.mask), t(inp.rewards), cu, cu_host)
    sa.grpo_loss(*args, group_size=inp.wl.group_size, workspace=ws)
    torch.cuda.synchronize()
    assert sa.sinkattn_get_device_status() == 6  # SINKATTN_ERR_TIMEOUT
    ws.zero_()
    stats, dlogp, adv = sa.grpo_loss(*args, group_size=inp.wl.group_size, workspace=ws)
    assert sa.sinkattn_get_device_status() == 0
    want = ref.grpo_loss(inp.logp.astype(np.float64), inp.logp_old.astype(np.float64), None, inp.mask,
                         inp.rewards.astype(np.float64), inp.cu_tokens, inp.wl.group_size)
    assert abs(float(stats[1]) - want["policy"]) <= 1e-5 * max(1.0, abs(want["policy"])) + 1e-3
