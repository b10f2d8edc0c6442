"""Seeded synthetic inputs for sink-aware attention.

This module is shared by the CPU oracle (``oracle/``) and the CUDA path
(``sink_aware_masked_gb300``).  It holds shapes, seeds and random draws only:
none of the attention arithmetic lives here.

Workloads follow the shapes of the memory study in "Efficient Reinforcement
Learning for Long-Horizon Tool-Use Agentic Tasks" (SinkFlex-RL), section 5
"Sink-aware FlexAttention": long multi-turn trajectories (up to 8192 tokens),
causal and sliding-window masks with an always-visible prefix, and one
learned sink logit per query head.  The pages name no attention shapes, so
the configurations below fix head_dim = 64 and a 64/8 GQA split.

Every tensor is drawn on the CPU from ``torch.Generator().manual_seed(seed)``
in the order q, k, v, dout, sink, then q/k/v/dout are rounded to bf16.  The
oracle receives the bf16-rounded values widened to float64, the GPU receives
the bf16 tensors, so both sides see identical inputs.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import numpy as np
import torch

# Encodes the unbounded window ("w = inf").
WINDOW_INF = -1


@dataclasses.dataclass(frozen=True)
class Workload:
    """One attention problem: packed sequences plus mask parameters."""

    name: str
    seqlens: tuple           # per-sequence token counts
    num_heads_q: int
    num_heads_kv: int
    head_dim: int
    window: int              # inclusive window w, or WINDOW_INF
    prefix: int              # always-visible prefix p
    causal: bool
    seed: int
    sink_dist: str           # "normal" (N(0,1)) or "uniform2" (U[-2, 2])
    uniform: bool = True     # all sequences the same length (batch layout)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def num_seqs(self) -> int:
        return len(self.seqlens)

    @property
    def total_tokens(self) -> int:
        return int(sum(self.seqlens))

    @property
    def max_seqlen(self) -> int:
        return int(max(self.seqlens)) if self.seqlens else 0

    def cu_seqlens(self) -> np.ndarray:
        cu = np.zeros(self.num_seqs + 1, dtype=np.int32)
        cu[1:] = np.cumsum(np.asarray(self.seqlens, dtype=np.int64))
        return cu

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# Sequence lengths of the packed-trajectory workload: eight multi-turn
# trajectories with lengths drawn once from U[1024, 8192]
# (torch.randint(1024, 8193, (8,), generator seeded with 5)) and written out
# so the workload does not depend on the RNG implementation.
VARLEN_LENGTHS = (6111, 5036, 1589, 6459, 1056, 6459, 3018, 2085)


def _uniform(name, B, S, hq, hkv, w, p, seed, sink_dist, d=64):
    return Workload(name, tuple([S] * B), hq, hkv, d, w, p, True, seed, sink_dist, True)


# The five workloads, in order.  Names describe the workload; the two
# 8192-token variants share inputs (same seed) and differ only in the mask,
# the two packed layers differ in mask and seed.
WORKLOADS = {
    "tiny_s128_w32_p4": _uniform("tiny_s128_w32_p4", 1, 128, 2, 2, 32, 4, 0, "normal"),
    "causal_gqa_s4096": _uniform("causal_gqa_s4096", 1, 4096, 64, 8, WINDOW_INF, 0, 2, "uniform2"),
    "window128_gqa_s4096": _uniform("window128_gqa_s4096", 1, 4096, 64, 8, 128, 0, 3, "uniform2"),
    "causal_gqa_b2_s8192": _uniform("causal_gqa_b2_s8192", 2, 8192, 64, 8, WINDOW_INF, 0, 4, "uniform2"),
    "window128_prefix4_gqa_b2_s8192": _uniform(
        "window128_prefix4_gqa_b2_s8192", 2, 8192, 64, 8, 128, 4, 4, "uniform2"),
    "varlen8_window128": Workload("varlen8_window128", VARLEN_LENGTHS, 64, 8, 64, 128, 0, True, 5,
                                  "uniform2", uniform=False),
    "varlen8_causal": Workload("varlen8_causal", VARLEN_LENGTHS, 64, 8, 64, WINDOW_INF, 0, True, 50,
                               "uniform2", uniform=False),
}


def custom(seqlens, hq, hkv, window=WINDOW_INF, prefix=0, causal=True, seed=0,
           sink_dist="normal", head_dim=64, name="custom") -> Workload:
    seqlens = tuple(int(s) for s in seqlens)
    uniform = len(set(seqlens)) <= 1
    return Workload(name, seqlens, hq, hkv, head_dim, window, prefix, causal, seed, sink_dist, uniform)


@dataclasses.dataclass
class Inputs:
    """Inputs of one workload.  ``*_bf16`` go to the GPU, ``*_f64`` to the oracle."""

    wl: Workload
    q_bf16: torch.Tensor     # [T, Hq, D]
    k_bf16: torch.Tensor     # [T, Hkv, D]
    v_bf16: torch.Tensor     # [T, Hkv, D]
    do_bf16: torch.Tensor    # [T, Hq, D]
    sink: torch.Tensor       # [Hq] float32
    q_f32: Optional[torch.Tensor] = None   # unrounded draws (tiny workload only)
    k_f32: Optional[torch.Tensor] = None
    v_f32: Optional[torch.Tensor] = None
    do_f32: Optional[torch.Tensor] = None

    def f64(self, name: str) -> np.ndarray:
        t = getattr(self, name + "_bf16") if name != "sink" else self.sink
        return t.to(torch.float64).numpy()


def make_inputs(wl: Workload, keep_f32: bool = False) -> Inputs:
    """Draw the inputs of ``wl`` from its seed (CPU, deterministic)."""
    g = torch.Generator().manual_seed(wl.seed)
    T, hq, hkv, d = wl.total_tokens, wl.num_heads_q, wl.num_heads_kv, wl.head_dim
    q = torch.randn((T, hq, d), generator=g, dtype=torch.float32)
    k = torch.randn((T, hkv, d), generator=g, dtype=torch.float32)
    v = torch.randn((T, hkv, d), generator=g, dtype=torch.float32)
    do = torch.randn((T, hq, d), generator=g, dtype=torch.float32)
    if wl.sink_dist == "normal":
        sink = torch.randn((hq,), generator=g, dtype=torch.float32)
    elif wl.sink_dist == "uniform2":
        sink = torch.rand((hq,), generator=g, dtype=torch.float32) * 4.0 - 2.0
    else:
        raise ValueError(wl.sink_dist)
    inp = Inputs(wl, q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16),
                 do.to(torch.bfloat16), sink)
    if keep_f32:
        inp.q_f32, inp.k_f32, inp.v_f32, inp.do_f32 = q, k, v, do
    return inp


def random_lengths(n: int, lo: int, hi: int, seed: int) -> List[int]:
    """Seeded sequence lengths, uniform in [lo, hi]."""
    g = torch.Generator().manual_seed(seed)
    return [int(x) for x in torch.randint(lo, hi + 1, (n,), generator=g)]


@dataclasses.dataclass
class DecodeInputs:
    """Inputs of one decode step: the key/value cache of every sequence and the
    queries of its last ``n`` positions (rows b * n ... b * n + n - 1)."""

    wl: Workload
    n: int
    q_bf16: torch.Tensor     # [B * n, Hq, D]
    k_bf16: torch.Tensor     # [T, Hkv, D]
    v_bf16: torch.Tensor     # [T, Hkv, D]
    sink: torch.Tensor       # [Hq] float32

    def f64(self, name: str) -> np.ndarray:
        t = getattr(self, name + "_bf16") if name != "sink" else self.sink
        return t.to(torch.float64).numpy()


def make_decode_inputs(wl: Workload, n: int) -> DecodeInputs:
    """Draw a decode step from the workload's seed: k, v, q, sink in that order."""
    g = torch.Generator().manual_seed(wl.seed)
    T, hq, hkv, d = wl.total_tokens, wl.num_heads_q, wl.num_heads_kv, wl.head_dim
    k = torch.randn((T, hkv, d), generator=g, dtype=torch.float32)
    v = torch.randn((T, hkv, d), generator=g, dtype=torch.float32)
    q = torch.randn((wl.num_seqs * n, hq, d), generator=g, dtype=torch.float32)
    if wl.sink_dist == "normal":
        sink = torch.randn((hq,), generator=g, dtype=torch.float32)
    elif wl.sink_dist == "uniform2":
        sink = torch.rand((hq,), generator=g, dtype=torch.float32) * 4.0 - 2.0
    else:
        raise ValueError(wl.sink_dist)
    return DecodeInputs(wl, n, q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16), sink)


# Rollout-side decode steps: one new query row per sequence against long
# cached histories (the policy samples turn by turn), on the same head
# layout.  name -> (workload holding the cached sequences, query rows per sequence).
DECODE_WORKLOADS = {
    "decode_b32_kv8192": (_uniform("decode_b32_kv8192", 32, 8192, 64, 8, WINDOW_INF, 0, 6, "uniform2"), 1),
    "decode_b32_kv8192_w128_p4": (
        _uniform("decode_b32_kv8192_w128_p4", 32, 8192, 64, 8, 128, 4, 6, "uniform2"), 1),
    "decode_varlen8": (Workload("decode_varlen8", VARLEN_LENGTHS, 64, 8, 64, WINDOW_INF, 0, True, 7,
                                "uniform2", uniform=False), 1),
    "decode_b8_kv32768_n4": (_uniform("decode_b8_kv32768_n4", 8, 32768, 64, 8, WINDOW_INF, 0, 8, "uniform2"), 4),
}


# ------------------------------------------------------------------ GRPO
@dataclasses.dataclass(frozen=True)
class GrpoWorkload:
    """One GRPO update batch: prompts x G rollouts of drawn token lengths."""

    name: str
    prompts: int
    group_size: int
    len_lo: int
    len_hi: int
    seed: int
    clip_eps: float = 0.2
    adv_eps: float = 1e-6
    kl_beta: float = 0.04


@dataclasses.dataclass
class GrpoInputs:
    wl: GrpoWorkload
    cu_tokens: np.ndarray    # int32 [R + 1]
    logp: np.ndarray         # float32 [T]
    logp_old: np.ndarray
    logp_ref: np.ndarray
    mask: np.ndarray         # uint8 [T]: optimised (policy-generated) tokens
    rewards: np.ndarray      # float32 [R]


def make_grpo_inputs(wl: GrpoWorkload) -> GrpoInputs:
    """Rollout lengths U[len_lo, len_hi]; each rollout alternates observation
    spans (not optimised) and action spans (optimised) of U[16, 256] tokens;
    logp_old = -Gamma(2, 1), logp = logp_old + N(0, 0.3), logp_ref = logp_old
    + N(0, 0.2); task rewards in {0, 1} (a group can be all-equal)."""
    rng = np.random.default_rng(wl.seed)
    R = wl.prompts * wl.group_size
    lens = rng.integers(wl.len_lo, wl.len_hi + 1, R)
    cu = np.zeros(R + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lens)
    T = int(cu[-1])
    logp_old = -rng.gamma(2.0, 1.0, T).astype(np.float32)
    logp = (logp_old + rng.normal(0.0, 0.3, T)).astype(np.float32)
    logp_ref = (logp_old + rng.normal(0.0, 0.2, T)).astype(np.float32)
    mask = np.zeros(T, dtype=np.uint8)
    for i in range(R):
        t, on = int(cu[i]), False
        while t < cu[i + 1]:
            span = int(rng.integers(16, 257))
            if on:
                mask[t:min(t + span, int(cu[i + 1]))] = 1
            t += span
            on = not on
    rewards = rng.integers(0, 2, R).astype(np.float32)
    return GrpoInputs(wl, cu, logp, logp_old, logp_ref, mask, rewards)


GRPO_WORKLOADS = {
    "grpo_64x8_traj1k8k": GrpoWorkload("grpo_64x8_traj1k8k", 64, 8, 1024, 8192, 9),
}
