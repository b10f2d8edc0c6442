"""Sequence-parallel sink-aware attention (Ulysses-style all-to-all).

Long trajectories are held sequence-sharded: rank r of a group of P owns a
contiguous run of the packed token stream (``shard_tokens[r]`` tokens, all
heads).  Attention needs every token of a sequence, so one all-to-all turns
the sequence sharding into head sharding before the attention call and one
turns it back afterwards; the backward does the same with the gradients.
This is the long-context scheme of the GPT-OSS agentic-RL retrospective
(section on sequence parallelism: an all-to-all before and after attention),
made sink-aware: rank r owns query heads [r Hq/P, (r+1) Hq/P), the key/value
heads they read ([r Hkv/P, (r+1) Hkv/P), contiguous GQA groups stay
together), their sink logits and their sink gradients.

The attention itself is one call of the library (``sinkattn_fwd`` /
``sinkattn_bwd``) over the whole packed stream for the rank's heads; this
module only moves tensors.  Requirements: Hq and Hkv divisible by P, every
rank passing the same problem description (the global sequence offsets,
mask, scale).  The exchange uses ``torch.distributed.all_to_all_single``;
on a gloo group, GPU tensors are staged through host memory.

Gradient of the sink: rank r returns the gradient of the whole loss (every
token) for its own heads and zeros for the others, so that summing dsink
over the group, as the usual gradient all-reduce of a replicated parameter
does, gives the full gradient once.
"""
from __future__ import annotations

from typing import Callable, Optional, Sequence

import torch
import torch.distributed as dist

from . import api


def _group_info(group):
    return dist.get_world_size(group), dist.get_rank(group)


def _a2a(send: torch.Tensor, send_splits, recv_splits, group) -> torch.Tensor:
    """all_to_all_single along dim 0 with explicit split sizes."""
    shape = (int(sum(recv_splits)),) + tuple(send.shape[1:])
    out = torch.empty(shape, dtype=send.dtype, device=send.device)
    send_splits = [int(x) for x in send_splits]
    recv_splits = [int(x) for x in recv_splits]
    if send.is_cuda and dist.get_backend(group) == "gloo":
        host = torch.empty(shape, dtype=send.dtype)
        dist.all_to_all_single(host, send.contiguous().cpu(), recv_splits, send_splits, group=group)
        out.copy_(host)
    else:
        dist.all_to_all_single(out, send.contiguous(), recv_splits, send_splits, group=group)
    return out


def seq_to_heads(x: torch.Tensor, shard_tokens: Sequence[int], group=None) -> torch.Tensor:
    """[T_r, H, D] (this rank's tokens, all heads) -> [T, H/P, D] (every
    token, this rank's heads)."""
    P, r = _group_info(group)
    T_r, H, D = x.shape
    hp = H // P
    send = x.reshape(T_r, P, hp, D).permute(1, 0, 2, 3).reshape(P * T_r, hp, D)
    return _a2a(send, [T_r] * P, shard_tokens, group)


def heads_to_seq(y: torch.Tensor, shard_tokens: Sequence[int], group=None) -> torch.Tensor:
    """[T, H/P, D] (every token, this rank's heads) -> [T_r, H, D]."""
    P, r = _group_info(group)
    T, hp, D = y.shape
    T_r = int(shard_tokens[r])
    recv = _a2a(y.contiguous(), shard_tokens, [T_r] * P, group)
    return recv.reshape(P, T_r, hp, D).permute(1, 0, 2, 3).reshape(T_r, P * hp, D)


def lse_heads_to_seq(lse: torch.Tensor, shard_tokens: Sequence[int], group=None) -> torch.Tensor:
    """[H/P, T] -> [H, T_r] (the log-sum-exp rows of this rank's tokens)."""
    hp = lse.shape[0]
    return heads_to_seq(lse.t().contiguous().reshape(-1, hp, 1), shard_tokens, group)[..., 0].t().contiguous()


def _check(q, k, sink, shard_tokens, P, r):
    T_r, H, D = q.shape
    hkv = k.shape[1]
    if len(shard_tokens) != P:
        raise ValueError(f"shard_tokens has {len(shard_tokens)} entries for a group of {P}")
    if int(shard_tokens[r]) != T_r or k.shape[0] != T_r:
        raise ValueError(f"rank {r} holds {T_r} query and {k.shape[0]} key tokens, shard_tokens says {shard_tokens[r]}")
    if H % P or hkv % P:
        raise ValueError(f"query heads ({H}) and key/value heads ({hkv}) must be divisible by the group size {P}")
    if sink.shape != (H,):
        raise ValueError(f"sink must have shape [{H}]")


def ulysses_forward(q, k, v, sink, *, shard_tokens: Sequence[int], group=None,
                    local_fwd: Optional[Callable] = None, **problem):
    """Forward on sequence-sharded q [T_r, Hq, 64], k, v [T_r, Hkv, 64] and
    the replicated sink [Hq].  ``problem`` describes the whole packed stream
    (as for ``api.sinkattn_fwd``).  Returns (o [T_r, Hq, 64], lse [Hq, T_r],
    saved), ``saved`` holding the head-sharded tensors the backward reuses."""
    P, r = _group_info(group)
    _check(q, k, sink, shard_tokens, P, r)
    local_fwd = local_fwd or api.sinkattn_fwd
    hp = q.shape[1] // P
    qh = seq_to_heads(q, shard_tokens, group)
    kh = seq_to_heads(k, shard_tokens, group)
    vh = seq_to_heads(v, shard_tokens, group)
    sh = sink[r * hp:(r + 1) * hp].contiguous()
    oh, lseh = local_fwd(qh, kh, vh, sh, **problem)
    o = heads_to_seq(oh, shard_tokens, group)
    lse = lse_heads_to_seq(lseh, shard_tokens, group)
    saved = dict(q=qh, k=kh, v=vh, sink=sh, o=oh, lse=lseh)
    return o, lse, saved


def ulysses_backward(saved, dout, *, shard_tokens: Sequence[int], num_heads_q: int, group=None,
                     local_bwd: Optional[Callable] = None, **problem):
    """Backward from dout [T_r, Hq, 64]: returns dq [T_r, Hq, 64], dk, dv
    [T_r, Hkv, 64] and dsink [Hq] (this rank's heads filled, zeros
    elsewhere)."""
    P, r = _group_info(group)
    local_bwd = local_bwd or api.sinkattn_bwd
    hp = num_heads_q // P
    doh = seq_to_heads(dout.contiguous(), shard_tokens, group)
    dqh, dkh, dvh, dsh = local_bwd(saved["q"], saved["k"], saved["v"], saved["o"], saved["lse"], doh, saved["sink"],
                                   **problem)
    dq = heads_to_seq(dqh, shard_tokens, group)
    dk = heads_to_seq(dkh, shard_tokens, group)
    dv = heads_to_seq(dvh, shard_tokens, group)
    dsink = torch.zeros(num_heads_q, dtype=dsh.dtype, device=dsh.device)
    dsink[r * hp:(r + 1) * hp] = dsh
    return dq, dk, dv, dsink


class UlyssesSinkAttention(torch.autograd.Function):
    """Autograd wrapper of ulysses_forward / ulysses_backward."""

    @staticmethod
    def forward(ctx, q, k, v, sink, shard_tokens, group, problem):
        o, lse, saved = ulysses_forward(q, k, v, sink, shard_tokens=shard_tokens, group=group, **problem)
        ctx.saved = saved
        ctx.cfg = (tuple(int(x) for x in shard_tokens), group, problem, q.shape[1])
        ctx.mark_non_differentiable(lse)
        return o, lse

    @staticmethod
    def backward(ctx, do, dlse):
        shard_tokens, group, problem, hq = ctx.cfg
        dq, dk, dv, dsink = ulysses_backward(ctx.saved, do, shard_tokens=shard_tokens, num_heads_q=hq, group=group,
                                             **problem)
        ctx.saved = None
        return dq, dk, dv, dsink, None, None, None


def ulysses_sink_attention(q, k, v, sink, *, shard_tokens: Sequence[int], group=None, **problem):
    """Differentiable sequence-parallel sink attention; returns this rank's
    output rows [T_r, Hq, 64]."""
    o, _ = UlyssesSinkAttention.apply(q, k, v, sink, shard_tokens, group, problem)
    return o
