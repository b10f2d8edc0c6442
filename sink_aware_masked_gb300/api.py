"""Thin PyTorch binding of the C ABI: argument marshalling only.

Every step of the computation runs in the CUDA kernels of libsinkattn.so.
PyTorch supplies device memory (outputs and workspace are allocated with
torch) and the current CUDA stream.  There is no CPU path: on a machine
without the built library or without a GPU these functions raise.

Tensors: q, o, dout, dq [T, Hq, 64] bf16; k, v, dk, dv [T, Hkv, 64] bf16;
lse [Hq, T] fp32; sink, dsink [Hq] fp32.  A uniform batch is given with
``num_seqs`` (T = num_seqs * seqlen); packed sequences with ``cu_seqlens``
(device int32 [B + 1]) and its host copy ``cu_seqlens_host``.
"""
from __future__ import annotations

import ctypes
import math
from typing import Optional, Sequence

import torch

from . import _lib

WINDOW_INF = -1


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


HEAD_DIM = 64


def _check(name: str, t: Optional[torch.Tensor], dtype: torch.dtype, shape=None, device=None) -> None:
    """Reject what the C ABI cannot see: it receives only a raw pointer, so a
    tensor of another dtype, layout, size or device would be read as
    garbage.  Checked in this order: shape, dtype, contiguity, same device as
    the call's first tensor (``device``); ``_on_gpu`` then checks that this
    device is a GPU."""
    if t is None:
        raise ValueError(f"{name} is required")
    if shape is not None:
        if t.dim() != len(shape) or any(s is not None and int(a) != int(s) for a, s in zip(t.shape, shape)):
            want = "[" + ", ".join("*" if s is None else str(int(s)) for s in shape) + "]"
            raise ValueError(f"{name} has shape {list(t.shape)}, expected {want}")
    if t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def _on_gpu(name: str, t: torch.Tensor) -> None:
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor (there is no CPU path)")


def _check_qkv(q, k, v, sink):
    """q [T, Hq, 64], k and v [T_kv, Hkv, 64] bf16 with Hq % Hkv == 0, sink [Hq] fp32, one CUDA device."""
    if q is None or k is None or q.dim() != 3 or k.dim() != 3:
        raise ValueError("q and k must be 3-D tensors [tokens, heads, head_dim]")
    if q.shape[2] != HEAD_DIM or k.shape[2] != HEAD_DIM:
        raise ValueError(f"head_dim must be {HEAD_DIM} (q: {q.shape[2]}, k: {k.shape[2]})")
    hq, hkv = q.shape[1], k.shape[1]
    if hkv < 1 or hq % hkv != 0:
        raise ValueError(f"query heads ({hq}) must be a multiple of key/value heads ({hkv})")
    dev = q.device
    _check("q", q, torch.bfloat16, (None, hq, HEAD_DIM), dev)
    _check("k", k, torch.bfloat16, (None, hkv, HEAD_DIM), dev)
    _check("v", v, torch.bfloat16, tuple(k.shape), dev)
    _check("sink", sink, torch.float32, (hq,), dev)
    return dev


def _stream() -> int:
    return torch.cuda.current_stream().cuda_stream


def make_problem(q: torch.Tensor, k: torch.Tensor, *, num_seqs: Optional[int] = None,
                 cu_seqlens: Optional[torch.Tensor] = None,
                 cu_seqlens_host: Optional[Sequence[int]] = None, max_seqlen: Optional[int] = None,
                 window: int = WINDOW_INF, prefix: int = 0, causal: bool = True,
                 scale: Optional[float] = None, total_tokens: Optional[int] = None):
    """Build the C problem struct; returns (struct, keep-alive objects).

    The sequences are those of q (T = q.shape[0]) unless ``total_tokens``
    says otherwise (decode: the key/value cache holds the sequences)."""
    _, hq, d = q.shape
    T = q.shape[0] if total_tokens is None else int(total_tokens)
    hkv = k.shape[1]
    keep = []
    if cu_seqlens is None:
        B = 1 if num_seqs is None else int(num_seqs)
        S = T // B if B > 0 else 0
        cu_dev = cu_host_ptr = None
    else:
        if cu_seqlens_host is None:
            raise ValueError("cu_seqlens_host (a host copy of cu_seqlens) is required with cu_seqlens")
        host = (ctypes.c_int32 * len(cu_seqlens_host))(*[int(x) for x in cu_seqlens_host])
        keep.append(host)
        B = len(cu_seqlens_host) - 1
        lens = [int(cu_seqlens_host[i + 1]) - int(cu_seqlens_host[i]) for i in range(B)]
        S = int(max_seqlen) if max_seqlen is not None else (max(lens) if lens else 0)
        cu_dev = cu_seqlens.data_ptr()
        cu_host_ptr = ctypes.cast(host, ctypes.c_void_p).value
    pr = _lib.Problem(
        num_seqs=B, seqlen=S, cu_seqlens=cu_dev, cu_seqlens_host=cu_host_ptr, total_tokens=T,
        num_heads_q=hq, num_heads_kv=hkv, head_dim=d, window=int(window), prefix=int(prefix),
        causal=1 if causal else 0, scale=float(scale if scale is not None else 1.0 / math.sqrt(d)))
    return pr, keep


def _check_cu(problem: dict, dev) -> None:
    cu = problem.get("cu_seqlens")
    if cu is not None:
        host = problem.get("cu_seqlens_host")
        n = None if host is None else len(host)
        _check("cu_seqlens", cu, torch.int32, (n,), dev)


def sinkattn_fwd(q, k, v, sink, *, o=None, lse=None, workspace=None, **problem):
    """Forward: returns (o, lse).  ``problem`` keys as in make_problem."""
    dev = _check_qkv(q, k, v, sink)
    T, hq, d = q.shape
    if k.shape[0] != T:
        raise ValueError(f"k and v hold {k.shape[0]} tokens, q holds {T}")
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((hq, T), dtype=torch.float32, device=q.device)
    _check("o", o, torch.bfloat16, tuple(q.shape), dev)
    _check("lse", lse, torch.float32, (hq, T), dev)
    _check_cu(problem, dev)
    _on_gpu("q", q)
    lib = _lib.load()
    pr, keep = make_problem(q, k, **problem)
    ws_bytes = lib.sinkattn_fwd_workspace_size(ctypes.byref(pr))
    if workspace is None and ws_bytes > 0:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    st = lib.sinkattn_fwd(ctypes.byref(pr), _ptr(q), _ptr(k), _ptr(v), _ptr(sink), _ptr(o), _ptr(lse),
                          _ptr(workspace), ws_bytes if workspace is not None else 0, _stream())
    _lib.check("sinkattn_fwd", st)
    return o, lse


def kernel_launches(q, k, which: str, **problem) -> int:
    """Kernel launches sinkattn_fwd (which="fwd") or sinkattn_bwd ("bwd") makes for this problem."""
    lib = _lib.load()
    pr, keep = make_problem(q, k, **problem)
    n = int(lib.sinkattn_kernel_launches(ctypes.byref(pr), {"fwd": 1, "bwd": 2}[which]))
    if n < 0:
        raise ValueError("kernel_launches: invalid problem")
    return n


def bwd_workspace_bytes(q, k, **problem) -> int:
    lib = _lib.load()
    pr, keep = make_problem(q, k, **problem)
    return int(lib.sinkattn_bwd_workspace_size(ctypes.byref(pr)))


def sinkattn_bwd(q, k, v, o, lse, dout, sink, *, dq=None, dk=None, dv=None, dsink=None, workspace=None,
                 **problem):
    """Backward: returns (dq, dk, dv, dsink)."""
    dev = _check_qkv(q, k, v, sink)
    T, hq, _ = q.shape
    if k.shape[0] != T:
        raise ValueError(f"k and v hold {k.shape[0]} tokens, q holds {T}")
    _check("o", o, torch.bfloat16, tuple(q.shape), dev)
    _check("dout", dout, torch.bfloat16, tuple(q.shape), dev)
    _check("lse", lse, torch.float32, (hq, T), dev)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    dsink = torch.empty_like(sink) if dsink is None else dsink
    _check("dq", dq, torch.bfloat16, tuple(q.shape), dev)
    _check("dk", dk, torch.bfloat16, tuple(k.shape), dev)
    _check("dv", dv, torch.bfloat16, tuple(k.shape), dev)
    _check("dsink", dsink, torch.float32, (hq,), dev)
    if workspace is not None:
        _check("workspace", workspace, torch.uint8, (None,), dev)
    _check_cu(problem, dev)
    _on_gpu("q", q)
    lib = _lib.load()
    pr, keep = make_problem(q, k, **problem)
    ws_bytes = int(lib.sinkattn_bwd_workspace_size(ctypes.byref(pr)))
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=q.device)
    st = lib.sinkattn_bwd(ctypes.byref(pr), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout),
                          _ptr(sink), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dsink), _ptr(workspace),
                          workspace.numel(), _stream())
    _lib.check("sinkattn_bwd", st)
    return dq, dk, dv, dsink


def decode_workspace_bytes(q, k, *, q_per_seq: int, **problem) -> int:
    lib = _lib.load()
    pr, keep = make_problem(q, k, total_tokens=k.shape[0], **problem)
    return int(lib.sinkattn_decode_workspace_size(ctypes.byref(pr), int(q_per_seq)))


def sinkattn_decode_fwd(q, k, v, sink, *, q_per_seq: int, o=None, lse=None, workspace=None, **problem):
    """Decode forward: returns (o, lse) for the last ``q_per_seq`` positions.

    k, v [T_kv, Hkv, 64] hold every cached position of each sequence
    (``num_seqs`` uniform sequences, or ``cu_seqlens``/``cu_seqlens_host``
    offsets into k and v); q [num_seqs * q_per_seq, Hq, 64] holds the queries
    of the last q_per_seq positions of each sequence in order.  Each output
    row equals the same row of sinkattn_fwd over the whole sequence.
    """
    dev = _check_qkv(q, k, v, sink)
    R, hq, d = q.shape
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((hq, R), dtype=torch.float32, device=q.device)
    _check("o", o, torch.bfloat16, tuple(q.shape), dev)
    _check("lse", lse, torch.float32, (hq, R), dev)
    if workspace is not None:
        _check("workspace", workspace, torch.uint8, (None,), dev)
    _check_cu(problem, dev)
    _on_gpu("q", q)
    lib = _lib.load()
    pr, keep = make_problem(q, k, total_tokens=k.shape[0], **problem)
    ws_bytes = int(lib.sinkattn_decode_workspace_size(ctypes.byref(pr), int(q_per_seq)))
    if workspace is None:
        # zero-filled: the chunk counters at its start must be zero (each call leaves them so)
        workspace = torch.zeros(max(ws_bytes, 16), dtype=torch.uint8, device=q.device)
    st = lib.sinkattn_decode_fwd(ctypes.byref(pr), int(q_per_seq), _ptr(q), _ptr(k), _ptr(v), _ptr(sink), _ptr(o),
                                 _ptr(lse), _ptr(workspace), workspace.numel(), _stream())
    _lib.check("sinkattn_decode_fwd", st)
    return o, lse


def _grpo_problem(cu_tokens, cu_tokens_host, group_size, clip_eps=0.2, adv_eps=1e-6, kl_beta=0.0):
    host = (ctypes.c_int32 * len(cu_tokens_host))(*[int(x) for x in cu_tokens_host])
    g = _lib.GrpoProblem(num_rollouts=len(cu_tokens_host) - 1, group_size=int(group_size),
                         cu_tokens=_ptr(cu_tokens),
                         cu_tokens_host=ctypes.cast(host, ctypes.c_void_p).value, total_tokens=int(cu_tokens_host[-1]),
                         clip_eps=float(clip_eps), adv_eps=float(adv_eps), kl_beta=float(kl_beta))
    return g, host


def grpo_workspace_bytes(cu_tokens, cu_tokens_host, *, group_size: int) -> int:
    """Workspace bytes of grpo_loss for these rollout offsets (device tensor and host list)."""
    lib = _lib.load()
    g, keep = _grpo_problem(cu_tokens, cu_tokens_host, group_size)
    n = int(lib.sinkattn_grpo_workspace_size(ctypes.byref(g)))
    if n == 0 and len(cu_tokens_host) > 1:
        raise ValueError("grpo_workspace_bytes: invalid rollout offsets or group size")
    return n


def grpo_loss(logp, logp_old, mask, rewards, cu_tokens, cu_tokens_host, *, group_size: int, clip_eps: float = 0.2,
              adv_eps: float = 1e-6, kl_beta: float = 0.0, logp_ref=None, dlogp=None, workspace=None, stats=None,
              advantages=None):
    """GRPO token loss: returns (stats [4] fp32, dlogp [T] fp32, advantages [R] fp32).

    stats = (loss, policy term, KL term, clipped fraction); all tensors on the
    GPU (logp/logp_old/logp_ref fp32 [T], mask uint8 [T], rewards fp32 [R],
    cu_tokens int32 [R + 1] with its host copy cu_tokens_host).  A caller
    that passes ``workspace`` (uint8, grpo_workspace_bytes long) zero-fills it
    once; each completed call leaves it reusable.  Without one, a zero-filled
    workspace is allocated per call.
    """
    R = len(cu_tokens_host) - 1
    dev = logp.device if isinstance(logp, torch.Tensor) else None
    _check("logp", logp, torch.float32, (None,), dev)
    T = logp.shape[0]
    _check("logp_old", logp_old, torch.float32, (T,), dev)
    if kl_beta:
        _check("logp_ref", logp_ref, torch.float32, (T,), dev)
    _check("mask", mask, torch.uint8, (T,), dev)
    _check("rewards", rewards, torch.float32, (R,), dev)
    _check("cu_tokens", cu_tokens, torch.int32, (R + 1,), dev)
    if dlogp is not None:
        _check("dlogp", dlogp, torch.float32, (T,), dev)
    if stats is not None:
        _check("stats", stats, torch.float32, (4,), dev)
    if advantages is not None:
        _check("advantages", advantages, torch.float32, (R,), dev)
    if workspace is not None:
        _check("workspace", workspace, torch.uint8, (None,), dev)
    _on_gpu("logp", logp)
    lib = _lib.load()
    g, keep = _grpo_problem(cu_tokens, cu_tokens_host, group_size, clip_eps, adv_eps, kl_beta)
    stats = torch.empty(4, dtype=torch.float32, device=logp.device) if stats is None else stats
    dlogp = torch.empty_like(logp) if dlogp is None else dlogp
    adv = torch.empty(R, dtype=torch.float32, device=logp.device) if advantages is None else advantages
    ws_bytes = int(lib.sinkattn_grpo_workspace_size(ctypes.byref(g)))
    if workspace is None:
        workspace = torch.zeros(max(ws_bytes, 16), dtype=torch.uint8, device=logp.device)
    st = lib.sinkattn_grpo_loss(ctypes.byref(g), _ptr(logp), _ptr(logp_old), _ptr(logp_ref), _ptr(mask), _ptr(rewards),
                                _ptr(stats), _ptr(dlogp), _ptr(adv), _ptr(workspace), workspace.numel(), _stream())
    _lib.check("sinkattn_grpo_loss", st)
    return stats, dlogp, adv


def sinkattn_varlen_plan(seqlens: torch.Tensor) -> torch.Tensor:
    """Device int32 lengths [B] -> device int32 offsets [B + 1]."""
    _check("seqlens", seqlens, torch.int32, (None,))
    _on_gpu("seqlens", seqlens)
    lib = _lib.load()
    cu = torch.empty(seqlens.numel() + 1, dtype=torch.int32, device=seqlens.device)
    _lib.check("sinkattn_varlen_plan",
               lib.sinkattn_varlen_plan(_ptr(seqlens), seqlens.numel(), _ptr(cu), _stream()))
    return cu


def sinkattn_pack(padded: torch.Tensor, cu_seqlens: torch.Tensor, total_tokens: int) -> torch.Tensor:
    """[B, Smax, H, D] bf16 -> [T, H, D] (rows past each length dropped)."""
    _check("padded", padded, torch.bfloat16, (None, None, None, None))
    B, Smax, H, D = padded.shape
    _check("cu_seqlens", cu_seqlens, torch.int32, (B + 1,), padded.device)
    _on_gpu("padded", padded)
    lib = _lib.load()
    packed = torch.empty((total_tokens, H, D), dtype=padded.dtype, device=padded.device)
    _lib.check("sinkattn_pack", lib.sinkattn_pack(_ptr(padded), _ptr(cu_seqlens), B, Smax, H, D,
                                                  _ptr(packed), _stream()))
    return packed


def sinkattn_unpack(packed: torch.Tensor, cu_seqlens: torch.Tensor, B: int, Smax: int) -> torch.Tensor:
    """[T, H, D] -> [B, Smax, H, D] with zero padding rows."""
    _check("packed", packed, torch.bfloat16, (None, None, None))
    T, H, D = packed.shape
    _check("cu_seqlens", cu_seqlens, torch.int32, (int(B) + 1,), packed.device)
    _on_gpu("packed", packed)
    lib = _lib.load()
    padded = torch.empty((B, Smax, H, D), dtype=packed.dtype, device=packed.device)
    _lib.check("sinkattn_unpack", lib.sinkattn_unpack(_ptr(packed), _ptr(cu_seqlens), B, Smax, H, D,
                                                      _ptr(padded), _stream()))
    return padded


def sinkattn_get_device_status() -> int:
    """Synchronise the current stream and return (and clear) the device status."""
    return int(_lib.load().sinkattn_get_device_status(_stream()))


PROFILE_FWD, PROFILE_BWD_MAIN, PROFILE_DECODE = 1, 2, 3


def sinkattn_set_profile_events(kind: int, start=None, stop=None) -> None:
    """Record torch.cuda.Event ``start``/``stop`` around the selected kernel
    (PROFILE_FWD, PROFILE_BWD_MAIN or PROFILE_DECODE) of every later call; None clears."""
    lib = _lib.load()
    ps = None if start is None else start.cuda_event
    pe = None if stop is None else stop.cuda_event
    if start is not None and (not ps or not pe):
        raise ValueError("record the events once before installing them (torch creates them lazily)")
    _lib.check("sinkattn_set_profile_events", lib.sinkattn_set_profile_events(kind, ps, pe))


class SinkAttention(torch.autograd.Function):
    """Autograd wrapper: forward and backward both run in libsinkattn.so."""

    @staticmethod
    def forward(ctx, q, k, v, sink, problem):
        o, lse = sinkattn_fwd(q, k, v, sink, **problem)
        ctx.save_for_backward(q, k, v, sink, o, lse)
        ctx.problem = problem
        ctx.mark_non_differentiable(lse)
        return o, lse

    @staticmethod
    def backward(ctx, do, dlse):
        q, k, v, sink, o, lse = ctx.saved_tensors
        dq, dk, dv, dsink = sinkattn_bwd(q, k, v, o, lse, do.contiguous(), sink, **ctx.problem)
        return dq, dk, dv, dsink, None


def sink_attention(q, k, v, sink, **problem):
    """Differentiable sink-aware attention; returns the output only."""
    o, _ = SinkAttention.apply(q, k, v, sink, problem)
    return o
