"""Peak device memory of one sink-aware attention layer (forward + backward):
this library against eager attention with an explicit sink column.

The pages compare an optimised sink-aware attention path with an eager
reference path by peak VRAM at 4096 and 8192 tokens, the eager path running
out of memory at 8192 (SinkFlex-RL summary page, paragraph on the peak-memory
study; abstract on the same page).  This module measures that quantity for a
single attention layer on the GPU.

Eager reference (a measurement baseline only; the library never uses it):
scores = scale * Q K^T in fp32 [B, Hq, S, S] with masked entries at -inf,
the sink logit appended as column S, softmax over S + 1 columns, and
O = P[..., :S] V (the zero-value sink contributes nothing to O), followed by
autograd's backward.  Its memory is quadratic in S; the library keeps every
buffer linear in S.

Run:  python -m studies.memstudy [--seqlens 4096 8192 16384]
"""
from __future__ import annotations

import argparse
import json
import math
from typing import Dict, Optional

import torch

from sink_aware_masked_gb300 import api


def eager_reference_layer(q, k, v, sink, dout, *, window: int = api.WINDOW_INF, prefix: int = 0,
                          scale: Optional[float] = None):
    """Eager sink attention for one uniform sequence batch, with backward.

    q, dout: [B, S, Hq, D]; k, v: [B, S, Hkv, D]; sink: [Hq].  Returns
    (o, dq, dk, dv, dsink) in fp32.  Keys k of query q are visible when
    k <= q and (q - k <= window or k < prefix); window < 0 is unbounded.
    """
    B, S, hq, D = q.shape
    hkv = k.shape[2]
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    qf = q.detach().float().requires_grad_(True)
    kf = k.detach().float().requires_grad_(True)
    vf = v.detach().float().requires_grad_(True)
    sf = sink.detach().float().requires_grad_(True)
    rep = hq // hkv
    kx = kf.repeat_interleave(rep, dim=2)  # GQA: query head h reads key/value head h // rep
    vx = vf.repeat_interleave(rep, dim=2)
    scores = torch.einsum("bqhd,bkhd->bhqk", qf, kx) * scale
    pos = torch.arange(S, device=q.device)
    dq_k = pos[:, None] - pos[None, :]
    vis = dq_k >= 0
    if window >= 0:
        vis = vis & ((dq_k <= window) | (pos[None, :] < prefix))
    scores = scores.masked_fill(~vis, float("-inf"))
    sink_col = sf.view(1, hq, 1, 1).expand(B, hq, S, 1)
    p = torch.softmax(torch.cat([scores, sink_col], dim=-1), dim=-1)
    o = torch.einsum("bhqk,bkhd->bqhd", p[..., :S], vx)
    o.backward(dout.float())
    return o.detach(), qf.grad, kf.grad, vf.grad, sf.grad


def eager_scores_bytes(B: int, S: int, hq: int) -> int:
    """Bytes of one fp32 [B, Hq, S, S + 1] tensor (the eager path holds several)."""
    return 4 * B * hq * S * (S + 1)


def _inputs(B, S, hq, hkv, D, seed, device):
    g = torch.Generator().manual_seed(seed)
    mk = lambda *shape: torch.randn(*shape, generator=g).to(torch.bfloat16).to(device)  # noqa: E731
    q, k, v, dout = mk(B, S, hq, D), mk(B, S, hkv, D), mk(B, S, hkv, D), mk(B, S, hq, D)
    sink = torch.randn(hq, generator=g).float().to(device)
    return q, k, v, dout, sink


def measure(S: int, *, B: int = 1, hq: int = 64, hkv: int = 8, D: int = 64, window: int = api.WINDOW_INF,
            prefix: int = 0, seed: int = 0, run_eager: bool = True) -> Dict:
    """Peak allocated bytes of one fwd+bwd of each path (inputs included)."""
    dev = torch.device("cuda")
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    q, k, v, dout, sink = _inputs(B, S, hq, hkv, D, seed, dev)
    inputs = sum(t.numel() * t.element_size() for t in (q, k, v, dout, sink))
    res = {"seqlen": S, "batch": B, "heads_q": hq, "heads_kv": hkv, "head_dim": D, "window": window,
           "prefix": prefix, "input_bytes": inputs}

    # Library: packed [T, H, D] views of the same inputs, fwd then bwd.
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats()
    problem = dict(num_seqs=B, window=window, prefix=prefix)
    qp, kp, vp, dp = (t.reshape(B * S, t.shape[2], D) for t in (q, k, v, dout))
    o, lse = api.sinkattn_fwd(qp, kp, vp, sink, **problem)
    dq, dk, dv, dsink = api.sinkattn_bwd(qp, kp, vp, o, lse, dp, sink, **problem)
    torch.cuda.synchronize()
    res["library_peak_bytes"] = int(torch.cuda.max_memory_allocated())
    lib_out = (o, dq, dk, dv, dsink)
    del o, lse, dq, dk, dv, dsink

    if run_eager:
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        torch.cuda.reset_peak_memory_stats()
        try:
            eo, edq, edk, edv, eds = eager_reference_layer(q, k, v, sink, dout, window=window, prefix=prefix)
            torch.cuda.synchronize()
            res["eager_peak_bytes"] = int(torch.cuda.max_memory_allocated())
            # Same computation: the library's bf16 outputs against eager fp32.
            res["max_abs_diff_o"] = float((lib_out[0].float().view_as(eo) - eo).abs().max())
            res["rel_diff_dsink"] = float((lib_out[4] - eds).abs().max() / eds.abs().max().clamp_min(1e-30))
            del eo, edq, edk, edv, eds
        except torch.cuda.OutOfMemoryError:
            res["eager_peak_bytes"] = None
            res["eager"] = "out of memory"
        torch.cuda.empty_cache()
    return res


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--seqlens", type=int, nargs="+", default=[4096, 8192, 16384])
    ap.add_argument("--window", type=int, default=api.WINDOW_INF)
    ap.add_argument("--prefix", type=int, default=0)
    ap.add_argument("--json", action="store_true", help="one JSON line per sequence length")
    args = ap.parse_args(argv)
    rows = []
    for S in args.seqlens:
        r = measure(S, window=args.window, prefix=args.prefix)
        rows.append(r)
        if args.json:
            print(json.dumps(r), flush=True)
    if not args.json:
        gb = lambda x: "OOM" if x is None else f"{x / 1e9:.2f}"  # noqa: E731
        print("| S | library peak GB | eager peak GB | eager / library | inputs GB |")
        print("|---|---|---|---|---|")
        for r in rows:
            e = r.get("eager_peak_bytes")
            ratio = "-" if e is None else f"{e / r['library_peak_bytes']:.1f}x"
            print(f"| {r['seqlen']} | {gb(r['library_peak_bytes'])} | {gb(e)} | {ratio} | {gb(r['input_bytes'])} |")
    return 0


if __name__ == "__main__":
    raise SystemExit(main())
