"""Helpers for comparing the CUDA path with the CPU oracle.

The oracle runs one query head per worker process (a ``spawn`` pool, safe to
start after CUDA is initialised) on float64 slices of the inputs, so that
full-size workloads can be checked on whole GQA groups in reasonable time.
"""
from __future__ import annotations

import multiprocessing as mp
import os

import numpy as np

# Parity bars: max abs error on O and lse, relative L2 on the gradients.
TOL = {"o": 1e-2, "lse": 1e-3, "dq": 2e-2, "dk": 2e-2, "dv": 2e-2, "dsink": 2e-2}


def _one_head(args):
    import oracle

    q, k, v, do, sink, cu, window, prefix, causal, scale = args
    return oracle.forward_backward(q, k, v, sink, do, cu, window, prefix, causal, scale)


_POOL = None


def _pool():
    global _POOL
    if _POOL is None:
        n = max(1, min(16, os.cpu_count() or 1))
        _POOL = mp.get_context("spawn").Pool(n)
    return _POOL


def oracle_heads(inp, wl, heads, parallel=True):
    """Oracle outputs for the query heads ``heads`` (float64).

    Returns dict with o [T, nh, D], lse [nh, T], dq [T, nh, D], dsink [nh] for
    the listed heads, and dk, dv [T, Hkv, D] holding the summed contributions
    of those heads (complete for a kv head when all its query heads are listed).
    """
    group = wl.num_heads_q // wl.num_heads_kv
    q = inp.f64("q")
    k = inp.f64("k")
    v = inp.f64("v")
    do = inp.f64("do")
    sink = inp.f64("sink")
    cu = wl.cu_seqlens()
    jobs = []
    for h in heads:
        g = h // group
        jobs.append((np.ascontiguousarray(q[:, h:h + 1]), np.ascontiguousarray(k[:, g:g + 1]),
                     np.ascontiguousarray(v[:, g:g + 1]), np.ascontiguousarray(do[:, h:h + 1]),
                     sink[h:h + 1].copy(), cu, wl.window, wl.prefix, wl.causal, wl.scale))
    if parallel and len(jobs) > 1:
        outs = _pool().map(_one_head, jobs)
    else:
        outs = [_one_head(j) for j in jobs]
    T, D = q.shape[0], q.shape[2]
    res = {"o": np.stack([r["o"][:, 0] for r in outs], 1), "lse": np.stack([r["lse"][0] for r in outs], 0),
           "dq": np.stack([r["dq"][:, 0] for r in outs], 1), "dsink": np.array([r["dsink"][0] for r in outs]),
           "dk": np.zeros((T, wl.num_heads_kv, D)), "dv": np.zeros((T, wl.num_heads_kv, D))}
    for h, r in zip(heads, outs):
        res["dk"][:, h // group] += r["dk"][:, 0]
        res["dv"][:, h // group] += r["dv"][:, 0]
    return res


def max_abs(a, b):
    return float(np.max(np.abs(np.asarray(a, np.float64) - np.asarray(b, np.float64)))) if np.size(a) else 0.0


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    nb = float(np.linalg.norm(b))
    if nb == 0.0:
        return float(np.linalg.norm(a))
    return float(np.linalg.norm(a - b) / nb)


def errors(gpu, ref, heads, kv_heads):
    """Error metrics of GPU results (torch tensors, all heads) against oracle
    results for ``heads`` (and complete dk/dv for ``kv_heads``)."""
    f = lambda t: t.detach().double().cpu().numpy()
    hs = list(heads)
    out = {
        "o": max_abs(f(gpu["o"])[:, hs], ref["o"]),
        "lse": max_abs(f(gpu["lse"])[hs], ref["lse"]),
        "dq": rel_l2(f(gpu["dq"])[:, hs], ref["dq"]),
        "dsink": rel_l2(f(gpu["dsink"])[hs], ref["dsink"]),
    }
    if kv_heads:
        out["dk"] = rel_l2(f(gpu["dk"])[:, kv_heads], ref["dk"][:, kv_heads])
        out["dv"] = rel_l2(f(gpu["dv"])[:, kv_heads], ref["dv"][:, kv_heads])
    return out


def assert_within(errs, label=""):
    bad = {k: v for k, v in errs.items() if not v <= TOL[k]}
    assert not bad, f"{label} parity failed: {bad} (all: {errs})"
