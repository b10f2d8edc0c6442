"""CPU float64 oracle for exact sink-aware attention, forward and backward.

TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's CPU
baseline may import or run this module.  The product path (the CUDA library
and its Python binding) never calls it and shares no code with it.

What it computes is the plain definition, written out with explicit score
matrices.  Sources, all from "Efficient Reinforcement Learning for
Long-Horizon Tool-Use Agentic Tasks" (SinkFlex-RL):

* Mask (summary page, paragraph on the sink-aware FlexAttention path):
  M[q, k] = [k <= q] and ([q - k <= w] or [k < p]); w is the local window,
  p the number of always-visible prefix positions; the same mask for every
  batch entry and head.
* Explicit sink (section 5, "zero-value sink equivalence"): a learned sink
  logit s_h whose value vector is zero joins the softmax as one more column,
      O = (sum_i e^{s_i} v_i + e^{s_h} * 0) / (sum_i e^{s_i} + e^{s_h}).
* Auxiliary log-sum-exp (summary page): l = log sum_i e^{s_i} over the real
  (unmasked) keys only, without the sink.
* Sink gradient dL/dS_h per head ("GPT-OSS agentic RL training" page,
  "FlashAttention v3 implementation"): obtained here as the softmax gradient
  of the appended sink column, summed over all rows of that head.

Readings where the pages are silent or garbled:
* scores are s = scale * <q, k>; the sink logit is compared with the scaled
  scores as is; l is the natural-log LSE of the scaled masked scores;
* the window is inclusive (w + 1 keys including the query itself);
  window = -1 means unbounded;
* causal = False drops the [k <= q] term literally;
* prefix positions are counted inside each packed sequence;
* GQA: query head h reads key/value head h // (Hq // Hkv);
* one sink logit per query head, shared by all sequences;
* sink = +inf gives alpha = 0, O = 0; sink = -inf gives plain attention;
* a row with no visible key (not reachable with causal masks and w >= 0)
  gets O = 0 and l = -inf.

Backward: with the extended probabilities P (real columns plus the sink
column) and dP_j = <dO, v_j> (zero for the sink column), the softmax gradient
is dS_j = P_j (dP_j - D) with D = sum_j P_j dP_j; then dQ = scale dS K,
dK = scale dS^T Q, dV = P^T dO, and dsink[h] = sum over rows of dS_sink.

Arrays: q, dout [T, Hq, D]; k, v [T, Hkv, D]; sink [Hq]; cu_seqlens [B + 1]
(token offsets of the packed sequences).  All float64 NumPy arrays.
``decode_forward`` evaluates the last few rows of each sequence against its
whole key/value history (the rollout-side forward).
Rows are handled in blocks of at most ``row_block`` queries to bound memory;
each row's softmax is independent, so blocking changes no arithmetic.
"""
from __future__ import annotations

import numpy as np

WINDOW_INF = -1


def visible(qpos: np.ndarray, kpos: np.ndarray, window: int, prefix: int, causal: bool) -> np.ndarray:
    """Boolean mask M[q, k] for within-sequence positions (summary page mask).

    qpos: [R] query positions, kpos: [C] key positions -> [R, C] booleans.
    """
    qq = qpos[:, None].astype(np.int64)
    kk = kpos[None, :].astype(np.int64)
    if window == WINDOW_INF:
        in_window = np.ones((qq.shape[0], kk.shape[1]), dtype=bool)
    else:
        in_window = (qq - kk) <= window
    in_prefix = kk < prefix
    m = in_window | in_prefix
    if causal:
        m = m & (kk <= qq)
    return m


def _extended_softmax(scores: np.ndarray, sink_logit: float):
    """Softmax over the real columns plus one appended sink column.

    scores: [R, C] with masked entries at -inf.  Returns (P_real [R, C],
    P_sink [R], lse_real [R]) where lse_real is the log-sum-exp of the real
    columns only.
    """
    R = scores.shape[0]
    ext = np.concatenate([scores, np.full((R, 1), sink_logit, dtype=np.float64)], axis=1)
    if np.isposinf(sink_logit):
        # The sink column dominates every row: all mass on the sink.
        p = np.zeros_like(ext)
        p[:, -1] = 1.0
    else:
        mx = np.max(ext, axis=1, keepdims=True)
        mx = np.where(np.isneginf(mx), 0.0, mx)      # whole row -inf (empty row, sink -inf)
        e = np.exp(ext - mx)
        z = np.sum(e, axis=1, keepdims=True)
        p = np.where(z > 0, e / np.where(z > 0, z, 1.0), 0.0)
    real_max = np.max(scores, axis=1) if scores.shape[1] else np.full(R, -np.inf)
    safe = np.where(np.isneginf(real_max), 0.0, real_max)
    with np.errstate(divide="ignore"):
        lse = np.log(np.sum(np.exp(scores - safe[:, None]), axis=1)) + safe
    lse = np.where(np.isneginf(real_max), -np.inf, lse)
    return p[:, :-1], p[:, -1], lse


def _check(q, k, v, sink, cu_seqlens):
    T, hq, d = q.shape
    assert k.shape[0] == T and v.shape == k.shape and k.shape[2] == d
    hkv = k.shape[1]
    assert hq % hkv == 0
    assert sink.shape == (hq,)
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    assert cu[0] == 0 and cu[-1] == T and np.all(np.diff(cu) >= 0)
    return T, hq, hkv, d, cu


def forward(q, k, v, sink, cu_seqlens, window=WINDOW_INF, prefix=0, causal=True, scale=None,
            heads=None, row_block=1024):
    """Return (o [T, Hq, D], lse [Hq, T]) for the query heads in ``heads``.

    Entries of heads outside ``heads`` are left as NaN.
    """
    out = forward_backward(q, k, v, sink, None, cu_seqlens, window, prefix, causal, scale,
                           heads=heads, row_block=row_block)
    return out["o"], out["lse"]


def forward_backward(q, k, v, sink, dout, cu_seqlens, window=WINDOW_INF, prefix=0, causal=True,
                     scale=None, heads=None, row_block=1024):
    """Forward and (if ``dout`` is given) backward of sink-aware attention.

    Returns a dict with o [T, Hq, D], lse [Hq, T] and, with dout,
    dq [T, Hq, D], dk, dv [T, Hkv, D], dsink [Hq].  With ``heads`` a subset
    of query heads, only those heads are computed; dk/dv then hold only the
    contributions of those heads and other heads' entries of o/lse/dq/dsink
    are NaN.
    """
    T, hq, hkv, d, cu = _check(q, k, v, sink, cu_seqlens)
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    group = hq // hkv
    heads = list(range(hq)) if heads is None else sorted(set(int(h) for h in heads))
    o = np.full((T, hq, d), np.nan)
    lse = np.full((hq, T), np.nan)
    with_bwd = dout is not None
    if with_bwd:
        dq = np.full((T, hq, d), np.nan)
        dk = np.zeros((T, hkv, d))
        dv = np.zeros((T, hkv, d))
        dsink = np.full(hq, np.nan)
    for h in heads:
        g = h // group
        if with_bwd:
            dsink[h] = 0.0
        for b in range(len(cu) - 1):
            t0, t1 = int(cu[b]), int(cu[b + 1])
            n = t1 - t0
            if n == 0:
                continue
            Q = q[t0:t1, h, :]
            K = k[t0:t1, g, :]
            V = v[t0:t1, g, :]
            kpos = np.arange(n)
            for r0 in range(0, n, row_block):
                r1 = min(n, r0 + row_block)
                qpos = np.arange(r0, r1)
                s = scale * (Q[r0:r1] @ K.T)
                s = np.where(visible(qpos, kpos, window, prefix, causal), s, -np.inf)
                p, p_sink, l = _extended_softmax(s, float(sink[h]))
                O = p @ V
                o[t0 + r0:t0 + r1, h, :] = O
                lse[h, t0 + r0:t0 + r1] = l
                if not with_bwd:
                    continue
                dO = dout[t0 + r0:t0 + r1, h, :]
                dp = dO @ V.T                                  # real columns
                dp_sink = np.zeros(r1 - r0)                    # value of the sink is zero
                D = np.sum(p * dp, axis=1) + p_sink * dp_sink  # sum_j P_j dP_j
                ds = p * (dp - D[:, None])
                ds_sink = p_sink * (dp_sink - D)
                dq[t0 + r0:t0 + r1, h, :] = scale * (ds @ K)
                dk[t0:t1, g, :] += scale * (ds.T @ Q[r0:r1])
                dv[t0:t1, g, :] += p.T @ dO
                dsink[h] += np.sum(ds_sink)
    res = {"o": o, "lse": lse}
    if with_bwd:
        res.update(dq=dq, dk=dk, dv=dv, dsink=dsink)
    return res


def decode_forward(q, k, v, sink, cu_kv, q_per_seq, window=WINDOW_INF, prefix=0, causal=True, scale=None):
    """Forward for the last ``q_per_seq`` positions of each packed sequence.

    The rollout-side (decode) forward of the same attention: sequence b keeps
    its L_b cached keys and values in k, v [T_kv, Hkv, D] at offsets cu_kv
    [B + 1], and q [B * n, Hq, D] (n = q_per_seq) holds the queries of its
    positions L_b - n ... L_b - 1 in that order.  Every row is the same row
    of ``forward`` over the whole sequence (rows are independent): same mask,
    explicit sink column and lse.  Returns (o [B * n, Hq, D], lse [Hq, B * n]).
    """
    T_kv, hkv, d = k.shape
    hq = q.shape[1]
    n = int(q_per_seq)
    cu = np.asarray(cu_kv, dtype=np.int64)
    B = len(cu) - 1
    assert n >= 1 and q.shape == (B * n, hq, d) and v.shape == k.shape and sink.shape == (hq,)
    assert hq % hkv == 0 and cu[0] == 0 and cu[-1] == T_kv and np.all(np.diff(cu) >= n)
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    group = hq // hkv
    o = np.zeros((B * n, hq, d))
    lse = np.zeros((hq, B * n))
    for b in range(B):
        t0, t1 = int(cu[b]), int(cu[b + 1])
        L = t1 - t0
        m = visible(np.arange(L - n, L), np.arange(L), window, prefix, causal)
        rows = slice(b * n, (b + 1) * n)
        for h in range(hq):
            g = h // group
            s = scale * (q[rows, h, :] @ k[t0:t1, g, :].T)
            s = np.where(m, s, -np.inf)
            p, _, l = _extended_softmax(s, float(sink[h]))
            o[rows, h, :] = p @ v[t0:t1, g, :]
            lse[h, rows] = l
    return o, lse


def unmasked_pairs(seqlens, num_heads_q, window=WINDOW_INF, prefix=0, causal=True) -> int:
    """Number of visible (query, key, query-head) triples, by enumerating the mask."""
    total = 0
    for n in seqlens:
        n = int(n)
        if n == 0:
            continue
        per_row = 0
        for r0 in range(0, n, 2048):
            r1 = min(n, r0 + 2048)
            per_row += int(np.count_nonzero(visible(np.arange(r0, r1), np.arange(n), window, prefix, causal)))
        total += per_row
    return total * int(num_heads_q)
